// Product-key scoring and exact top-k for a whole sequence (all B*T tokens, both
// queries) on CUDA cores.
//
// One CTA takes `tok_per_cta` consecutive tokens of one head: 2*tok_per_cta query
// rows (row 2t = write query, 2t+1 = read query).  Phase 1 computes every factor
// score of those rows into shared memory as a tiled product of the query rows with
// the sub-key table (32 rows x 256 sub-keys per pass, 32-wide slices of d_sub staged
// in shared memory, 4x8 outputs per thread), with the accurate accumulation of
// sdm_common.cuh so that the float32 scores are (almost always) correctly rounded.
// Phase 2 gives each warp whole rows for row_topk (sdm_topk.cuh).
#include "sdm_common.cuh"
#include "sdm_internal.h"
#include "sdm_topk.cuh"

namespace sdm {

namespace {

constexpr int kDK = 32;        // d_sub slice per stage
constexpr int kNT = 256;       // sub-keys per pass
constexpr int kRT = 32;        // query rows per pass (= max rows per CTA)
constexpr int kRM = 4, kAM = 8;

template <int EF, int EC, typename ACT>
__global__ void __launch_bounds__(kThreads)
    topk_kernel(const __grid_constant__ TopkArgs a, const __grid_constant__ CandidateList cl) {
  extern __shared__ __align__(16) unsigned char smem[];
  const KeyGeometry &g = a.g;
  const int h = blockIdx.y;
  const int64_t tok0 = (int64_t)blockIdx.x * a.tok_per_cta;
  const int ntok = (int)min((int64_t)a.tok_per_cta, a.BT - tok0);
  const int nrows = 2 * ntok;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int ntot = g.ntot, d_sub = g.d_sub;
  const int64_t qdim = (int64_t)g.F * d_sub;

  float *scores = reinterpret_cast<float *>(smem);                       // [2*tok_per_cta][ntot]
  uint32_t *cand = reinterpret_cast<uint32_t *>(scores + (size_t)2 * a.tok_per_cta * ntot);
  unsigned char *scratch = reinterpret_cast<unsigned char *>(cand + cl.n[0] + cl.n[1]);
  scratch = reinterpret_cast<unsigned char *>(((uintptr_t)scratch + 15) & ~(uintptr_t)15);
  float *qs = reinterpret_cast<float *>(scratch);                        // [kRT][kDK]
  float *ks = qs + kRT * kDK;                                            // [kDK][kNT + 1]
  RowScratch *rs = reinterpret_cast<RowScratch *>(scratch);              // [8] in phase 2

  for (int i = tid; i < cl.n[0]; i += kThreads) cand[i] = cl.tup[0][i];
  for (int i = tid; i < cl.n[1]; i += kThreads) cand[cl.n[0] + i] = cl.tup[1][i];

  const ACT *q[2] = {static_cast<const ACT *>(a.q[0]), static_cast<const ACT *>(a.q[1])};
  const ACT *K = static_cast<const ACT *>(a.subkeys) + (int64_t)h * ntot * d_sub;
  const int tr = tid >> 5, ta = tid & 31;

  // ---- phase 1: factor scores
  for (int f = 0; f < g.F; ++f) {
    for (int a0 = 0; a0 < g.nf[f]; a0 += kNT) {
      Acc2 acc[kRM][kAM];
#pragma unroll
      for (int i = 0; i < kRM; ++i)
#pragma unroll
        for (int j = 0; j < kAM; ++j) acc[i][j] = Acc2{0.0f, 0.0f};
      for (int d0 = 0; d0 < d_sub; d0 += kDK) {
        const int dk = min(kDK, d_sub - d0);
        for (int e = tid; e < kRT * kDK; e += kThreads) {
          const int r = e / kDK, dd = e % kDK;
          float v = 0.0f;
          if (r < nrows && dd < dk) {
            const int64_t tok = tok0 + (r >> 1);
            v = to_f32(q[r & 1][(tok * a.H + h) * qdim + (int64_t)f * d_sub + d0 + dd]);
          }
          qs[r * kDK + dd] = v;
        }
        for (int e = tid; e < kNT * kDK; e += kThreads) {
          const int aa = e / kDK, dd = e % kDK;
          const int arow = a0 + aa;
          float v = 0.0f;
          if (arow < g.nf[f] && dd < dk) v = to_f32(K[(int64_t)(g.off[f] + arow) * d_sub + d0 + dd]);
          ks[dd * (kNT + 1) + aa] = v;
        }
        __syncthreads();
        if constexpr (sizeof(ACT) == 2) {
          float blk[kRM][kAM];
#pragma unroll
          for (int i = 0; i < kRM; ++i)
#pragma unroll
            for (int j = 0; j < kAM; ++j) blk[i][j] = 0.0f;
          for (int dd = 0; dd < dk; ++dd) {
            float qv[kRM], kv[kAM];
#pragma unroll
            for (int i = 0; i < kRM; ++i) qv[i] = qs[(tr * kRM + i) * kDK + dd];
#pragma unroll
            for (int j = 0; j < kAM; ++j) kv[j] = ks[dd * (kNT + 1) + ta + 32 * j];
#pragma unroll
            for (int i = 0; i < kRM; ++i)
#pragma unroll
              for (int j = 0; j < kAM; ++j) blk[i][j] = __fmaf_rn(qv[i], kv[j], blk[i][j]);
          }
#pragma unroll
          for (int i = 0; i < kRM; ++i)
#pragma unroll
            for (int j = 0; j < kAM; ++j) two_sum_into(acc[i][j], blk[i][j]);
        } else {
          for (int dd = 0; dd < dk; ++dd) {
            float qv[kRM], kv[kAM];
#pragma unroll
            for (int i = 0; i < kRM; ++i) qv[i] = qs[(tr * kRM + i) * kDK + dd];
#pragma unroll
            for (int j = 0; j < kAM; ++j) kv[j] = ks[dd * (kNT + 1) + ta + 32 * j];
#pragma unroll
            for (int i = 0; i < kRM; ++i)
#pragma unroll
              for (int j = 0; j < kAM; ++j) dot2_step(acc[i][j], qv[i], kv[j]);
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int i = 0; i < kRM; ++i) {
        const int r = tr * kRM + i;
#pragma unroll
        for (int j = 0; j < kAM; ++j) {
          const int arow = a0 + ta + 32 * j;
          if (r < nrows && arow < g.nf[f]) scores[r * ntot + g.off[f] + arow] = acc2_value(acc[i][j]);
        }
      }
    }
  }
  __syncthreads();

  // ---- phase 2: one warp per row
  for (int r = warp; r < nrows; r += kThreads / 32) {
    const int qsel = r & 1;
    const int64_t row = (tok0 + (r >> 1)) * a.H + h;
    const int k = g.k[qsel];
    row_topk<EF, EC>(scores + (size_t)r * ntot, g, qsel, cand + (qsel ? cl.n[0] : 0), cl.n[qsel],
                     rs[warp], a.idx[qsel] + row * k, a.wt[qsel] + row * k);
  }
}

template <int EF, int EC>
cudaError_t launch_topk_t(const TopkArgs &a, const CandidateList &cl, int act_dtype,
                          int64_t smem, cudaStream_t st) {
  dim3 grid((unsigned)((a.BT + a.tok_per_cta - 1) / a.tok_per_cta), (unsigned)a.H);
  if (act_dtype == SDM_BF16) {
    auto kern = topk_kernel<EF, EC, __nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>(a, cl);
  } else {
    auto kern = topk_kernel<EF, EC, float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>(a, cl);
  }
  return cudaGetLastError();
}

}  // namespace

// Shared memory of phase 1 tiles; phase 2's per-warp scratch reuses it.
int64_t topk_scratch_bytes() {
  const int64_t p1 = (int64_t)(kRT * kDK + kDK * (kNT + 1)) * 4;
  const int64_t p2 = (int64_t)(kThreads / 32) * sizeof(RowScratch);
  return p1 > p2 ? p1 : p2;
}

cudaError_t launch_topk(const TopkArgs &a, const CandidateList &cl, int act_dtype, int EF,
                        int EC, int64_t smem, cudaStream_t st) {
  if (a.BT == 0 || a.H == 0) return cudaSuccess;
#define SDM_TOPK_CASE(ef, ec) \
  if (EF == ef && EC == ec) return launch_topk_t<ef, ec>(a, cl, act_dtype, smem, st);
  SDM_TOPK_CASE(2, 4) SDM_TOPK_CASE(2, 8) SDM_TOPK_CASE(2, 16) SDM_TOPK_CASE(2, 32)
  SDM_TOPK_CASE(8, 4) SDM_TOPK_CASE(8, 8) SDM_TOPK_CASE(8, 16) SDM_TOPK_CASE(8, 32)
#undef SDM_TOPK_CASE
  return cudaErrorInvalidValue;
}

}  // namespace sdm
