// Product-key factor scores on CUDA cores (any activation type and sub-key width): the
// op's scorer where the tensor-core one does not apply (a factor width that is not a
// multiple of 16, bfloat16 queries whose d_sub is not a multiple of 64), and on request of
// the test hook that compares the two.
//
// s_f[a] = <q[f*d_sub:(f+1)*d_sub], K_f[a]> for both queries of every token and head
// (product-key memory, Lample et al., cited in the sparse-delta-memory README).  One CTA
// takes 16 consecutive tokens of one head = 32 query rows (row 2t = write query, 2t+1 =
// read query) and computes every factor score of those rows as a tiled product with
// the sub-key table: 32-wide slices of d_sub and 256 sub-keys at a time are staged in
// shared memory, 4x8 outputs per thread.  Accumulation follows the block order of
// score_block (sdm_topk.cuh): compensated for float32 inputs, FMA blocks of 32 folded
// into a TwoSum pair for bfloat16, so that the decode kernel's scores are the same bits.
#include "sdm_common.cuh"
#include "sdm_internal.h"
#include "sdm_topk.cuh"

namespace sdm {

namespace {

constexpr int kDK = 32;        // d_sub slice per stage (= the bfloat16 FMA block)
constexpr int kNT = 256;       // sub-keys per pass
constexpr int kRT = 32;        // query rows per CTA
constexpr int kTok = kRT / 2;  // tokens per CTA
constexpr int kRM = 4, kAM = 8;
constexpr int kLoadBatch = 8;  // global loads in flight per thread while staging a tile

template <typename ACT>
__global__ void __launch_bounds__(kThreads) score_simt_kernel(const __grid_constant__ ScoreArgs a) {
  __shared__ float qs[kRT * kDK];
  __shared__ float ks[kDK * (kNT + 1)];
  const KeyGeometry &g = a.g;
  const int h = blockIdx.y;
  const int64_t tok0 = (int64_t)blockIdx.x * kTok;
  const int ntok = (int)min((int64_t)kTok, a.BT - tok0);
  const int nrows = 2 * ntok;
  const int tid = threadIdx.x;
  const int ntot = g.ntot, d_sub = g.d_sub;
  const int64_t qdim = (int64_t)g.F * d_sub;
  const ACT *q[2] = {static_cast<const ACT *>(a.q[0]), static_cast<const ACT *>(a.q[1])};
  const ACT *K = static_cast<const ACT *>(a.subkeys) + (int64_t)h * ntot * d_sub;
  const int tr = tid >> 5, ta = tid & 31;
  const int64_t rows_per_q = a.BT * a.H;

  for (int f = 0; f < g.F; ++f) {
    for (int a0 = 0; a0 < g.nf[f]; a0 += kNT) {
      Acc2 acc[kRM][kAM];
#pragma unroll
      for (int i = 0; i < kRM; ++i)
#pragma unroll
        for (int j = 0; j < kAM; ++j) acc[i][j] = Acc2{0.0f, 0.0f};
      for (int d0 = 0; d0 < d_sub; d0 += kDK) {
        const int dk = min(kDK, d_sub - d0);
        // stage the query slice [kRT][kDK] (4 loads per thread, issued together)
        {
          float t[kRT * kDK / kThreads];
#pragma unroll
          for (int i = 0; i < kRT * kDK / kThreads; ++i) {
            const int e = tid + i * kThreads;
            const int r = e / kDK, dd = e % kDK;
            t[i] = 0.0f;
            if (r < nrows && dd < dk) {
              const int64_t tok = tok0 + (r >> 1);
              t[i] = to_f32(q[r & 1][(tok * a.H + h) * qdim + (int64_t)f * d_sub + d0 + dd]);
            }
          }
#pragma unroll
          for (int i = 0; i < kRT * kDK / kThreads; ++i) qs[tid + i * kThreads] = t[i];
        }
        // stage the sub-key slice transposed, ks[dd][aa] (batches of loads in flight)
        for (int i0 = 0; i0 < kNT * kDK / kThreads; i0 += kLoadBatch) {
          float t[kLoadBatch];
#pragma unroll
          for (int i = 0; i < kLoadBatch; ++i) {
            const int e = tid + (i0 + i) * kThreads;
            const int aa = e / kDK, dd = e % kDK;
            const int arow = a0 + aa;
            t[i] = (arow < g.nf[f] && dd < dk) ? to_f32(K[(int64_t)(g.off[f] + arow) * d_sub + d0 + dd]) : 0.0f;
          }
#pragma unroll
          for (int i = 0; i < kLoadBatch; ++i) {
            const int e = tid + (i0 + i) * kThreads;
            ks[(e % kDK) * (kNT + 1) + e / kDK] = t[i];
          }
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
        if (r >= nrows) continue;
        const int64_t row = (tok0 + (r >> 1)) * a.H + h;
        float *out = a.scores + ((int64_t)(r & 1) * rows_per_q + row) * ntot + g.off[f];
#pragma unroll
        for (int j = 0; j < kAM; ++j) {
          const int arow = a0 + ta + 32 * j;
          if (arow < g.nf[f]) out[arow] = acc2_value(acc[i][j]);
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_score_simt(const ScoreArgs &a, int act_dtype, cudaStream_t st) {
  if (a.BT == 0 || a.H == 0) return cudaSuccess;
  dim3 grid((unsigned)((a.BT + kTok - 1) / kTok), (unsigned)a.H);
  if (act_dtype == SDM_BF16)
    score_simt_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(a);
  else
    score_simt_kernel<float><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sdm
