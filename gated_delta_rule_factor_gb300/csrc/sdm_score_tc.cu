// Product-key factor scores on the 5th-generation tensor cores (bfloat16 inputs).
//
// For one query kind, head h and factor f the scores are a dense product
//   S[m, a] = sum_d Q[m, f*d_sub + d] * K_f[a, d],   m = token (B*T of them), a < n_f,
// (product-key memory, Lample et al., cited in the sparse-delta-memory README); at the
// README layer shape that is 8 products of 8192 x 256 x 512, 17.2 GFLOP in all.  One CTA
// computes a 128 x N tile (N <= 256, a whole factor at the layer shape):
//   * one thread issues TMA loads of 64-wide d_sub slices of Q (128 rows) and K_f (N rows)
//     into a 4-stage ring of 128-byte-swizzled shared-memory tiles;
//   * one thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, 128 x N x 16 per
//     instruction) accumulating in tensor memory, and commits each stage back to the
//     loader through an mbarrier;
//   * four warps read the accumulator out of tensor memory (tcgen05.ld, one row per
//     thread) and store float32 scores.
// bfloat16 products are exact in float32; the tensor core's float32 accumulation order is
// its own, so these scores can differ from a correctly rounded dot product in the last
// bits (the selection parity rule allows for that at near ties).
// Every mbarrier wait is bounded: on time-out the kernel records SDM_DEVERR_TIMEOUT,
// stops issuing work, waits (bounded) for its own copies and frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kTcM = 128;         // tokens per tile (MMA M)
constexpr int kTcK = 64;          // bf16 per k-block = one 128-byte swizzle row
constexpr int kTcStages = 4;
constexpr int kTcMaxN = 256;
constexpr int kTcThreads = 128;

struct TcArgs {
  CUtensorMap tq[2];   // q_w, q_r viewed as [BT rows][H*F*d_sub] bf16
  CUtensorMap tk;      // subkeys viewed as [H*ntot rows][d_sub] bf16
  float *scores;
  int32_t *err;
  int64_t BT;
  int32_t H, F, d_sub, ntot;
  int32_t nf[SDM_MAX_FACTORS], off[SDM_MAX_FACTORS];
  int32_t n_tile;      // MMA N (multiple of 16, <= 256)
  int32_t n_tiles;     // N tiles per factor (max over factors)
};

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int32_t x, int32_t y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled bf16 tile whose rows
// are 128 bytes and whose 8-row groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);            // start address
  d |= (uint64_t)1u << 16;                            // leading byte offset (unused here)
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;      // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1u << 46;                            // descriptor version
  d |= (uint64_t)2u << 61;                            // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, A = B = bf16, D = fp32, both K-major, M x N.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kTcThreads, 1) score_tc_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int N = a.n_tile;
  const int a_bytes = kTcM * 128, b_bytes = N * 128;
  unsigned char *tiles_a = smem;                                   // [stages][128 rows][128 B]
  unsigned char *tiles_b = smem + kTcStages * a_bytes;             // [stages][N rows][128 B]
  uint64_t *bars = reinterpret_cast<uint64_t *>(tiles_b + kTcStages * b_bytes);
  uint64_t *full = bars, *empty = bars + kTcStages, *done = bars + 2 * kTcStages;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kTcStages + 1);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int yb = blockIdx.y;
  const int nt = yb % a.n_tiles;
  yb /= a.n_tiles;
  const int f = yb % a.F;
  yb /= a.F;
  const int h = yb % a.H;
  const int qsel = yb / a.H;
  const int n0 = nt * N;
  if (n0 >= a.nf[f]) return;                     // uniform over the CTA
  const int nvalid = min(N, a.nf[f] - n0);
  const int64_t m0 = (int64_t)blockIdx.x * kTcM;
  const int nk = a.d_sub / kTcK;
  const uint32_t tmem_cols = N <= 32 ? 32 : (N <= 64 ? 64 : (N <= 128 ? 128 : 256));

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(tmem_slot)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer
    const CUtensorMap *tq = &a.tq[qsel];
    const int32_t qx0 = h * a.F * a.d_sub + f * a.d_sub;
    const int32_t ky = h * a.ntot + a.off[f] + n0;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kTcStages, use = kb / kTcStages;
      if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1)) {
        raise_error(a.err, SDM_DEVERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      mbar_expect_tx(&full[s], (uint32_t)(a_bytes + b_bytes));
      tma_load_2d(tiles_a + s * a_bytes, tq, qx0 + kb * kTcK, (int32_t)m0, &full[s]);
      tma_load_2d(tiles_b + s * b_bytes, &a.tk, kb * kTcK, ky, &full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    const uint32_t idesc = mma_idesc(kTcM, N);
    bool ok = true;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kTcStages, use = kb / kTcStages;
      if (!mbar_wait(&full[s], use & 1)) {
        raise_error(a.err, SDM_DEVERR_TIMEOUT);
        *abort_flag = 1;
        ok = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
      const uint32_t sa = smem_addr(tiles_a + s * a_bytes), sb = smem_addr(tiles_b + s * b_bytes);
#pragma unroll
      for (int kk = 0; kk < kTcK / 16; ++kk)
        mma_bf16(tmem, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32), idesc, (kb | kk) ? 1u : 0u);
      mma_commit(&empty[s]);
    }
    if (ok) mma_commit(done);
  }
  __syncwarp();

  // ---- epilogue: TMEM lane = tile row = 32 * warp + lane
  const bool ok = mbar_wait(done, 0);
  if (!ok && tid == 0) raise_error(a.err, SDM_DEVERR_TIMEOUT);
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
  if (ok && !*abort_flag) {
    const int64_t m = m0 + warp * 32 + lane;
    const int64_t rows_per_q = a.BT * a.H;
    float *out = a.scores + ((int64_t)qsel * rows_per_q + m * a.H + h) * a.ntot + a.off[f] + n0;
    for (int c0 = 0; c0 < N; c0 += 32) {
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
      if (m < a.BT) {
        if (c0 + 32 <= nvalid) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4 *>(out + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
          for (int i = 0; i < 32 && c0 + i < nvalid; ++i) out[c0 + i] = v[i];
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(tmem_cols) : "memory");
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool score_tc_supported(const KeyGeometry &g, int act_dtype) {
  if (act_dtype != SDM_BF16 || g.d_sub % kTcK != 0) return false;
  for (int f = 0; f < g.F; ++f)
    if (g.nf[f] % 16 != 0) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_score_tc(const ScoreArgs &s, cudaStream_t st) {
  if (s.BT == 0 || s.H == 0) return cudaSuccess;
  TcArgs a{};
  const KeyGeometry &g = s.g;
  const uint64_t qcols = (uint64_t)s.H * g.F * g.d_sub;
  int maxnf = 0;
  for (int f = 0; f < g.F; ++f) maxnf = maxnf > g.nf[f] ? maxnf : g.nf[f];
  a.n_tile = maxnf < kTcMaxN ? maxnf : kTcMaxN;
  a.n_tiles = (maxnf + a.n_tile - 1) / a.n_tile;
  if (!make_map(&a.tq[0], s.q[0], qcols, (uint64_t)s.BT, kTcK, kTcM) ||
      !make_map(&a.tq[1], s.q[1], qcols, (uint64_t)s.BT, kTcK, kTcM) ||
      !make_map(&a.tk, s.subkeys, (uint64_t)g.d_sub, (uint64_t)s.H * g.ntot, kTcK, (uint32_t)a.n_tile))
    return cudaErrorInvalidValue;
  a.scores = s.scores;
  a.err = s.err;
  a.BT = s.BT;
  a.H = s.H;
  a.F = g.F;
  a.d_sub = g.d_sub;
  a.ntot = g.ntot;
  for (int f = 0; f < SDM_MAX_FACTORS; ++f) {
    a.nf[f] = g.nf[f];
    a.off[f] = g.off[f];
  }
  const int64_t smem = 1024 + (int64_t)kTcStages * (kTcM + a.n_tile) * 128 + 256;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(score_tc_kernel), smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((s.BT + kTcM - 1) / kTcM), (unsigned)(2 * s.H * g.F * a.n_tiles));
  score_tc_kernel<<<grid, kTcThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sdm
