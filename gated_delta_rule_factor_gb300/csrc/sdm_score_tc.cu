// Product-key factor scores on the 5th-generation tensor cores.
//
// For one query kind, head h and factor f the scores are a dense product
//   S[m, a] = sum_d Q[m, f*d_sub + d] * K_f[a, d],   m = token (B*T of them), a < n_f,
// (product-key memory, Lample et al., cited in the sparse-delta-memory README); at the
// README layer shape that is 8 products of 8192 x 256 x 512, 17.2 GFLOP in all.  One CTA
// computes a 128 x N tile (N <= 256, a whole factor at the layer shape):
//   * one thread issues TMA loads of 64-wide d_sub slices of Q (128 rows) and K_f (N rows)
//     into a ring of 128-byte-swizzled shared-memory tiles;
//   * one thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, 128 x N x 16 per
//     instruction) accumulating in tensor memory, and commits each stage back to the
//     loader through an mbarrier;
//   * four warps read the accumulator out of tensor memory (tcgen05.ld, one row per
//     thread) and store float32 scores.
// bfloat16 products are exact in float32; the tensor core's float32 accumulation order is
// its own, so these scores can differ from a correctly rounded dot product in the last
// bits (the selection parity rule allows for that at near ties).
//
// float32 inputs take the same path through an error-free splitting in the manner of
// Ozaki et al. (error-free transformation of matrix products into products that the
// hardware computes exactly).  split_kernel scales each query segment and each sub-key row
// by a power of two, 2^-e with e the exponent of the row's largest magnitude, and cuts
// the scaled values into four fixed-point slices of 8 bits: x = 2^(e-7) * (n0 + n1 2^-8 +
// n2 2^-16 + n3 2^-24) + (a remainder below 2^(e-31)), with integers |n0| <= 256 and
// |n1|, |n2|, |n3| <= 128, all exact in bfloat16.  Level L of the product keeps the slice
// pairs (i, L - i), L <= 3: its products are integers below 2^16 and its sum over d_sub
// terms stays below 1.5 * 2^16 * d_sub, so for d_sub <= 128 every level accumulates
// exactly in its own float32 tensor-memory accumulator whatever the order.  The epilogue
// joins the four levels exactly in a 64-bit integer, converts it to float32 with one
// rounding and scales by 2^(e_q + e_k - 38): the correctly rounded score of the sum with
// the slice pairs of level >= 4 and the remainders left out (below 2^-29 * d_sub *
// max|q| * max|k| together).  The parts are padded with zeros to a multiple of 64.
// Every mbarrier wait is bounded: on time-out the kernel records SDM_DEVERR_TIMEOUT,
// stops issuing work, waits (bounded) for its own copies and frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kTcM = 128;         // tokens per tile (MMA M)
constexpr int kTcK = 64;          // bf16 per k-block = one 128-byte swizzle row
constexpr int kTcMaxStages = 4;
constexpr int kTcMaxN = 256;
constexpr int kTcSplitMaxN = 64;    // four level accumulators of <= 64 columns: 256 TMEM columns
constexpr int kSplitParts = 4;
constexpr int kTcThreads = 128;
constexpr int64_t kTcStageBudget = 200 * 1024;

struct TcArgs {
  CUtensorMap tq[2];   // q_w, q_r viewed as [BT rows][H*F*PARTS*dp] bf16
  CUtensorMap tk;      // subkeys viewed as [H*ntot rows][PARTS*dp] bf16
  float *scores;
  int32_t *err;
  int64_t BT;
  int32_t H, F, ntot;
  int32_t dp;          // width of one part in the rows above (d_sub, or d_sub padded to 64)
  int32_t nk;          // 64-wide k blocks per part
  int32_t stages;      // ring depth (<= kTcMaxStages)
  int32_t nf[SDM_MAX_FACTORS], off[SDM_MAX_FACTORS];
  int32_t n_tile;      // MMA N (multiple of 16, <= 256; <= 64 for split inputs)
  int32_t n_tiles;     // N tiles per factor (max over factors)
  const int32_t *qexp, *kexp;   // split inputs: segment exponents (SplitArgs)
};

// The split inputs of float32 scoring: four integer slices per value, zero-padded to dp,
// and the power-of-two exponent of every segment.
struct SplitArgs {
  const float *q[2];        // [BT, H*F*d_sub]
  const float *subkeys;     // [H*ntot, d_sub]
  __nv_bfloat16 *qs;        // [2][BT][H*F][4][dp]
  __nv_bfloat16 *ks;        // [H*ntot][4][dp]
  int32_t *qexp;            // [2][BT][H*F]
  int32_t *kexp;            // [H*ntot]
  int64_t BT;
  int32_t HF, d_sub, dp, krows;
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

// 2^k as a float32 for -126 <= k <= 127 (exact), else 0.
__device__ __forceinline__ float pow2f(int k) {
  return (k >= -126 && k <= 127) ? __uint_as_float((uint32_t)(k + 127) << 23) : 0.0f;
}

// x * 2^k, exact whenever the result is a normal float32.
__device__ __forceinline__ float scale2(float x, int k) {
  const float p = pow2f(k);
  return p != 0.0f ? x * p : ldexpf(x, k);
}

// Eight lanes per segment (a query's factor slice, or a sub-key row), eight consecutive
// values per lane and 64-wide column block: the largest magnitude m gives e with m in
// [2^e, 2^(e+1)) (e = 0 for an all-zero segment); each value scaled by 2^(7-e) lies in
// [-256, 256] and is cut into its nearest integer n0 and three further 8-bit integer
// digits of the remainders, each step exact in float32; every slice is stored as eight
// bfloat16 (16 bytes).
__global__ void __launch_bounds__(256) split_kernel(const __grid_constant__ SplitArgs a) {
  const int lane = threadIdx.x & 31, sub8 = lane & 7;
  const unsigned gmask = 0xffu << (lane & 24);
  const int64_t qrows = 2 * a.BT * a.HF, total = qrows + a.krows;
  const int64_t ngroups = ((int64_t)gridDim.x * blockDim.x) >> 3;
  const bool vec = (a.d_sub & 7) == 0;
  for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 3; row < total; row += ngroups) {
    const float *src;
    __nv_bfloat16 *dst;
    int32_t *ex;
    if (row < qrows) {                     // row = (qsel * BT + token) * HF + hf
      const int64_t qsel = row / (a.BT * a.HF), rem = row % (a.BT * a.HF);
      src = a.q[qsel] + rem * a.d_sub;
      dst = a.qs + row * kSplitParts * a.dp;
      ex = a.qexp + row;
    } else {
      const int64_t kr = row - qrows;
      src = a.subkeys + kr * a.d_sub;
      dst = a.ks + kr * kSplitParts * a.dp;
      ex = a.kexp + kr;
    }
    auto load8 = [&](int d0, float (&v)[8]) {
      if (vec && d0 < a.d_sub) {
        const float4 lo = *reinterpret_cast<const float4 *>(src + d0);
        const float4 hi = *reinterpret_cast<const float4 *>(src + d0 + 4);
        v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
        v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = d0 + j < a.d_sub ? src[d0 + j] : 0.0f;
      }
    };
    float m = 0.0f;
    for (int d0 = 8 * sub8; d0 < a.d_sub; d0 += 64) {
      float v[8];
      load8(d0, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(gmask, m, o));
    int e = 0;
    if (m > 0.0f) {
      int E;
      frexpf(m, &E);                       // m = f 2^E, f in [0.5, 1)
      e = E - 1;
    }
    if (sub8 == 0) *ex = e;
    for (int d0 = 8 * sub8; d0 < a.dp; d0 += 64) {
      float v[8];
      load8(d0, v);
      __align__(16) __nv_bfloat16 p[kSplitParts][8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float r = scale2(v[j], 7 - e);
#pragma unroll
        for (int q = 0; q < kSplitParts; ++q) {
          const float n = rintf(r);
          p[q][j] = __float2bfloat16_rn(n);
          r = (r - n) * 256.0f;
        }
      }
#pragma unroll
      for (int q = 0; q < kSplitParts; ++q)
        *reinterpret_cast<uint4 *>(dst + q * a.dp + d0) = *reinterpret_cast<const uint4 *>(p[q]);
    }
  }
}

// PARTS = 1: bfloat16 inputs, one accumulator.  PARTS = 4: the split float32 inputs; the
// stage holds the four slices of the Q slice and of the K_f slice, and level L's
// accumulator takes TMEM columns [L C, L C + N), C = N rounded up to 32 so that every
// 32-column read stays inside the allocation.
template <int PARTS>
__global__ void __launch_bounds__(kTcThreads, 1) score_tc_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int N = a.n_tile;
  const int a_bytes = kTcM * 128, b_bytes = N * 128;
  const int stage_bytes = PARTS * (a_bytes + b_bytes);   // [PARTS A tiles][PARTS B tiles]
  const int stages = a.stages;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + stages * stage_bytes);
  uint64_t *full = bars, *empty = bars + kTcMaxStages, *done = bars + 2 * kTcMaxStages;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kTcMaxStages + 1);
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
  const int nk = a.nk;
  const int lvl_col = (N + 31) & ~31;            // column stride of the level accumulators
  const int acc_cols = PARTS == 1 ? N : 4 * lvl_col;
  const uint32_t tmem_cols = acc_cols <= 32 ? 32 : (acc_cols <= 64 ? 64 : (acc_cols <= 128 ? 128 : 256));

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
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
    const int32_t qx0 = (h * a.F + f) * PARTS * a.dp;
    const int32_t ky = h * a.ntot + a.off[f] + n0;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % stages, use = kb / stages;
      if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1)) {
        raise_error(a.err, SDM_DEVERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      unsigned char *st = smem + s * stage_bytes;
      mbar_expect_tx(&full[s], (uint32_t)stage_bytes);
#pragma unroll
      for (int p = 0; p < PARTS; ++p) {
        tma_load_2d(st + p * a_bytes, tq, qx0 + p * a.dp + kb * kTcK, (int32_t)m0, &full[s]);
        tma_load_2d(st + PARTS * a_bytes + p * b_bytes, &a.tk, p * a.dp + kb * kTcK, ky, &full[s]);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    const uint32_t idesc = mma_idesc(kTcM, N);
    bool ok = true;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % stages, use = kb / stages;
      if (!mbar_wait(&full[s], use & 1)) {
        raise_error(a.err, SDM_DEVERR_TIMEOUT);
        *abort_flag = 1;
        ok = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
      const uint32_t sa = smem_addr(smem + s * stage_bytes), sb = sa + PARTS * a_bytes;
#pragma unroll
      for (int kk = 0; kk < kTcK / 16; ++kk) {
        if (PARTS == 1) {
          mma_bf16(tmem, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32), idesc, (kb | kk) ? 1u : 0u);
        } else {
          // level L = i + j of the slice pair (i, j), L <= 3
          constexpr int pi[10] = {0, 0, 1, 0, 1, 2, 0, 1, 2, 3}, pj[10] = {0, 1, 0, 2, 1, 0, 3, 2, 1, 0};
          constexpr int lv[10] = {0, 1, 1, 2, 2, 2, 3, 3, 3, 3}, first[10] = {1, 1, 0, 1, 0, 0, 1, 0, 0, 0};
#pragma unroll
          for (int c = 0; c < 10; ++c)
            mma_bf16(tmem + (uint32_t)(lv[c] * lvl_col), sw128_desc(sa + pi[c] * a_bytes + kk * 32),
                     sw128_desc(sb + pj[c] * b_bytes + kk * 32), idesc, ((kb | kk) || !first[c]) ? 1u : 0u);
        }
      }
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
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int32_t eq = PARTS == 1 || m >= a.BT ? 0 : a.qexp[(qsel * a.BT + m) * a.H * a.F + h * a.F + f];
    const int32_t *ek = PARTS == 1 ? nullptr : a.kexp + h * a.ntot + a.off[f] + n0;
    for (int c0 = 0; c0 < N; c0 += 32) {
      float v[32];
      tmem_ld32(lane_base + (uint32_t)c0, v);
      if (PARTS == kSplitParts) {
        // join the exact level sums X = sum_L acc_L 2^(8 (3 - L)) as a 64-bit integer (each
        // acc_L converted to 32 bits), then X = H 2^24 + Lo with H and Lo exact in float32,
        // so one float32 addition rounds X correctly; then the exact scale 2^(e_q + e_k - 38)
        long long tot[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) tot[i] = (long long)__float2int_rn(v[i]) << 24;
#pragma unroll
        for (int L = 1; L < 4; ++L) {
          tmem_ld32(lane_base + (uint32_t)(L * lvl_col + c0), v);
#pragma unroll
          for (int i = 0; i < 32; ++i) tot[i] += (long long)__float2int_rn(v[i]) << (8 * (3 - L));
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int32_t e = c0 + i < nvalid ? ek[c0 + i] : 0;
          const float hi = (float)(int32_t)(tot[i] >> 24), lo = (float)(int32_t)(tot[i] & 0xffffff);
          v[i] = scale2(__fmaf_rn(hi, 16777216.0f, lo), eq + e - 38);
        }
      }
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

int32_t split_width(const KeyGeometry &g) { return (g.d_sub + kTcK - 1) / kTcK * kTcK; }

int tc_n_tile(const KeyGeometry &g, int act_dtype) {
  int maxnf = 0;
  for (int f = 0; f < g.F; ++f) maxnf = maxnf > g.nf[f] ? maxnf : g.nf[f];
  const int cap = act_dtype == SDM_F32 ? kTcSplitMaxN : kTcMaxN;
  return maxnf < cap ? maxnf : cap;
}

// Slices [segments][4][dp] bf16, then the segments' exponents (int32), 256-byte aligned.
int64_t split_slice_bytes(const KeyGeometry &g, int64_t BT, int64_t H) {
  return ((2 * BT * H * g.F + H * g.ntot) * kSplitParts * (int64_t)split_width(g) * 2 + 255) & ~int64_t(255);
}

}  // namespace

int64_t score_split_bytes(const KeyGeometry &g, int64_t BT, int64_t H, int act_dtype) {
  if (act_dtype != SDM_F32) return 0;
  return split_slice_bytes(g, BT, H) + (2 * BT * H * g.F + H * g.ntot) * 4;
}

bool score_tc_supported(const KeyGeometry &g, int64_t H, int act_dtype) {
  if (act_dtype == SDM_BF16) {
    if (g.d_sub % kTcK != 0) return false;
  } else if (act_dtype != SDM_F32) {
    return false;
  }
  int maxnf = 0;
  for (int f = 0; f < g.F; ++f) {
    if (g.nf[f] % 16 != 0) return false;
    maxnf = maxnf > g.nf[f] ? maxnf : g.nf[f];
  }
  const int nt = tc_n_tile(g, act_dtype);
  if (2 * H * g.F * ((maxnf + nt - 1) / nt) > 65535) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_score_tc(const ScoreArgs &s, int act_dtype, cudaStream_t st) {
  if (s.BT == 0 || s.H == 0) return cudaSuccess;
  TcArgs a{};
  const KeyGeometry &g = s.g;
  const bool split = act_dtype == SDM_F32;
  const int parts = split ? kSplitParts : 1;
  a.dp = split ? split_width(g) : g.d_sub;
  a.nk = a.dp / kTcK;
  const void *q0 = s.q[0], *q1 = s.q[1], *keys = s.subkeys;
  if (split) {
    if (!s.split) return cudaErrorInvalidValue;
    SplitArgs sp{};
    sp.q[0] = static_cast<const float *>(s.q[0]);
    sp.q[1] = static_cast<const float *>(s.q[1]);
    sp.subkeys = static_cast<const float *>(s.subkeys);
    sp.BT = s.BT;
    sp.HF = s.H * g.F;
    sp.d_sub = g.d_sub;
    sp.dp = a.dp;
    sp.krows = s.H * g.ntot;
    const int64_t qrows = 2 * s.BT * sp.HF;
    sp.qs = static_cast<__nv_bfloat16 *>(s.split);
    sp.ks = sp.qs + qrows * kSplitParts * (int64_t)a.dp;
    sp.qexp = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(s.split) + split_slice_bytes(g, s.BT, s.H));
    sp.kexp = sp.qexp + qrows;
    const int64_t blocks = std::min<int64_t>((qrows + sp.krows + 31) / 32, 16384);  // 32 segments a block
    split_kernel<<<(unsigned)blocks, 256, 0, st>>>(sp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    q0 = sp.qs;
    q1 = sp.qs + s.BT * sp.HF * kSplitParts * (int64_t)a.dp;
    keys = sp.ks;
    a.qexp = sp.qexp;
    a.kexp = sp.kexp;
  }
  const uint64_t qcols = (uint64_t)s.H * g.F * parts * a.dp;
  int maxnf = 0;
  for (int f = 0; f < g.F; ++f) maxnf = maxnf > g.nf[f] ? maxnf : g.nf[f];
  a.n_tile = tc_n_tile(g, act_dtype);
  a.n_tiles = (maxnf + a.n_tile - 1) / a.n_tile;
  if (!make_map(&a.tq[0], q0, qcols, (uint64_t)s.BT, kTcK, kTcM) ||
      !make_map(&a.tq[1], q1, qcols, (uint64_t)s.BT, kTcK, kTcM) ||
      !make_map(&a.tk, keys, (uint64_t)parts * a.dp, (uint64_t)s.H * g.ntot, kTcK, (uint32_t)a.n_tile))
    return cudaErrorInvalidValue;
  a.scores = s.scores;
  a.err = s.err;
  a.BT = s.BT;
  a.H = s.H;
  a.F = g.F;
  a.ntot = g.ntot;
  for (int f = 0; f < SDM_MAX_FACTORS; ++f) {
    a.nf[f] = g.nf[f];
    a.off[f] = g.off[f];
  }
  const int64_t stage_bytes = (int64_t)parts * (kTcM + a.n_tile) * 128;
  a.stages = (int32_t)std::max<int64_t>(1, std::min<int64_t>({(int64_t)kTcMaxStages, kTcStageBudget / stage_bytes,
                                                               (int64_t)a.nk}));
  const int64_t smem = 1024 + a.stages * stage_bytes + 256;
  const void *kern = split ? reinterpret_cast<const void *>(score_tc_kernel<kSplitParts>)
                           : reinterpret_cast<const void *>(score_tc_kernel<1>);
  cudaError_t e = raise_smem_limit(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((s.BT + kTcM - 1) / kTcM), (unsigned)(2 * s.H * g.F * a.n_tiles));
  if (split)
    score_tc_kernel<kSplitParts><<<grid, kTcThreads, smem, st>>>(a);
  else
    score_tc_kernel<1><<<grid, kTcThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sdm
