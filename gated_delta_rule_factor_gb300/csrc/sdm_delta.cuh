// Per-token gated delta-rule write and weighted read.
//
// For one token with forget gate alpha, input gate beta, value v and the W selected
// rows M[i_j] with weights w_j (a reading of the gated delta rule of Yang et al., cited
// in the sparse-delta-memory README, restricted to the selected rows):
//   m_j = alpha * M[i_j]
//   p   = sum_j w_j m_j
//   M[i_j] <- m_j + w_j * beta * (v - p)          (rounded to the bank type)
// and then the read over the R selected rows: y = sum_j r_j M[i^r_j].  Every column is
// independent.  All of it is float32 with a fixed operation order, so results are
// bitwise repeatable and independent of how tokens are staged.
//
// Two layouts:
//   * delta_write_staged / weighted_read_staged (the decode kernel): a warp owns NCG
//     16-byte column groups (lane % NCG) and splits the rows over RG = 32 / NCG row
//     groups (lane / NCG): row j belongs to row group j % RG and is accumulated in
//     increasing j; the RG partial sums are combined by an xor butterfly.  Each lane
//     fetches all of its rows into shared memory with cp.async at once (one memory round
//     trip per sum) and reads back only what it fetched.
//   * token_blocks2 (the write/read kernel, rows in shared memory), below.
#pragma once

#include "sdm_common.cuh"

namespace sdm {

// 16-byte raw row chunk <-> float32 lanes.
template <typename BANK>
__device__ __forceinline__ void unpack16(const uint4 &u, float (&out)[Vec16<BANK>::N]) {
  const BANK *e = reinterpret_cast<const BANK *>(&u);
#pragma unroll
  for (int i = 0; i < Vec16<BANK>::N; ++i) out[i] = to_f32(e[i]);
}

// stage: this warp's rows, NCG * 16 bytes each (at least n rows); src(j): row j's 16
// bytes of this lane's column group in global memory.  valid == false (a column group
// past d_v) fetches and stores nothing; its lanes' sums are not used.
template <int NCG, class SrcRow>
__device__ __forceinline__ void stage_rows(int n, bool valid, unsigned char *stage, SrcRow src) {
  constexpr int RG = 32 / NCG, RB = NCG * 16;
  const int lane = threadIdx.x & 31, rg = lane / NCG;
  unsigned char *mine = stage + (lane % NCG) * 16;
  if (valid)
#pragma unroll 4
    for (int j = rg; j < n; j += RG) cp_async16(mine + j * RB, src(j));
  cp_async_commit();
  cp_async_wait_all();
}

template <typename BANK, int NCG>
__device__ __forceinline__ void staged_row(const unsigned char *stage, int j, float (&out)[Vec16<BANK>::N]) {
  const int lane = threadIdx.x & 31;
  unpack16<BANK>(*reinterpret_cast<const uint4 *>(stage + j * (NCG * 16) + (lane % NCG) * 16), out);
}

template <int NCG, int VEC>
__device__ __forceinline__ void row_group_butterfly(float (&x)[VEC]) {
#pragma unroll
  for (int o = NCG; o < 32; o <<= 1)
#pragma unroll
    for (int c = 0; c < VEC; ++c) x[c] = __fadd_rn(x[c], __shfl_xor_sync(0xffffffffu, x[c], o));
}

// The gated delta-rule write of W rows: p = sum_j w_j alpha m_j, then
// m_j <- alpha m_j + w_j beta (v - p), stored through dst(j).
template <typename BANK, int NCG, class SrcRow, class DstRow>
__device__ __forceinline__ void delta_write_staged(int W, const float *w, float alpha, float beta,
                                                   const float (&v)[Vec16<BANK>::N], bool valid,
                                                   unsigned char *stage, SrcRow src, DstRow dst) {
  constexpr int VEC = Vec16<BANK>::N, RG = 32 / NCG;
  const int rg = (threadIdx.x & 31) / NCG;
  stage_rows<NCG>(W, valid, stage, src);
  float acc[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) acc[c] = 0.0f;
  for (int j = rg; j < W; j += RG) {
    const float wj = w[j];
    float r[VEC];
    staged_row<BANK, NCG>(stage, j, r);
#pragma unroll
    for (int c = 0; c < VEC; ++c) acc[c] = __fmaf_rn(wj, __fmul_rn(alpha, r[c]), acc[c]);
  }
  row_group_butterfly<NCG>(acc);
  float d[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) d[c] = __fmul_rn(beta, __fsub_rn(v[c], acc[c]));
  if (!valid) return;
  for (int j = rg; j < W; j += RG) {
    const float wj = w[j];
    float r[VEC];
    staged_row<BANK, NCG>(stage, j, r);
#pragma unroll
    for (int c = 0; c < VEC; ++c) r[c] = __fmaf_rn(wj, d[c], __fmul_rn(alpha, r[c]));
    store_vec16<BANK>(dst(j), r);
  }
}

// The weighted read y = sum_j r_j m_j of R rows fetched through src(j).
template <typename BANK, int NCG, class SrcRow>
__device__ __forceinline__ void weighted_read_staged(int R, const float *r, bool valid, unsigned char *stage,
                                                     SrcRow src, float (&y)[Vec16<BANK>::N]) {
  constexpr int VEC = Vec16<BANK>::N, RG = 32 / NCG;
  const int rg = (threadIdx.x & 31) / NCG;
  stage_rows<NCG>(R, valid, stage, src);
#pragma unroll
  for (int c = 0; c < VEC; ++c) y[c] = 0.0f;
  for (int j = rg; j < R; j += RG) {
    const float rj = r[j];
    float m[VEC];
    staged_row<BANK, NCG>(stage, j, m);
#pragma unroll
    for (int c = 0; c < VEC; ++c) y[c] = __fmaf_rn(rj, m[c], y[c]);
  }
  row_group_butterfly<NCG>(y);
}

// ------------------------------------------------------------------------------------
// Block-ordered token step of the write/read kernel, two warps per row slice.
//
// Summation order.  The n rows of a sum (n = W for the prediction p, n = R for the
// read y) are cut into 8 consecutive blocks of B8 = ceil(n / 8) rows; block k is summed
// in increasing j into a_k and the block sums are combined as
//   ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7)).
// The order depends on n alone: not on the stage length, nor on the column slicing.
//
// Layout.  Lane % 8 owns VEC consecutive elements of the slice (the slice is 8*VEC
// elements wide) and warp wsel's row group rg = lane / 8 owns block k = 4*wsel + rg: a
// lane adds its block, two xor steps inside the warp give (a0+a1)+(a2+a3) in warp 0 and
// (a4+a5)+(a6+a7) in warp 1, and the warps swap those through shared memory (xch:
// [2 warps][8 column groups][VEC] floats) on a 64-thread named barrier `bar`.  IEEE
// addition is commutative, so both partners of every step hold the same bits.
// JB >= B8: register slot s holds row k*B8 + s.
template <int BYTES>
struct RawVec;
template <>
struct RawVec<16> { using T = uint4; };
template <>
struct RawVec<8> { using T = uint2; };
template <>
struct RawVec<4> { using T = uint32_t; };
template <>
struct RawVec<2> { using T = uint16_t; };

// VEC elements of BANK <-> float32.
template <typename BANK, int VEC>
struct LaneRow {
  using Raw = typename RawVec<VEC * (int)sizeof(BANK)>::T;
  __device__ __forceinline__ static Raw load(const unsigned char *p) { return *reinterpret_cast<const Raw *>(p); }
  __device__ __forceinline__ static void unpack(const Raw &r, float (&out)[VEC]) {
    const BANK *e = reinterpret_cast<const BANK *>(&r);
#pragma unroll
    for (int i = 0; i < VEC; ++i) out[i] = to_f32(e[i]);
  }
  __device__ __forceinline__ static void store(unsigned char *p, const float (&in)[VEC]) {
    Raw r;
    BANK *e = reinterpret_cast<BANK *>(&r);
#pragma unroll
    for (int i = 0; i < VEC; ++i) e[i] = from_f32<BANK>(in[i]);
    *reinterpret_cast<Raw *>(p) = r;
  }
};

template <int JB>
struct BlockSlots1 {
  int b8, j0, n;
  __device__ __forceinline__ BlockSlots1(int n_, int k) : b8((n_ + 7) >> 3), j0(k * ((n_ + 7) >> 3)), n(n_) {}
  __device__ __forceinline__ int ref(int s) const { return j0 + s; }
  __device__ __forceinline__ bool has(int s) const { return s < b8 && j0 + s < n; }
};

template <int VEC>
__device__ __forceinline__ void pair_tree(const float (&a)[VEC], float (&out)[VEC], float *xch, int wsel, int bar) {
  const int lane = threadIdx.x & 31;
  float x[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) {
    x[c] = __fadd_rn(a[c], __shfl_xor_sync(0xffffffffu, a[c], 8));
    x[c] = __fadd_rn(x[c], __shfl_xor_sync(0xffffffffu, x[c], 16));
  }
  float *mine = xch + (wsel * 8 + (lane & 7)) * VEC;
  const float *theirs = xch + ((wsel ^ 1) * 8 + (lane & 7)) * VEC;
  if (lane < 8) {
    if constexpr (VEC % 4 == 0) {
#pragma unroll
      for (int c = 0; c < VEC; c += 4)
        *reinterpret_cast<float4 *>(mine + c) = make_float4(x[c], x[c + 1], x[c + 2], x[c + 3]);
    } else if constexpr (VEC == 2) {
      *reinterpret_cast<float2 *>(mine) = make_float2(x[0], x[1]);
    } else {
      mine[0] = x[0];
    }
  }
  named_barrier(bar, 64);
  float o[VEC];
  if constexpr (VEC % 4 == 0) {
#pragma unroll
    for (int c = 0; c < VEC; c += 4) {
      const float4 q = *reinterpret_cast<const float4 *>(theirs + c);
      o[c] = q.x;
      o[c + 1] = q.y;
      o[c + 2] = q.z;
      o[c + 3] = q.w;
    }
  } else if constexpr (VEC == 2) {
    const float2 q = *reinterpret_cast<const float2 *>(theirs);
    o[0] = q.x;
    o[1] = q.y;
  } else {
    o[0] = theirs[0];
  }
#pragma unroll
  for (int c = 0; c < VEC; ++c) out[c] = __fadd_rn(x[c], o[c]);
}

template <typename BANK, int VEC, int JB>
__device__ __forceinline__ void pair_read(const BlockSlots1<JB> &rs, const uint16_t *rm_r, const float *wt_r,
                                          const unsigned char *rows, int RB, float (&b)[VEC]) {
  using LR = LaneRow<BANK, VEC>;
#pragma unroll
  for (int s0 = 0; s0 < JB; s0 += 4) {
    typename LR::Raw raw[4];
    float wr[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int s = s0 + q;
      if (rs.has(s)) {
        raw[q] = LR::load(rows + (int)rm_r[rs.ref(s)] * RB);
        wr[q] = wt_r[rs.ref(s)];
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (rs.has(s0 + q)) {
        float m[VEC];
        LR::unpack(raw[q], m);
#pragma unroll
        for (int c = 0; c < VEC; ++c) b[c] = __fmaf_rn(wr[q], m[c], b[c]);
      }
    }
  }
}

// One token: the gated delta-rule write of its W rows, then the read of its R rows, with
// the arithmetic of delta_write_staged / weighted_read_staged per element and the block order
// above for both sums.  rm / wt: the token's row references (stage-buffer row indices)
// and weights, W write entries then R read entries; rows: the stage buffer offset by this
// lane's column group; RB: the row slice in bytes.  When the token reads none of the rows
// it writes (overlap == false) the read runs before the write: those rows hold the same
// values before and after it.  FULL: W == R == 8 * JB.  The read's exchange barrier comes
// after the row stores, so it also orders this token's writes before the next token's
// loads in the other warp.
template <typename BANK, int VEC, int JB, bool FULL = false>
__device__ __forceinline__ void token_blocks2(int W, int R, const uint16_t *rm, const float *wt, float alpha,
                                              float beta, const float (&v)[VEC], unsigned char *rows, int RB,
                                              bool overlap, float (&y)[VEC], float *xch_p, float *xch_y, int wsel,
                                              int bar) {
  using LR = LaneRow<BANK, VEC>;
  if constexpr (FULL) W = R = 8 * JB;
  const int k = 4 * wsel + ((threadIdx.x & 31) >> 3);
  const BlockSlots1<JB> ws(W, k), rs(R, k);
  int ow[JB];
  float ww[JB];
  typename LR::Raw rw[JB];
#pragma unroll
  for (int s = 0; s < JB; ++s) {
    ow[s] = ws.has(s) ? (int)rm[ws.ref(s)] * RB : 0;
    ww[s] = ws.has(s) ? wt[ws.ref(s)] : 0.0f;
  }
#pragma unroll
  for (int s = 0; s < JB; ++s)
    if (ws.has(s)) rw[s] = LR::load(rows + ow[s]);
  float b[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) b[c] = 0.0f;
  if (!overlap) pair_read<BANK, VEC, JB>(rs, rm + W, wt + W, rows, RB, b);

  float a[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) a[c] = 0.0f;
#pragma unroll
  for (int s = 0; s < JB; ++s) {
    if (ws.has(s)) {
      float m[VEC];
      LR::unpack(rw[s], m);
#pragma unroll
      for (int c = 0; c < VEC; ++c) a[c] = __fmaf_rn(ww[s], __fmul_rn(alpha, m[c]), a[c]);
    }
  }
  float p[VEC], d[VEC];
  pair_tree<VEC>(a, p, xch_p, wsel, bar);
#pragma unroll
  for (int c = 0; c < VEC; ++c) d[c] = __fmul_rn(beta, __fsub_rn(v[c], p[c]));
#pragma unroll
  for (int s = 0; s < JB; ++s) {
    if (ws.has(s)) {
      float m[VEC];
      LR::unpack(rw[s], m);
#pragma unroll
      for (int c = 0; c < VEC; ++c) m[c] = __fmaf_rn(ww[s], d[c], __fmul_rn(alpha, m[c]));
      LR::store(rows + ow[s], m);
    }
  }
  if (overlap) {
    named_barrier(bar, 64);
    pair_read<BANK, VEC, JB>(rs, rm + W, wt + W, rows, RB, b);
  }
  pair_tree<VEC>(b, y, xch_y, wsel, bar);
}

}  // namespace sdm
