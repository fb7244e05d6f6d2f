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
//   * piece_token (the write/read kernel, rows in shared memory), below.
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
// Token step of the write/read kernel: one warp per 32-byte piece of every row.
//
// Columns are independent, so each compute warp of the write/read kernel owns a 32-byte
// piece of every row of its CTA's column slice and runs the tokens on it alone: no two
// compute warps ever wait for each other.  Lane = 2*rg + c: c picks the 16-byte half of
// the piece (VEC = 16 / sizeof(BANK) columns), rg (0..15) a block of rows.
//
// Summation order.  The n rows of a sum (n = W for the prediction p, n = R for the read
// y) are cut into 16 consecutive blocks of B16 = ceil(n / 16) rows; lane rg sums block
// rg in increasing j, and an xor butterfly over the rg bits (lane xor 2, 4, 8, 16)
// combines the block sums as a balanced binary tree in block order,
//   (((s0+s1)+(s2+s3))+((s4+s5)+(s6+s7))) + (((s8+s9)+(s10+s11))+((s12+s13)+(s14+s15))),
// which leaves the same bits in every lane (IEEE addition is commutative).  The order
// depends on n alone: not on the stage length, the column slice or the warp.
//
// Shared-memory addresses.  rm holds, per reference, the row's offset o in the stage
// buffer (sdm_internal.h, PlanLayout); this lane's 16 bytes of that row sit at
// o ^ wc, wc = (warp << 5) | (c << 4).  The planner gives the rows of blocks 4q..4q+3
// four different colors (bits 5-6 of o), so the eight lanes of a quarter-warp, which
// read block rows 4q..4q+3 at once, hit eight different 16-byte bank groups.

template <typename BANK>
struct PieceRow {
  static constexpr int VEC = 16 / (int)sizeof(BANK);
  __device__ __forceinline__ static void unpack(const uint4 &r, float (&out)[VEC]) {
    const BANK *e = reinterpret_cast<const BANK *>(&r);
#pragma unroll
    for (int i = 0; i < VEC; ++i) out[i] = to_f32(e[i]);
  }
  __device__ __forceinline__ static uint4 pack(const float (&in)[VEC]) {
    uint4 r;
    BANK *e = reinterpret_cast<BANK *>(&r);
#pragma unroll
    for (int i = 0; i < VEC; ++i) e[i] = from_f32<BANK>(in[i]);
    return r;
  }
};

// The butterfly over the 16 row blocks (lane bits 1-4).
template <int VEC>
__device__ __forceinline__ void block_tree(float (&x)[VEC]) {
#pragma unroll
  for (int o = 2; o < 32; o <<= 1)
#pragma unroll
    for (int c = 0; c < VEC; ++c) x[c] = __fadd_rn(x[c], __shfl_xor_sync(0xffffffffu, x[c], o));
}

// Offsets and weights of this lane's rows of one sum (block rg of n references rm / wt).
// FULL: n == 64 (B16 = 4, read as 8- and 16-byte vectors).  Rows past the block or past
// n get offset 0 and weight 0 and are never touched (has(s) is false for them).
template <int JB, bool FULL>
struct BlockRows {
  int off[JB];
  float w[JB];
  int j0;                                         // first row of this block
  int nb;                                         // rows of this block
  __device__ __forceinline__ BlockRows(int n, int rg, const uint16_t *rm, const float *wt, uint32_t wc) {
    if constexpr (FULL) {
      static_assert(JB == 4, "FULL blocks hold 4 rows");
      const uint2 o4 = *reinterpret_cast<const uint2 *>(rm + 4 * rg);
      const uint32_t wc2 = wc | (wc << 16);
      const uint32_t x = o4.x ^ wc2, y = o4.y ^ wc2;
      off[0] = (int)(x & 0xffffu);
      off[1] = (int)(x >> 16);
      off[2] = (int)(y & 0xffffu);
      off[3] = (int)(y >> 16);
      const float4 w4 = *reinterpret_cast<const float4 *>(wt + 4 * rg);
      w[0] = w4.x;
      w[1] = w4.y;
      w[2] = w4.z;
      w[3] = w4.w;
      j0 = 4 * rg;
      nb = 4;
    } else {
      const int b16 = (n + 15) >> 4;
      j0 = rg * b16;
      nb = min(b16, max(n - j0, 0));
#pragma unroll
      for (int s = 0; s < JB; ++s) {
        const bool h = s < nb;
        off[s] = h ? (int)((uint32_t)rm[j0 + s] ^ wc) : 0;
        w[s] = h ? wt[j0 + s] : 0.0f;
      }
    }
  }
  __device__ __forceinline__ bool has(int s) const { return FULL ? true : s < nb; }
};

// One token on this warp's pieces of the stage buffer `rows`: the gated delta-rule write
// of its W rows, then the read of its R rows (after the write: the token's own update is
// visible).  rm / wt: the token's W write then R read references (offsets o, weights).
// When the token reads none of the rows it writes (overlap == false) the read rows are
// fetched before the write: those rows hold the same values before and after it.  y is
// left in every lane.  snap(j, raw) receives this lane's 16 bytes of write row j before
// the write (the backward's snapshot).  The caller orders tokens with __syncwarp().
template <typename BANK, int JB, bool FULL, class Snap>
__device__ __forceinline__ void piece_token(int W, int R, const uint16_t *rm, const float *wt, float alpha,
                                            float beta, const float (&v)[PieceRow<BANK>::VEC], unsigned char *rows,
                                            uint32_t wc, bool overlap, float (&y)[PieceRow<BANK>::VEC], Snap &&snap) {
  using PR = PieceRow<BANK>;
  constexpr int VEC = PR::VEC;
  if constexpr (FULL) W = R = 64;
  const int rg = (threadIdx.x & 31) >> 1;
  const BlockRows<JB, FULL> wr_(W, rg, rm, wt, wc);
  uint4 rw[JB];
#pragma unroll
  for (int s = 0; s < JB; ++s)
    if (wr_.has(s)) rw[s] = *reinterpret_cast<const uint4 *>(rows + wr_.off[s]);
  const BlockRows<JB, FULL> rd(R, rg, rm + W, wt + W, wc);
  uint4 rr[JB];
  if (!overlap) {
#pragma unroll
    for (int s = 0; s < JB; ++s)
      if (rd.has(s)) rr[s] = *reinterpret_cast<const uint4 *>(rows + rd.off[s]);
  }
#pragma unroll
  for (int s = 0; s < JB; ++s)
    if (wr_.has(s)) snap(wr_.j0 + s, rw[s]);
  // p = sum_j w_j (alpha m_j)
  float am[JB][VEC];
  float a[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) a[c] = 0.0f;
#pragma unroll
  for (int s = 0; s < JB; ++s) {
    if (wr_.has(s)) {
      float m[VEC];
      PR::unpack(rw[s], m);
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        am[s][c] = __fmul_rn(alpha, m[c]);
        a[c] = __fmaf_rn(wr_.w[s], am[s][c], a[c]);
      }
    }
  }
  block_tree<VEC>(a);
  // m_j <- alpha m_j + w_j beta (v - p)
  float d[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) d[c] = __fmul_rn(beta, __fsub_rn(v[c], a[c]));
#pragma unroll
  for (int s = 0; s < JB; ++s) {
    if (wr_.has(s)) {
      float m[VEC];
#pragma unroll
      for (int c = 0; c < VEC; ++c) m[c] = __fmaf_rn(wr_.w[s], d[c], am[s][c]);
      *reinterpret_cast<uint4 *>(rows + wr_.off[s]) = PR::pack(m);
    }
  }
  if (overlap) {
    __syncwarp();
#pragma unroll
    for (int s = 0; s < JB; ++s)
      if (rd.has(s)) rr[s] = *reinterpret_cast<const uint4 *>(rows + rd.off[s]);
  }
  // y = sum_j r_j m_j
#pragma unroll
  for (int c = 0; c < VEC; ++c) y[c] = 0.0f;
#pragma unroll
  for (int s = 0; s < JB; ++s) {
    if (rd.has(s)) {
      float m[VEC];
      PR::unpack(rr[s], m);
#pragma unroll
      for (int c = 0; c < VEC; ++c) y[c] = __fmaf_rn(rd.w[s], m[c], y[c]);
    }
  }
  block_tree<VEC>(y);
}

}  // namespace sdm
