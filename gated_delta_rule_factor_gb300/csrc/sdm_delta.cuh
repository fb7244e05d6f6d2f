// Per-token gated delta-rule write and weighted read over a column slice, by one warp
// (shared by the write/read kernel, which keeps rows in shared memory, and the decode
// kernel, which works on the bank in global memory, so both do identical arithmetic).
//
// For one token with forget gate alpha, input gate beta, value v and the W selected
// rows M[i_j] with weights w_j (a reading of the gated delta rule of Yang et al., cited
// in the sparse-delta-memory README, restricted to the selected rows):
//   m_j = alpha * M[i_j]
//   p   = sum_j w_j m_j
//   M[i_j] <- m_j + w_j * beta * (v - p)          (rounded to the bank type)
// and then the read over the R selected rows: y = sum_j r_j M[i^r_j].
// Every column is independent, so a warp owns NCG 16-byte column groups (lane % NCG)
// and splits the rows of the token over RG = 32 / NCG row groups (lane / NCG): row j
// belongs to row group j % RG and is accumulated in increasing j; the RG partial sums
// are combined by an xor butterfly.  All of it is float32 with fixed operation order,
// so results are bitwise repeatable and independent of how tokens are staged.
//
// Rows are fetched kJB at a time per lane (independent loads in flight) because the
// token chain is latency-bound: one warp walks the tokens of a stream in order.
#pragma once

#include "sdm_common.cuh"

namespace sdm {

constexpr int kJB = 8;  // rows in flight per lane

// 16-byte raw row chunk <-> float32 lanes.
template <typename BANK>
__device__ __forceinline__ void unpack16(const uint4 &u, float (&out)[Vec16<BANK>::N]) {
  const BANK *e = reinterpret_cast<const BANK *>(&u);
#pragma unroll
  for (int i = 0; i < Vec16<BANK>::N; ++i) out[i] = to_f32(e[i]);
}

template <typename BANK, int NCG, class SrcRow, class DstRow>
__device__ __forceinline__ void delta_write_cols(int W, const float *w, float alpha, float beta,
                                                 const float (&v)[Vec16<BANK>::N], SrcRow src,
                                                 DstRow dst) {
  constexpr int VEC = Vec16<BANK>::N, RG = 32 / NCG;
  const int rg = (threadIdx.x & 31) / NCG;
  float acc[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) acc[c] = 0.0f;
  for (int j0 = rg; j0 < W; j0 += RG * kJB) {
    uint4 raw[kJB];
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < W) raw[b] = *reinterpret_cast<const uint4 *>(src(j));
    }
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < W) {
        const float wj = w[j];
        float r[VEC];
        unpack16<BANK>(raw[b], r);
#pragma unroll
        for (int c = 0; c < VEC; ++c) acc[c] = __fmaf_rn(wj, __fmul_rn(alpha, r[c]), acc[c]);
      }
    }
  }
#pragma unroll
  for (int o = NCG; o < 32; o <<= 1)
#pragma unroll
    for (int c = 0; c < VEC; ++c) acc[c] = __fadd_rn(acc[c], __shfl_xor_sync(0xffffffffu, acc[c], o));
  float d[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) d[c] = __fmul_rn(beta, __fsub_rn(v[c], acc[c]));
  for (int j0 = rg; j0 < W; j0 += RG * kJB) {
    uint4 raw[kJB];
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < W) raw[b] = *reinterpret_cast<const uint4 *>(src(j));
    }
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < W) {
        const float wj = w[j];
        float r[VEC];
        unpack16<BANK>(raw[b], r);
#pragma unroll
        for (int c = 0; c < VEC; ++c) r[c] = __fmaf_rn(wj, d[c], __fmul_rn(alpha, r[c]));
        store_vec16<BANK>(dst(j), r);
      }
    }
  }
}

template <typename BANK, int NCG, class SrcRow>
__device__ __forceinline__ void weighted_read_cols(int R, const float *r, SrcRow src,
                                                   float (&y)[Vec16<BANK>::N]) {
  constexpr int VEC = Vec16<BANK>::N, RG = 32 / NCG;
  const int rg = (threadIdx.x & 31) / NCG;
#pragma unroll
  for (int c = 0; c < VEC; ++c) y[c] = 0.0f;
  for (int j0 = rg; j0 < R; j0 += RG * kJB) {
    uint4 raw[kJB];
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < R) raw[b] = *reinterpret_cast<const uint4 *>(src(j));
    }
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < R) {
        const float rj = r[j];
        float m[VEC];
        unpack16<BANK>(raw[b], m);
#pragma unroll
        for (int c = 0; c < VEC; ++c) y[c] = __fmaf_rn(rj, m[c], y[c]);
      }
    }
  }
#pragma unroll
  for (int o = NCG; o < 32; o <<= 1)
#pragma unroll
    for (int c = 0; c < VEC; ++c) y[c] = __fadd_rn(y[c], __shfl_xor_sync(0xffffffffu, y[c], o));
}

// The row references of one token that one lane handles: row group rg takes the refs
// j = rg + b*RG, b < kJB (valid while j < W, resp. j < R).
struct LaneRefs {
  int uw[kJB], ur[kJB];      // row byte offsets in the stage buffer
};

// One token, when each lane holds at most kJB write rows and kJB read rows (W, R <=
// RG*kJB).  Same arithmetic, in the same order, as delta_write_cols followed by
// weighted_read_cols.  When the token reads no row it writes (overlap == false) its
// read rows are fetched together with the write rows and both reductions run side by
// side: the rows it reads hold the same values before and after its write.
template <typename BANK, int NCG>
__device__ __forceinline__ void token_write_read(int W, int R, const LaneRefs &ref, const float *w,
                                                 float alpha, float beta, const float (&v)[Vec16<BANK>::N],
                                                 unsigned char *rows, bool overlap, float (&y)[Vec16<BANK>::N]) {
  constexpr int VEC = Vec16<BANK>::N, RG = 32 / NCG;
  const int rg = (threadIdx.x & 31) / NCG;
  uint4 rw[kJB], rr[kJB];
  struct {
    float ww[kJB], wr[kJB];
  } wt;
#pragma unroll
  for (int b = 0; b < kJB; ++b) {
    const int j = rg + b * RG;
    wt.ww[b] = j < W ? w[j] : 0.0f;
    wt.wr[b] = j < R ? w[W + j] : 0.0f;
  }
#pragma unroll
  for (int b = 0; b < kJB; ++b)
    if (rg + b * RG < W) rw[b] = *reinterpret_cast<const uint4 *>(rows + ref.uw[b]);
  if (!overlap) {
#pragma unroll
    for (int b = 0; b < kJB; ++b)
      if (rg + b * RG < R) rr[b] = *reinterpret_cast<const uint4 *>(rows + ref.ur[b]);
  }
  float acc[VEC], ya[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) acc[c] = ya[c] = 0.0f;
#pragma unroll
  for (int b = 0; b < kJB; ++b) {
    if (rg + b * RG < W) {
      float r[VEC];
      unpack16<BANK>(rw[b], r);
#pragma unroll
      for (int c = 0; c < VEC; ++c) acc[c] = __fmaf_rn(wt.ww[b], __fmul_rn(alpha, r[c]), acc[c]);
    }
  }
  if (!overlap) {
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      if (rg + b * RG < R) {
        float m[VEC];
        unpack16<BANK>(rr[b], m);
#pragma unroll
        for (int c = 0; c < VEC; ++c) ya[c] = __fmaf_rn(wt.wr[b], m[c], ya[c]);
      }
    }
#pragma unroll
    for (int o = NCG; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        acc[c] = __fadd_rn(acc[c], __shfl_xor_sync(0xffffffffu, acc[c], o));
        ya[c] = __fadd_rn(ya[c], __shfl_xor_sync(0xffffffffu, ya[c], o));
      }
  } else {
#pragma unroll
    for (int o = NCG; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < VEC; ++c) acc[c] = __fadd_rn(acc[c], __shfl_xor_sync(0xffffffffu, acc[c], o));
  }
  float d[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) d[c] = __fmul_rn(beta, __fsub_rn(v[c], acc[c]));
#pragma unroll
  for (int b = 0; b < kJB; ++b) {
    if (rg + b * RG < W) {
      float r[VEC];
      unpack16<BANK>(rw[b], r);
#pragma unroll
      for (int c = 0; c < VEC; ++c) r[c] = __fmaf_rn(wt.ww[b], d[c], __fmul_rn(alpha, r[c]));
      store_vec16<BANK>(reinterpret_cast<BANK *>(rows + ref.uw[b]), r);
    }
  }
  if (overlap) {
    __syncwarp();
#pragma unroll
    for (int b = 0; b < kJB; ++b)
      if (rg + b * RG < R) rr[b] = *reinterpret_cast<const uint4 *>(rows + ref.ur[b]);
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      if (rg + b * RG < R) {
        float m[VEC];
        unpack16<BANK>(rr[b], m);
#pragma unroll
        for (int c = 0; c < VEC; ++c) ya[c] = __fmaf_rn(wt.wr[b], m[c], ya[c]);
      }
    }
#pragma unroll
    for (int o = NCG; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < VEC; ++c) ya[c] = __fadd_rn(ya[c], __shfl_xor_sync(0xffffffffu, ya[c], o));
  }
#pragma unroll
  for (int c = 0; c < VEC; ++c) y[c] = ya[c];
}

// ------------------------------------------------------------------------------------
// Block-ordered token step of the write/read kernel on a 128-byte row slice (one warp).
//
// Summation order.  The n rows of a sum (n = W for the prediction p, n = R for the
// read y) are cut into 8 consecutive blocks of B8 = ceil(n / 8) rows; block k is summed
// in increasing j into a_k and the block sums are combined as
//   ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7)).
// The order depends on n alone: not on the stage length, nor on the column slicing.
//
// Lane layout.  Lane % 8 is a 16-byte column group of the slice (8 x 16 = 128 bytes)
// and lane / 8 = rg a row group that owns blocks 2rg and 2rg+1, so a lane adds its own
// pair and two xor steps (8 and 16 lanes apart) finish the tree; IEEE addition is
// commutative, so both partners of a step hold the same bits afterwards.
//
// JB = the most rows one lane holds, >= 2 * B8 for both sums.  Register slot s < JB/2
// holds row 2rg*B8 + s (block 2rg), slot JB/2 + s holds row 2rg*B8 + B8 + s (block
// 2rg+1); slots past the block or past n hold nothing.
template <int JB>
struct BlockSlots {
  static constexpr int H = JB / 2;
  int b8, j0, n;
  __device__ __forceinline__ BlockSlots(int n_, int rg) : b8((n_ + 7) >> 3), j0(2 * rg * ((n_ + 7) >> 3)), n(n_) {}
  __device__ __forceinline__ int ref(int s) const { return j0 + (s < H ? s : b8 + s - H); }
  __device__ __forceinline__ bool has(int s) const { return (s < H ? s : s - H) < b8 && ref(s) < n; }
};

template <int VEC>
__device__ __forceinline__ void block_tree(const float (&a0)[VEC], const float (&a1)[VEC], float (&out)[VEC]) {
#pragma unroll
  for (int c = 0; c < VEC; ++c) {
    float x = __fadd_rn(a0[c], a1[c]);
    x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, 8));
    out[c] = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, 16));
  }
}

// Accumulates the read rows of the token (slots of `rs`) into b0 / b1.
template <typename BANK, int JB>
__device__ __forceinline__ void block_read(const BlockSlots<JB> &rs, const uint16_t *rm_r, const float *wt_r,
                                           const unsigned char *rows, float (&b0)[Vec16<BANK>::N],
                                           float (&b1)[Vec16<BANK>::N]) {
  constexpr int VEC = Vec16<BANK>::N, H = JB / 2, RB = 128;
#pragma unroll
  for (int s0 = 0; s0 < JB; s0 += 4) {
    uint4 raw[4];
    float wr[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int s = s0 + q;
      if (rs.has(s)) {
        raw[q] = *reinterpret_cast<const uint4 *>(rows + (int)rm_r[rs.ref(s)] * RB);
        wr[q] = wt_r[rs.ref(s)];
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int s = s0 + q;
      if (rs.has(s)) {
        float m[VEC];
        unpack16<BANK>(raw[q], m);
        float(&b)[VEC] = s < H ? b0 : b1;
#pragma unroll
        for (int c = 0; c < VEC; ++c) b[c] = __fmaf_rn(wr[q], m[c], b[c]);
      }
    }
  }
}

// One token: the gated delta-rule write of its W rows, then the read of its R rows,
// with the arithmetic of delta_write_cols / weighted_read_cols per element and the
// block order above for both sums.  rm / wt: the token's row references (stage-buffer
// row indices) and weights, W write entries then R read entries; rows: the stage
// buffer offset by this lane's 16-byte column group.  When the token reads none of the
// rows it writes (overlap == false) the read runs before the write: those rows hold
// the same values before and after it.
// FULL: W == R == 4 * JB, every slot of every lane holds a row (no predicates).
template <typename BANK, int JB, bool FULL = false>
__device__ __forceinline__ void token_blocks(int W, int R, const uint16_t *rm, const float *wt, float alpha,
                                             float beta, const float (&v)[Vec16<BANK>::N], unsigned char *rows,
                                             bool overlap, float (&y)[Vec16<BANK>::N]) {
  constexpr int VEC = Vec16<BANK>::N, H = JB / 2, RB = 128;
  if constexpr (FULL) W = R = 4 * JB;
  const int rg = (threadIdx.x & 31) >> 3;
  const BlockSlots<JB> ws(W, rg), rs(R, rg);
  int ow[JB];
  float ww[JB];
  uint4 rw[JB];
#pragma unroll
  for (int s = 0; s < JB; ++s) {
    ow[s] = ws.has(s) ? (int)rm[ws.ref(s)] * RB : 0;
    ww[s] = ws.has(s) ? wt[ws.ref(s)] : 0.0f;
  }
#pragma unroll
  for (int s = 0; s < JB; ++s)
    if (ws.has(s)) rw[s] = *reinterpret_cast<const uint4 *>(rows + ow[s]);
  float b0[VEC], b1[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) b0[c] = b1[c] = 0.0f;
  if (!overlap) block_read<BANK, JB>(rs, rm + W, wt + W, rows, b0, b1);

  float a0[VEC], a1[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) a0[c] = a1[c] = 0.0f;
#pragma unroll
  for (int s = 0; s < JB; ++s) {
    if (ws.has(s)) {
      float m[VEC];
      unpack16<BANK>(rw[s], m);
      float(&a)[VEC] = s < H ? a0 : a1;
#pragma unroll
      for (int c = 0; c < VEC; ++c) a[c] = __fmaf_rn(ww[s], __fmul_rn(alpha, m[c]), a[c]);
    }
  }
  float p[VEC], d[VEC];
  block_tree<VEC>(a0, a1, p);
#pragma unroll
  for (int c = 0; c < VEC; ++c) d[c] = __fmul_rn(beta, __fsub_rn(v[c], p[c]));
#pragma unroll
  for (int s = 0; s < JB; ++s) {
    if (ws.has(s)) {
      float m[VEC];
      unpack16<BANK>(rw[s], m);
#pragma unroll
      for (int c = 0; c < VEC; ++c) m[c] = __fmaf_rn(ww[s], d[c], __fmul_rn(alpha, m[c]));
      store_vec16<BANK>(reinterpret_cast<BANK *>(rows + ow[s]), m);
    }
  }
  if (overlap) {
    __syncwarp();
    block_read<BANK, JB>(rs, rm + W, wt + W, rows, b0, b1);
  }
  block_tree<VEC>(b0, b1, y);
}

// ------------------------------------------------------------------------------------
// The same token step with the rows split between two warps (same summation order, so
// the results are bitwise those of token_blocks).  Warp wsel's row group rg owns block
// k = 4*wsel + rg alone: a lane adds its block, two xor steps inside the warp give
// (a0+a1)+(a2+a3) in warp 0 and (a4+a5)+(a6+a7) in warp 1, and the warps swap those
// through shared memory (xch: [2 warps][8 column groups][VEC] floats) on a 64-thread
// named barrier `bar`.  JB >= B8: register slot s holds row k*B8 + s.
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
#pragma unroll
    for (int c = 0; c < VEC; c += 4)
      *reinterpret_cast<float4 *>(mine + c) = make_float4(x[c], x[c + 1], x[c + 2], x[c + 3]);
  }
  named_barrier(bar, 64);
#pragma unroll
  for (int c = 0; c < VEC; c += 4) {
    const float4 o = *reinterpret_cast<const float4 *>(theirs + c);
    out[c] = __fadd_rn(x[c], o.x);
    out[c + 1] = __fadd_rn(x[c + 1], o.y);
    out[c + 2] = __fadd_rn(x[c + 2], o.z);
    out[c + 3] = __fadd_rn(x[c + 3], o.w);
  }
}

template <typename BANK, int JB>
__device__ __forceinline__ void pair_read(const BlockSlots1<JB> &rs, const uint16_t *rm_r, const float *wt_r,
                                          const unsigned char *rows, float (&b)[Vec16<BANK>::N]) {
  constexpr int VEC = Vec16<BANK>::N, RB = 128;
#pragma unroll
  for (int s0 = 0; s0 < JB; s0 += 4) {
    uint4 raw[4];
    float wr[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int s = s0 + q;
      if (rs.has(s)) {
        raw[q] = *reinterpret_cast<const uint4 *>(rows + (int)rm_r[rs.ref(s)] * RB);
        wr[q] = wt_r[rs.ref(s)];
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (rs.has(s0 + q)) {
        float m[VEC];
        unpack16<BANK>(raw[q], m);
#pragma unroll
        for (int c = 0; c < VEC; ++c) b[c] = __fmaf_rn(wr[q], m[c], b[c]);
      }
    }
  }
}

// FULL: W == R == 8 * JB.  The read's exchange barrier comes after the row stores, so it
// also orders this token's writes before the next token's loads in the other warp.
template <typename BANK, int JB, bool FULL = false>
__device__ __forceinline__ void token_blocks2(int W, int R, const uint16_t *rm, const float *wt, float alpha,
                                              float beta, const float (&v)[Vec16<BANK>::N], unsigned char *rows,
                                              bool overlap, float (&y)[Vec16<BANK>::N], float *xch_p, float *xch_y,
                                              int wsel, int bar) {
  constexpr int VEC = Vec16<BANK>::N, RB = 128;
  if constexpr (FULL) W = R = 8 * JB;
  const int k = 4 * wsel + ((threadIdx.x & 31) >> 3);
  const BlockSlots1<JB> ws(W, k), rs(R, k);
  int ow[JB];
  float ww[JB];
  uint4 rw[JB];
#pragma unroll
  for (int s = 0; s < JB; ++s) {
    ow[s] = ws.has(s) ? (int)rm[ws.ref(s)] * RB : 0;
    ww[s] = ws.has(s) ? wt[ws.ref(s)] : 0.0f;
  }
#pragma unroll
  for (int s = 0; s < JB; ++s)
    if (ws.has(s)) rw[s] = *reinterpret_cast<const uint4 *>(rows + ow[s]);
  float b[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) b[c] = 0.0f;
  if (!overlap) pair_read<BANK, JB>(rs, rm + W, wt + W, rows, b);

  float a[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) a[c] = 0.0f;
#pragma unroll
  for (int s = 0; s < JB; ++s) {
    if (ws.has(s)) {
      float m[VEC];
      unpack16<BANK>(rw[s], m);
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
      unpack16<BANK>(rw[s], m);
#pragma unroll
      for (int c = 0; c < VEC; ++c) m[c] = __fmaf_rn(ww[s], d[c], __fmul_rn(alpha, m[c]));
      store_vec16<BANK>(reinterpret_cast<BANK *>(rows + ow[s]), m);
    }
  }
  if (overlap) {
    named_barrier(bar, 64);
    pair_read<BANK, JB>(rs, rm + W, wt + W, rows, b);
  }
  pair_tree<VEC>(b, y, xch_y, wsel, bar);
}

}  // namespace sdm
