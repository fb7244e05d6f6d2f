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

}  // namespace sdm
