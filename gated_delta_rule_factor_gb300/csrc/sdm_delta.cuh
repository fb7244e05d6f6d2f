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
    float r[kJB][VEC];
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < W) load_vec16<BANK>(src(j), r[b]);
    }
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < W) {
        const float wj = w[j];
#pragma unroll
        for (int c = 0; c < VEC; ++c) acc[c] = __fmaf_rn(wj, __fmul_rn(alpha, r[b][c]), acc[c]);
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
    float r[kJB][VEC];
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < W) load_vec16<BANK>(src(j), r[b]);
    }
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < W) {
        const float wj = w[j];
#pragma unroll
        for (int c = 0; c < VEC; ++c) r[b][c] = __fmaf_rn(wj, d[c], __fmul_rn(alpha, r[b][c]));
        store_vec16<BANK>(dst(j), r[b]);
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
    float m[kJB][VEC];
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < R) load_vec16<BANK>(src(j), m[b]);
    }
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int j = j0 + b * RG;
      if (j < R) {
        const float rj = r[j];
#pragma unroll
        for (int c = 0; c < VEC; ++c) y[c] = __fmaf_rn(rj, m[b][c], y[c]);
      }
    }
  }
#pragma unroll
  for (int o = NCG; o < 32; o <<= 1)
#pragma unroll
    for (int c = 0; c < VEC; ++c) y[c] = __fadd_rn(y[c], __shfl_xor_sync(0xffffffffu, y[c], o));
}

}  // namespace sdm
