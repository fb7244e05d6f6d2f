// Single-token decode step: scoring, exact top-k, gated delta-rule write and read for
// every stream in one launch (one CTA per stream), copying or in place.
//
// lumen PR #29 ("a state holds only itself, and a step can give it up") observes that
// returning a fresh table per stream costs O(B*N*d_v) per step against O(B*(W+R)*d_v)
// of arithmetic, and lets a caller that will not read the old state donate it so that
// the successor is written into the same buffers; both forms run one body and agree
// bit for bit.  Here the donated form touches only the W written rows; the copying
// form runs the same arithmetic with bank_out as the destination and also copies
// every unwritten row (each row is read once and written once).
#pragma once

#include "sdm_common.cuh"
#include "sdm_delta.cuh"
#include "sdm_internal.h"
#include "sdm_topk.cuh"

namespace sdm {
namespace dec {

constexpr int kDecodeNCG = 8;  // 16-byte column groups per warp

template <int EF, int EC, typename ACT, typename BANK>
__global__ void __launch_bounds__(kThreads)
    decode_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CandidateList cl) {
  constexpr int VEC = Vec16<BANK>::N;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ __align__(16) RowScratch rs[2];
  __shared__ int32_t sel_idx[2][SDM_MAX_K];
  __shared__ float sel_wt[2][SDM_MAX_K];
  __shared__ int32_t wsorted[SDM_MAX_K];
  __shared__ uint8_t read_written[SDM_MAX_K];
  __shared__ __align__(16) uint4 dummy_src, dummy_dst;

  const KeyGeometry &g = a.g;
  const int64_t s = blockIdx.x;
  const int64_t b = s / a.H, h = s % a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qdim = g.F * g.d_sub;
  const int W = g.k[0], R = g.k[1];

  float *qf = reinterpret_cast<float *>(smem);                 // [2][qdim]
  float *scores = qf + 2 * qdim;                                // [2][ntot]
  uint32_t *cand = reinterpret_cast<uint32_t *>(scores + 2 * g.ntot);

  const ACT *q0 = static_cast<const ACT *>(a.q[0]) + s * qdim;
  const ACT *q1 = static_cast<const ACT *>(a.q[1]) + s * qdim;
  for (int i = tid; i < qdim; i += kThreads) {
    qf[i] = to_f32(q0[i]);
    qf[qdim + i] = to_f32(q1[i]);
  }
  for (int i = tid; i < cl.n[0]; i += kThreads) cand[i] = cl.tup[0][i];
  for (int i = tid; i < cl.n[1]; i += kThreads) cand[cl.n[0] + i] = cl.tup[1][i];
  if (tid == 0) {
    dummy_src = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();

  // factor scores of both queries
  const ACT *K = static_cast<const ACT *>(a.subkeys) + h * (int64_t)g.ntot * g.d_sub;
  for (int o = tid; o < 2 * g.ntot; o += kThreads) {
    const int qsel = o / g.ntot, arow = o % g.ntot;
    int f = 0;
    while (f + 1 < g.F && arow >= g.off[f + 1]) ++f;
    scores[o] = score_dot<ACT>(qf + qsel * qdim + f * g.d_sub, K + (int64_t)arow * g.d_sub, g.d_sub);
  }
  __syncthreads();

  // exact top-k: warp 0 the write query, warp 1 the read query
  if (warp < 2) {
    row_topk<EF, EC>(scores + warp * g.ntot, g, warp, cand + (warp ? cl.n[0] : 0), cl.n[warp], rs[warp],
                     sel_idx[warp], sel_wt[warp]);
    const int k = g.k[warp];
    for (int j = lane; j < k; j += 32) {
      if (sel_idx[warp][j] < 0 || sel_idx[warp][j] >= a.N) {
        raise_error(a.err, SDM_DEVERR_SLOT_RANGE);
        sel_idx[warp][j] = 0;
      }
      if (a.idx[warp]) a.idx[warp][s * k + j] = sel_idx[warp][j];
      if (a.wt[warp]) a.wt[warp][s * k + j] = sel_wt[warp][j];
    }
  }
  __syncthreads();
  // written slots in ascending order (distinct, so the rank is a position)
  for (int j = tid; j < W; j += kThreads) {
    const int32_t x = sel_idx[0][j];
    int rank = 0;
    for (int i = 0; i < W; ++i) rank += sel_idx[0][i] < x;
    wsorted[rank] = x;
  }
  __syncthreads();
  auto is_written = [&](int64_t slot) -> bool {
    int lo = 0, hi = W;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (wsorted[mid] < slot) lo = mid + 1; else hi = mid;
    }
    return lo < W && wsorted[lo] == slot;
  };
  for (int j = tid; j < R; j += kThreads) read_written[j] = is_written(sel_idx[1][j]) ? 1 : 0;
  __syncthreads();

  // write and read, column blocks of kDecodeNCG 16-byte groups per warp
  const BANK *bin = static_cast<const BANK *>(a.bank_in) +
                    (a.bank_in_shared ? h : s) * a.N * a.d_v;
  BANK *bout = static_cast<BANK *>(a.bank_out) + s * a.N * a.d_v;
  const float alpha = a.gates[2 * s], beta = a.gates[2 * s + 1];
  const ACT *kv = static_cast<const ACT *>(a.k_val) + s * a.d_v;
  ACT *yo = static_cast<ACT *>(a.y) + s * a.d_v;
  const int64_t block_cols = (int64_t)kDecodeNCG * VEC;
  const int cg = lane % kDecodeNCG;
  for (int64_t cb = warp; cb * block_cols < a.d_v; cb += kThreads / 32) {
    const int64_t col = cb * block_cols + cg * VEC;
    const bool valid = col < a.d_v;
    auto wsrc = [&](int j) -> const BANK * {
      return valid ? bin + (int64_t)sel_idx[0][j] * a.d_v + col : reinterpret_cast<const BANK *>(&dummy_src);
    };
    auto wdst = [&](int j) -> BANK * {
      return valid ? bout + (int64_t)sel_idx[0][j] * a.d_v + col : reinterpret_cast<BANK *>(&dummy_dst);
    };
    auto rsrc = [&](int j) -> const BANK * {
      if (!valid) return reinterpret_cast<const BANK *>(&dummy_src);
      const int64_t slot = sel_idx[1][j];
      return (read_written[j] ? static_cast<const BANK *>(bout) : bin) + slot * a.d_v + col;
    };
    float v[VEC];
    if (valid) {
      load_vec<ACT, VEC>(kv + col, v);
    } else {
#pragma unroll
      for (int c = 0; c < VEC; ++c) v[c] = 0.0f;
    }
    delta_write_cols<BANK, kDecodeNCG>(W, sel_wt[0], alpha, beta, v, wsrc, wdst);
    __syncwarp();
    float out[VEC];
    weighted_read_cols<BANK, kDecodeNCG>(R, sel_wt[1], rsrc, out);
    if (valid && lane < kDecodeNCG) store_vec<ACT, VEC>(yo + col, out);
    __syncwarp();
  }

  // copying form: every unwritten row of bank_in -> bank_out
  if (a.copy_rest) {
    const int64_t row_chunks = a.d_v * (int64_t)sizeof(BANK) / 16;
    for (int64_t n = warp; n < a.N; n += kThreads / 32) {
      if (is_written(n)) continue;
      const uint4 *src = reinterpret_cast<const uint4 *>(bin + n * a.d_v);
      uint4 *dst = reinterpret_cast<uint4 *>(bout + n * a.d_v);
      for (int64_t c = lane; c < row_chunks; c += 32) dst[c] = src[c];
    }
  }
}

// Launches decode_kernel for one (ACT, BANK) pair and the sort widths (EF, EC).
template <typename ACT, typename BANK>
cudaError_t launch_decode_dt(const DecodeArgs &a, const CandidateList &cl, int EF, int EC, int64_t smem,
                             cudaStream_t st) {
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(a.B * a.H), kThreads, smem, st>>>(a, cl);
    return cudaGetLastError();
  };
  if (EF == 2 && EC == 2) return go(decode_kernel<2, 2, ACT, BANK>);
  if (EF == 4 && EC == 4) return go(decode_kernel<4, 4, ACT, BANK>);
  return cudaErrorInvalidValue;
}

// One translation unit per (ACT, BANK) pair instantiates it (sdm_decode_<act>_<bank>.cu).
cudaError_t launch_decode_f32_f32(const DecodeArgs &, const CandidateList &, int, int, int64_t, cudaStream_t);
cudaError_t launch_decode_f32_bf16(const DecodeArgs &, const CandidateList &, int, int, int64_t, cudaStream_t);
cudaError_t launch_decode_bf16_f32(const DecodeArgs &, const CandidateList &, int, int, int64_t, cudaStream_t);
cudaError_t launch_decode_bf16_bf16(const DecodeArgs &, const CandidateList &, int, int, int64_t, cudaStream_t);

}  // namespace dec
}  // namespace sdm
