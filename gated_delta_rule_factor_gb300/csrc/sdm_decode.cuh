// Single-token decode step: scoring, exact top-k, gated delta-rule write and read for
// every stream in one launch (one CTA per stream), copying or in place.
//
// The lumen decode notes (PR #29) point out that handing back a fresh table per stream
// costs O(B*N*d_v) per step while the arithmetic is O(B*(W+R)*d_v), and let a caller
// that no longer needs the old state donate it, so that the successor is written into
// the same buffers; both forms run one body and agree bit for bit.  Here the donated
// form touches only the W written rows.  The copying form streams the whole table into
// bank_out with bulk copies while the other warps score and select, then runs the same
// write with bank_out as the destination (the written rows are copied, then replaced).
#pragma once

#include "sdm_common.cuh"
#include "sdm_delta.cuh"
#include "sdm_internal.h"
#include "sdm_topk.cuh"

namespace sdm {
namespace dec {

constexpr int kDecodeWarps = kThreads / 32;
constexpr int kSelectWarp = 4;                 // warps 4..7 select (two per query)
constexpr int kBarSelect = 1;                  // named barrier of the selecting warps
constexpr int kCopyWarp = 2;                   // streams the copy meanwhile
constexpr int kScoreRows = kDecodeScoreRows;   // sub-key rows per scoring tile (two queries each)
constexpr int kScoreCols = kDecodeScoreCols;   // sub-key columns per scoring tile
static_assert(kScoreCols == kBf16Block, "a scoring tile is one block of the bfloat16 dot product");
static_assert(2 * kScoreRows == kThreads, "one thread per (query, tile row)");
constexpr int kCopyStages = 3;
constexpr uint32_t kCopyChunk = (uint32_t)(kDecodeCopyRingBytes / kCopyStages);  // bytes per copy stage

// Streams `bytes` (a multiple of 16, both ends 16-byte aligned) from src to dst through
// kCopyStages shared-memory stages with bulk copies; one thread.  Every copy has landed
// and every write is performed when it returns; false if a wait gave up.
__device__ __forceinline__ bool copy_table(unsigned char *ring, uint64_t *bar, const unsigned char *src,
                                           unsigned char *dst, int64_t bytes) {
  const int64_t n = (bytes + kCopyChunk - 1) / kCopyChunk;
  auto size = [&](int64_t i) -> uint32_t { return (uint32_t)min((int64_t)kCopyChunk, bytes - i * kCopyChunk); };
  auto issue = [&](int64_t i) {
    const int st = (int)(i % kCopyStages);
    mbar_expect_tx(&bar[st], size(i));
    bulk_load(ring + st * kCopyChunk, src + i * kCopyChunk, size(i), &bar[st]);
  };
  fence_proxy_async_shared();  // the ring held the scoring tile (generic accesses)
  int64_t issued = 0, landed = 0;
  for (; issued < n && issued < kCopyStages; ++issued) issue(issued);
  bool ok = true;
  for (int64_t i = 0; i < n; ++i) {
    const int st = (int)(i % kCopyStages);
    if (!mbar_wait(&bar[st], (uint32_t)(i / kCopyStages) & 1u)) {
      ok = false;
      break;
    }
    landed = i + 1;
    fence_proxy_async_shared();
    bulk_store(dst + i * kCopyChunk, ring + st * kCopyChunk, size(i));
    bulk_commit();
    if (i >= 1 && issued < n) {  // the stage of chunk i - 1 takes chunk i - 1 + kCopyStages
      bulk_wait_read_pending<1>();
      issue(issued++);
    }
  }
  for (int64_t i = landed; i < issued; ++i)  // after a failed wait: loads still in flight
    mbar_wait(&bar[i % kCopyStages], (uint32_t)(i / kCopyStages) & 1u);
  bulk_wait_all();
  fence_proxy_async_global();  // generic stores to bank_out (the write) come after the copy
  fence_proxy_async_shared();  // and generic accesses to the ring (the row stage)
  return ok;
}

// One CTA per stream: all warps score, warps kSelectWarp .. kSelectWarp + 3 select
// (in the copying form warp kCopyWarp copies the whole table bank_in -> bank_out
// meanwhile), all warps write and read.  The selection stays off warp 0: measured on
// GB300, the same selection code ran about six times slower on warp 0 than on any
// other warp of this kernel.
template <int EF, int EC, typename ACT, typename BANK>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CandidateList cl) {
  constexpr int VEC = Vec16<BANK>::N;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ __align__(16) RowScratch rs[2];
  __shared__ int32_t sel_idx[2][SDM_MAX_K];
  __shared__ float sel_wt[2][SDM_MAX_K];
  __shared__ int32_t wsorted[SDM_MAX_K];
  __shared__ uint8_t read_written[SDM_MAX_K];
  __shared__ __align__(8) uint64_t copy_bar[kCopyStages];
  __shared__ uint64_t part_keys[2][32 * EC];  // part 1's best candidate keys per query

  const KeyGeometry &g = a.g;
  const int64_t s = blockIdx.x;
  const int64_t h = s % a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qdim = g.F * g.d_sub;
  const int W = g.k[0], R = g.k[1];
  // this stream's tables (computed where they are used, to keep them out of the
  // selection's registers)
  auto table_in = [&]() { return static_cast<const BANK *>(a.bank_in) + (a.bank_in_shared ? h : s) * a.N * a.d_v; };
  auto table_out = [&]() { return static_cast<BANK *>(a.bank_out) + s * a.N * a.d_v; };

  // region: the scoring tile, then the copy ring (copying form), then the row stage
  float(*ktile)[kScoreCols + 1] = reinterpret_cast<float(*)[kScoreCols + 1]>(smem);
  unsigned char *ring = smem;
  // the read query starts one float after the write query's end: the two rows are read
  // together by neighbouring lanes, and this puts their words in different banks
  const int qpitch = qdim + 1;
  float *qf = reinterpret_cast<float *>(smem + a.region_bytes);  // [2][qpitch]
  float *scores = qf + 2 * qpitch;                              // [2][ntot]
  uint32_t *cand = reinterpret_cast<uint32_t *>(scores + 2 * g.ntot);

  const ACT *q0 = static_cast<const ACT *>(a.q[0]) + s * qdim;
  const ACT *q1 = static_cast<const ACT *>(a.q[1]) + s * qdim;
  for (int i = tid; i < qdim; i += kThreads) {
    qf[i] = to_f32(q0[i]);
    qf[qpitch + i] = to_f32(q1[i]);
  }
  for (int i = tid; i < cl.n[0]; i += kThreads) cand[i] = cl.tup[0][i];
  for (int i = tid; i < cl.n[1]; i += kThreads) cand[cl.n[0] + i] = cl.tup[1][i];
  if (a.copy_rest && tid == kCopyWarp * 32) {
    for (int i = 0; i < kCopyStages; ++i) mbar_init(&copy_bar[i], 1);
    mbar_init_fence();
  }
  __syncthreads();

  // factor scores of both queries: the sub-keys pass through shared memory in tiles of
  // kScoreRows rows x kScoreCols columns (coalesced loads, the next tile in flight while
  // this one is used); each thread folds each tile into its sum in block order.
  const ACT *K = static_cast<const ACT *>(a.subkeys) + h * (int64_t)g.ntot * g.d_sub;
  constexpr int kPer = kScoreRows * kScoreCols / kThreads;  // tile elements per thread
  for (int r0 = 0; r0 < g.ntot; r0 += kScoreRows) {
    const int nr = min(kScoreRows, g.ntot - r0);
    // thread t: row t / 2 of query t % 2, so that the rows in use (at most rows_t per
    // query) fill the low warps, one per SM sub-partition, instead of two per query
    const int row = tid >> 1, qsel = tid & 1, arow = r0 + row;
    int f = 0;
    while (f + 1 < g.F && arow >= g.off[f + 1]) ++f;
    const float *qrow = qf + qsel * qpitch + f * g.d_sub;
    float pre[kPer];
    auto fetch = [&](int d0) {
      const int nc = min(kScoreCols, g.d_sub - d0);
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = tid + k * kThreads, rr = i / kScoreCols, cc = i % kScoreCols;
        pre[k] = (rr < nr && cc < nc) ? to_f32(K[(int64_t)(r0 + rr) * g.d_sub + d0 + cc]) : 0.0f;
      }
    };
    fetch(0);
    Acc2 acc{0.0f, 0.0f};
    for (int d0 = 0; d0 < g.d_sub; d0 += kScoreCols) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = tid + k * kThreads;
        ktile[i / kScoreCols][i % kScoreCols] = pre[k];
      }
      __syncthreads();
      if (d0 + kScoreCols < g.d_sub) fetch(d0 + kScoreCols);
      if (row < nr) score_block<sizeof(ACT) == 2>(acc, qrow + d0, &ktile[row][0], min(kScoreCols, g.d_sub - d0));
      __syncthreads();
    }
    if (row < nr) scores[qsel * g.ntot + arow] = acc2_value(acc);
  }
  __syncthreads();

  // exact top-k on warps kSelectWarp .. kSelectWarp + 3: warp (q, part) = (w / 2, w % 2)
  // with w = warp - kSelectWarp sorts the factors part, part + 2, ... of query q, then
  // keeps the best of its part of q's candidate tuples; part 0 merges part 1's list
  // into its own (exact: the keys are unique) and computes the weights.  The result is
  // the one row_topk gives on one warp.
  if (warp >= kSelectWarp && warp < kSelectWarp + 4) {
    int w = warp - kSelectWarp;
    asm volatile("" : "+r"(w));  // one body for every selecting warp, not one per warp
    const int q = w >> 1, part = w & 1;
    for (int f = part; f < g.F; f += 2) factor_topk<EF>(scores + q * g.ntot, g, q, f, rs[q]);
    named_barrier(kBarSelect, 4 * 32);
    const int n = cl.n[q];
    const int mid = min(n, (n / 2 + 32 * EC - 1) / (32 * EC) * (32 * EC));  // whole chunks first
    uint64_t ck[EC];
    candidate_topk<EC>(cand + (q ? cl.n[0] : 0), part ? mid : 0, part ? n : mid, g, rs[q], ck);
    if (part == 1) {
#pragma unroll
      for (int e = 0; e < EC; ++e) part_keys[q][lane * EC + e] = ck[e];
    }
    named_barrier(kBarSelect, 4 * 32);
    if (part == 0) {
      uint64_t other[EC];
#pragma unroll
      for (int e = 0; e < EC; ++e) other[e] = part_keys[q][lane * EC + e];
      warp_merge_top_desc<EC>(ck, other);
      finish_topk<EC>(ck, g, q, rs[q], sel_idx[q], sel_wt[q]);
      const int k = g.k[q];
      for (int j = lane; j < k; j += 32) {
        if (sel_idx[q][j] < 0 || sel_idx[q][j] >= a.N) {
          raise_error(a.err, SDM_DEVERR_SLOT_RANGE);
          sel_idx[q][j] = 0;
        }
        if (a.idx[q]) a.idx[q][s * k + j] = sel_idx[q][j];
        if (a.wt[q]) a.wt[q][s * k + j] = sel_wt[q][j];
      }
    }
  } else if (warp == kCopyWarp && a.copy_rest) {
    // bank_out <- bank_in, all rows: the write below then replaces the written ones.
    // test_stall_copy: wait instead on stage 0's barrier, which nothing arrives at, so
    // that the bounded wait gives up (no copy issued, nothing left in flight).
    if (lane == 0) {
      const bool ok = a.test_stall_copy
                          ? mbar_wait(&copy_bar[0], 0)
                          : copy_table(ring, copy_bar, reinterpret_cast<const unsigned char *>(table_in()),
                                       reinterpret_cast<unsigned char *>(table_out()),
                                       a.N * a.d_v * (int64_t)sizeof(BANK));
      if (!ok) raise_error(a.err, SDM_DEVERR_TIMEOUT);
    }
    __syncwarp();
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

  // write and read, column blocks of kDecodeNCG 16-byte groups per warp, rows staged in
  // this warp's part of the region
  const BANK *bin = table_in();
  BANK *bout = table_out();
  unsigned char *stage = smem + (int64_t)warp * (W > R ? W : R) * kDecodeRowSlice;
  const float alpha = a.gates[2 * s], beta = a.gates[2 * s + 1];
  const ACT *kv = static_cast<const ACT *>(a.k_val) + s * a.d_v;
  ACT *yo = static_cast<ACT *>(a.y) + s * a.d_v;
  const int64_t block_cols = (int64_t)kDecodeNCG * VEC;
  const int cg = lane % kDecodeNCG;
  for (int64_t cb = warp; cb * block_cols < a.d_v; cb += kDecodeWarps) {
    const int64_t col = cb * block_cols + cg * VEC;
    const bool valid = col < a.d_v;
    auto wsrc = [&](int j) -> const BANK * { return bin + (int64_t)sel_idx[0][j] * a.d_v + col; };
    auto wdst = [&](int j) -> BANK * { return bout + (int64_t)sel_idx[0][j] * a.d_v + col; };
    auto rsrc = [&](int j) -> const BANK * {
      return (read_written[j] ? static_cast<const BANK *>(bout) : bin) + (int64_t)sel_idx[1][j] * a.d_v + col;
    };
    float v[VEC];
    if (valid) {
      load_vec<ACT, VEC>(kv + col, v);
    } else {
#pragma unroll
      for (int c = 0; c < VEC; ++c) v[c] = 0.0f;
    }
    delta_write_staged<BANK, kDecodeNCG>(W, sel_wt[0], alpha, beta, v, valid, stage, wsrc, wdst);
    __syncwarp();  // the written rows are in bank_out before any lane reads them back
    float out[VEC];
    weighted_read_staged<BANK, kDecodeNCG>(R, sel_wt[1], valid, stage, rsrc, out);
    if (valid && lane < kDecodeNCG) store_vec<ACT, VEC>(yo + col, out);
    __syncwarp();
  }
}

// Launches one decode_kernel instance.
template <int EF, int EC, typename ACT, typename BANK>
cudaError_t launch_decode_k(const DecodeArgs &a, const CandidateList &cl, int64_t smem, cudaStream_t st) {
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(decode_kernel<EF, EC, ACT, BANK>), smem);
  if (e != cudaSuccess) return e;
  decode_kernel<EF, EC, ACT, BANK><<<(unsigned)(a.B * a.H), kThreads, smem, st>>>(a, cl);
  return cudaGetLastError();
}

// Launches decode_kernel for one (ACT, BANK) pair and the sort widths (EF, EC).
template <typename ACT, typename BANK>
cudaError_t launch_decode_dt(const DecodeArgs &a, const CandidateList &cl, int EF, int EC, int64_t smem,
                             cudaStream_t st) {
  if (EF == 2 && EC == 2) return launch_decode_k<2, 2, ACT, BANK>(a, cl, smem, st);
  if (EF == 4 && EC == 4) return launch_decode_k<4, 4, ACT, BANK>(a, cl, smem, st);
  return cudaErrorInvalidValue;
}

// One translation unit per (ACT, BANK) pair instantiates it (sdm_decode_<act>_<bank>.cu).
cudaError_t launch_decode_f32_f32(const DecodeArgs &, const CandidateList &, int, int, int64_t, cudaStream_t);
cudaError_t launch_decode_f32_bf16(const DecodeArgs &, const CandidateList &, int, int, int64_t, cudaStream_t);
cudaError_t launch_decode_bf16_f32(const DecodeArgs &, const CandidateList &, int, int, int64_t, cudaStream_t);
cudaError_t launch_decode_bf16_bf16(const DecodeArgs &, const CandidateList &, int, int, int64_t, cudaStream_t);

}  // namespace dec
}  // namespace sdm
