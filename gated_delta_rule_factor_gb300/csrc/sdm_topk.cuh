// Exact product-key top-k of one query row, by one warp (shared by the sequence
// top-k kernel and the decode kernel so that both select identically).
//
// Product-key memory (Lample et al., cited in the sparse-delta-memory README) scores
// each factor's sub-keys separately; the slot score is the float32 sum of the factor
// scores, and ties go to the larger rank sum, then the larger first rank
// (sparse-delta-memory CHANGELOG, 2.0.0 > Upgrading from v1).  A factor's rank is its
// ascending score rank, equal scores ordered by index, so "larger rank" means
// "earlier in the factor's best-first order".
//
// Exactness of the pruning: let each factor be sorted best first and describe a slot
// by its positions (p_1..p_F) in those orders.  Any tuple p' <= p position-wise scores
// at least as high (float addition is monotone in each operand) and, if the scores
// tie, has the larger rank sum.  The prod(p_f + 1) - 1 tuples below p therefore all
// beat p, so p can only be among the top k if prod(p_f + 1) <= k.  The surviving
// candidates are ranked with one 64-bit key:
//   bits 63..32  slot score (order-preserving bits)
//   bits 31..24  255 - sum_f p_f      (larger rank sum first)
//   bits 23..16  255 - p_1            (larger first rank first)
//   bits 15..8   255 - p_2, bits 7..0  255 - p_3   (then the next ranks)
// Distinct tuples get distinct keys (p_4 = sum - p_1 - p_2 - p_3), so the order is
// total and the selection unique.  Every p_f and sum_f p_f is <= k - 1 <= 255.
#pragma once

#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

// Per-warp scratch: best-first factor scores and indices, [F][SDM_MAX_K] each, and the
// keys of the candidates that pass the pruning bound.
constexpr int kSurvivorCap = 2 * SDM_MAX_K;
struct RowScratch {
  float fs[SDM_MAX_FACTORS * SDM_MAX_K];
  int32_t fi[SDM_MAX_FACTORS * SDM_MAX_K];
  uint64_t surv[kSurvivorCap];
};

// The 32*E best keys of a list of n keys, best first: chunks of 32*E keys (made by
// make(first index, keys)) are sorted two at a time and merged into the running best.
template <int E, class Make>
__device__ __forceinline__ void top_of_chunks(int n, Make make, uint64_t (&best)[E]) {
  constexpr int P = 32 * E;
  bool have = false;
  int c0 = 0;
  for (; c0 + P < n; c0 += 2 * P) {
    uint64_t ka[E], kb[E];
    make(c0, ka);
    make(c0 + P, kb);
    warp_sort_desc2<E>(ka, kb);
    if (!have) {
#pragma unroll
      for (int e = 0; e < E; ++e) best[e] = ka[e];
      have = true;
    } else {
      warp_merge_top_desc<E>(best, ka);
    }
    warp_merge_top_desc<E>(best, kb);
  }
  if (c0 < n) {
    uint64_t ka[E];
    make(c0, ka);
    warp_sort_desc<E>(ka);
    if (!have) {
#pragma unroll
      for (int e = 0; e < E; ++e) best[e] = ka[e];
    } else {
      warp_merge_top_desc<E>(best, ka);
    }
  }
}

// The phases of one row's selection, each run by one warp: factor_topk for every
// factor, then candidate_topk over the candidate tuples (or a part of them, whose best
// lists warp_merge_top_desc can merge, since the keys are unique), then finish_topk.

// Best-first order of factor f, kept to its first min(k, n_f) positions (sc.fs, sc.fi).
template <int EF>
__device__ __forceinline__ void factor_topk(const float *scores, const KeyGeometry &g, int qsel, int f,
                                            RowScratch &sc) {
  const int lane = threadIdx.x & 31;
  const int nf = g.nf[f];
  const float *s = scores + g.off[f];
  uint64_t best[EF];
  top_of_chunks<EF>(nf, [&](int c0, uint64_t(&key)[EF]) {
#pragma unroll
    for (int e = 0; e < EF; ++e) {
      const int a = c0 + lane * EF + e;
      key[e] = (a < nf) ? ((uint64_t)ordered_bits(s[a]) << 32) | (uint32_t)a : 0ull;
    }
  }, best);
  const int kf = g.kf[qsel][f];
#pragma unroll
  for (int e = 0; e < EF; ++e) {
    const int pos = lane * EF + e;
    if (pos < kf) {
      sc.fs[f * SDM_MAX_K + pos] = from_ordered_bits((uint32_t)(best[e] >> 32));
      sc.fi[f * SDM_MAX_K + pos] = (int32_t)(uint32_t)(best[e] & 0xffffffffu);
    }
  }
}

// The need-th largest of the warp's values (v[i] of lane l is value l + 32 i; those with ok
// false do not count), 1 <= need <= their number: a radix select over 8-bit digits, from
// the top, with exact integer counters in hist (256 ints of the warp's scratch).
template <int KPL>
__device__ __forceinline__ uint32_t warp_kth_largest(const uint32_t (&v)[KPL], const bool (&ok)[KPL], int need,
                                                     int *hist) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0, pmask = 0;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
#pragma unroll
    for (int j = 0; j < 8; ++j) hist[lane * 8 + j] = 0;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < KPL; ++i)
      if (ok[i] && (v[i] & pmask) == prefix) atomicAdd(&hist[(v[i] >> shift) & 255u], 1);
    __syncwarp();
    // bins from the top digit down: lane l holds digits 255 - 8l - j, j = 0..7
    int c[8], run = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = hist[255 - 8 * lane - j];
      run += c[j];
    }
    int before = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, before, o);
      if (lane >= o) before += x;
    }
    before -= run;                                    // values in higher digits (earlier lanes)
    int digit = -1, above = 0, acc = before;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (digit < 0 && acc + c[j] >= need) {
        digit = 255 - 8 * lane - j;
        above = acc;
      }
      acc += c[j];
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, digit >= 0)) - 1;   // the first digit reaching need
    digit = __shfl_sync(0xffffffffu, digit, src);
    above = __shfl_sync(0xffffffffu, above, src);
    prefix |= (uint32_t)digit << shift;
    pmask |= 255u << shift;
    need -= above;
    __syncwarp();
  }
  return prefix;
}

// factor_topk for a factor of 129 to 256 sub-keys and kf <= 64 (the sequence path's row
// selection, one warp per row with its own scratch): the score bits of the kf-th largest
// key are found first (warp_kth_largest, its counters in the row's survivor buffer, free
// until the candidate phase), and only the keys whose score bits reach them (every key of
// the top kf, plus any key tied with the kf-th on score) are sorted as before: the same
// kf keys in the same order.
__device__ __forceinline__ void factor_topk_radix(const float *scores, const KeyGeometry &g, int qsel, int f,
                                                  RowScratch &sc) {
  constexpr int KPL = 8;                              // keys per lane (n_f <= 256)
  const int lane = threadIdx.x & 31;
  const int nf = g.nf[f], kf = g.kf[qsel][f];
  const float *s = scores + g.off[f];
  uint32_t hi[KPL];
  bool ok[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int a = lane + 32 * i;
    ok[i] = a < nf;
    hi[i] = ok[i] ? ordered_bits(s[a]) : 0u;
  }
  const uint32_t T = warp_kth_largest<KPL>(hi, ok, kf, reinterpret_cast<int *>(sc.surv));
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const bool keep = ok[i] && hi[i] >= T;
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (keep) sc.surv[cnt + __popc(m & ((1u << lane) - 1u))] = ((uint64_t)hi[i] << 32) | (uint32_t)(lane + 32 * i);
    cnt += __popc(m);
  }
  __syncwarp();
  uint64_t best[2];
  top_of_chunks<2>(cnt, [&](int c0, uint64_t(&key)[2]) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = c0 + lane * 2 + e;
      key[e] = i < cnt ? sc.surv[i] : 0ull;
    }
  }, best);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int pos = lane * 2 + e;
    if (pos < kf) {
      sc.fs[f * SDM_MAX_K + pos] = from_ordered_bits((uint32_t)(best[e] >> 32));
      sc.fi[f * SDM_MAX_K + pos] = (int32_t)(uint32_t)(best[e] & 0xffffffffu);
    }
  }
  __syncwarp();
}

// Slot score of a position tuple (byte f = p_f): the float32 sum of its factor scores,
// left to right.
__device__ __forceinline__ float tuple_score(uint32_t t, const KeyGeometry &g, const RowScratch &sc) {
  float S = sc.fs[t & 255];
  if (g.F > 1) S = __fadd_rn(S, sc.fs[SDM_MAX_K + ((t >> 8) & 255)]);
  if (g.F > 2) S = __fadd_rn(S, sc.fs[2 * SDM_MAX_K + ((t >> 16) & 255)]);
  if (g.F > 3) S = __fadd_rn(S, sc.fs[3 * SDM_MAX_K + (t >> 24)]);
  return S;
}

// The 64-bit key of a position tuple with score S (layout above).
__device__ __forceinline__ uint64_t tuple_key(uint32_t t, float S) {
  const uint32_t p0 = t & 255, p1 = (t >> 8) & 255, p2 = (t >> 16) & 255, p3 = t >> 24;
  const uint32_t sum = p0 + p1 + p2 + p3;
  const uint32_t low = ((255u - sum) << 24) | ((255u - p0) << 16) | ((255u - p1) << 8) | (255u - p2);
  return ((uint64_t)ordered_bits(S) << 32) | low;
}

// Candidate tuples cand[c0, c1), keyed and kept best first (k <= 32 * EC); an empty
// range gives all-zero keys, which order after every real key.
template <int EC>
__device__ __forceinline__ void candidate_topk(const uint32_t *cand, int c0, int c1, const KeyGeometry &g,
                                               const RowScratch &sc, uint64_t (&ck)[EC]) {
  const int lane = threadIdx.x & 31;
  if (c1 <= c0) {
#pragma unroll
    for (int e = 0; e < EC; ++e) ck[e] = 0ull;
    return;
  }
  top_of_chunks<EC>(c1 - c0, [&](int b0, uint64_t(&kk)[EC]) {
#pragma unroll
    for (int e = 0; e < EC; ++e) {
      const int c = c0 + b0 + lane * EC + e;
      if (c < c1) {
        const uint32_t t = cand[c];
        kk[e] = tuple_key(t, tuple_score(t, g, sc));
      } else {
        kk[e] = 0ull;
      }
    }
  }, ck);
}

// candidate_topk over all ncand tuples, sorting only those that can be among the k
// best.  Every slot of a box of at least k tuples scores at least the box's corner
// (float addition is monotone in each operand), so the k-th best slot score is at
// least tau, the best corner score of `boxes`; a tuple scoring below tau cannot be
// selected.  The others are gathered (up to kSurvivorCap of them; past that, all
// tuples are sorted) and sorted with the same keys, so the result is the same.
template <int EC>
__device__ __forceinline__ void candidate_topk_pruned(const uint32_t *cand, int ncand, const uint32_t *boxes,
                                                      int nbox, const KeyGeometry &g, RowScratch &sc,
                                                      uint64_t (&ck)[EC]) {
  const int lane = threadIdx.x & 31;
  float tau = -INFINITY;
  if (lane < nbox) tau = tuple_score(boxes[lane], g, sc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tau = fmaxf(tau, __shfl_xor_sync(0xffffffffu, tau, o));
  int cnt = 0;
  for (int c0 = 0; c0 < ncand; c0 += 32) {
    const int c = c0 + lane;
    uint64_t key = 0ull;
    bool keep = false;
    if (c < ncand) {
      const uint32_t t = cand[c];
      const float S = tuple_score(t, g, sc);
      keep = S >= tau;
      key = tuple_key(t, S);
    }
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    const int pos = cnt + __popc(m & ((1u << lane) - 1u));
    if (keep && pos < kSurvivorCap) sc.surv[pos] = key;
    cnt += __popc(m);
  }
  __syncwarp();
  if (cnt > kSurvivorCap) {
    candidate_topk<EC>(cand, 0, ncand, g, sc, ck);
    return;
  }
  if (EC == 2 && cnt > 64) {
    // more than one chunk: keep only the keys whose score bits reach the 64th largest's
    // (the best 64 keys are among them), as factor_topk_radix does
    constexpr int KPL = kSurvivorCap / 32;
    uint64_t kv[KPL];
    uint32_t hi[KPL];
    bool ok[KPL];
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int j = lane + 32 * i;
      ok[i] = j < cnt;
      kv[i] = ok[i] ? sc.surv[j] : 0ull;
      hi[i] = (uint32_t)(kv[i] >> 32);
    }
    __syncwarp();
    const uint32_t T = warp_kth_largest<KPL>(hi, ok, 64, reinterpret_cast<int *>(sc.surv));
    int kept = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const bool keep = ok[i] && hi[i] >= T;
      const unsigned m = __ballot_sync(0xffffffffu, keep);
      if (keep) sc.surv[kept + __popc(m & ((1u << lane) - 1u))] = kv[i];
      kept += __popc(m);
    }
    __syncwarp();
    cnt = kept;
  }
  top_of_chunks<EC>(cnt, [&](int b0, uint64_t(&kk)[EC]) {
#pragma unroll
    for (int e = 0; e < EC; ++e) {
      const int i = b0 + lane * EC + e;
      kk[e] = i < cnt ? sc.surv[i] : 0ull;
    }
  }, ck);
  __syncwarp();
}

// Softmax weights of the k best keys (fixed summation order) and their slot ids.
template <int EC>
__device__ __forceinline__ void finish_topk(const uint64_t (&ck)[EC], const KeyGeometry &g, int qsel,
                                            const RowScratch &sc, int32_t *idx_out, float *wt_out) {
  const int lane = threadIdx.x & 31;
  const int k = g.k[qsel];
  const float S0 = from_ordered_bits((uint32_t)(__shfl_sync(0xffffffffu, ck[0], 0) >> 32));
  float ex[EC];
  float part = 0.0f;
#pragma unroll
  for (int e = 0; e < EC; ++e) {
    const int pos = lane * EC + e;
    ex[e] = 0.0f;
    if (pos < k) {
      const float S = from_ordered_bits((uint32_t)(ck[e] >> 32));
      ex[e] = expf(__fsub_rn(S, S0));
      part = __fadd_rn(part, ex[e]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, o));
#pragma unroll
  for (int e = 0; e < EC; ++e) {
    const int pos = lane * EC + e;
    if (pos < k) {
      const uint32_t low = (uint32_t)(ck[e] & 0xffffffffu);
      const int sum = 255 - (int)(low >> 24);
      const int p0 = 255 - (int)((low >> 16) & 255);
      const int p1 = 255 - (int)((low >> 8) & 255);
      const int p2 = 255 - (int)(low & 255);
      const int p3 = sum - p0 - p1 - p2;
      int64_t slot = sc.fi[p0];
      if (g.F > 1) slot = slot * g.nf[1] + sc.fi[SDM_MAX_K + p1];
      if (g.F > 2) slot = slot * g.nf[2] + sc.fi[2 * SDM_MAX_K + p2];
      if (g.F > 3) slot = slot * g.nf[3] + sc.fi[3 * SDM_MAX_K + p3];
      idx_out[pos] = (int32_t)slot;
      wt_out[pos] = __fdiv_rn(ex[e], part);
    }
  }
  __syncwarp();
}

// One row by one warp.  scores: the row's ntot factor scores (shared memory), factor f
// at g.off[f]; qsel: 0 = write query (k = W), 1 = read query (k = R); cand: the
// candidate tuples of this query kind (shared memory), ncand entries.  Writes k slot
// ids (best first) to idx_out and their softmax weights to wt_out.
template <int EF, int EC>
__device__ __forceinline__ void row_topk(const float *scores, const KeyGeometry &g, int qsel,
                                         const uint32_t *cand, int ncand, const uint32_t *boxes, int nbox,
                                         RowScratch &sc, int32_t *idx_out, float *wt_out) {
  for (int f = 0; f < g.F; ++f) {
    // (for at most 128 keys the chunk sorts are already short: the radix passes cost more)
    if (EF == 2 && g.nf[f] > 128 && g.nf[f] <= 256) factor_topk_radix(scores, g, qsel, f, sc);
    else factor_topk<EF>(scores, g, qsel, f, sc);
  }
  __syncwarp();
  uint64_t ck[EC];
  candidate_topk_pruned<EC>(cand, ncand, boxes, nbox, g, sc, ck);
  finish_topk<EC>(ck, g, qsel, sc, idx_out, wt_out);
}

// Terms [0, n) of one factor score folded into acc, n <= kBf16Block: one block of the
// bfloat16 dot product (BF16) or n compensated float32 steps (accurate accumulation as
// described in sdm_common.cuh); k holds sub-key values of the activation type, read as
// float32.  A factor score <q, k> over d_sub terms is the blocks starting at 0,
// kBf16Block, 2 * kBf16Block, ... folded in order into Acc2{0, 0}, then acc2_value.
template <bool BF16, typename KT>
__device__ __forceinline__ void score_block(Acc2 &acc, const float *q, const KT *k, int n) {
  if constexpr (BF16) {
    float blk = 0.0f;
#pragma unroll 8
    for (int d = 0; d < n; ++d) blk = __fmaf_rn(q[d], to_f32(k[d]), blk);
    two_sum_into(acc, blk);
  } else {
#pragma unroll 8
    for (int d = 0; d < n; ++d) dot2_step(acc, q[d], to_f32(k[d]));
  }
}

}  // namespace sdm
