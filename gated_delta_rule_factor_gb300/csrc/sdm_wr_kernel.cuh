// The write/read kernel template (included by the translation units that instantiate
// it).
//
// Parallel axes: streams (b, h) are independent, and so is every bank column (the
// update of a column reads only that column, see sdm_delta.cuh).  One CTA owns one
// stream and a slice of CW columns (CW * elem = 16..128 bytes of every row) and runs
// the stream's tokens in order.  Tokens are staged G at a time; the chunk plan
// (sdm_plan.cu) lists the distinct rows of each stage.
//
// Warp roles (one CTA):
//   2 compute warps: the tokens of the current stage on the shared-memory rows, with the
//               block-ordered token step (sdm_delta.cuh token_blocks2);
//   8 loader warps (4 when two CTAs share an SM): fetch the next stage's rows, its token data and the stage record
//               after it, all with 16-byte cp.async on the LSU path (a bulk/TMA copy per
//               row slice costs more than it saves at this granularity); once the compute
//               warps signal (barrier 5) that the current stage's next-to-last token is
//               done, write back the current stage's dirty rows its last token leaves
//               alone, and after the stage the rest of them, while the next stage's rows
//               are still landing.  More loader warps keep more row requests in flight.
//   every warp copies the rows carried over from the previous stage.
// Two row buffers alternate between stages; rows shared by consecutive stages are
// copied across buffers instead of re-read, because the bank copy may be stale.  Stage
// records use three buffers (in use / rows being fetched / record being fetched).
#pragma once

#include "sdm_common.cuh"
#include "sdm_delta.cuh"
#include "sdm_internal.h"

namespace sdm {
namespace wr {


struct TokLayout {
  int64_t wts, gates, v, bytes;  // offsets inside one token-data buffer
};

__host__ __device__ inline int64_t align16(int64_t x) { return (x + 15) & ~int64_t(15); }

__host__ __device__ inline TokLayout tok_layout(int G, int W, int R, int CW, int act_elem) {
  TokLayout t;
  t.wts = 0;
  t.gates = align16((int64_t)G * (W + R) * 4);
  t.v = t.gates + align16((int64_t)G * 2 * 4);
  t.bytes = t.v + align16((int64_t)G * CW * act_elem);
  return t;
}

// A CTA owns a slice of CW columns (CW * elem = 16..128 bytes of every row): two compute
// warps and LW loader warps (8 when one CTA runs per SM, 4 when two share an SM, so that
// their registers fit).  Lane % 8 of a compute warp owns VB = CW / 8 consecutive columns.
template <typename BANK, int CW, int LW_ = 8>
struct WrGeometry {
  static constexpr int VB = CW / 8;                   // columns per compute lane
  static constexpr int RB = CW * (int)sizeof(BANK);   // row slice bytes
  static constexpr int NCW = 2;                       // compute warps (rows split)
  static constexpr int LW = LW_;                      // loader warps
  static constexpr int NTHR = 32 * (NCW + LW);
  static_assert(CW % 8 == 0 && RB >= 16 && RB <= 128 && (RB & (RB - 1)) == 0, "column slice");
};

// JB = the most rows a compute lane holds (one of the 8 row blocks of a token);
// FULL: W == R == 8 * JB, fixed at compile time.
template <typename BANK, typename ACT, int CW, int JB, bool FULL = false, int LW = 8>
__global__ void __launch_bounds__(WrGeometry<BANK, CW, LW>::NTHR)
    write_read_kernel(const __grid_constant__ WriteReadArgs a) {
  using Geo = WrGeometry<BANK, CW, LW>;
  constexpr int kLoaderThreads = 32 * Geo::LW;
  constexpr int VB = Geo::VB, NCW = Geo::NCW, NTHR = Geo::NTHR, RB = Geo::RB;
  constexpr int CPR = RB / 16;                        // 16-byte chunks per row slice

  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ __align__(16) float xch[2 * 2 * 8 * VB];  // the two compute warps' partial sums
  const PlanLayout &lay = a.lay;
  const int L = lay.L, G = lay.G, S = lay.n_stages;
  const int W = a.W, R = a.R, WR = W + R;
  const int64_t s = blockIdx.y;
  const int slice = blockIdx.x;
  const int64_t b = s / a.H, h = s % a.H;
  const int64_t c0 = (int64_t)slice * CW;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool is_loader = warp >= NCW;

  // Buffer addresses are computed, not kept in an indexed array, so that they stay
  // shared-memory addresses for the compiler.
  auto rowbuf = [&](int i) -> unsigned char * { return smem + (int64_t)(i & 1) * L * RB; };
  unsigned char *plans = smem + 2 * (int64_t)L * RB;
  const TokLayout tl = tok_layout(G, W, R, CW, (int)sizeof(ACT));
  auto tokbuf = [&](int i) -> unsigned char * { return plans + 3 * lay.rec_bytes + (int64_t)(i & 1) * tl.bytes; };

  BANK *bank = static_cast<BANK *>(a.bank) + s * a.N * a.d_v;   // this stream's table
  const ACT *kv = static_cast<const ACT *>(a.k_val);
  ACT *y = static_cast<ACT *>(a.y);
  const unsigned char *records = a.records + s * (int64_t)S * lay.rec_bytes;

  auto plan_of = [&](int g) -> unsigned char * { return plans + (int64_t)(g % 3) * lay.rec_bytes; };
  auto hdr_ok = [&](const int32_t *hdr) -> bool {
    return hdr[0] >= 0 && hdr[0] <= L && hdr[1] >= 0 && hdr[1] <= L && hdr[2] >= 0 && hdr[2] <= L &&
           hdr[3] >= 0 && hdr[3] <= L && hdr[4] >= 0 && hdr[4] <= hdr[1] && hdr[5] >= 0 && hdr[5] <= hdr[3];
  };

  constexpr int VBYTES = CW * (int)sizeof(ACT);      // value bytes per token (>= 16)

  // ---- loader helpers (threads of the loader warps).  Every copy is a 16-byte cp.async
  // (or 8/4-byte for the gates and unaligned weights) on the LSU path: CPR lanes take
  // one row slice, so one warp request covers whole 128-byte lines.
  const int ltid = tid - 32 * NCW;
  const int sub = ltid % CPR, grp = ltid / CPR;       // chunk of a row, row group
  constexpr int GRP = kLoaderThreads / CPR;           // row slices per loader pass
  const int64_t row_pitch = a.d_v * (int64_t)sizeof(BANK);
  auto fetch_record = [&](int g) {
    const unsigned char *src = records + (int64_t)g * lay.rec_bytes;
    unsigned char *dst = plan_of(g);
    for (int64_t i = ltid; i < lay.rec_bytes / 16; i += kLoaderThreads) cp_async16(dst + i * 16, src + i * 16);
  };
  // Rows of stage g's load list with index in [lo, hi) (the last hdr[4] entries are the
  // rows of stage g-2, which must wait for that stage's write-back).
  auto fetch_rows = [&](int g, bool early, bool late) {
    const unsigned char *rec = plan_of(g);
    const int32_t *hdr = reinterpret_cast<const int32_t *>(rec);
    const int n_load = hdr_ok(hdr) ? hdr[1] : 0;
    const int n_late = hdr_ok(hdr) ? hdr[4] : 0;
    const int lo = early ? 0 : n_load - n_late, hi = late ? n_load : n_load - n_late;
    const int32_t *load_slot = reinterpret_cast<const int32_t *>(rec + lay.off_load_slot);
    const uint16_t *load_u = reinterpret_cast<const uint16_t *>(rec + lay.off_load_u);
    unsigned char *dst = rowbuf(g & 1) + sub * 16;
    const unsigned char *src = reinterpret_cast<const unsigned char *>(bank + c0) + sub * 16;
#pragma unroll 4
    for (int e = lo + grp; e < hi; e += GRP) {
      const int32_t slot = load_slot[e];
      const int u = load_u[e];
      if (u >= L || slot < 0 || slot >= a.N) {
        raise_error(a.err, SDM_DEVERR_PLAN);
        continue;
      }
      cp_async16(dst + (int64_t)u * RB, src + (int64_t)slot * row_pitch);
    }
  };
  auto fetch_tokens = [&](int g) {
    const int64_t t0 = (int64_t)g * G;
    const int nt = (int)min((int64_t)G, a.T - t0);
    unsigned char *tb = tokbuf(g & 1);
    float *wts = reinterpret_cast<float *>(tb + tl.wts);
    if (a.tok_bulk) {                                  // weights in 16-byte pieces
      const int wq = W / 4, rq = R / 4;
      for (int i = ltid; i < nt * (wq + rq); i += kLoaderThreads) {
        const int t = i / (wq + rq), q = i % (wq + rq);
        const int64_t row = (b * a.T + t0 + t) * a.H + h;
        if (q < wq) cp_async16(wts + t * WR + 4 * q, a.wt[0] + row * W + 4 * q);
        else cp_async16(wts + t * WR + W + 4 * (q - wq), a.wt[1] + row * R + 4 * (q - wq));
      }
    } else {
      for (int i = ltid; i < nt * WR; i += kLoaderThreads) {
        const int t = i / WR, j = i % WR;
        const int64_t row = (b * a.T + t0 + t) * a.H + h;
        const float *src_w = (j < W) ? a.wt[0] + row * W + j : a.wt[1] + row * R + (j - W);
        cp_async4(wts + i, src_w);
      }
    }
    float *gt = reinterpret_cast<float *>(tb + tl.gates);
    for (int i = ltid; i < nt; i += kLoaderThreads) {
      const int64_t row = (b * a.T + t0 + i) * a.H + h;
      cp_async8(gt + 2 * i, a.gates + row * 2);
    }
    unsigned char *vb = tb + tl.v;
    for (int i = ltid; i < nt * (VBYTES / 16); i += kLoaderThreads) {
      const int t = i / (VBYTES / 16), c = i % (VBYTES / 16);
      const int64_t row = (b * a.T + t0 + t) * a.H + h;
      cp_async16(vb + (int64_t)t * VBYTES + c * 16,
                 reinterpret_cast<const unsigned char *>(kv + row * a.d_v + c0) + c * 16);
    }
  };
  // Dirty rows of stage g back to the bank (CPR lanes per row slice, 16-byte stores).
  // Dirty rows of stage g back to the bank: early = the rows its last token does not
  // write (stored while that token runs), late = the rest (stored after the stage).
  auto write_back = [&](int g, bool early) {
    const unsigned char *rec = plan_of(g);
    const int32_t *hdr = reinterpret_cast<const int32_t *>(rec);
    const bool ok = hdr_ok(hdr);
    const int n_all = ok ? hdr[3] : 0, n_late = ok ? hdr[5] : 0;
    const int lo = early ? 0 : n_all - n_late, n_wb = early ? n_all - n_late : n_all;
    const int32_t *wb_slot = reinterpret_cast<const int32_t *>(rec + lay.off_wb_slot);
    const uint16_t *wb_u = reinterpret_cast<const uint16_t *>(rec + lay.off_wb_u);
    const unsigned char *src = rowbuf(g & 1) + sub * 16;
    unsigned char *dst = reinterpret_cast<unsigned char *>(bank + c0) + sub * 16;
#pragma unroll 4
    for (int e = lo + grp; e < n_wb; e += GRP) {
      const int32_t slot = wb_slot[e];
      const int u = wb_u[e];
      if (u >= L || slot < 0 || slot >= a.N) {
        raise_error(a.err, SDM_DEVERR_PLAN);
        continue;
      }
      *reinterpret_cast<uint4 *>(dst + (int64_t)slot * row_pitch) = *reinterpret_cast<const uint4 *>(src + (int64_t)u * RB);
    }
  };

  auto fetch_stage = [&](int g) {
    fetch_rows(g, true, true);
    fetch_tokens(g);
  };
  // ---- prologue: record 0, then stage 0 and record 1
  if (is_loader) {
    fetch_record(0);
    cp_async_commit();
    cp_async_wait_all();
    named_barrier(1, kLoaderThreads);
    fetch_stage(0);
    if (S > 1) fetch_record(1);
    cp_async_commit();
  }

  for (int g = 0; g < S; ++g) {
    if (is_loader) cp_async_wait_all();
    named_barrier(2, NTHR);                                      // stage g resident
    const unsigned char *rec = plan_of(g);
    {
      // rows shared with stage g-1 come from its buffer (the bank may still be stale);
      // every warp of the CTA copies
      const int32_t *hdr = reinterpret_cast<const int32_t *>(rec);
      const bool ok = hdr_ok(hdr);
      if (!ok && tid == 0) raise_error(a.err, SDM_DEVERR_PLAN);
      const int n_carry = ok ? hdr[2] : 0;
      const uint32_t *carry = reinterpret_cast<const uint32_t *>(rec + lay.off_carry);
      const unsigned char *from = rowbuf((g + 1) & 1);
      unsigned char *to = rowbuf(g & 1);
      for (int i = tid; i < n_carry * CPR; i += NTHR) {
        const int e = i / CPR, c = i % CPR;
        const int u = carry[e] & 0xffff, src = carry[e] >> 16;
        if (u >= L || src >= L) {
          raise_error(a.err, SDM_DEVERR_PLAN);
          continue;
        }
        *reinterpret_cast<uint4 *>(to + (int64_t)u * RB + c * 16) =
            *reinterpret_cast<const uint4 *>(from + (int64_t)src * RB + c * 16);
      }
    }
    named_barrier(3, NTHR);                                      // carries in place

    if (!is_loader) {
      // ---- compute: tokens of stage g in order; both compute warps work on the same
      // column groups, the token's row blocks split between them (token_blocks2); warp 0
      // stores y
      const uint16_t *refmap = reinterpret_cast<const uint16_t *>(rec + lay.off_refmap);
      const uint8_t *tokflag = rec + lay.off_tokflag;
      const unsigned char *tb = tokbuf(g);
      const float *wts = reinterpret_cast<const float *>(tb + tl.wts);
      const float *gt = reinterpret_cast<const float *>(tb + tl.gates);
      const ACT *vv = reinterpret_cast<const ACT *>(tb + tl.v);
      const int cl = lane & 7;                                 // column group in the slice
      unsigned char *rows = rowbuf(g) + cl * VB * (int)sizeof(BANK);
      const int64_t t0 = (int64_t)g * G;
      const int nt = (int)min((int64_t)G, a.T - t0);
      ACT *ybase = y + ((b * a.T + t0) * a.H + h) * a.d_v + c0 + cl * VB;
      const int64_t ystep = (int64_t)a.H * a.d_v;
      if (nt <= 1) named_barrier_arrive(5, kLoaderThreads + 32 * NCW);
      for (int t = 0; t < nt; ++t) {
        float v[VB], out[VB];
        load_vec<ACT, VB>(vv + t * CW + cl * VB, v);
        token_blocks2<BANK, VB, JB, FULL>(W, R, refmap + t * WR, wts + t * WR, gt[2 * t], gt[2 * t + 1], v, rows,
                                          RB, tokflag[t] != 0, out, xch, xch + 2 * 8 * VB, warp, 6);
        if (warp == 0 && lane < 8) store_vec<ACT, VB>(ybase + t * ystep, out);
        __syncwarp();
        if (t == nt - 2) named_barrier_arrive(5, kLoaderThreads + 32 * NCW);  // rows the last token leaves alone are final
      }
    } else {
      // ---- loaders: fetch stage g+1 into its buffer (stage g-1's, fully written back at
      // the end of that stage) and record g+2, then store the rows of stage g its last
      // token leaves alone once the compute warps are past its next-to-last token
      if (g + 1 < S) fetch_stage(g + 1);
      if (g + 2 < S) fetch_record(g + 2);
      cp_async_commit();
      named_barrier(5, kLoaderThreads + 32 * NCW);             // stage g's next-to-last token done
      write_back(g, true);
    }
    named_barrier(4, NTHR);                                      // stage g computed
    // the rest of stage g's dirty rows go back while the next stage's rows land; the next
    // stage barrier orders these stores before any later load of the same rows
    if (is_loader) write_back(g, false);
  }
}

// Launches the instance for the shape: W = R = 64 fixed at compile time, else the
// smallest JB >= ceil(max(W, R) / 8); 4 loader warps when two CTAs share an SM.
template <typename BANK, typename ACT, int CW, int LW>
cudaError_t launch_cw_lw(const WriteReadArgs &a, int64_t streams, int64_t smem, cudaStream_t st) {
  const dim3 grid((unsigned)a.slices, (unsigned)streams);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, WrGeometry<BANK, CW, LW>::NTHR, smem, st>>>(a);
    return cudaGetLastError();
  };
  const int n = a.W > a.R ? a.W : a.R;
  const int per_lane = (n + 7) / 8;
  if (a.W == 64 && a.R == 64) return go(write_read_kernel<BANK, ACT, CW, 8, true, LW>);
  if (per_lane <= 4) return go(write_read_kernel<BANK, ACT, CW, 4, false, LW>);
  if (per_lane <= 8) return go(write_read_kernel<BANK, ACT, CW, 8, false, LW>);
  if (per_lane <= 16) return go(write_read_kernel<BANK, ACT, CW, 16, false, LW>);
  return cudaErrorInvalidValue;
}

template <typename BANK, typename ACT, int CW>
cudaError_t launch_cw(const WriteReadArgs &a, int64_t streams, int64_t smem, cudaStream_t st) {
  if (a.two_per_sm) return launch_cw_lw<BANK, ACT, CW, 4>(a, streams, smem, st);
  return launch_cw_lw<BANK, ACT, CW, 8>(a, streams, smem, st);
}

}  // namespace wr
}  // namespace sdm
