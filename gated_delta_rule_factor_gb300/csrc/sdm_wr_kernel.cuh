// The write/read kernel template (included by the translation units that instantiate
// it).
//
// Parallel axes: streams (b, h) are independent, and so is every bank column (the
// update of a column reads only that column, see sdm_delta.cuh).  One CTA owns one
// stream and a slice of RB = 32*NCW bytes of every row; each of its NCW compute warps
// owns a 32-byte piece of that slice and runs the stream's tokens in order on it, with
// no synchronisation between compute warps.  Tokens are staged G at a time; the chunk
// plan (sdm_plan.cu) lists the distinct rows of each stage.
//
// Pipeline.  Three row buffers (stage g uses buffer g % 3), each with the stage's
// per-reference offsets and token data (weights, gates, value slice); a ring of five
// row-list records (stages g-1 .. g+3 of loader iteration g).  Three mbarriers per
// buffer:
//   full[b]  stage g's bank rows, offsets and token data have landed (issued two stages
//            ahead; every loader waits for its own copies, then one thread arrives);
//   recs[b]  loader iteration g has made the row lists of stages g+1 and g+2 visible
//            and finished reading stage g-1's buffer for its write-back (one arrival,
//            after the loaders' barrier);
//   done[b]  every compute warp has finished stage g and copied out of buffer g the
//            rows stages g+1 and g+2 carry over (one arrival per warp, after __syncwarp).
// mbarrier arrivals are shared-memory atomics that serialize, so each is made once per
// group of threads that a barrier or __syncwarp has already ordered.
// Loader iteration g: fetch the row lists of stage g+3; wait done[g-1] and write stage
// g-1's dirty rows back; arrive on recs; fetch stage g+2's bank rows into buffer
// (g+2) % 3 (stage g-1's, now free); wait until stage g+1's rows have landed and
// arrive on full.  (A cp.async-tracked mbarrier arrival per thread measured as costly
// as waiting for the copies.)  Compute warps, stage g: wait full[g], run the
// tokens, wait recs(g), copy this stage's rows that stage g+1 (carry 1) or stage g+2
// (carry 2, rows g+1 does not hold) needs into their buffers, arrive on done.  The
// bank is never read stale: a row one of the two previous stages holds is carried in
// shared memory, and any older row was written back before the fetch.  No memory round
// trip lies between one stage's end and the next stage's start.  With one compute warp
// per CTA the loaders make the carries instead (kLoaderHandOn): after done[g-1] they copy
// the rows stage g takes over, arrive on full[g], then copy those stage g+1 takes over.
// Every wait is bounded (2 s of %globaltimer); a wait that runs out records
// SDM_DEVERR_TIMEOUT and sets a shared abort flag that every other wait also watches.
#pragma once

#include "sdm_common.cuh"
#include "sdm_delta.cuh"
#include "sdm_internal.h"

namespace sdm {
namespace wr {

constexpr int kRowBufs = 3;      // row / compute-record / token-data buffers
constexpr int kLoaderRecs = 5;   // loader records: stages g-1 .. g+3 of loader iteration g
constexpr int kBatch = 4;        // list entries whose copies one thread issues together

// Value slice of a stage's tokens (the only per-CTA token data; weights and gates come
// with the compute record).  cols: the CTA's bank columns (RB / bank element bytes).
__host__ __device__ inline int64_t align16(int64_t x) { return (x + 15) & ~int64_t(15); }
__host__ __device__ inline int64_t vals_bytes(int G, int cols, int act_elem) {
  return align16((int64_t)G * cols * act_elem);
}

struct SmemLayout {
  int64_t rows, crec, tok, lrec, bars, bytes;
};

__host__ __device__ inline SmemLayout smem_layout(const PlanLayout &lay, int bank_elem, int act_elem) {
  SmemLayout m;
  m.rows = 0;
  m.crec = m.rows + (int64_t)kRowBufs * lay.L * lay.RB;
  m.tok = m.crec + kRowBufs * lay.crec_bytes;
  m.lrec = m.tok + kRowBufs * vals_bytes(lay.G, lay.RB / bank_elem, act_elem);
  m.bars = m.lrec + kLoaderRecs * lay.lrec_bytes;
  m.bytes = m.bars + 3 * kRowBufs * 8 + 16;           // full[3], recs[3], done[3], flags
  return m;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}

// cp.async without a compiler memory clobber, for the loaders' row copies: the compiler
// may then batch the row-list reads around them.  The destination is read only after a
// cp.async.wait_group and a barrier (both with memory clobbers), so no access that the
// clobber would order is affected.
__device__ __forceinline__ void cp_async16_rows(uint32_t dst_smem, const void *src_gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst_smem), "l"(src_gmem));
}

// Bounded wait for the phase of `bar` with the given parity that also gives up as soon
// as another warp has set the abort flag.  false: gave up.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, volatile int32_t *abort_flag) {
  const uint32_t addr = smem_addr(bar);
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 63) == 63) {
      if (*abort_flag) return false;
      const uint64_t now = global_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > kWaitLimitNs) return false;
    }
  }
}

template <int NCW, int LW>
struct WrGeometry {
  static constexpr int RB = 32 * NCW;                 // row slice bytes of the CTA
  static constexpr int CPR = RB / 16;                 // 16-byte chunks per row slice
  static constexpr int NL = 32 * LW;                  // loader threads
  static constexpr int NTHR = 32 * (NCW + LW);
  static_assert(NL % CPR == 0, "loader threads cover whole row slices");
};

// JB: the most rows a lane holds per sum (ceil(max(W, R) / 16)); FULL: W == R == 64.
// Four loader warps mean the launch plans two CTAs per SM, whose registers must fit.
template <typename BANK, typename ACT, int NCW, int JB, bool FULL, int LW>
__global__ void __launch_bounds__(WrGeometry<NCW, LW>::NTHR, LW == 4 ? 2 : 1)
    write_read_kernel(const __grid_constant__ WriteReadArgs a) {
  using Geo = WrGeometry<NCW, LW>;
  constexpr int RB = Geo::RB, CPR = Geo::CPR, NL = Geo::NL;
  constexpr int VEC = PieceRow<BANK>::VEC;            // columns per lane
  constexpr int PC = 2 * VEC;                         // columns per warp piece
  constexpr int COLS = NCW * PC;                      // columns per CTA
  extern __shared__ __align__(128) unsigned char smem[];

  const PlanLayout &lay = a.lay;
  const int L = lay.L, G = lay.G, S = lay.n_stages;
  const int W = a.W, R = a.R, WR = W + R;
  const int64_t s = blockIdx.y;
  const int slice = blockIdx.x;
  const int64_t b = s / a.H, h = s % a.H;
  const int64_t c0 = (int64_t)slice * COLS;                   // first column of the slice
  const int valid_chunks = min(CPR, (a.row_bytes - slice * RB) / 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool is_loader = warp >= NCW;

  // One compute warp per CTA: the loaders, otherwise idle while it runs the tokens, copy
  // the rows each stage hands on (the compute warps do it themselves when there are more).
  constexpr bool kLoaderHandOn = NCW == 1;
  const SmemLayout sl = smem_layout(lay, (int)sizeof(BANK), (int)sizeof(ACT));
  const int64_t vbytes = vals_bytes(G, COLS, (int)sizeof(ACT));
  auto rowbuf = [&](int g) -> unsigned char * { return smem + sl.rows + (int64_t)(g % kRowBufs) * L * RB; };
  auto crecbuf = [&](int g) -> unsigned char * { return smem + sl.crec + (int64_t)(g % kRowBufs) * lay.crec_bytes; };
  auto tokbuf = [&](int g) -> unsigned char * { return smem + sl.tok + (int64_t)(g % kRowBufs) * vbytes; };
  auto lrecbuf = [&](int g) -> unsigned char * { return smem + sl.lrec + (int64_t)(g % kLoaderRecs) * lay.lrec_bytes; };
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + sl.bars);
  uint64_t *recs = full + kRowBufs;
  uint64_t *done = recs + kRowBufs;
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(done + kRowBufs);
  volatile int32_t *loader_go = abort_flag + 1;                 // written by loader thread 0 only

  BANK *bank = static_cast<BANK *>(a.bank) + s * a.N * a.d_v;   // this stream's table
  const unsigned char *lrecs = a.lrecs + s * (int64_t)S * lay.lrec_bytes;
  const unsigned char *crecs = a.crecs + s * (int64_t)S * lay.crec_bytes;
  const int64_t row_pitch = a.d_v * (int64_t)sizeof(BANK);
  const int64_t row_limit = (int64_t)L * RB;                    // offsets o must stay below

  if (tid == 0) {
    for (int i = 0; i < kRowBufs; ++i) {
      mbar_init(&full[i], 1);      // loader thread 0, after the loaders' copies landed
      mbar_init(&recs[i], 1);      // loader thread 0, after the loader barrier
      mbar_init(&done[i], NCW);    // lane 0 of each compute warp, after __syncwarp
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  if (S == 0) return;

  if (is_loader) {
    // ------------------------------------------------------------------ loaders
    const int lt = tid - 32 * NCW;
    const int sub = lt % CPR, grp = lt / CPR;          // chunk of a row slice, row group
    constexpr int GRP = NL / CPR;                      // row slices per loader pass
    const unsigned char *bank_slice = reinterpret_cast<const unsigned char *>(bank + c0) + sub * 16;
    auto loader_bar = [&] { named_barrier(1, NL); };
    const int lrec_chunks = (int)(lay.lrec_bytes / 16), crec_chunks = (int)(lay.crec_bytes / 16);
    auto fetch_lrec = [&](int g) {
      const unsigned char *src = lrecs + (int64_t)g * lay.lrec_bytes;
      unsigned char *dst = lrecbuf(g);
      for (int i = lt; i < lrec_chunks; i += NL) cp_async16(dst + i * 16, src + i * 16);
    };
    auto hdr_ok = [&](const int32_t *hdr) {
      return hdr[0] >= 0 && hdr[0] <= L && hdr[1] >= 0 && hdr[1] <= hdr[0] && hdr[2] >= 0 && hdr[3] >= 0 &&
             hdr[2] + hdr[3] <= hdr[0] && hdr[4] >= 0 && hdr[4] <= hdr[0];
    };
    // Row offsets (16-byte units) must stay inside the stream's table, shared-memory
    // offsets inside the stage buffer; a bad entry is skipped and reported.
    const uint32_t lim16 = (uint32_t)((uint64_t)a.N * (uint64_t)row_pitch / 16);
    const uint32_t olim = (uint32_t)row_limit;
    const uint32_t sub16 = (uint32_t)sub << 4;
    // stage g's bank rows (the first n_load row-list entries)
    auto fetch_rows = [&](int g) {
      const unsigned char *rec = lrecbuf(g);
      const int32_t *hdr = reinterpret_cast<const int32_t *>(rec);
      const bool ok = hdr_ok(hdr);
      if (!ok && lt == 0) raise_error(a.err, SDM_DEVERR_PLAN);
      const int n_load = ok ? hdr[1] : 0;
      const uint2 *ent = reinterpret_cast<const uint2 *>(rec + lay.off_ent);
      const uint32_t dst = smem_addr(rowbuf(g));
      if (sub >= valid_chunks) return;
      // kBatch entries read first, then their copies issued back to back
      for (int e0 = grp; e0 < n_load; e0 += kBatch * GRP) {
        uint2 v[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) v[k] = e0 + k * GRP < n_load ? ent[e0 + k * GRP] : make_uint2(0u, 0u);
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          if (e0 + k * GRP >= n_load) break;
          if (v[k].x < lim16 && v[k].y < olim) cp_async16_rows(dst + (v[k].y ^ sub16), bank_slice + (size_t)v[k].x * 16);
          else raise_error(a.err, SDM_DEVERR_PLAN);
        }
      }
    };
    // stage g's compute record (offsets, flags, weights, gates: one contiguous copy) and
    // this slice's values of its tokens.  Each thread's share of the values is the same
    // every stage: worked out once.
    constexpr int VCH = COLS * (int)sizeof(ACT) / 16;                      // value chunks per token
    const int vch = (int)min((int64_t)VCH, (a.d_v - c0) * (int64_t)sizeof(ACT) / 16);
    const int tv_t = lt / VCH, tv_c = lt % VCH;
    const ACT *kv = static_cast<const ACT *>(a.k_val);
    auto fetch_stage_data = [&](int g) {
      const unsigned char *src = crecs + (int64_t)g * lay.crec_bytes;
      unsigned char *dst = crecbuf(g);
      for (int i = lt; i < crec_chunks; i += NL) cp_async16(dst + i * 16, src + i * 16);
      const int64_t t0 = (int64_t)g * G;
      const int nt = (int)min((int64_t)G, a.T - t0);
      if (tv_c < vch) {
        unsigned char *vb = tokbuf(g) + tv_c * 16;
        const unsigned char *kvs = reinterpret_cast<const unsigned char *>(kv + c0) + tv_c * 16;
        const int64_t tstep = (int64_t)a.H * a.d_v * (int64_t)sizeof(ACT);
        const unsigned char *src_t = kvs + ((b * a.T + t0) * a.H + h) * a.d_v * (int64_t)sizeof(ACT);
        for (int t = tv_t; t < nt; t += NL / VCH)
          cp_async16(vb + (int64_t)t * COLS * sizeof(ACT), src_t + (int64_t)t * tstep);
      }
    };
    auto write_back = [&](int g) {
      const unsigned char *rec = lrecbuf(g);
      const int32_t *hdr = reinterpret_cast<const int32_t *>(rec);
      const int n_wb = hdr_ok(hdr) ? hdr[4] : 0;
      const uint2 *wb = reinterpret_cast<const uint2 *>(rec + lay.off_wb);
      const unsigned char *src = rowbuf(g);
      unsigned char *dst = reinterpret_cast<unsigned char *>(bank + c0) + sub * 16;
      if (sub >= valid_chunks) return;
      // kBatch entries, then their rows out of shared memory, then the stores
      for (int e0 = grp; e0 < n_wb; e0 += kBatch * GRP) {
        uint2 v[kBatch];
        uint4 r[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) v[k] = e0 + k * GRP < n_wb ? wb[e0 + k * GRP] : make_uint2(lim16, olim);
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
          if (v[k].x < lim16 && v[k].y < olim) r[k] = *reinterpret_cast<const uint4 *>(src + (v[k].y ^ sub16));
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          if (e0 + k * GRP >= n_wb) break;
          if (v[k].x < lim16 && v[k].y < olim) *reinterpret_cast<uint4 *>(dst + (size_t)v[k].x * 16) = r[k];
          else raise_error(a.err, SDM_DEVERR_PLAN);
        }
      }
    };
    // Waits for the compute warps to finish stage g (one thread waits, all loaders learn
    // the outcome at the loader barrier); false: give up.
    // (The decision is published in loader_go, which only this thread writes, so that
    // every loader reads the same value even if a compute warp raises the abort flag
    // meanwhile; the next write of loader_go comes after another loader barrier.)
    auto wait_done = [&](int g) -> bool {
      if (lt == 0) {
        bool ok = !*abort_flag && wait_phase(&done[g % kRowBufs], (uint32_t)(g / kRowBufs) & 1u, abort_flag);
        if (!ok && !*abort_flag) {
          raise_error(a.err, SDM_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        *loader_go = ok ? 1 : 0;
      }
      loader_bar();
      return *loader_go != 0;
    };

    // Loader hand-on (kLoaderHandOn): stage g's rows that stage g+1 (second == false) or
    // stage g+2 (second == true) takes over, copied out of buffer g once the compute warps
    // are done with it, kBatch list entries per thread at a time, each thread one 16-byte
    // chunk of a row slice.
    auto hand_on_rows = [&](int g, bool second) {
      const unsigned char *rec = lrecbuf(g);
      const int32_t *hdr = reinterpret_cast<const int32_t *>(rec);
      if (!hdr_ok(hdr)) return;
      const int n1 = hdr[2], n = second ? hdr[2] + hdr[3] : hdr[2];
      const uint2 *out = reinterpret_cast<const uint2 *>(rec + lay.off_out);
      const unsigned char *src = rowbuf(g);
      if (sub >= valid_chunks) return;
      for (int e0 = (second ? n1 : 0) + grp; e0 < n; e0 += kBatch * GRP) {
        uint32_t cv[kBatch];
        uint4 r[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) cv[k] = e0 + k * GRP < n ? out[e0 + k * GRP].x : 0u;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const uint32_t os = cv[k] >> 16;
          if (e0 + k * GRP < n && os < olim) r[k] = *reinterpret_cast<const uint4 *>(src + (os ^ sub16));
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int e = e0 + k * GRP;
          if (e >= n) break;
          const uint32_t od = cv[k] & 0xffffu, os = cv[k] >> 16;
          if (od < olim && os < olim) *reinterpret_cast<uint4 *>((e < n1 ? rowbuf(g + 1) : rowbuf(g + 2)) + (od ^ sub16)) = r[k];
          else raise_error(a.err, SDM_DEVERR_PLAN);
        }
      }
    };

    if constexpr (kLoaderHandOn) {
      // Iteration g: wait until the compute warps are done with stage g-1, copy the rows
      // stage g takes over from it, wait for stage g's bank rows and arrive on full[g]
      // (stage g is then complete); then copy the rows stage g+1 takes over from stage g-1
      // (before full[g+1], in the next iteration), write stage g-1's dirty rows back, and
      // fetch the row lists of stage g+3 and the rows of stage g+2 into buffer g-1.
      // Group order: A(g) = row lists of stage g+3, R(g) = stage g+2's rows.
      for (int g = 0; g < 3 && g < S; ++g) fetch_lrec(g);
      cp_async_commit();
      cp_async_wait_all();
      loader_bar();
      for (int g = 0; g < 2; ++g) {
        if (g < S) {
          fetch_rows(g);
          fetch_stage_data(g);
        }
        cp_async_commit();                                       // R(-2), R(-1)
      }
      bool alive = true;
      for (int g = 0; g < S; ++g) {
        if (g + 3 < S) fetch_lrec(g + 3);
        cp_async_commit();                                       // A(g)
        if (g >= 1) {
          alive = wait_done(g - 1);
          if (!alive) break;
          hand_on_rows(g - 1, false);
          cp_async_wait_pending<3>();                            // R(g-2): stage g's rows
        } else {
          cp_async_wait_pending<2>();                            // R(-2): stage 0's rows
        }
        loader_bar();                                            // carries and rows of stage g in place
        if (lt == 0) mbar_arrive(&full[g % kRowBufs]);
        if (g >= 1) {
          hand_on_rows(g - 1, true);
          write_back(g - 1);
        }
        cp_async_wait_pending<2>();                              // A(g-1): row lists of stage g+2
        loader_bar();                                            // buffer g-1 read; lists visible
        if (g + 2 < S) {
          fetch_rows(g + 2);
          fetch_stage_data(g + 2);
        }
        cp_async_commit();                                       // R(g)
      }
      if (alive && wait_done(S - 1)) write_back(S - 1);
      cp_async_wait_all();
    } else {
    // prologue: row lists 0..2, then the bank rows of stages 0 and 1
    for (int g = 0; g < 3 && g < S; ++g) fetch_lrec(g);
    cp_async_commit();
    cp_async_wait_all();
    loader_bar();
    for (int g = 0; g < 2; ++g) {
      if (g < S) {
        fetch_rows(g);
        fetch_stage_data(g);
      }
      cp_async_commit();
    }
    cp_async_wait_pending<1>();                                  // stage 0 landed
    loader_bar();
    if (lt == 0) mbar_arrive(&full[0]);

    // Iteration g.  Group order: A(g) = row lists of stage g+3, R(g) = stage g+2's rows.
    bool alive = true;
    for (int g = 0; g < S; ++g) {
      if (g + 3 < S) fetch_lrec(g + 3);
      cp_async_commit();                                         // A(g)
      if (g >= 1) {
        alive = wait_done(g - 1);
        if (!alive) break;
        write_back(g - 1);
      }
      cp_async_wait_pending<2>();                                // A(g-1): row lists of stage g+2
      loader_bar();                                              // write-back reads done; lists visible
      if (g + 1 < S && lt == 0) mbar_arrive(&recs[g % kRowBufs]);
      if (g + 2 < S) {
        fetch_rows(g + 2);
        fetch_stage_data(g + 2);
      }
      cp_async_commit();                                         // R(g)
      cp_async_wait_pending<1>();                                // R(g-1): stage g+1 landed
      loader_bar();
      if (g + 1 < S && lt == 0) mbar_arrive(&full[(g + 1) % kRowBufs]);
    }
    if (alive && wait_done(S - 1)) write_back(S - 1);
    cp_async_wait_all();
    }
    return;
  }

  // -------------------------------------------------------------------- compute warps
  const int rg = lane >> 1, c = lane & 1;
  const uint32_t wc = ((uint32_t)warp << 5) | ((uint32_t)c << 4);
  const int col = warp * PC + c * VEC;                           // this lane's first column in the slice
  const bool lane_valid = (2 * warp + c) < valid_chunks;
  ACT *y = static_cast<ACT *>(a.y);
  // The snapshot of this warp's piece: rows of one token contiguous, [T][P][W][PC].
  const bool snap_on = a.snap != nullptr;
  const int snap_elem = a.snap_bf16 ? 2 : 4;
  const int64_t snap_pcs = (int64_t)PC * snap_elem;                // bytes of one row piece
  const int64_t snap_row_step = (int64_t)W * snap_pcs;             // one (token, piece)
  const int64_t snap_tok_step = (int64_t)a.pieces * snap_row_step; // one token
  const int piece = slice * NCW + warp;
  const int64_t snap_lane = (int64_t)c * VEC * snap_elem;
  auto snap_store = [&](unsigned char *dst, const uint4 &raw) {
    dst += snap_lane;
    if constexpr (sizeof(BANK) == 4) {
      if (a.snap_bf16) {
        float x[VEC];
        PieceRow<BANK>::unpack(raw, x);
        store_vec<__nv_bfloat16, VEC>(reinterpret_cast<__nv_bfloat16 *>(dst), x);
      } else {
        *reinterpret_cast<uint4 *>(dst) = raw;
      }
    } else {
      if (a.snap_bf16) {
        *reinterpret_cast<uint4 *>(dst) = raw;
      } else {
        float x[VEC];
        PieceRow<BANK>::unpack(raw, x);
        store_vec<float, VEC>(reinterpret_cast<float *>(dst), x);
      }
    }
  };
  const int64_t ystep = (int64_t)a.H * a.d_v;
  // every lane waits (and acquires what the barrier publishes); the warp gives up as one.
  // (Letting lane 0 spin alone and the others check once measured ten times slower token
  // steps afterwards on GB300, so every lane spins.)
  auto wait_bar = [&](uint64_t *bar, int g) -> bool {
    const bool ok = __all_sync(0xffffffffu, wait_phase(&bar[g % kRowBufs], (uint32_t)(g / kRowBufs) & 1u,
                                                       abort_flag));
    if (!ok && lane == 0) {
      if (!*abort_flag) raise_error(a.err, SDM_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
    return ok;
  };
  // Rows this stage hands on (its own record's out list, visible since the end of stage
  // g-1): {o_dst | o_src << 16}; the first 32 entries are read into registers at the
  // stage's start, two per lane pair, so the copies at its end cost one round trip.
  struct Handoff {
    int n1 = 0, n2 = 0;
    uint32_t e[2] = {0, 0};
  };
  auto handoff_of = [&](int g) -> Handoff {
    Handoff hf;
    const unsigned char *rec = lrecbuf(g);
    const int32_t *hdr = reinterpret_cast<const int32_t *>(rec);
    const bool ok = hdr[0] >= 0 && hdr[0] <= L && hdr[2] >= 0 && hdr[3] >= 0 && hdr[2] + hdr[3] <= hdr[0];
    if (!ok) return hf;
    hf.n1 = hdr[2];
    hf.n2 = hdr[3];
    const uint2 *out = reinterpret_cast<const uint2 *>(rec + lay.off_out);
    if (rg < hf.n1 + hf.n2) hf.e[0] = out[rg].x;
    if (rg + 16 < hf.n1 + hf.n2) hf.e[1] = out[rg + 16].x;
    return hf;
  };
  auto copy_piece = [&](uint32_t cv, unsigned char *to, const unsigned char *from) {
    const uint32_t od = (cv & 0xffffu) ^ wc, os = (cv >> 16) ^ wc;
    if (od >= (uint32_t)row_limit || os >= (uint32_t)row_limit) {
      raise_error(a.err, SDM_DEVERR_PLAN);
      return;
    }
    *reinterpret_cast<uint4 *>(to + od) = *reinterpret_cast<const uint4 *>(from + os);
  };
  // Entries a compute lane copies together: 1 where the launch caps registers at 128 (512
  // threads per SM), where the batch's registers measured as spills in the token step.
  constexpr int HB = Geo::NTHR * (LW == 4 ? 2 : 1) >= 512 ? 1 : kBatch;
  auto hand_on = [&](int g, const Handoff &hf) {
    const unsigned char *rows = rowbuf(g);
    const uint2 *out = reinterpret_cast<const uint2 *>(lrecbuf(g) + lay.off_out);
    const int n = hf.n1 + hf.n2;
    for (int e = rg, k = 0; e < n && k < 2; e += 16, ++k)
      copy_piece(hf.e[k], e < hf.n1 ? rowbuf(g + 1) : rowbuf(g + 2), rows);
    // the rest HB entries at a time: offsets, then the pieces, then the stores
    for (int e0 = rg + 32; e0 < n; e0 += HB * 16) {
      uint32_t cv[HB];
      uint4 r[HB];
#pragma unroll
      for (int k = 0; k < HB; ++k) cv[k] = e0 + 16 * k < n ? out[e0 + 16 * k].x : 0u;
#pragma unroll
      for (int k = 0; k < HB; ++k) {
        const uint32_t os = (cv[k] >> 16) ^ wc;
        if (e0 + 16 * k < n && os < (uint32_t)row_limit) r[k] = *reinterpret_cast<const uint4 *>(rows + os);
      }
#pragma unroll
      for (int k = 0; k < HB; ++k) {
        const int e = e0 + 16 * k;
        if (e >= n) break;
        const uint32_t od = (cv[k] & 0xffffu) ^ wc, os = (cv[k] >> 16) ^ wc;
        if (od >= (uint32_t)row_limit || os >= (uint32_t)row_limit) {
          raise_error(a.err, SDM_DEVERR_PLAN);
          continue;
        }
        *reinterpret_cast<uint4 *>((e < hf.n1 ? rowbuf(g + 1) : rowbuf(g + 2)) + od) = r[k];
      }
    }
  };
  for (int g = 0; g < S; ++g) {
    if (!wait_bar(full, g)) return;
    const Handoff hf = kLoaderHandOn ? Handoff{} : handoff_of(g);
    const unsigned char *cr = crecbuf(g);
    const uint16_t *refmap = reinterpret_cast<const uint16_t *>(cr + lay.off_refmap);
    const uint8_t *tokflag = cr + lay.off_tokflag;
    const float *wts = reinterpret_cast<const float *>(cr + lay.off_wts);
    const float *gt = reinterpret_cast<const float *>(cr + lay.off_gates);
    const ACT *vv = reinterpret_cast<const ACT *>(tokbuf(g));
    unsigned char *rows = rowbuf(g);
    const int64_t t0 = (int64_t)g * G;
    const int nt = (int)min((int64_t)G, a.T - t0);
    ACT *ybase = y + ((b * a.T + t0) * a.H + h) * a.d_v + c0 + col;
    unsigned char *snap_tok = snap_on ? a.snap + ((s * a.T + t0) * a.pieces + piece) * snap_row_step : nullptr;
    for (int t = 0; t < nt; ++t) {
      float v[VEC], out[VEC];
      load_vec<ACT, VEC>(vv + t * COLS + col, v);
      const float2 ab = *reinterpret_cast<const float2 *>(gt + 2 * t);
      piece_token<BANK, JB, FULL>(W, R, refmap + t * WR, wts + t * WR, ab.x, ab.y, v, rows, wc, tokflag[t] != 0,
                                  out, [&](int j, const uint4 &raw) {
                                    if (snap_on && lane_valid) snap_store(snap_tok + (int64_t)j * snap_pcs, raw);
                                  });
      if (snap_on) snap_tok += snap_tok_step;
      if (rg == 0 && lane_valid) store_vec<ACT, VEC>(ybase + t * ystep, out);
      __syncwarp();
    }
    // rows the next two stages take over: copy this warp's pieces out of buffer g (into
    // buffer g+2 only once the loaders have written back stage g-1 from it: recs(g))
    if (!kLoaderHandOn && g + 1 < S) {
      if (!wait_bar(recs, g)) return;
      hand_on(g, hf);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&done[g % kRowBufs]);
  }
}

// Launches the instance for the shape: W = R = 64 fixed at compile time, else up to 8
// rows per lane and sum (W, R <= 128).
template <typename BANK, typename ACT, int NCW, int LW>
cudaError_t launch_ncw_lw(const WriteReadArgs &a, int64_t streams, int64_t smem, cudaStream_t st) {
  const dim3 grid((unsigned)a.slices, (unsigned)streams);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, WrGeometry<NCW, LW>::NTHR, smem, st>>>(a);
    return cudaGetLastError();
  };
  if (a.W == 64 && a.R == 64) return go(write_read_kernel<BANK, ACT, NCW, 4, true, LW>);
  if (a.W <= 128 && a.R <= 128) return go(write_read_kernel<BANK, ACT, NCW, 8, false, LW>);
  return cudaErrorInvalidValue;
}

template <typename BANK, typename ACT>
cudaError_t launch_types(const WriteReadArgs &a, int64_t streams, const WriteReadLaunch &l, cudaStream_t st) {
  if (l.NCW == 4 && l.LW == 8) return launch_ncw_lw<BANK, ACT, 4, 8>(a, streams, l.smem_bytes, st);
  if (l.NCW == 4 && l.LW == 4) return launch_ncw_lw<BANK, ACT, 4, 4>(a, streams, l.smem_bytes, st);
  if (l.NCW == 8 && l.LW == 8) return launch_ncw_lw<BANK, ACT, 8, 8>(a, streams, l.smem_bytes, st);
  if (l.NCW == 1 && l.LW == 8) return launch_ncw_lw<BANK, ACT, 1, 8>(a, streams, l.smem_bytes, st);
  if (l.NCW == 1 && l.LW == 4) return launch_ncw_lw<BANK, ACT, 1, 4>(a, streams, l.smem_bytes, st);
  return cudaErrorInvalidValue;
}

}  // namespace wr
}  // namespace sdm
