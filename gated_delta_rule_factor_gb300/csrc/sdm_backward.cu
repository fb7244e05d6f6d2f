// The backward of the write/read op: gradients of a scalar loss L with respect to the
// initial bank, the values, the gates (alpha, beta), both queries and the sub-keys,
// deterministic (no float atomics: every sum runs in a fixed order) and restoring the
// bank in place from the forward's snapshot (sparse-delta-memory CHANGELOG > 2.0.0 >
// New: deterministic sparse backward; > Behavior changes: the first backward restores
// the bank in place; > Package: bf16 snapshots).
//
// The chain rule through one token (alpha, beta, value v, write rows X_j = M[i_j] before
// the write, m_j = alpha X_j, p = sum_j w_j m_j, u = v - p, M'[i_j] = m_j + beta w_j u,
// read y = sum_j r_j M'[i^r_j]), with G = dL/dM' over the whole table and dy = dL/dy:
//   read:  dr_j = <dy, M'[i^r_j]>;   G[i^r_j] += r_j dy
//   write: G_j = G[i_j];  dv = beta sum_j w_j G_j;  dp = -dv;  dm_j = G_j + w_j dp
//          dw_j = beta <G_j, u> + <dp, m_j>;  dbeta = sum_j w_j <G_j, u>
//          dalpha = sum_j <dm_j, X_j>;  G[i_j] <- alpha dm_j;  M[i_j] <- X_j (restore)
//   softmax: dS_j = w_j (dw_j - sum_k w_k dw_k)  (the same for the read weights)
//   scores:  ds_f[a] = sum of dS_j over the selected slots whose factor-f index is a;
//            dq_f = sum_a ds_f[a] K_f[a],  dK_f[a] += ds_f[a] q_f.
// Tokens are taken from last to first, so the bank always holds the state after the
// token being undone.  Every per-column quantity (G, dv, u) depends on its own column
// only; the sums over columns (dr_j, dw_j, dalpha, dbeta) feed nothing back into the
// sweep.  So the sweep splits the columns over independent warps, each of which writes
// its partial column sums, and a second kernel adds the partials in a fixed order.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kSweepWarps = kSweepCtaWarps;      // warps per CTA of the sweep (adjacent pieces of the rows)
// The CTA's warps add their partial column sums in shared memory (in warp order, once per
// token, behind a CTA barrier) and store one record per CTA instead of one per warp.
constexpr bool kSweepCombine = kSweepCtaRecord;
constexpr int kPartMax = (2 * SDM_MAX_K + 2 + 3) & ~3;   // the largest partial record (floats)
// 16-byte stage slots per lane: JB snapshot rows (two slots each), JB read rows and the
// float32 G of the read and write rows (VEC / 4 slots each)
__host__ __device__ constexpr int sweep_slots(int JB, int VEC) { return JB * (3 + 2 * (VEC / 4)); }
constexpr int kReduceWarps = 4;
constexpr int kFlagWarps = kThreads / 32;

// ---------------------------------------------------------------- read-after-write flags

// flags[s*T + t] = 1 when token t of stream s reads a row it also writes: the sweep then
// orders the read's gradient update before the write's loads of the same rows.
__global__ void __launch_bounds__(kThreads) bwd_flags_kernel(const __grid_constant__ BackwardArgs a) {
  __shared__ int32_t wids[kFlagWarps][SDM_MAX_K];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows = a.B * a.T * a.H;
  for (int64_t r = (int64_t)blockIdx.x * kFlagWarps + warp; r < rows; r += (int64_t)gridDim.x * kFlagWarps) {
    const int32_t *iw = a.idx[0] + r * a.W, *ir = a.idx[1] + r * a.R;
    for (int j = lane; j < a.W; j += 32) wids[warp][j] = iw[j];
    __syncwarp();
    bool hit = false;
    for (int j = lane; j < a.R; j += 32) {
      const int32_t x = ir[j];
      for (int i = 0; i < a.W; ++i) hit |= wids[warp][i] == x;
    }
    const bool any = __any_sync(0xffffffffu, hit);
    if (lane == 0) {
      const int64_t h = r % a.H, bt = r / a.H, b = bt / a.T, t = bt % a.T;
      a.flags[(b * a.H + h) * a.T + t] = any ? 1 : 0;
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- sweep

template <int V>
__device__ __forceinline__ void load_f32v(const float *p, float (&o)[V]) {
#pragma unroll
  for (int i = 0; i < V; i += 4) {
    const float4 x = __ldcg(reinterpret_cast<const float4 *>(p + i));
    o[i] = x.x;
    o[i + 1] = x.y;
    o[i + 2] = x.z;
    o[i + 3] = x.w;
  }
}

template <int V>
__device__ __forceinline__ void store_f32v(float *p, const float (&x)[V]) {
#pragma unroll
  for (int i = 0; i < V; i += 4) *reinterpret_cast<float4 *>(p + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
}

template <int V>
__device__ __forceinline__ void load_act(const void *base, int64_t e, bool bf16, float (&o)[V]) {
  if (bf16) load_vec<__nv_bfloat16, V>(static_cast<const __nv_bfloat16 *>(base) + e, o);
  else load_vec<float, V>(static_cast<const float *>(base) + e, o);
}

// The sum over the row blocks of a warp (the lane bits above the column group's), a
// balanced tree in block order.
template <int CG, int V>
__device__ __forceinline__ void row_block_sum(float (&x)[V]) {
#pragma unroll
  for (int o = CG; o < 32; o <<= 1)
#pragma unroll
    for (int c = 0; c < V; ++c) x[c] = __fadd_rn(x[c], __shfl_xor_sync(0xffffffffu, x[c], o));
}

// This lane's rows of one selection of token row r: block rg of ceil(n / RG) rows (RG row
// groups per warp).  FULL: n == 64, JB = 64 / RG rows read as vectors.  A slot id
// outside [0, N) is reported and its row skipped.
template <int RG, int JB, bool FULL>
struct LaneRefs {
  int32_t idx[JB];
  float w[JB];
  int j0, nb;
  __device__ __forceinline__ void load(const int32_t *ids, const float *wts, int n, int rg) {
    if constexpr (FULL) {
      static_assert(JB * RG == 64 && (JB == 2 || JB == 4), "FULL lanes hold 2 or 4 rows");
      j0 = JB * rg;
      nb = JB;
      if constexpr (JB == 4) {
        const int4 i4 = *reinterpret_cast<const int4 *>(ids + j0);
        const float4 w4 = *reinterpret_cast<const float4 *>(wts + j0);
        idx[0] = i4.x;
        idx[1] = i4.y;
        idx[2] = i4.z;
        idx[3] = i4.w;
        w[0] = w4.x;
        w[1] = w4.y;
        w[2] = w4.z;
        w[3] = w4.w;
      } else {
        const int2 i2 = *reinterpret_cast<const int2 *>(ids + j0);
        const float2 w2 = *reinterpret_cast<const float2 *>(wts + j0);
        idx[0] = i2.x;
        idx[1] = i2.y;
        w[0] = w2.x;
        w[1] = w2.y;
      }
    } else {
      const int bk = (n + RG - 1) / RG;
      j0 = rg * bk;
      nb = min(bk, max(n - j0, 0));
#pragma unroll
      for (int s = 0; s < JB; ++s) {
        idx[s] = s < nb ? ids[j0 + s] : 0;
        w[s] = s < nb ? wts[j0 + s] : 0.0f;
      }
    }
  }
  __device__ __forceinline__ bool has(int s, int64_t N) const {
    return (FULL || s < nb) && idx[s] >= 0 && (int64_t)idx[s] < N;
  }
};

template <int RG, int JB, bool FULL>
struct TokenRefs {
  LaneRefs<RG, JB, FULL> wr, rd;
  float2 ab;
  int flag;
};

// One warp per (stream, piece p of CG 16-byte column groups of every bank row): lane =
// CG*rg + c, c picks the column group (VEC columns), rg (RG = 32 / CG of them) a block of
// consecutive rows of each sum.  The warp runs the stream's tokens from last to first on
// its columns alone; its global-memory traffic is ordered by __syncwarp between
// dependent phases (the bank and G entries of one column are only ever touched by this
// warp).  The snapshot is read in the forward's layout (32-byte pieces).
template <typename BANK, int CG, int JB, bool FULL>
__global__ void __launch_bounds__(32 * kSweepWarps) bwd_sweep_kernel(const __grid_constant__ BackwardArgs a) {
  constexpr int VEC = 16 / (int)sizeof(BANK);
  constexpr int RG = 32 / CG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p = blockIdx.x * kSweepWarps + warp;    // this warp's column piece
  const int64_t s = blockIdx.y;
  if (*a.snap_hdr != kSnapshotArmed) {          // no snapshot to undo: touch nothing
    if (lane == 0 && p == 0) raise_error(a.err, SDM_DEVERR_SNAPSHOT);
    return;
  }
  if (!kSweepCombine && p >= a.Pw) return;       // (with the combine, idle warps add zeros)
  const int W = FULL ? 64 : a.W, R = FULL ? 64 : a.R;
  const int rg = lane / CG, c = lane % CG;
  const int64_t col = ((int64_t)p * CG + c) * VEC;
  const bool valid = col < a.d_v;               // false for a whole warp past the last piece
  const int64_t b = s / a.H, h = s % a.H;
  const int64_t N = a.N, d_v = a.d_v;
  BANK *bank = static_cast<BANK *>(a.bank) + s * N * d_v + col;
  float *grad = a.grad + s * N * d_v + col;
  const bool sbf = a.snap_bf16 != 0;
  const int se = sbf ? 2 : 4;
  const int64_t pcs = 2 * VEC * se;                  // snapshot bytes of a row's 32-byte piece
  const int64_t p32 = col / (2 * VEC), half = (col / VEC) & 1;
  const unsigned char *snap_sp = a.snap + ((s * a.T) * a.P32 + p32) * (int64_t)W * pcs + half * VEC * se;
  const int64_t snap_tstep = (int64_t)a.P32 * W * pcs;
  const bool abf = a.act_bf16 != 0;
  __shared__ __align__(16) float comb[2][kSweepWarps][kPartMax];
  // stage slots of a lane (16-byte chunks): snapshot rows (2 each), read rows, their G
  // (GC each), write rows' G (GC each)
  constexpr int GC = VEC / 4;
  extern __shared__ __align__(16) unsigned char sweep_smem[];
  unsigned char *stg = sweep_smem + ((int64_t)warp * sweep_slots(JB, VEC) * 32 + lane) * 16;
  auto sx = [&](int q, int hh) { return (int64_t)(2 * q + hh) * 512; };
  auto sm_ = [&](int q) { return (int64_t)(2 * JB + q) * 512; };
  auto sgr = [&](int q, int hh) { return (int64_t)(3 * JB + GC * q + hh) * 512; };
  auto sgw = [&](int q, int hh) { return (int64_t)((3 + GC) * JB + GC * q + hh) * 512; };

  auto refs_of = [&](int64_t t) {
    TokenRefs<RG, JB, FULL> k;
    const int64_t r = (b * a.T + t) * a.H + h;
    k.wr.load(a.idx[0] + r * W, a.wt[0] + r * W, W, rg);
    k.rd.load(a.idx[1] + r * R, a.wt[1] + r * R, R, rg);
    k.ab = *reinterpret_cast<const float2 *>(a.gates + 2 * r);
    k.flag = a.flags[s * a.T + t];
    return k;
  };

  TokenRefs<RG, JB, FULL> cur = refs_of(a.T - 1);
  for (int64_t t = a.T - 1; t >= 0; --t) {
    const TokenRefs<RG, JB, FULL> nxt = t > 0 ? refs_of(t - 1) : cur;
    const int64_t r = (b * a.T + t) * a.H + h;
    const LaneRefs<RG, JB, FULL> &wr_ = cur.wr, &rd = cur.rd;
    bool bad = false;
    float dyv[VEC], vv[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) dyv[i] = vv[i] = 0.0f;
    if (valid) {
      load_act<VEC>(a.dy, r * d_v + col, abf, dyv);
      load_act<VEC>(a.k_val, r * d_v + col, abf, vv);
    }
    // rows before the write (the snapshot), and the read rows after it with their G: in
    // through cp.async into this lane's stage slots ([slot][lane] 16-byte chunks; plain
    // 16-byte register gathers measured slower, held back by how many a warp keeps in
    // flight), then into registers
    float xw[JB][VEC], mr[JB][VEC], gr[JB][VEC], gw[JB][VEC];
    const unsigned char *snap_t = snap_sp + t * snap_tstep;
#pragma unroll
    for (int q = 0; q < JB; ++q)
#pragma unroll
      for (int i = 0; i < VEC; ++i) xw[q][i] = mr[q][i] = gr[q][i] = gw[q][i] = 0.0f;
    // the token's rows come in through cp.async into this lane's slots of the stage
    // area ([slot][lane] 16-byte chunks), then into registers
    const int xbytes = VEC * se;
#pragma unroll
    for (int q = 0; q < JB; ++q) {
      if (valid && wr_.has(q, N)) {
        const unsigned char *sp = snap_t + (int64_t)(wr_.j0 + q) * pcs;
        if (xbytes == 8) cp_async8(stg + sx(q, 0), sp);
        else {
          cp_async16(stg + sx(q, 0), sp);
          if (xbytes == 32) cp_async16(stg + sx(q, 1), sp + 16);
        }
        if (!cur.flag)
#pragma unroll
          for (int hh = 0; hh < GC; ++hh) cp_async16(stg + sgw(q, hh), grad + (int64_t)wr_.idx[q] * d_v + 4 * hh);
      }
      if (valid && rd.has(q, N)) {
        cp_async16(stg + sm_(q), bank + (int64_t)rd.idx[q] * d_v);
#pragma unroll
        for (int hh = 0; hh < GC; ++hh) cp_async16(stg + sgr(q, hh), grad + (int64_t)rd.idx[q] * d_v + 4 * hh);
      }
    }
    cp_async_commit();
    cp_async_wait_all();
#pragma unroll
    for (int q = 0; q < JB; ++q) {
      if (valid && wr_.has(q, N)) {
        if (sbf) load_vec<__nv_bfloat16, VEC>(reinterpret_cast<const __nv_bfloat16 *>(stg + sx(q, 0)), xw[q]);
        else if (VEC == 4) load_vec<float, VEC>(reinterpret_cast<const float *>(stg + sx(q, 0)), xw[q]);
        else {
          float lo[4], hi[4];
          load_vec<float, 4>(reinterpret_cast<const float *>(stg + sx(q, 0)), lo);
          load_vec<float, 4>(reinterpret_cast<const float *>(stg + sx(q, 1)), hi);
#pragma unroll
          for (int i = 0; i < 4 && i + 4 < VEC + 4; ++i) {
            xw[q][i] = lo[i];
            if (i + 4 < VEC) xw[q][i + 4] = hi[i];
          }
        }
        if (!cur.flag)
#pragma unroll
          for (int hh = 0; hh < GC; ++hh) {
            float x4[4];
            load_vec<float, 4>(reinterpret_cast<const float *>(stg + sgw(q, hh)), x4);
#pragma unroll
            for (int i = 0; i < 4; ++i) gw[q][4 * hh + i] = x4[i];
          }
      }
      if (valid && rd.has(q, N)) {
        load_vec<BANK, VEC>(reinterpret_cast<const BANK *>(stg + sm_(q)), mr[q]);
#pragma unroll
        for (int hh = 0; hh < GC; ++hh) {
          float x4[4];
          load_vec<float, 4>(reinterpret_cast<const float *>(stg + sgr(q, hh)), x4);
#pragma unroll
          for (int i = 0; i < 4; ++i) gr[q][4 * hh + i] = x4[i];
        }
      }
    }

    auto load_write_grads = [&] {
#pragma unroll
      for (int q = 0; q < JB; ++q)
        if (valid && wr_.has(q, N)) load_f32v<VEC>(grad + (int64_t)wr_.idx[q] * d_v, gw[q]);
    };
    // read: dr_j = <dy, M'[i^r_j]>, G[i^r_j] += r_j dy
    float drp[JB];
#pragma unroll
    for (int q = 0; q < JB; ++q) {
      drp[q] = 0.0f;
      if (!rd.has(q, N)) {
        if (!FULL && q < rd.nb) bad = true;
        continue;
      }
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        drp[q] = __fmaf_rn(dyv[i], mr[q][i], drp[q]);
        gr[q][i] = __fmaf_rn(rd.w[q], dyv[i], gr[q][i]);
      }
      if (valid) store_f32v<VEC>(grad + (int64_t)rd.idx[q] * d_v, gr[q]);
    }
    if (cur.flag) {                                 // the write's rows see the read's update
      __syncwarp();
      load_write_grads();
    }
    // write: p = sum_j w_j (alpha X_j) and sum_j w_j G_j over the token's W rows
    const float alpha = cur.ab.x, beta = cur.ab.y;
    float sp_[VEC], sg[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) sp_[i] = sg[i] = 0.0f;
#pragma unroll
    for (int q = 0; q < JB; ++q) {
      if (!wr_.has(q, N)) {
        if (!FULL && q < wr_.nb) bad = true;
        continue;
      }
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        sp_[i] = __fmaf_rn(wr_.w[q], __fmul_rn(alpha, xw[q][i]), sp_[i]);
        sg[i] = __fmaf_rn(wr_.w[q], gw[q][i], sg[i]);
      }
    }
    row_block_sum<CG, VEC>(sp_);
    row_block_sum<CG, VEC>(sg);
    float dv[VEC], u[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      dv[i] = __fmul_rn(beta, sg[i]);
      u[i] = __fsub_rn(vv[i], sp_[i]);
    }
    float dwp[JB];
    float dap = 0.0f, dbp = 0.0f;
#pragma unroll
    for (int q = 0; q < JB; ++q) {
      dwp[q] = 0.0f;
      if (!wr_.has(q, N)) continue;
      float gu = 0.0f, dpm = 0.0f, gn[VEC];
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const float dm = __fmaf_rn(-wr_.w[q], dv[i], gw[q][i]);          // G_j + w_j dp
        gu = __fmaf_rn(gw[q][i], u[i], gu);
        dpm = __fmaf_rn(-dv[i], __fmul_rn(alpha, xw[q][i]), dpm);         // <dp, m_j>
        dap = __fmaf_rn(dm, xw[q][i], dap);
        gn[i] = __fmul_rn(alpha, dm);
      }
      dwp[q] = __fmaf_rn(beta, gu, dpm);
      dbp = __fmaf_rn(wr_.w[q], gu, dbp);
      if (valid) {
        store_f32v<VEC>(grad + (int64_t)wr_.idx[q] * d_v, gn);
        store_vec<BANK, VEC>(bank + (int64_t)wr_.idx[q] * d_v, xw[q]);
      }
    }
    if (rg == 0 && valid) store_f32v<VEC>(a.d_kv + r * d_v + col, dv);
    // partial column sums of this piece: the row sums over its two halves, dalpha and
    // dbeta over the whole warp (a fixed butterfly)
#pragma unroll
    for (int o = 1; o < CG; o <<= 1)
#pragma unroll
      for (int q = 0; q < JB; ++q) {
        dwp[q] = __fadd_rn(dwp[q], __shfl_xor_sync(0xffffffffu, dwp[q], o));
        drp[q] = __fadd_rn(drp[q], __shfl_xor_sync(0xffffffffu, drp[q], o));
      }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      dap = __fadd_rn(dap, __shfl_xor_sync(0xffffffffu, dap, o));
      dbp = __fadd_rn(dbp, __shfl_xor_sync(0xffffffffu, dbp, o));
    }
    // this warp's record: its own slot of the part buffer, or its row of the CTA's
    // shared-memory buffer (two, alternating by token, so one barrier a token suffices)
    float *pp = kSweepCombine ? comb[t & 1][warp] : a.part + ((s * a.T + t) * a.P + p) * (int64_t)a.PS;
    if constexpr (FULL && JB == 4) {
      if (c == 0) *reinterpret_cast<float4 *>(pp + wr_.j0) = make_float4(dwp[0], dwp[1], dwp[2], dwp[3]);
      if (c == CG - 1) *reinterpret_cast<float4 *>(pp + W + rd.j0) = make_float4(drp[0], drp[1], drp[2], drp[3]);
    } else if constexpr (FULL && JB == 2) {
      if (c == 0) *reinterpret_cast<float2 *>(pp + wr_.j0) = make_float2(dwp[0], dwp[1]);
      if (c == CG - 1) *reinterpret_cast<float2 *>(pp + W + rd.j0) = make_float2(drp[0], drp[1]);
    } else {
      if (c == 0) {
#pragma unroll
        for (int q = 0; q < JB; ++q)
          if (q < wr_.nb) pp[wr_.j0 + q] = dwp[q];
      }
      if (c == CG - 1) {
#pragma unroll
        for (int q = 0; q < JB; ++q)
          if (q < rd.nb) pp[W + rd.j0 + q] = drp[q];
      }
    }
    if (lane == 0) {
      pp[W + R] = dap;
      pp[W + R + 1] = dbp;
    }
    if (FULL) {
#pragma unroll
      for (int q = 0; q < JB; ++q) bad |= !wr_.has(q, N) || !rd.has(q, N);
    }
    if (bad) raise_error(a.err, SDM_DEVERR_SLOT_RANGE);
    if constexpr (kSweepCombine) {
      // every warp's record is in shared memory and its global stores are ordered before
      // the next token's loads (the barrier orders the CTA's memory traffic); the CTA's
      // threads then add the records in warp order and store the CTA's one
      named_barrier(1, 32 * kSweepWarps);
      const int n_tot = W + R + 2;
      float *dst = a.part + ((s * a.T + t) * a.P + blockIdx.x) * (int64_t)a.PS;
      for (int v = threadIdx.x; v < n_tot; v += 32 * kSweepWarps) {
        float acc = comb[t & 1][0][v];
#pragma unroll
        for (int w = 1; w < kSweepWarps; ++w) acc = __fadd_rn(acc, comb[t & 1][w][v]);
        dst[v] = acc;
      }
    } else {
      __syncwarp();                                 // this token's stores before the next one's loads
    }
    cur = nxt;
  }
}

// ---------------------------------------------------------------- reduction

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float load_act1(const void *base, int64_t e, bool bf16) {
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[e]) : static_cast<const float *>(base)[e];
}

// Eight consecutive elements of an activation row (16 bytes of bfloat16, 32 of float32).
__device__ __forceinline__ void load_act8(const void *base, int64_t e, bool bf16, float (&o)[8]) {
  if (bf16) load_vec<__nv_bfloat16, 8>(static_cast<const __nv_bfloat16 *>(base) + e, o);
  else load_vec<float, 8>(static_cast<const float *>(base) + e, o);
}

// One warp per token row r = (b*T + t)*H + h.
__global__ void __launch_bounds__(32 * kReduceWarps, 4) bwd_reduce_kernel(const __grid_constant__ BackwardArgs a) {
  __shared__ float tot[kReduceWarps][2 * SDM_MAX_K + 4];
  __shared__ float dsrow[kReduceWarps][SDM_MAX_FACTOR_DIM];
  __shared__ int32_t nz[kReduceWarps][SDM_MAX_K];
  constexpr int kJ = SDM_MAX_K / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows = a.B * a.T * a.H, BT = a.B * a.T;
  const int W = a.W, R = a.R, n_tot = W + R + 2;
  const KeyGeometry &g = a.g;
  const int d_sub = g.d_sub;
  const bool abf = a.act_bf16 != 0;
  const bool vec8 = (d_sub % 8) == 0;
  for (int64_t r = (int64_t)blockIdx.x * kReduceWarps + warp; r < rows; r += (int64_t)gridDim.x * kReduceWarps) {
    const int64_t h = r % a.H, bt = r / a.H, b = bt / a.T, t = bt % a.T, s = b * a.H + h;
    // 1. the per-piece partial sums, added in piece order
    const float *pp = a.part + (s * a.T + t) * (int64_t)a.P * a.PS;
    for (int v = lane; v < n_tot; v += 32) {
      float acc = 0.0f;
#pragma unroll 8
      for (int p = 0; p < a.P; ++p) acc = __fadd_rn(acc, pp[(int64_t)p * a.PS + v]);
      tot[warp][v] = acc;
    }
    __syncwarp();
    if (lane == 0) {
      a.d_gates[2 * r] = tot[warp][W + R];
      a.d_gates[2 * r + 1] = tot[warp][W + R + 1];
    }
    for (int kind = 0; kind < 2; ++kind) {
      const int k = kind ? R : W;
      const float *wts = a.wt[kind] + r * k;
      const int32_t *ids = a.idx[kind] + r * k;
      const float *dw = tot[warp] + (kind ? W : 0);
      // 2. softmax backward: dS_j = w_j (dw_j - sum_k w_k dw_k); lane holds j = 32 i + lane
      float sw = 0.0f;
      for (int j = lane; j < k; j += 32) sw = __fmaf_rn(wts[j], dw[j], sw);
      sw = warp_sum(sw);
      float dSj[kJ];
      int32_t idj[kJ];
#pragma unroll
      for (int i = 0; i < kJ; ++i) {
        const int j = lane + 32 * i;
        dSj[i] = j < k ? __fmul_rn(wts[j], __fsub_rn(dw[j], sw)) : 0.0f;
        idj[i] = j < k ? ids[j] : -1;
      }
      int64_t stride = 1;
      for (int f = g.F - 1; f >= 0; --f) {
        const int n = g.nf[f];
        float *drow = dsrow[warp];
        for (int x = lane; x < n; x += 32) drow[x] = 0.0f;
        __syncwarp();
        // 3. ds_f[x] = sum of dS_j over the slots whose factor-f index is x, in a fixed
        // order: within each group of 32 slots (j = 32 i + lane) the slots sharing x are
        // added in lane order by the first of them, and the groups in increasing i.
#pragma unroll
        for (int i = 0; i < kJ; ++i) {
          if (32 * i < k) {
            const int32_t id = idj[i];
            const bool in = id >= 0 && (int64_t)id < a.N;
            const int x = in ? (int)(((int64_t)id / stride) % n) : -1 - lane;   // a bad slot stays alone
            const unsigned grp = __match_any_sync(0xffffffffu, x);
            float sum = 0.0f;
            for (unsigned m = grp; m; m &= m - 1) sum = __fadd_rn(sum, __shfl_sync(grp, dSj[i], __ffs(m) - 1));
            if (in && __ffs(grp) - 1 == lane) drow[x] = __fadd_rn(drow[x], sum);
            __syncwarp();
          }
        }
        // the dense row for the sub-key gradient, and the indices with a nonzero ds, ascending
        float *dsg = a.ds + ((h * 2 + kind) * BT + bt) * (int64_t)g.ntot + g.off[f];
        int nnz = 0;
        for (int x0 = 0; x0 < n; x0 += 32) {
          const int x = x0 + lane;
          const float v = x < n ? drow[x] : 0.0f;
          if (x < n) dsg[x] = v;
          const unsigned m = __ballot_sync(0xffffffffu, v != 0.0f);
          if (v != 0.0f) nz[warp][nnz + __popc(m & ((1u << lane) - 1u))] = x;
          nnz += __popc(m);                         // at most k: only selected indices are nonzero
        }
        __syncwarp();
        // 4. dq_f[d] = sum over those indices (ascending) of ds_f[x] K_f[x][d]
        const int64_t krow0 = (h * g.ntot + g.off[f]) * (int64_t)d_sub;
        float *dq = a.d_q[kind] + r * (int64_t)g.F * d_sub + (int64_t)f * d_sub;
        if (vec8) {
          for (int d = 8 * lane; d < d_sub; d += 256) {
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
            for (int q = 0; q < nnz; ++q) {
              const int x = nz[warp][q];
              const float dx = drow[x];
              float kv[8];
              load_act8(a.subkeys, krow0 + (int64_t)x * d_sub + d, abf, kv);
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[e] = __fmaf_rn(dx, kv[e], acc[e]);
            }
            store_f32v<8>(dq + d, acc);
          }
        } else {
          for (int d = lane; d < d_sub; d += 32) {
            float acc = 0.0f;
            for (int q = 0; q < nnz; ++q) {
              const int x = nz[warp][q];
              acc = __fmaf_rn(drow[x], load_act1(a.subkeys, krow0 + (int64_t)x * d_sub + d, abf), acc);
            }
            dq[d] = acc;
          }
        }
        __syncwarp();
        stride *= n;
      }
    }
  }
}

// ---------------------------------------------------------------- sub-key gradient

constexpr int kTileA = 64, kTileD = 64, kTileK = 16;

// Split ks of the tile (a-block, d-block) of head h and factor f:
//   dk_part[ks][h][off_f + x][d] = sum over k in the split, increasing, of
//   ds[h][k][off_f + x] * q_kind[row(k)][f*d_sub + d],  k = kind*BT + bt.
// blockIdx.x enumerates (h, f, a-block, d-block); blockIdx.y = ks.
__global__ void __launch_bounds__(256) bwd_subkey_tiles_kernel(const __grid_constant__ BackwardArgs a) {
  __shared__ __align__(16) float As[kTileK][kTileA];
  __shared__ __align__(16) float Bs[kTileK][kTileD];
  const KeyGeometry &g = a.g;
  const int d_sub = g.d_sub;
  const int td = (d_sub + kTileD - 1) / kTileD;
  int per_head = 0;
  for (int f = 0; f < g.F; ++f) per_head += (g.nf[f] + kTileA - 1) / kTileA * td;
  const int h = blockIdx.x / per_head;
  int rem = blockIdx.x % per_head, f = 0;
  while (rem >= (g.nf[f] + kTileA - 1) / kTileA * td) {
    rem -= (g.nf[f] + kTileA - 1) / kTileA * td;
    ++f;
  }
  const int n = g.nf[f];
  const int a0 = (rem / td) * kTileA, d0 = (rem % td) * kTileD;
  const int64_t BT = a.B * a.T, K = 2 * BT;
  const int64_t k_begin = (int64_t)blockIdx.y * a.k_chunk;
  const int64_t k_end = min(K, k_begin + a.k_chunk);
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const bool abf = a.act_bf16 != 0;
  const int64_t qw = (int64_t)g.F * d_sub;                     // query row width
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  const float *dsh = a.ds + (int64_t)h * K * g.ntot + g.off[f];
  for (int64_t k0 = k_begin; k0 < k_end; k0 += kTileK) {
    {
      const int kk = tid >> 4, c4 = (tid & 15) * 4;
      const int64_t k = k0 + kk;
      const bool kin = k < k_end;
      float av[4], bv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int x = a0 + c4 + e;
        av[e] = (kin && x < n) ? dsh[k * g.ntot + x] : 0.0f;
      }
      const int kind = k >= BT ? 1 : 0;
      const int64_t bt = k - kind * BT;
      const int64_t row = bt * a.H + h;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = d0 + c4 + e;
        bv[e] = (kin && d < d_sub) ? load_act1(a.q[kind], row * qw + (int64_t)f * d_sub + d, abf) : 0.0f;
      }
      *reinterpret_cast<float4 *>(&As[kk][c4]) = make_float4(av[0], av[1], av[2], av[3]);
      *reinterpret_cast<float4 *>(&Bs[kk][c4]) = make_float4(bv[0], bv[1], bv[2], bv[3]);
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kTileK; ++kk) {
      const float4 a4 = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
      const float4 b4 = *reinterpret_cast<const float4 *>(&Bs[kk][tx * 4]);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  float *out = a.dk_part + (((int64_t)blockIdx.y * a.H + h) * g.ntot + g.off[f]) * d_sub;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int x = a0 + ty * 4 + i;
    if (x >= n) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int d = d0 + tx * 4 + j;
      if (d < d_sub) out[(int64_t)x * d_sub + d] = acc[i][j];
    }
  }
}

// d_subkeys = sum of the splits in split order.
__global__ void __launch_bounds__(kThreads) bwd_subkey_sum_kernel(const __grid_constant__ BackwardArgs a) {
  const int64_t total = a.H * (int64_t)a.g.ntot * a.g.d_sub;
  for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < total; e += (int64_t)gridDim.x * kThreads) {
    float acc = 0.0f;
    for (int ks = 0; ks < a.KS; ++ks) acc = __fadd_rn(acc, a.dk_part[(int64_t)ks * total + e]);
    a.d_subkeys[e] = acc;
  }
}

// W = R = 64 fixed at compile time (two rows per lane and sum), else up to four.
template <typename BANK, int JB, bool FULL>
cudaError_t launch_sweep_jb(const BackwardArgs &a, cudaStream_t st) {
  const dim3 grid((unsigned)((a.Pw + kSweepWarps - 1) / kSweepWarps), (unsigned)(a.B * a.H));
  const int64_t smem = (int64_t)kSweepWarps * sweep_slots(JB, 16 / (int)sizeof(BANK)) * 32 * 16;
  auto kern = bwd_sweep_kernel<BANK, kSweepCG, JB, FULL>;
  const cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, 32 * kSweepWarps, smem, st>>>(a);
  return cudaGetLastError();
}

template <typename BANK>
cudaError_t launch_sweep_t(const BackwardArgs &a, cudaStream_t st) {
  if (a.W == 64 && a.R == 64) return launch_sweep_jb<BANK, 64 / (32 / kSweepCG), true>(a, st);
  return launch_sweep_jb<BANK, SDM_MAX_K / (32 / kSweepCG), false>(a, st);
}

unsigned grid_for(int64_t items, int per_block) {
  int64_t b = (items + per_block - 1) / per_block;
  if (b > 65535LL * 16) b = 65535LL * 16;
  return (unsigned)(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_bwd_flags(const BackwardArgs &a, cudaStream_t st) {
  const int64_t rows = a.B * a.T * a.H;
  if (rows == 0) return cudaSuccess;
  bwd_flags_kernel<<<grid_for(rows, kFlagWarps), kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_sweep(const BackwardArgs &a, int bank_dtype, cudaStream_t st) {
  if (a.B * a.H == 0 || a.T == 0 || a.P == 0) return cudaSuccess;
  return bank_dtype == SDM_BF16 ? launch_sweep_t<__nv_bfloat16>(a, st) : launch_sweep_t<float>(a, st);
}

cudaError_t launch_bwd_reduce(const BackwardArgs &a, cudaStream_t st) {
  const int64_t rows = a.B * a.T * a.H;
  if (rows == 0) return cudaSuccess;
  bwd_reduce_kernel<<<grid_for(rows, kReduceWarps), 32 * kReduceWarps, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_subkeys(const BackwardArgs &a, cudaStream_t st) {
  const int64_t total = a.H * (int64_t)a.g.ntot * a.g.d_sub;
  if (total == 0) return cudaSuccess;
  if (a.B * a.T > 0) {
    const int td = (a.g.d_sub + kTileD - 1) / kTileD;
    int per_head = 0;
    for (int f = 0; f < a.g.F; ++f) per_head += (a.g.nf[f] + kTileA - 1) / kTileA * td;
    bwd_subkey_tiles_kernel<<<dim3((unsigned)(per_head * a.H), (unsigned)a.KS), 256, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  bwd_subkey_sum_kernel<<<grid_for(total, kThreads), kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sdm
