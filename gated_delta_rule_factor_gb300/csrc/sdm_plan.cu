// Chunk planner: turns the selected slot ids of each stage (G consecutive tokens of
// one stream) into the row movement plan the write/read kernel executes.
//
// Tokens of a stream must see every earlier token's writes, including writes to the
// same row inside one stage.  The write/read kernel therefore keeps each stage's rows
// in shared memory, one copy per distinct row, and runs the tokens in order on those
// copies.  The plan says, per stage: which distinct rows it touches (sorted slot ids),
// where each of the stage's references lives among them, which rows come from the
// bank and which are carried over from the previous stage's copies (the bank may
// still hold a stale value for those), and which rows go back to the bank after the
// stage (the ones it dirtied or carried in, unless the next stage carries them on).
// Everything is integer work with fixed orders (bitonic sort of (slot, ref) keys,
// ordered prefix sums), so plans are bitwise repeatable and no float atomics exist.
//
// plan_sort: per stage, sort and deduplicate its G*(W+R) references.
// plan_link: per stage, compare with the neighbouring stages and emit the record.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

// Exclusive prefix sum over the block's threads (kThreads = 256); returns the prefix
// and writes the block total to *total.
__device__ __forceinline__ int block_scan_exclusive(int x, int *warp_sums, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < kThreads / 32) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kThreads / 32) warp_sums[lane] = w;   // inclusive warp totals
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + v - x;
  *total = warp_sums[kThreads / 32 - 1];
  __syncthreads();
  return before;
}

__device__ __forceinline__ int find_sorted(const int32_t *a, int n, int32_t key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < key) lo = mid + 1; else hi = mid;
  }
  return (lo < n && a[lo] == key) ? lo : -1;
}

__global__ void __launch_bounds__(kThreads) plan_sort_kernel(const __grid_constant__ PlanArgs a, int P) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t *keys = reinterpret_cast<uint64_t *>(smem);            // [P]
  uint8_t *wr = reinterpret_cast<uint8_t *>(keys + P);              // [P], 4-byte aligned
  const int P4 = (P + 3) & ~3;                                      // wr is updated by words
  uint8_t *tokflag = wr + P4;                                       // [G]
  __shared__ int warp_sums[kThreads / 32];

  const PlanLayout &lay = a.lay;
  const int g = blockIdx.x;
  const int64_t s = blockIdx.y;
  const int64_t b = s / a.H, h = s % a.H;
  const int WR = a.W + a.R;
  const int64_t t0 = (int64_t)g * lay.G;
  const int nt = (int)min((int64_t)lay.G, a.T - t0);
  const int L = nt * WR;
  const int tid = threadIdx.x;

  for (int i = tid; i < P4; i += kThreads) wr[i] = 0;
  for (int i = tid; i < P; i += kThreads) {
    uint64_t key = ~0ull;
    if (i < L) {
      const int64_t t = t0 + i / WR;
      const int j = i % WR;
      const int64_t row = (b * a.T + t) * a.H + h;
      int32_t slot = (j < a.W) ? a.idx[0][row * a.W + j] : a.idx[1][row * a.R + (j - a.W)];
      if (slot < 0 || (int64_t)slot >= a.N) {
        raise_error(a.err, SDM_DEVERR_SLOT_RANGE);
        slot = 0;
      }
      key = ((uint64_t)(uint32_t)slot << 16) | (uint32_t)i;
    }
    keys[i] = key;
  }
  for (int i = tid; i < lay.G; i += kThreads) tokflag[i] = 0;
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P / 2; i += kThreads) {
        const int lo = ((i & ~(j - 1)) << 1) | (i & (j - 1)), hi = lo + j;   // j is a power of two
        const bool asc = (lo & k) == 0;
        const uint64_t x = keys[lo], y = keys[hi];
        if ((x > y) == asc) { keys[lo] = y; keys[hi] = x; }
      }
      __syncthreads();
    }
  }

  // distinct rows: each thread takes a contiguous run of sorted positions
  const int ept = (L + kThreads - 1) / kThreads;
  const int i0 = min(L, tid * ept), i1 = min(L, i0 + ept);
  int nfirst = 0;
  for (int i = i0; i < i1; ++i)
    nfirst += (i == 0 || (keys[i] >> 16) != (keys[i - 1] >> 16)) ? 1 : 0;
  int n_u;
  int u = block_scan_exclusive(nfirst, warp_sums, &n_u) - 1;

  const int64_t stage = s * lay.n_stages + g;
  int32_t *uniq = a.uniq + stage * lay.L;
  uint16_t *refmap = reinterpret_cast<uint16_t *>(a.records + stage * lay.rec_bytes + lay.off_refmap);
  for (int i = i0; i < i1; ++i) {
    const uint32_t slot = (uint32_t)(keys[i] >> 16);
    if (i == 0 || slot != (uint32_t)(keys[i - 1] >> 16)) {
      ++u;
      uniq[u] = (int32_t)slot;
    }
    const int ref = (int)(keys[i] & 0xffffu);
    refmap[ref] = (uint16_t)u;
    if (ref % WR < a.W) {
      // bit 0: written in this stage; bit 1: written by the stage's last token (such rows
      // can only be written back once the whole stage is done).  A row's refs may be
      // split between threads, hence the word-wide atomic OR.
      const uint32_t bits = (ref / WR == nt - 1) ? 3u : 1u;
      atomicOr(reinterpret_cast<unsigned int *>(wr + (u & ~3)), bits << (8 * (u & 3)));
      // a token's refs to one row are adjacent in (slot, ref) order, its write before its
      // read: a read ref of the same token right after this write ref means overlap
      if (i + 1 < L && (keys[i + 1] >> 16) == slot) {
        const int ref2 = (int)(keys[i + 1] & 0xffffu);
        if (ref2 / WR == ref / WR) tokflag[ref / WR] = 1;
      }
    }
  }
  __syncthreads();
  uint8_t *tf = a.records + stage * lay.rec_bytes + lay.off_tokflag;
  for (int i = tid; i < nt; i += kThreads) tf[i] = tokflag[i];
  uint8_t *written = a.written + stage * lay.L;
  for (int i = tid; i < n_u; i += kThreads) written[i] = wr[i];
  if (tid == 0) a.nuniq[stage] = n_u;
}

__global__ void __launch_bounds__(kThreads) plan_link_kernel(const __grid_constant__ PlanArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const PlanLayout &lay = a.lay;
  int32_t *prev = reinterpret_cast<int32_t *>(smem);       // [L]
  int32_t *next = prev + lay.L;                             // [L]
  int32_t *prev2 = next + lay.L;                            // [L]
  __shared__ int warp_sums[kThreads / 32];

  const int g = blockIdx.x;
  const int64_t s = blockIdx.y;
  const int S = lay.n_stages;
  const int64_t stage = s * S + g;
  const int tid = threadIdx.x;
  const int n_prev = g > 0 ? a.nuniq[stage - 1] : 0;
  const int n_cur = a.nuniq[stage];
  const int n_next = g + 1 < S ? a.nuniq[stage + 1] : 0;
  const int n_prev2 = g > 1 ? a.nuniq[stage - 2] : 0;
  for (int i = tid; i < n_prev2; i += kThreads) prev2[i] = a.uniq[(stage - 2) * lay.L + i];
  for (int i = tid; i < n_prev; i += kThreads) prev[i] = a.uniq[(stage - 1) * lay.L + i];
  for (int i = tid; i < n_next; i += kThreads) next[i] = a.uniq[(stage + 1) * lay.L + i];
  __syncthreads();

  const int32_t *cur = a.uniq + stage * lay.L;
  const uint8_t *written = a.written + stage * lay.L;
  const int ept = (n_cur + kThreads - 1) / kThreads;
  const int u0 = min(n_cur, tid * ept), u1 = min(n_cur, u0 + ept);
  // A row loaded here that stage g-2 also held may have been written back at the end of
  // stage g-2, which the write/read kernel only waits for late: such loads go last.
  // Write-backs are listed rows-the-last-token-did-not-write first: the kernel stores
  // those while the stage's last token still runs, the rest ("wb late") after it.
  int c_load = 0, c_late = 0, c_carry = 0, c_wb = 0, c_wbl = 0;
  for (int u = u0; u < u1; ++u) {
    const int32_t slot = cur[u];
    const int src = find_sorted(prev, n_prev, slot);
    const bool out = find_sorted(next, n_next, slot) >= 0;
    const bool late = src < 0 && find_sorted(prev2, n_prev2, slot) >= 0;
    c_load += src < 0 && !late;
    c_late += late;
    c_carry += src >= 0;
    const bool wb = (written[u] || src >= 0) && !out;
    c_wb += wb && !(written[u] & 2);
    c_wbl += wb && (written[u] & 2);
  }
  int n_load, n_late, n_carry, n_wb_early, n_wb_late;
  int o_load = block_scan_exclusive(c_load, warp_sums, &n_load);
  int o_late = n_load + block_scan_exclusive(c_late, warp_sums, &n_late);
  int o_carry = block_scan_exclusive(c_carry, warp_sums, &n_carry);
  int o_wb = block_scan_exclusive(c_wb, warp_sums, &n_wb_early);
  int o_wbl = n_wb_early + block_scan_exclusive(c_wbl, warp_sums, &n_wb_late);
  const int n_wb = n_wb_early + n_wb_late;

  unsigned char *rec = a.records + stage * lay.rec_bytes;
  int32_t *load_slot = reinterpret_cast<int32_t *>(rec + lay.off_load_slot);
  uint16_t *load_u = reinterpret_cast<uint16_t *>(rec + lay.off_load_u);
  uint32_t *carry = reinterpret_cast<uint32_t *>(rec + lay.off_carry);
  int32_t *wb_slot = reinterpret_cast<int32_t *>(rec + lay.off_wb_slot);
  uint16_t *wb_u = reinterpret_cast<uint16_t *>(rec + lay.off_wb_u);
  for (int u = u0; u < u1; ++u) {
    const int32_t slot = cur[u];
    const int src = find_sorted(prev, n_prev, slot);
    const bool out = find_sorted(next, n_next, slot) >= 0;
    if (src < 0) {
      const bool late = find_sorted(prev2, n_prev2, slot) >= 0;
      int &o = late ? o_late : o_load;
      load_slot[o] = slot;
      load_u[o] = (uint16_t)u;
      ++o;
    } else {
      carry[o_carry] = (uint32_t)u | ((uint32_t)src << 16);
      ++o_carry;
    }
    if ((written[u] || src >= 0) && !out) {
      int &o = (written[u] & 2) ? o_wbl : o_wb;
      wb_slot[o] = slot;
      wb_u[o] = (uint16_t)u;
      ++o;
    }
  }
  if (tid == 0) {
    int32_t *hdr = reinterpret_cast<int32_t *>(rec);
    hdr[0] = n_cur;
    hdr[1] = n_load + n_late;
    hdr[2] = n_carry;
    hdr[3] = n_wb;
    hdr[4] = n_late;
    hdr[5] = n_wb_late;
  }
}

}  // namespace

cudaError_t launch_plan_sort(const PlanArgs &a, int64_t streams, int P, cudaStream_t st) {
  if (streams == 0 || a.lay.n_stages == 0) return cudaSuccess;
  const int64_t smem = (int64_t)P * 8 + ((P + 3) & ~3) + a.lay.G;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(plan_sort_kernel), smem);
  if (e != cudaSuccess) return e;
  plan_sort_kernel<<<dim3((unsigned)a.lay.n_stages, (unsigned)streams), kThreads, smem, st>>>(a, P);
  return cudaGetLastError();
}

cudaError_t launch_plan_link(const PlanArgs &a, int64_t streams, cudaStream_t st) {
  if (streams == 0 || a.lay.n_stages == 0) return cudaSuccess;
  const int64_t smem = (int64_t)a.lay.L * 12;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(plan_link_kernel), smem);
  if (e != cudaSuccess) return e;
  plan_link_kernel<<<dim3((unsigned)a.lay.n_stages, (unsigned)streams), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sdm
