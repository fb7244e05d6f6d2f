// Chunk planner: turns the selected slot ids of each stage (G consecutive tokens of
// one stream) into the row movement plan the write/read kernel executes (record
// layout in sdm_internal.h, PlanLayout).
//
// Tokens of a stream must see every earlier token's writes, including writes to the
// same row inside one stage.  The write/read kernel therefore keeps each stage's rows
// in shared memory, one copy per distinct row, and runs the tokens in order on those
// copies.  The plan says, per stage: which distinct rows it touches (sorted slot ids),
// where each of the stage's references lives among them, which rows come from the
// bank and which are carried over from the copies of one of the two previous stages
// (the bank may still hold a stale value for those), and which rows go back to the
// bank after the stage (the ones it dirtied or carried in, unless one of the next two
// stages carries them on).
// Everything is integer work with fixed orders (bitonic sort of (slot, ref) keys,
// ordered prefix sums), so plans are bitwise repeatable and no float atomics exist.
//
// plan_sort: per stage, sort and deduplicate its G*(W+R) references; give every
//            distinct row its shared-memory offset o (slot u, bank color) and every
//            reference the offset of its row.
// plan_link: per stage, compare with the two stages before and after it and emit the
//            row lists (bank loads, carries, write-backs).
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

// Bank color of a reference: the write/read kernel's lane rg reads the rows of block rg
// (16 consecutive blocks of ceil(n/16) references of the token's write or read list),
// and the lanes of blocks 4q..4q+3 read at the same time, so block k's rows get color
// k mod 4.  A row referenced several times takes the color of its first reference.
__device__ __forceinline__ int ref_color(int j, int W, int R) {
  if (j < W) return (j / ((W + 15) >> 4)) & 3;
  return ((j - W) / ((R + 15) >> 4)) & 3;
}

__global__ void __launch_bounds__(kThreads) plan_sort_kernel(const __grid_constant__ PlanArgs a, int P) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t *keys = reinterpret_cast<uint64_t *>(smem);            // [P]
  uint8_t *wr = reinterpret_cast<uint8_t *>(keys + P);              // [P], 4-byte aligned
  const int P4 = (P + 3) & ~3;                                      // wr is updated by words
  uint16_t *uo_s = reinterpret_cast<uint16_t *>(wr + P4);           // [P]
  uint8_t *tokflag = reinterpret_cast<uint8_t *>(uo_s + P);         // [G]
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
  const int u_before = block_scan_exclusive(nfirst, warp_sums, &n_u) - 1;

  const int64_t stage = s * lay.n_stages + g;
  int32_t *uniq = a.uniq + stage * lay.L;
  uint16_t *uo = a.uo + stage * lay.L;
  unsigned char *crec = a.crecs + stage * lay.crec_bytes;
  uint16_t *refmap = reinterpret_cast<uint16_t *>(crec + lay.off_refmap);
  // pass 1: each distinct row's slot, offset and written flag; per-token overlap flags
  int u = u_before;
  for (int i = i0; i < i1; ++i) {
    const uint32_t slot = (uint32_t)(keys[i] >> 16);
    const int ref = (int)(keys[i] & 0xffffu);
    if (i == 0 || slot != (uint32_t)(keys[i - 1] >> 16)) {
      ++u;
      uniq[u] = (int32_t)slot;
      const int o = u * lay.RB + ((ref_color(ref % WR, a.W, a.R) & lay.cmask) << 5);
      uo_s[u] = (uint16_t)o;
      uo[u] = (uint16_t)o;
    }
    if (ref % WR < a.W) {
      // a row's refs may be split between threads, hence the word-wide atomic OR
      atomicOr(reinterpret_cast<unsigned int *>(wr + (u & ~3)), 1u << (8 * (u & 3)));
      // a token's refs to one row are adjacent in (slot, ref) order, its write before its
      // read: a read ref of the same token right after this write ref means overlap
      if (i + 1 < L && (keys[i + 1] >> 16) == slot) {
        const int ref2 = (int)(keys[i + 1] & 0xffffu);
        if (ref2 / WR == ref / WR) tokflag[ref / WR] = 1;
      }
    }
  }
  __syncthreads();
  // pass 2: every reference gets its row's offset
  u = u_before;
  for (int i = i0; i < i1; ++i) {
    if (i == 0 || (keys[i] >> 16) != (keys[i - 1] >> 16)) ++u;
    refmap[keys[i] & 0xffffu] = uo_s[u];
  }
  uint8_t *tf = crec + lay.off_tokflag;
  for (int i = tid; i < nt; i += kThreads) tf[i] = tokflag[i];
  // the stage's weights and gates, next to the offsets, so that the write/read kernel
  // fetches everything its compute warps read per stage with one contiguous copy
  float *wts = reinterpret_cast<float *>(crec + lay.off_wts);
  for (int i = tid; i < L; i += kThreads) {
    const int64_t row = (b * a.T + t0 + i / WR) * a.H + h;
    const int j = i % WR;
    wts[i] = j < a.W ? a.wt[0][row * a.W + j] : a.wt[1][row * a.R + (j - a.W)];
  }
  float *gts = reinterpret_cast<float *>(crec + lay.off_gates);
  for (int i = tid; i < 2 * nt; i += kThreads) gts[i] = a.gates[((b * a.T + t0 + i / 2) * a.H + h) * 2 + (i & 1)];
  uint8_t *written = a.written + stage * lay.L;
  for (int i = tid; i < n_u; i += kThreads) written[i] = wr[i];
  if (tid == 0) a.nuniq[stage] = n_u;
}

__global__ void __launch_bounds__(kThreads) plan_link_kernel(const __grid_constant__ PlanArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const PlanLayout &lay = a.lay;
  int32_t *prev = reinterpret_cast<int32_t *>(smem);       // [L] slots of stage g-1
  int32_t *prev2 = prev + lay.L;                            // [L] g-2
  int32_t *next = prev2 + lay.L;                            // [L] g+1
  int32_t *next2 = next + lay.L;                            // [L] g+2
  uint16_t *uo_next = reinterpret_cast<uint16_t *>(next2 + lay.L);   // [L]
  uint16_t *uo_next2 = uo_next + lay.L;                              // [L]
  __shared__ int warp_sums[kThreads / 32];

  const int g = blockIdx.x;
  const int64_t s = blockIdx.y;
  const int S = lay.n_stages;
  const int64_t stage = s * S + g;
  const int tid = threadIdx.x;
  const int n_prev = g > 0 ? a.nuniq[stage - 1] : 0;
  const int n_prev2 = g > 1 ? a.nuniq[stage - 2] : 0;
  const int n_cur = a.nuniq[stage];
  const int n_next = g + 1 < S ? a.nuniq[stage + 1] : 0;
  const int n_next2 = g + 2 < S ? a.nuniq[stage + 2] : 0;
  for (int i = tid; i < n_prev; i += kThreads) prev[i] = a.uniq[(stage - 1) * lay.L + i];
  for (int i = tid; i < n_prev2; i += kThreads) prev2[i] = a.uniq[(stage - 2) * lay.L + i];
  for (int i = tid; i < n_next; i += kThreads) {
    next[i] = a.uniq[(stage + 1) * lay.L + i];
    uo_next[i] = a.uo[(stage + 1) * lay.L + i];
  }
  for (int i = tid; i < n_next2; i += kThreads) {
    next2[i] = a.uniq[(stage + 2) * lay.L + i];
    uo_next2[i] = a.uo[(stage + 2) * lay.L + i];
  }
  __syncthreads();

  const int32_t *cur = a.uniq + stage * lay.L;
  const uint16_t *uo_cur = a.uo + stage * lay.L;
  const uint8_t *written = a.written + stage * lay.L;
  const int ept = (n_cur + kThreads - 1) / kThreads;
  const int u0 = min(n_cur, tid * ept), u1 = min(n_cur, u0 + ept);
  // The bank may be stale for a row that one of the two previous stages holds (their
  // write-backs come later): such a row arrives by a copy in shared memory from the
  // latest stage that holds it, made at that stage's end, so this stage fetches from
  // the bank only rows neither previous stage holds.  It hands its own rows on the same
  // way: to stage g+1 the rows g+1 holds, to stage g+2 the rows g+2 holds and g+1 does
  // not.  A row goes back to the bank after this stage if it is dirty here (written, or
  // handed in) and is not handed on.
  int c_load = 0, c_o1 = 0, c_o2 = 0, c_wb = 0;
  for (int u = u0; u < u1; ++u) {
    const int32_t slot = cur[u];
    const bool in1 = find_sorted(prev, n_prev, slot) >= 0;
    const bool in2 = !in1 && find_sorted(prev2, n_prev2, slot) >= 0;
    const bool out1 = find_sorted(next, n_next, slot) >= 0;
    const bool out2 = !out1 && find_sorted(next2, n_next2, slot) >= 0;
    c_load += !in1 && !in2;
    c_o1 += out1;
    c_o2 += out2;
    c_wb += (written[u] || in1 || in2) && !out1 && !out2;
  }
  int n_load, n_o1, n_o2, n_wb;
  int o_load = block_scan_exclusive(c_load, warp_sums, &n_load);
  int o_o1 = block_scan_exclusive(c_o1, warp_sums, &n_o1);
  int o_o2 = n_o1 + block_scan_exclusive(c_o2, warp_sums, &n_o2);
  int o_wb = block_scan_exclusive(c_wb, warp_sums, &n_wb);

  unsigned char *lrec = a.lrecs + stage * lay.lrec_bytes;
  uint2 *ent = reinterpret_cast<uint2 *>(lrec + lay.off_ent);
  uint2 *out = reinterpret_cast<uint2 *>(lrec + lay.off_out);
  uint2 *wb = reinterpret_cast<uint2 *>(lrec + lay.off_wb);
  for (int u = u0; u < u1; ++u) {
    const int32_t slot = cur[u];
    const uint32_t row16 = (uint32_t)slot * a.pitch16;     // < 2^32 (checked on the host)
    const bool in = find_sorted(prev, n_prev, slot) >= 0 || find_sorted(prev2, n_prev2, slot) >= 0;
    const int dst1 = find_sorted(next, n_next, slot);
    const int dst2 = dst1 < 0 ? find_sorted(next2, n_next2, slot) : -1;
    if (!in) ent[o_load++] = make_uint2(row16, uo_cur[u]);
    if (dst1 >= 0) out[o_o1++] = make_uint2((uint32_t)uo_next[dst1] | ((uint32_t)uo_cur[u] << 16), 0u);
    if (dst2 >= 0) out[o_o2++] = make_uint2((uint32_t)uo_next2[dst2] | ((uint32_t)uo_cur[u] << 16), 0u);
    if ((written[u] || in) && dst1 < 0 && dst2 < 0) wb[o_wb++] = make_uint2(row16, uo_cur[u]);
  }
  if (tid == 0) {
    int32_t *hdr = reinterpret_cast<int32_t *>(lrec);
    hdr[0] = n_cur;
    hdr[1] = n_load;
    hdr[2] = n_o1;
    hdr[3] = n_o2;
    hdr[4] = n_wb;
  }
}

}  // namespace

cudaError_t launch_plan_sort(const PlanArgs &a, int64_t streams, int P, cudaStream_t st) {
  if (streams == 0 || a.lay.n_stages == 0) return cudaSuccess;
  const int64_t smem = (int64_t)P * 8 + ((P + 3) & ~3) + (int64_t)P * 2 + a.lay.G;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(plan_sort_kernel), smem);
  if (e != cudaSuccess) return e;
  plan_sort_kernel<<<dim3((unsigned)a.lay.n_stages, (unsigned)streams), kThreads, smem, st>>>(a, P);
  return cudaGetLastError();
}

cudaError_t launch_plan_link(const PlanArgs &a, int64_t streams, cudaStream_t st) {
  if (streams == 0 || a.lay.n_stages == 0) return cudaSuccess;
  const int64_t smem = (int64_t)a.lay.L * 20;   // four slot lists and two offset lists
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(plan_link_kernel), smem);
  if (e != cudaSuccess) return e;
  plan_link_kernel<<<dim3((unsigned)a.lay.n_stages, (unsigned)streams), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sdm
