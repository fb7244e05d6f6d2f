// Host side of the SDM C ABI: argument checks, configuration, workspace layout,
// launches, kernel-side error read-back and per-kernel timing.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/sdm.h"
#include "sdm_internal.h"

using namespace sdm;

cudaError_t sdm::raise_smem_limit(const void *kernel, int64_t smem) {
  struct Raised {
    const void *kernel;
    int dev;
    int64_t smem;
  };
  static std::mutex mu;
  static std::vector<Raised> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (Raised &r : done) {
    if (r.kernel != kernel || r.dev != dev) continue;
    if (r.smem >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) r.smem = smem;
    return e;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) done.push_back({kernel, dev, smem});
  return e;
}

namespace {

// ---------------------------------------------------------------- error reporting

thread_local char g_msg[512] = "";

sdm_status fail(sdm_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

sdm_status ok() {
  g_msg[0] = '\0';
  return SDM_OK;
}

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_test_stall_decode_copy{0};  // sdm_test_stall_decode_copy
std::atomic<int> g_test_slice_bytes{0};        // sdm_test_force_write_read_layout
std::atomic<int> g_test_stage_tokens{0};
std::atomic<int> g_test_simt_scorer{0};        // sdm_test_force_simt_scorer

// ---------------------------------------------------------------- profiling

constexpr int kProfSlots = 4096;
struct ProfState {
  std::mutex mu;
  bool active = false;
  bool created = false;
  std::vector<cudaEvent_t> start, stop;
  std::vector<int> kind;
  int used = 0;
} g_prof;

bool prof_acquire(int kind, cudaEvent_t *start, cudaEvent_t *stop) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.active || g_prof.used >= kProfSlots) return false;
  const int i = g_prof.used++;
  g_prof.kind[i] = kind;
  *start = g_prof.start[i];
  *stop = g_prof.stop[i];
  return true;
}

template <class Launch>
sdm_status run_kernel(int kind, cudaStream_t st, const char *name, Launch &&launch) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  const bool prof = prof_acquire(kind, &e0, &e1);
  if (prof) cudaEventRecord(e0, st);
  const cudaError_t e = launch();
  if (prof) cudaEventRecord(e1, st);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return fail(SDM_ERR_CUDA, "%s launch failed: %s", name, cudaGetErrorString(e));
  return SDM_OK;
}

// A launch of library code (cuBLASLt): timed like the library's kernels, not counted by
// sdm_launch_count.  launch() returns nullptr or the reason it failed.
template <class Launch>
sdm_status run_library(int kind, cudaStream_t st, const char *name, Launch &&launch) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  const bool prof = prof_acquire(kind, &e0, &e1);
  if (prof) cudaEventRecord(e0, st);
  const char *why = launch();
  if (prof) cudaEventRecord(e1, st);
  if (why) return fail(SDM_ERR_CUDA, "%s: %s", name, why);
  return SDM_OK;
}

// ---------------------------------------------------------------- shape checks

int64_t elem_bytes(int32_t dt) { return dt == SDM_BF16 ? 2 : 4; }

sdm_status check_dtype(int32_t dt, const char *what) {
  if (dt == SDM_F16) return fail(SDM_ERR_UNSUPPORTED, "%s: float16 is not supported", what);
  if (dt != SDM_F32 && dt != SDM_BF16) return fail(SDM_ERR_INVALID_ARG, "%s: unknown dtype %d", what, dt);
  return SDM_OK;
}

// Position tuples (p_1..p_F), p_f < kf_f, prod(p_f + 1) <= k, lexicographic.
void enumerate_candidates(int F, const int32_t *kf, int k, std::vector<uint32_t> &out) {
  out.clear();
  int p[SDM_MAX_FACTORS] = {0, 0, 0, 0};
  // iterative odometer with pruning on the product
  std::vector<uint32_t> tmp;
  struct Rec {
    static void go(int f, int F, const int32_t *kf, int k, int64_t prod, int *p, std::vector<uint32_t> &o) {
      if (f == F) {
        uint32_t t = 0;
        for (int i = 0; i < F; ++i) t |= (uint32_t)p[i] << (8 * i);
        o.push_back(t);
        return;
      }
      for (int x = 0; x < kf[f]; ++x) {
        if (prod * (x + 1) > k) break;
        p[f] = x;
        go(f + 1, F, kf, k, prod * (x + 1), p, o);
        if (o.size() > (size_t)SDM_MAX_CANDIDATES) return;
      }
      p[f] = 0;
    }
  };
  Rec::go(0, F, kf, k, 1, p, out);
}

struct Derived {
  int64_t N = 0;
  int32_t ntot = 0;
  KeyGeometry g{};
  CandidateList *cl = nullptr;  // filled on demand
};

sdm_status check_shape(const sdm_shape *sh, bool decode, Derived *d) {
  if (!sh) return fail(SDM_ERR_INVALID_ARG, "shape is NULL");
  if (sh->B < 0 || sh->T < 0 || sh->H < 0) return fail(SDM_ERR_INVALID_ARG, "B, T, H must be >= 0");
  if (decode && sh->T != 1) return fail(SDM_ERR_INVALID_ARG, "decode step needs T == 1 (got %lld)", (long long)sh->T);
  if (!decode && sh->B * sh->H > 65535)
    return fail(SDM_ERR_UNSUPPORTED, "B*H = %lld streams exceeds 65535", (long long)(sh->B * sh->H));
  sdm_status st;
  if ((st = check_dtype(sh->act_dtype, "act_dtype")) != SDM_OK) return st;
  if ((st = check_dtype(sh->bank_dtype, "bank_dtype")) != SDM_OK) return st;
  if (sh->F < 1) return fail(SDM_ERR_INVALID_ARG, "F must be >= 1");
  if (sh->F > SDM_MAX_FACTORS) return fail(SDM_ERR_UNSUPPORTED, "F = %d > %d factors", sh->F, SDM_MAX_FACTORS);
  int64_t N = 1;
  int32_t ntot = 0;
  for (int f = 0; f < sh->F; ++f) {
    const int32_t n = sh->factor_dims[f];
    if (n < 1) return fail(SDM_ERR_INVALID_ARG, "factor_dims[%d] = %d < 1", f, n);
    if (n > SDM_MAX_FACTOR_DIM) return fail(SDM_ERR_UNSUPPORTED, "factor_dims[%d] = %d > %d", f, n, SDM_MAX_FACTOR_DIM);
    N *= n;
    ntot += n;
  }
  if (N > 0x7fffffffLL) return fail(SDM_ERR_UNSUPPORTED, "N = %lld slots exceeds 2^31 - 1", (long long)N);
  // the write/read kernel addresses a stream's table in 16-byte units with 32 bits
  if (sh->d_v > 0 && N * sh->d_v * elem_bytes(sh->bank_dtype) / 16 > 0xffffffffLL)
    return fail(SDM_ERR_UNSUPPORTED, "one stream's table (N * d_v) exceeds 64 GiB");
  if (sh->d_sub < 1) return fail(SDM_ERR_INVALID_ARG, "d_sub must be >= 1");
  if (sh->d_sub > SDM_MAX_SUBKEY_DIM) return fail(SDM_ERR_UNSUPPORTED, "d_sub = %lld > %d", (long long)sh->d_sub, SDM_MAX_SUBKEY_DIM);
  if (sh->d_v < 1) return fail(SDM_ERR_INVALID_ARG, "d_v must be >= 1");
  if (sh->d_v > SDM_MAX_HEAD_DIM) return fail(SDM_ERR_UNSUPPORTED, "head dim d_v = %lld > 2^20", (long long)sh->d_v);
  if (sh->d_v % 8 != 0) return fail(SDM_ERR_UNSUPPORTED, "d_v = %lld is not a multiple of 8 (16-byte rows)", (long long)sh->d_v);
  if (sh->W < 1 || sh->R < 1) return fail(SDM_ERR_INVALID_ARG, "W and R must be >= 1");
  if (sh->W > N || sh->R > N)
    return fail(SDM_ERR_INVALID_ARG, "more writes or reads per token (W=%d, R=%d) than slots (N=%lld)", sh->W, sh->R, (long long)N);
  if (sh->W > SDM_MAX_K || sh->R > SDM_MAX_K)
    return fail(SDM_ERR_UNSUPPORTED, "W=%d or R=%d above the compiled limit %d", sh->W, sh->R, SDM_MAX_K);
  if (!decode && (sh->chunk_size < 1 || sh->chunk_size > SDM_MAX_CHUNK))
    return fail(SDM_ERR_INVALID_ARG, "chunk_size = %d outside [1, %d]", sh->chunk_size, SDM_MAX_CHUNK);
  if (d) {
    d->N = N;
    d->ntot = ntot;
    KeyGeometry &g = d->g;
    g.F = sh->F;
    g.d_sub = (int32_t)sh->d_sub;
    g.ntot = ntot;
    int off = 0;
    for (int f = 0; f < SDM_MAX_FACTORS; ++f) {
      g.nf[f] = f < sh->F ? sh->factor_dims[f] : 1;
      g.off[f] = off;
      if (f < sh->F) off += sh->factor_dims[f];
    }
    g.k[0] = sh->W;
    g.k[1] = sh->R;
    for (int q = 0; q < 2; ++q)
      for (int f = 0; f < SDM_MAX_FACTORS; ++f) g.kf[q][f] = f < sh->F ? std::min(g.k[q], g.nf[f]) : 1;
  }
  return SDM_OK;
}

// Boxes of at least k position tuples, by corner: the first F-1 sides run over powers of
// two (and the full width kf), the last side is the least that reaches k tuples.
void enumerate_boxes(int F, const int32_t *kf, int k, std::vector<uint32_t> &out) {
  out.clear();
  int a[SDM_MAX_FACTORS] = {1, 1, 1, 1};
  struct Rec {
    static void go(int f, int F, const int32_t *kf, int k, int64_t prod, int *a, std::vector<uint32_t> &o) {
      if (o.size() >= 32) return;
      if (f == F - 1) {
        const int64_t last = (k + prod - 1) / prod;
        if (last < 1 || last > kf[f]) return;
        a[f] = (int)last;
        uint32_t t = 0;
        for (int i = 0; i < F; ++i) t |= (uint32_t)(a[i] - 1) << (8 * i);
        if (std::find(o.begin(), o.end(), t) == o.end()) o.push_back(t);
        return;
      }
      for (int x = 1;; x <<= 1) {
        const int side = x < kf[f] ? x : kf[f];
        a[f] = side;
        go(f + 1, F, kf, k, prod * side, a, o);
        if (side == kf[f]) break;
      }
    }
  };
  Rec::go(0, F, kf, k, 1, a, out);
}

sdm_status build_candidates(const Derived &d, CandidateList *cl) {
  std::vector<uint32_t> v;
  for (int q = 0; q < 2; ++q) {
    enumerate_candidates(d.g.F, d.g.kf[q], d.g.k[q], v);
    if (v.size() > (size_t)SDM_MAX_CANDIDATES)
      return fail(SDM_ERR_UNSUPPORTED, "k = %d has more than %d product-key candidates", d.g.k[q], SDM_MAX_CANDIDATES);
    cl->n[q] = (int32_t)v.size();
    std::copy(v.begin(), v.end(), cl->tup[q]);
    enumerate_boxes(d.g.F, d.g.kf[q], d.g.k[q], v);
    cl->nbox[q] = (int32_t)v.size();
    std::copy(v.begin(), v.end(), cl->box[q]);
  }
  return SDM_OK;
}

int pow2_at_least(int64_t x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Sort width of a factor (EF) and of the candidate list (EC), in keys per lane: both are
// sorted in chunks of 32*E keys merged into a running best 32*E (k <= 32*E), which keeps
// the selection kernels' register use low enough for several CTAs per SM.  E = 2 when
// both k are at most 64 (fewer compare-exchange steps per key), else 4 (k <= 128).
void sort_widths(const Derived &d, const CandidateList &, int *EF, int *EC) {
  const int kmax = std::max(d.g.k[0], d.g.k[1]);
  *EF = kmax <= 64 ? 2 : 4;
  *EC = *EF;
}

// ---------------------------------------------------------------- plan / kernel config

constexpr int kMaxStageRefs = 4096;

int64_t a16(int64_t x) { return (x + 15) & ~int64_t(15); }

PlanLayout plan_layout(int G, int W, int R, int64_t T, int RB) {
  PlanLayout p{};
  p.G = G;
  p.L = G * (W + R);
  p.n_stages = (int32_t)((T + G - 1) / G);
  p.RB = RB;
  p.cmask = RB >= 128 ? 3 : 0;
  const int64_t L = p.L;
  int64_t o = 32;                                    // n_u, n_load, n_c1, n_c2, n_wb
  p.off_ent = o;       o = a16(o + 8 * L);
  p.off_out = o;       o = a16(o + 8 * L);
  p.off_wb = o;        o = a16(o + 8 * L);
  p.lrec_bytes = o;
  o = 0;
  p.off_refmap = o;    o = a16(o + 2 * L);
  p.off_tokflag = o;   o = a16(o + G);
  p.off_wts = o;       o = a16(o + 4 * L);
  p.off_gates = o;     o = a16(o + 8 * (int64_t)G);
  p.crec_bytes = o;
  return p;
}

struct WrChoice {
  int NCW = 1, LW = 8;
  int slices = 0;
  PlanLayout lay{};
  int64_t smem = 0;
};

constexpr int64_t kSmemOneCta = 220 * 1024;
constexpr int64_t kSmemTwoCta = 110 * 1024;

// Compute warps per CTA the kernel is compiled for (each owns 32 bytes of every row).
constexpr int kNcwChoices[] = {8, 4, 1};

int64_t row_bytes_of(const sdm_shape *sh) { return sh->d_v * elem_bytes(sh->bank_dtype); }

// Longest stage (tokens) whose buffers fit `budget` bytes of shared memory; 0 if not even
// one token fits.  Row offsets are 16-bit: L * RB <= 65536.
int stage_tokens(const sdm_shape *sh, int RB, int64_t budget) {
  const int WR = sh->W + sh->R;
  int gmax = (int)std::min<int64_t>(sh->chunk_size, std::max<int64_t>(sh->T, 1));
  gmax = std::min(gmax, kMaxStageRefs / WR);
  gmax = std::min(gmax, 65536 / (WR * RB));
  for (int G = gmax; G >= 1; --G) {
    const PlanLayout lay = plan_layout(G, sh->W, sh->R, sh->T, RB);
    if (write_read_smem_bytes(lay, (int)elem_bytes(sh->bank_dtype), (int)elem_bytes(sh->act_dtype)) <=
        budget)
      return G;
  }
  return 0;
}

WrChoice configure(const sdm_shape *sh, int ncw, bool two_per_sm, int forced_g) {
  WrChoice c;
  c.NCW = ncw;
  if (ncw == 8) two_per_sm = false;                  // 512 threads: one CTA per SM
  const int RB = 32 * ncw;
  c.slices = (int)((row_bytes_of(sh) + RB - 1) / RB);
  int G = two_per_sm ? stage_tokens(sh, RB, kSmemTwoCta) : 0;
  if (G == 0) {                                      // one CTA per SM (the only choice for NCW = 8)
    two_per_sm = false;
    G = stage_tokens(sh, RB, kSmemOneCta);
  }
  c.LW = two_per_sm ? 4 : 8;
  if (forced_g > 0 && forced_g < G) G = forced_g;
  G = std::max(G, 1);
  c.lay = plan_layout(G, sh->W, sh->R, sh->T, RB);
  c.smem = write_read_smem_bytes(c.lay, (int)elem_bytes(sh->bank_dtype), (int)elem_bytes(sh->act_dtype));
  return c;
}

// The widest slice (most compute warps per CTA) that still gives at least 0.8 CTAs per
// SM; two CTAs per SM (four loader warps each) when there are more CTAs than SMs.
WrChoice choose_write_read(const sdm_shape *sh, int sm_count) {
  const int64_t streams = sh->B * sh->H, rb = row_bytes_of(sh);
  int ncw = 1;
  const int forced = g_test_slice_bytes.load();
  if (forced == 32 || forced == 128 || forced == 256) {
    ncw = forced / 32;
  } else {
    for (int n : kNcwChoices) {
      if (n > 1 && 32 * n > rb) continue;
      const int64_t ctas = streams * ((rb + 32 * n - 1) / (32 * n));
      if (ctas * 10 >= (int64_t)sm_count * 8) {
        ncw = n;
        break;
      }
    }
  }
  for (;;) {
    const int64_t ctas = streams * ((rb + 32 * ncw - 1) / (32 * ncw));
    const WrChoice c = configure(sh, ncw, ctas > sm_count, g_test_stage_tokens.load());
    if (c.smem <= kSmemOneCta || ncw == 1) return c;
    ncw = ncw == 8 ? 4 : 1;                          // not even one token fits: a narrower slice
  }
}

// ---------------------------------------------------------------- workspace layout

constexpr int64_t kHeaderBytes = 256;

int64_t a256(int64_t x) { return (x + 255) & ~int64_t(255); }

struct WsLayout {
  int64_t idx_w, wt_w, idx_r, wt_r;  // selection outputs kept here when the caller passes NULL
  int64_t scores;                    // factor scores [2, B*T*H, sum n_f] float32
  int64_t split;                     // bf16 parts of float32 queries and sub-keys (scorer)
  int64_t uniq, nuniq, uo, written, lrecs, crecs;
  int64_t total;
};

WsLayout ws_layout(const sdm_shape *sh, const PlanLayout &lay) {
  WsLayout w{};
  const int64_t rows = sh->B * sh->T * sh->H;
  const int64_t stages = sh->B * sh->H * (int64_t)lay.n_stages;
  int64_t o = kHeaderBytes;
  w.idx_w = o; o = a256(o + rows * sh->W * 4);
  w.wt_w = o;  o = a256(o + rows * sh->W * 4);
  w.idx_r = o; o = a256(o + rows * sh->R * 4);
  w.wt_r = o;  o = a256(o + rows * sh->R * 4);
  int64_t ntot = 0;
  for (int f = 0; f < sh->F && f < SDM_MAX_FACTORS; ++f) ntot += sh->factor_dims[f];
  w.scores = o; o = a256(o + 2 * rows * ntot * 4);
  KeyGeometry kg{};
  kg.F = (int32_t)sh->F;
  kg.d_sub = (int32_t)sh->d_sub;
  kg.ntot = (int32_t)ntot;
  w.split = o; o = a256(o + score_split_bytes(kg, sh->B * sh->T, sh->H, sh->act_dtype));
  w.uniq = o;  o = a256(o + stages * lay.L * 4);
  w.nuniq = o; o = a256(o + stages * 4);
  w.uo = o;    o = a256(o + stages * lay.L * 2);
  w.written = o; o = a256(o + stages * lay.L);
  w.lrecs = o; o = a256(o + stages * lay.lrec_bytes);
  w.crecs = o; o = a256(o + stages * lay.crec_bytes);
  w.total = o;
  return w;
}

// The size depends only on the shape: the maximum over every slice width and stage
// length the launch may pick on any device (stage lengths forced down by the test hook
// included).
int64_t write_read_ws_bytes(const sdm_shape *sh) {
  int64_t best = kHeaderBytes;
  for (int ncw : kNcwChoices)
    for (bool two : {false, true}) {
      const WrChoice c = configure(sh, ncw, two, 0);
      for (int g = 1; g <= c.lay.G; ++g)
        best = std::max(best, ws_layout(sh, plan_layout(g, sh->W, sh->R, sh->T, 32 * ncw)).total);
    }
  return best;
}

// ---------------------------------------------------------------- pointer checks

bool aligned(const void *p, int64_t a) { return ((uintptr_t)p % (uintptr_t)a) == 0; }

struct Range {
  const void *p;
  int64_t n;
  const char *name;
};

bool overlap(const Range &a, const Range &b) {
  if (!a.p || !b.p || a.n <= 0 || b.n <= 0) return false;
  const uintptr_t a0 = (uintptr_t)a.p, a1 = a0 + (uintptr_t)a.n;
  const uintptr_t b0 = (uintptr_t)b.p, b1 = b0 + (uintptr_t)b.n;
  return a0 < b1 && b0 < a1;
}

int g_sm_count_cache[64] = {0};

sdm_status sm_count(int *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64 && g_sm_count_cache[dev] > 0) {
    *out = g_sm_count_cache[dev];
    return SDM_OK;
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64) g_sm_count_cache[dev] = n;
  *out = n;
  return SDM_OK;
}

// The tensor-core scorer takes factor widths that are multiples of 16, and bfloat16
// inputs whose d_sub is a multiple of 64 or float32 inputs of any d_sub
// (sdm_test_force_simt_scorer forces the CUDA-core one).
bool use_tensor_cores(const Derived &d, const sdm_shape *sh) {
  if (g_test_simt_scorer.load()) return false;
  return score_tc_supported(d.g, sh->H, sh->act_dtype);
}

// Per-device side stream and fork / join events of write_read_impl, created on first use
// and kept for the life of the process.  A call holds `mu` from recording the fork to
// recording the join.  If another call re-records the join before this call's main
// stream waits on it, the wait also covers that later copy (the side stream runs the
// copies in order): it can only wait longer, never too little.
struct SideStream {
  cudaStream_t st = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex mu;
};
SideStream g_side[64];
std::mutex g_side_mu;

sdm_status side_stream(SideStream **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(SDM_ERR_UNSUPPORTED, "device ordinal %d is not supported", dev);
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream &s = g_side[dev];
  if (!s.st) {
    e = cudaStreamCreateWithFlags(&s.st, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      s.st = nullptr;
      return fail(SDM_ERR_CUDA, "side stream set-up: %s", cudaGetErrorString(e));
    }
  }
  *out = &s;
  return SDM_OK;
}

// The write/read op.  side_copy: run the learned-table copy on the library's side stream
// of the device, concurrently with scoring, selection and planning (they touch no bank
// row), and join it before the write/read kernel.
// Snapshot of a training forward: where its data starts (after the header) and its type.
struct SnapOut {
  unsigned char *data;
  int32_t bf16;
};

int64_t snapshot_pieces(const sdm_shape *sh) { return (sh->d_v * elem_bytes(sh->bank_dtype) + 31) / 32; }

int64_t snapshot_bytes_of(const sdm_shape *sh, int32_t snap_dtype) {
  const int64_t pc = 32 / elem_bytes(sh->bank_dtype);          // bank columns of a piece
  return kSnapshotHeaderBytes +
         sh->B * sh->H * sh->T * snapshot_pieces(sh) * (int64_t)sh->W * pc * elem_bytes(snap_dtype);
}

sdm_status write_read_impl(const sdm_shape *sh, const void *q_w, const void *q_r, const void *k_val,
                           const float *gates, const void *subkeys, const void *bank_init, void *bank,
                           void *y, int32_t *idx_w, float *wt_w, int32_t *idx_r, float *wt_r,
                           void *workspace, size_t workspace_bytes, sdm_stream_t stream, bool side_copy,
                           const SnapOut *snap = nullptr) {
  Derived d;
  sdm_status st = check_shape(sh, false, &d);
  if (st != SDM_OK) return st;
  static thread_local CandidateList cl;
  if ((st = build_candidates(d, &cl)) != SDM_OK) return st;

  const int64_t ab = elem_bytes(sh->act_dtype), sb = elem_bytes(sh->bank_dtype);
  const int64_t rows = sh->B * sh->T * sh->H;
  const int64_t qbytes = rows * sh->F * sh->d_sub * ab;
  const Range r_qw{q_w, qbytes, "q_w"}, r_qr{q_r, qbytes, "q_r"}, r_kv{k_val, rows * sh->d_v * ab, "k_val"};
  const Range r_g{gates, rows * 2 * 4, "gates"}, r_sk{subkeys, sh->H * d.ntot * sh->d_sub * ab, "subkeys"};
  const Range r_bi{bank_init, sh->H * d.N * sh->d_v * sb, "bank_init"};
  const Range r_b{bank, sh->B * sh->H * d.N * sh->d_v * sb, "bank"};
  const Range r_y{y, rows * sh->d_v * ab, "y"};
  const Range r_iw{idx_w, rows * sh->W * 4, "idx_w"}, r_ww{wt_w, rows * sh->W * 4, "wt_w"};
  const Range r_ir{idx_r, rows * sh->R * 4, "idx_r"}, r_wr{wt_r, rows * sh->R * 4, "wt_r"};
  const int64_t need_ws = write_read_ws_bytes(sh);
  const Range r_ws{workspace, (int64_t)workspace_bytes, "workspace"};

  if (rows > 0) {
    const Range req[] = {r_qw, r_qr, r_kv, r_g, r_sk, r_b, r_y};
    for (const Range &r : req)
      if (!r.p) return fail(SDM_ERR_INVALID_ARG, "%s is NULL", r.name);
  } else if (!bank && sh->B * sh->H > 0) {
    return fail(SDM_ERR_INVALID_ARG, "bank is NULL");
  }
  const Range al16[] = {r_qw, r_qr, r_kv, r_sk, r_bi, r_b, r_y};
  for (const Range &r : al16)
    if (r.p && !aligned(r.p, 16)) return fail(SDM_ERR_INVALID_ARG, "%s is not 16-byte aligned", r.name);
  if (gates && !aligned(gates, 8)) return fail(SDM_ERR_INVALID_ARG, "gates is not 8-byte aligned");
  const Range al4[] = {r_iw, r_ww, r_ir, r_wr};
  for (const Range &r : al4)
    if (r.p && !aligned(r.p, 4)) return fail(SDM_ERR_INVALID_ARG, "%s is not 4-byte aligned", r.name);
  if (!workspace) return fail(SDM_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 16)) return fail(SDM_ERR_WORKSPACE, "workspace is not 16-byte aligned");
  if ((int64_t)workspace_bytes < need_ws)
    return fail(SDM_ERR_WORKSPACE, "workspace has %zu bytes, needs %lld", workspace_bytes, (long long)need_ws);

  // outputs must not overlap inputs or each other
  const Range ins[] = {r_qw, r_qr, r_kv, r_g, r_sk, r_bi};
  const Range outs[] = {r_b, r_y, r_iw, r_ww, r_ir, r_wr, r_ws};
  for (const Range &o : outs)
    for (const Range &i : ins)
      if (overlap(o, i)) return fail(SDM_ERR_ALIAS, "%s overlaps %s", o.name, i.name);
  for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i)
    for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
      if (overlap(outs[i], outs[j])) return fail(SDM_ERR_ALIAS, "%s overlaps %s", outs[i].name, outs[j].name);

  int sms = 0;
  if ((st = sm_count(&sms)) != SDM_OK) return st;
  const WrChoice wc = choose_write_read(sh, sms);
  const WsLayout wl = ws_layout(sh, wc.lay);
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  int32_t *err = reinterpret_cast<int32_t *>(ws);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

  cudaError_t ce = cudaMemsetAsync(err, 0, sizeof(int32_t), cs);
  if (ce != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(ce));

  const int64_t streams = sh->B * sh->H;
  SideStream *side = nullptr;
  if (bank_init && streams > 0) {
    BankCopyArgs bc{bank_init, bank, sh->B, d.N * sh->d_v * sb, sh->H};
    cudaStream_t copy_st = cs;
    if (side_copy && rows > 0) {
      if ((st = side_stream(&side)) != SDM_OK) return st;
      side->mu.lock();
      ce = cudaEventRecord(side->fork, cs);
      if (ce == cudaSuccess) ce = cudaStreamWaitEvent(side->st, side->fork, 0);
      if (ce != cudaSuccess) {
        side->mu.unlock();
        return fail(SDM_ERR_CUDA, "side stream fork: %s", cudaGetErrorString(ce));
      }
      copy_st = side->st;
    }
    st = run_kernel(SDM_KERNEL_BANK_COPY, copy_st, "bank_copy", [&] { return launch_bank_copy(bc, sms, copy_st); });
    if (side) {
      ce = cudaEventRecord(side->join, side->st);
      side->mu.unlock();
      if (ce != cudaSuccess) return fail(SDM_ERR_CUDA, "side stream join: %s", cudaGetErrorString(ce));
    }
    if (st != SDM_OK) return st;
  }
  if (rows == 0) return ok();

  int32_t *iw = idx_w ? idx_w : reinterpret_cast<int32_t *>(ws + wl.idx_w);
  float *ww = wt_w ? wt_w : reinterpret_cast<float *>(ws + wl.wt_w);
  int32_t *ir = idx_r ? idx_r : reinterpret_cast<int32_t *>(ws + wl.idx_r);
  float *wr = wt_r ? wt_r : reinterpret_cast<float *>(ws + wl.wt_r);

  // 1. factor scores of both queries, then the exact top-k of every row
  int EF, EC;
  sort_widths(d, cl, &EF, &EC);
  float *scores = reinterpret_cast<float *>(ws + wl.scores);
  ScoreArgs sa{};
  sa.q[0] = q_w;
  sa.q[1] = q_r;
  sa.subkeys = subkeys;
  sa.scores = scores;
  sa.split = ws + wl.split;
  sa.err = err;
  sa.BT = sh->B * sh->T;
  sa.H = (int32_t)sh->H;
  sa.g = d.g;
  const bool tc = use_tensor_cores(d, sh);
  if ((st = run_kernel(SDM_KERNEL_SCORE, cs, tc ? "score_tc" : "score_simt", [&] {
         return tc ? launch_score_tc(sa, sh->act_dtype, cs) : launch_score_simt(sa, sh->act_dtype, cs);
       })) != SDM_OK)
    return st;
  SelectArgs se{};
  se.scores = scores;
  se.idx[0] = iw;
  se.idx[1] = ir;
  se.wt[0] = ww;
  se.wt[1] = wr;
  se.err = err;
  se.rows = rows;
  se.g = d.g;
  if ((st = run_kernel(SDM_KERNEL_SELECT, cs, "select", [&] { return launch_select(se, cl, EF, EC, sms, cs); })) !=
      SDM_OK)
    return st;

  // 2. chunk plan
  PlanArgs pa{};
  pa.idx[0] = iw;
  pa.idx[1] = ir;
  pa.wt[0] = ww;
  pa.wt[1] = wr;
  pa.gates = gates;
  pa.uniq = reinterpret_cast<int32_t *>(ws + wl.uniq);
  pa.nuniq = reinterpret_cast<int32_t *>(ws + wl.nuniq);
  pa.uo = reinterpret_cast<uint16_t *>(ws + wl.uo);
  pa.written = ws + wl.written;
  pa.lrecs = ws + wl.lrecs;
  pa.crecs = ws + wl.crecs;
  pa.err = err;
  pa.T = sh->T;
  pa.H = (int32_t)sh->H;
  pa.W = sh->W;
  pa.R = sh->R;
  pa.N = d.N;
  pa.pitch16 = (uint32_t)(sh->d_v * sb / 16);
  pa.lay = wc.lay;
  const int P = pow2_at_least(wc.lay.L);
  if ((st = run_kernel(SDM_KERNEL_PLAN_SORT, cs, "plan_sort", [&] { return launch_plan_sort(pa, streams, P, cs); })) != SDM_OK)
    return st;
  if ((st = run_kernel(SDM_KERNEL_PLAN_LINK, cs, "plan_link", [&] { return launch_plan_link(pa, streams, cs); })) != SDM_OK)
    return st;

  // 3. fused gather / delta update / read
  WriteReadArgs wa{};
  wa.k_val = k_val;
  wa.lrecs = ws + wl.lrecs;
  wa.crecs = ws + wl.crecs;
  wa.bank = bank;
  wa.y = y;
  wa.err = err;
  wa.T = sh->T;
  wa.N = d.N;
  wa.d_v = sh->d_v;
  wa.H = (int32_t)sh->H;
  wa.W = sh->W;
  wa.R = sh->R;
  wa.slices = wc.slices;
  wa.row_bytes = (int32_t)(sh->d_v * sb);
  wa.lay = wc.lay;
  wa.snap = snap ? snap->data : nullptr;
  wa.snap_bf16 = snap ? snap->bf16 : 0;
  wa.pieces = (int32_t)snapshot_pieces(sh);
  const WriteReadLaunch wl_launch{wc.NCW, wc.LW, wc.smem};
  if (side) {                                          // the bank copy must land first
    ce = cudaStreamWaitEvent(cs, side->join, 0);
    if (ce != cudaSuccess) return fail(SDM_ERR_CUDA, "side stream join: %s", cudaGetErrorString(ce));
  }
  if ((st = run_kernel(SDM_KERNEL_WRITE_READ, cs, "write_read", [&] {
         return launch_write_read(wa, streams, sh->bank_dtype, sh->act_dtype, wl_launch, cs);
       })) != SDM_OK)
    return st;
  return ok();
}

// ---------------------------------------------------------------- backward

constexpr int64_t kSubkeyChunk = 1024;        // rows of K = 2*B*T per split of the sub-key gradient

struct BwdLayout {
  int64_t flags, part, ds, dk_part, total;
  int64_t P, PS, KS, Pw;
};

BwdLayout bwd_layout(const sdm_shape *sh, const Derived &d) {
  BwdLayout w{};
  const int64_t S = sh->B * sh->H, BT = sh->B * sh->T;
  w.Pw = (sh->d_v * elem_bytes(sh->bank_dtype) + 16 * kSweepCG - 1) / (16 * kSweepCG);
  w.P = kSweepCtaRecord ? (w.Pw + kSweepCtaWarps - 1) / kSweepCtaWarps : w.Pw;
  w.PS = bwd_part_stride(sh->W, sh->R);
  w.KS = (2 * BT + kSubkeyChunk - 1) / kSubkeyChunk;
  int64_t o = kHeaderBytes;
  w.flags = o;   o = a256(o + S * sh->T);
  w.part = o;    o = a256(o + S * sh->T * w.P * w.PS * 4);
  w.ds = o;      o = a256(o + sh->H * 2 * BT * (int64_t)d.ntot * 4);
  w.dk_part = o; o = a256(o + w.KS * sh->H * (int64_t)d.ntot * sh->d_sub * 4);
  w.total = o;
  return w;
}

sdm_status check_snapshot_dtype(int32_t dt) {
  if (dt == SDM_F16) return fail(SDM_ERR_UNSUPPORTED, "snapshot_dtype: float16 is not supported");
  if (dt != SDM_F32 && dt != SDM_BF16) return fail(SDM_ERR_INVALID_ARG, "snapshot_dtype: unknown dtype %d", dt);
  return SDM_OK;
}

sdm_status backward_impl(const sdm_shape *sh, const void *q_w, const void *q_r, const void *k_val,
                         const float *gates, const void *subkeys, const int32_t *idx_w, const float *wt_w,
                         const int32_t *idx_r, const float *wt_r, void *snapshot, size_t snapshot_bytes,
                         int32_t snap_dtype, void *bank, const void *dy, float *dbank, float *d_k_val,
                         float *d_gates, float *d_q_w, float *d_q_r, float *d_subkeys, void *workspace,
                         size_t workspace_bytes, sdm_stream_t stream) {
  Derived d;
  sdm_status st = check_shape(sh, false, &d);
  if (st != SDM_OK) return st;
  if ((st = check_snapshot_dtype(snap_dtype)) != SDM_OK) return st;
  const int64_t ab = elem_bytes(sh->act_dtype), sb = elem_bytes(sh->bank_dtype);
  const int64_t rows = sh->B * sh->T * sh->H;
  const int64_t qbytes = rows * sh->F * sh->d_sub * ab;
  const int64_t table = sh->B * sh->H * d.N * sh->d_v;
  const int64_t skbytes = sh->H * d.ntot * sh->d_sub;
  const Range r_qw{q_w, qbytes, "q_w"}, r_qr{q_r, qbytes, "q_r"}, r_kv{k_val, rows * sh->d_v * ab, "k_val"};
  const Range r_g{gates, rows * 2 * 4, "gates"}, r_sk{subkeys, skbytes * ab, "subkeys"};
  const Range r_iw{idx_w, rows * sh->W * 4, "idx_w"}, r_ww{wt_w, rows * sh->W * 4, "wt_w"};
  const Range r_ir{idx_r, rows * sh->R * 4, "idx_r"}, r_wr{wt_r, rows * sh->R * 4, "wt_r"};
  const Range r_dy{dy, rows * sh->d_v * ab, "dy"};
  const Range r_snap{snapshot, (int64_t)snapshot_bytes, "snapshot"};
  const Range r_b{bank, table * sb, "bank"}, r_db{dbank, table * 4, "dbank"};
  const Range r_dkv{d_k_val, rows * sh->d_v * 4, "d_k_val"}, r_dg{d_gates, rows * 2 * 4, "d_gates"};
  const Range r_dqw{d_q_w, rows * sh->F * sh->d_sub * 4, "d_q_w"}, r_dqr{d_q_r, rows * sh->F * sh->d_sub * 4, "d_q_r"};
  const Range r_dsk{d_subkeys, skbytes * 4, "d_subkeys"};
  const Range r_ws{workspace, (int64_t)workspace_bytes, "workspace"};
  const int64_t need_snap = snapshot_bytes_of(sh, snap_dtype);
  const BwdLayout bl = bwd_layout(sh, d);

  const Range all[] = {r_qw, r_qr, r_kv, r_g, r_sk, r_iw, r_ww, r_ir, r_wr, r_dy, r_snap,
                       r_b, r_db, r_dkv, r_dg, r_dqw, r_dqr, r_dsk};
  if (rows > 0) {
    for (const Range &r : all)
      if (!r.p) return fail(SDM_ERR_INVALID_ARG, "%s is NULL", r.name);
  } else if (!snapshot || (!d_subkeys && skbytes > 0)) {
    return fail(SDM_ERR_INVALID_ARG, "%s is NULL", snapshot ? "d_subkeys" : "snapshot");
  }
  for (const Range &r : all)
    if (r.p && !aligned(r.p, r.p == gates ? 8 : 16))
      return fail(SDM_ERR_INVALID_ARG, "%s is not %d-byte aligned", r.name, r.p == gates ? 8 : 16);
  if ((int64_t)snapshot_bytes < need_snap)
    return fail(SDM_ERR_INVALID_ARG, "snapshot has %zu bytes, needs %lld", snapshot_bytes, (long long)need_snap);
  if (!workspace) return fail(SDM_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 16)) return fail(SDM_ERR_WORKSPACE, "workspace is not 16-byte aligned");
  if ((int64_t)workspace_bytes < bl.total)
    return fail(SDM_ERR_WORKSPACE, "workspace has %zu bytes, needs %lld", workspace_bytes, (long long)bl.total);
  const Range ins[] = {r_qw, r_qr, r_kv, r_g, r_sk, r_iw, r_ww, r_ir, r_wr, r_dy};
  const Range outs[] = {r_snap, r_b, r_db, r_dkv, r_dg, r_dqw, r_dqr, r_dsk, r_ws};
  for (const Range &o : outs)
    for (const Range &i : ins)
      if (overlap(o, i)) return fail(SDM_ERR_ALIAS, "%s overlaps %s", o.name, i.name);
  for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i)
    for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
      if (overlap(outs[i], outs[j])) return fail(SDM_ERR_ALIAS, "%s overlaps %s", outs[i].name, outs[j].name);

  unsigned char *ws = static_cast<unsigned char *>(workspace);
  int32_t *err = reinterpret_cast<int32_t *>(ws);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t ce = cudaMemsetAsync(err, 0, sizeof(int32_t), cs);
  if (ce != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(ce));

  BackwardArgs a{};
  a.idx[0] = idx_w;
  a.idx[1] = idx_r;
  a.wt[0] = wt_w;
  a.wt[1] = wt_r;
  a.gates = gates;
  a.q[0] = q_w;
  a.q[1] = q_r;
  a.k_val = k_val;
  a.dy = dy;
  a.subkeys = subkeys;
  a.snap = static_cast<const unsigned char *>(snapshot) + kSnapshotHeaderBytes;
  a.snap_hdr = static_cast<const int32_t *>(snapshot);
  a.flags = ws + bl.flags;
  a.bank = bank;
  a.grad = dbank;
  a.d_kv = d_k_val;
  a.d_gates = d_gates;
  a.d_q[0] = d_q_w;
  a.d_q[1] = d_q_r;
  a.d_subkeys = d_subkeys;
  a.part = reinterpret_cast<float *>(ws + bl.part);
  a.ds = reinterpret_cast<float *>(ws + bl.ds);
  a.dk_part = reinterpret_cast<float *>(ws + bl.dk_part);
  a.err = err;
  a.B = sh->B;
  a.T = sh->T;
  a.N = d.N;
  a.d_v = sh->d_v;
  a.H = (int32_t)sh->H;
  a.W = sh->W;
  a.R = sh->R;
  a.P = (int32_t)bl.P;
  a.Pw = (int32_t)bl.Pw;
  a.P32 = (int32_t)snapshot_pieces(sh);
  a.PS = (int32_t)bl.PS;
  a.act_bf16 = sh->act_dtype == SDM_BF16;
  a.snap_bf16 = snap_dtype == SDM_BF16;
  a.KS = (int32_t)bl.KS;
  a.k_chunk = kSubkeyChunk;
  a.g = d.g;

  if (rows > 0) {
    if ((st = run_kernel(SDM_KERNEL_BWD_FLAGS, cs, "bwd_flags", [&] { return launch_bwd_flags(a, cs); })) != SDM_OK)
      return st;
    if ((st = run_kernel(SDM_KERNEL_BWD_SWEEP, cs, "bwd_sweep",
                         [&] { return launch_bwd_sweep(a, sh->bank_dtype, cs); })) != SDM_OK)
      return st;
  }
  // the snapshot is spent: a second backward through it is refused
  ce = cudaMemsetAsync(snapshot, 0, sizeof(int32_t), cs);
  if (ce != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(ce));
  if (rows > 0 &&
      (st = run_kernel(SDM_KERNEL_BWD_REDUCE, cs, "bwd_reduce", [&] { return launch_bwd_reduce(a, cs); })) != SDM_OK)
    return st;
  if ((st = run_kernel(SDM_KERNEL_BWD_SUBKEY, cs, "bwd_subkeys", [&] { return launch_bwd_subkeys(a, cs); })) !=
      SDM_OK)
    return st;
  return ok();
}

// sdm_write_read_train's checks and work (also the op of the layer's training forward).
sdm_status train_forward_impl(const sdm_shape *sh, const void *q_w, const void *q_r, const void *k_val,
                              const float *gates, const void *subkeys, const void *bank_init, void *bank, void *y,
                              int32_t *idx_w, float *wt_w, int32_t *idx_r, float *wt_r, void *snapshot,
                              size_t snapshot_bytes, int32_t snapshot_dtype, void *workspace, size_t workspace_bytes,
                              sdm_stream_t stream) {
  sdm_status st = check_shape(sh, false, nullptr);
  if (st != SDM_OK) return st;
  if ((st = check_snapshot_dtype(snapshot_dtype)) != SDM_OK) return st;
  const int64_t rows = sh->B * sh->T * sh->H;
  if (!snapshot) return fail(SDM_ERR_INVALID_ARG, "snapshot is NULL");
  if (!aligned(snapshot, 16)) return fail(SDM_ERR_INVALID_ARG, "snapshot is not 16-byte aligned");
  const int64_t need = snapshot_bytes_of(sh, snapshot_dtype);
  if ((int64_t)snapshot_bytes < need)
    return fail(SDM_ERR_INVALID_ARG, "snapshot has %zu bytes, needs %lld", snapshot_bytes, (long long)need);
  const Range r_snap{snapshot, (int64_t)snapshot_bytes, "snapshot"};
  const Range sel[] = {{idx_w, rows * sh->W * 4, "idx_w"}, {wt_w, rows * sh->W * 4, "wt_w"},
                       {idx_r, rows * sh->R * 4, "idx_r"}, {wt_r, rows * sh->R * 4, "wt_r"}};
  for (const Range &r : sel) {
    if (rows > 0 && !r.p) return fail(SDM_ERR_INVALID_ARG, "%s is NULL (the backward reads it)", r.name);
    if (r.p && !aligned(r.p, 16)) return fail(SDM_ERR_INVALID_ARG, "%s is not 16-byte aligned", r.name);
  }
  Derived d;
  check_shape(sh, false, &d);
  const int64_t ab = elem_bytes(sh->act_dtype), sb = elem_bytes(sh->bank_dtype);
  const Range others[] = {{q_w, rows * sh->F * sh->d_sub * ab, "q_w"}, {q_r, rows * sh->F * sh->d_sub * ab, "q_r"},
                          {k_val, rows * sh->d_v * ab, "k_val"}, {gates, rows * 8, "gates"},
                          {subkeys, sh->H * d.ntot * sh->d_sub * ab, "subkeys"},
                          {bank_init, sh->H * d.N * sh->d_v * sb, "bank_init"},
                          {bank, sh->B * sh->H * d.N * sh->d_v * sb, "bank"}, {y, rows * sh->d_v * ab, "y"},
                          sel[0], sel[1], sel[2], sel[3],
                          {workspace, (int64_t)workspace_bytes, "workspace"}};
  for (const Range &o : others)
    if (overlap(r_snap, o)) return fail(SDM_ERR_ALIAS, "snapshot overlaps %s", o.name);
  const SnapOut so{static_cast<unsigned char *>(snapshot) + kSnapshotHeaderBytes, snapshot_dtype == SDM_BF16};
  st = write_read_impl(sh, q_w, q_r, k_val, gates, subkeys, bank_init, bank, y, idx_w, wt_w, idx_r, wt_r,
                       workspace, workspace_bytes, stream, true, &so);
  if (st != SDM_OK) return st;
  // armed for one backward, once the forward's kernels are done (stream order)
  const cudaError_t ce = cudaMemsetAsync(snapshot, 0x5a, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(ce));
  return ok();
}

// ---------------------------------------------------------------- the layer around the op

struct LayerLayout {
  int64_t op_ws, q_w, q_r, k_val, gates, y, gemm, total;
};

LayerLayout layer_layout(const sdm_shape *sh, const Derived &d) {
  LayerLayout w{};
  const int64_t rows = sh->B * sh->T * sh->H, ab = elem_bytes(sh->act_dtype);
  int64_t o = 0;
  w.op_ws = o;  o = a256(o + write_read_ws_bytes(sh));
  w.q_w = o;    o = a256(o + rows * d.g.F * sh->d_sub * ab);
  w.q_r = o;    o = a256(o + rows * d.g.F * sh->d_sub * ab);
  w.k_val = o;  o = a256(o + rows * sh->d_v * ab);
  w.gates = o;  o = a256(o + rows * 2 * 4);
  w.y = o;      o = a256(o + rows * sh->d_v * ab);
  w.gemm = o;   o = a256(o + kLayerGemmWorkspace);
  w.total = o;
  return w;
}

sdm_status layer_impl(const sdm_shape *sh, int64_t dim, const void *x, const void *w_qw, const void *w_qr,
                      const void *w_v, const void *w_g, const void *w_o, const void *subkeys,
                      const void *bank_init, void *bank, void *out, void *q_w, void *q_r, void *k_val,
                      float *gates, void *y, void *workspace, size_t workspace_bytes, sdm_stream_t stream,
                      const sdm_layer_saved *saved = nullptr) {
  Derived d;
  sdm_status st = check_shape(sh, false, &d);
  if (st != SDM_OK) return st;
  if (dim < 1) return fail(SDM_ERR_INVALID_ARG, "dim must be >= 1");
  if (saved && sh->B * sh->T * sh->H > 0 &&
      !(saved->q_w && saved->q_r && saved->k_val && saved->gates && saved->y))
    return fail(SDM_ERR_INVALID_ARG, "saved: the intermediates are required for training");
  const int64_t ab = elem_bytes(sh->act_dtype), BT = sh->B * sh->T, rows = BT * sh->H;
  const int64_t dq = (int64_t)d.g.F * sh->d_sub * sh->H;            // query width of a token
  const int64_t dv = sh->d_v * sh->H;
  const LayerLayout ll = layer_layout(sh, d);
  const Range r_x{x, BT * dim * ab, "x"}, r_out{out, BT * dim * ab, "out"};
  const Range r_wqw{w_qw, dq * dim * ab, "w_qw"}, r_wqr{w_qr, dq * dim * ab, "w_qr"};
  const Range r_wv{w_v, dv * dim * ab, "w_v"}, r_wg{w_g, 2 * sh->H * dim * ab, "w_g"}, r_wo{w_o, dim * dv * ab, "w_o"};
  const Range r_ws{workspace, (int64_t)workspace_bytes, "workspace"};
  if (rows > 0) {
    const Range req[] = {r_x, r_out, r_wqw, r_wqr, r_wv, r_wg, r_wo};
    for (const Range &r : req)
      if (!r.p) return fail(SDM_ERR_INVALID_ARG, "%s is NULL", r.name);
  }
  const Range al[] = {r_x, r_out, r_wqw, r_wqr, r_wv, r_wg, r_wo, {q_w, 1, "q_w"}, {q_r, 1, "q_r"},
                      {k_val, 1, "k_val"}, {gates, 1, "gates"}, {y, 1, "y"}};
  for (const Range &r : al)
    if (r.p && !aligned(r.p, 16)) return fail(SDM_ERR_INVALID_ARG, "%s is not 16-byte aligned", r.name);
  if (!workspace) return fail(SDM_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(SDM_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if ((int64_t)workspace_bytes < ll.total)
    return fail(SDM_ERR_WORKSPACE, "workspace has %zu bytes, needs %lld", workspace_bytes, (long long)ll.total);
  const Range ins[] = {r_x, r_wqw, r_wqr, r_wv, r_wg, r_wo};
  const Range outs[] = {r_out, r_ws, {q_w, rows * d.g.F * sh->d_sub * ab, "q_w"},
                        {q_r, rows * d.g.F * sh->d_sub * ab, "q_r"}, {k_val, rows * sh->d_v * ab, "k_val"},
                        {gates, rows * 8, "gates"}, {y, rows * sh->d_v * ab, "y"}};
  for (const Range &o : outs)
    for (const Range &i : ins)
      if (overlap(o, i)) return fail(SDM_ERR_ALIAS, "%s overlaps %s", o.name, i.name);
  for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i)
    for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
      if (overlap(outs[i], outs[j])) return fail(SDM_ERR_ALIAS, "%s overlaps %s", outs[i].name, outs[j].name);

  unsigned char *ws = static_cast<unsigned char *>(workspace);
  void *qw = q_w ? q_w : ws + ll.q_w, *qr = q_r ? q_r : ws + ll.q_r, *kv = k_val ? k_val : ws + ll.k_val;
  float *gt = gates ? gates : reinterpret_cast<float *>(ws + ll.gates);
  void *yy = y ? y : ws + ll.y;
  void *gws = ws + ll.gemm;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int sms = 0;
  if ((st = sm_count(&sms)) != SDM_OK) return st;
  const int adt = sh->act_dtype;
  if (rows > 0) {
    // input projections, then the gates
    if ((st = run_library(SDM_KERNEL_LAYER_GEMM, cs, "layer q_w projection", [&] {
           return layer_gemm(w_qw, x, qw, dq, BT, dim, adt, gws, kLayerGemmWorkspace, cs);
         })) != SDM_OK)
      return st;
    if ((st = run_library(SDM_KERNEL_LAYER_GEMM, cs, "layer q_r projection", [&] {
           return layer_gemm(w_qr, x, qr, dq, BT, dim, adt, gws, kLayerGemmWorkspace, cs);
         })) != SDM_OK)
      return st;
    if ((st = run_library(SDM_KERNEL_LAYER_GEMM, cs, "layer value projection", [&] {
           return layer_gemm(w_v, x, kv, dv, BT, dim, adt, gws, kLayerGemmWorkspace, cs);
         })) != SDM_OK)
      return st;
    if ((st = run_kernel(SDM_KERNEL_LAYER_GATES, cs, "layer_gates", [&] {
           return launch_layer_gates(x, w_g, gt, BT, dim, (int32_t)(2 * sh->H), adt, sms, cs);
         })) != SDM_OK)
      return st;
  }
  // the op (with the training forward's snapshot and selections when training)
  if (saved) st = train_forward_impl(sh, qw, qr, kv, gt, subkeys, bank_init, bank, yy, saved->idx_w, saved->wt_w,
                                     saved->idx_r, saved->wt_r, saved->snapshot, saved->snapshot_bytes,
                                     saved->snapshot_dtype, ws + ll.op_ws, (size_t)(ll.q_w - ll.op_ws), stream);
  else st = write_read_impl(sh, qw, qr, kv, gt, subkeys, bank_init, bank, yy, nullptr, nullptr, nullptr, nullptr,
                            ws + ll.op_ws, (size_t)(ll.q_w - ll.op_ws), stream, true);
  if (st != SDM_OK) return st;
  if (rows > 0 &&
      (st = run_library(SDM_KERNEL_LAYER_GEMM, cs, "layer output projection", [&] {
         return layer_gemm(w_o, yy, out, dim, BT, dv, adt, gws, kLayerGemmWorkspace, cs);
       })) != SDM_OK)
    return st;
  return ok();
}

// ---------------------------------------------------------------- the layer's backward

struct LayerBwdLayout {
  int64_t op_ws, dY, d_qw, d_qr, d_kv, d_g, gcat, wcat, gemm, total;
  int64_t dq, dv, ng, K, Kp;
};

LayerBwdLayout layer_bwd_layout(const sdm_shape *sh, const Derived &d, int64_t dim) {
  LayerBwdLayout w{};
  const int64_t BT = sh->B * sh->T, ab = elem_bytes(sh->act_dtype);
  w.dq = (int64_t)d.g.F * sh->d_sub * sh->H;
  w.dv = sh->d_v * sh->H;
  w.ng = 2 * sh->H;
  w.K = 2 * w.dq + w.dv + w.ng;
  w.Kp = (w.K + 7) / 8 * 8;          // row stride of G and rows of W: 16-byte multiples (zero padding)
  int64_t o = 0;
  w.op_ws = o; o = a256(o + bwd_layout(sh, d).total);
  w.dY = o;    o = a256(o + BT * w.dv * ab);
  w.d_qw = o;  o = a256(o + BT * w.dq * 4);
  w.d_qr = o;  o = a256(o + BT * w.dq * 4);
  w.d_kv = o;  o = a256(o + BT * w.dv * 4);
  w.d_g = o;   o = a256(o + BT * w.ng * 4);
  w.gcat = o;  o = a256(o + BT * w.Kp * ab);
  w.wcat = o;  o = a256(o + w.Kp * dim * ab);
  w.gemm = o;  o = a256(o + kLayerGemmWorkspace);
  w.total = o;
  return w;
}

sdm_status layer_backward_impl(const sdm_shape *sh, int64_t dim, const void *x, const void *w_qw, const void *w_qr,
                               const void *w_v, const void *w_g, const void *w_o, const void *subkeys, void *bank,
                               const void *dout, const sdm_layer_saved *sv, const sdm_layer_grads *gr,
                               void *workspace, size_t workspace_bytes, sdm_stream_t stream) {
  Derived d;
  sdm_status st = check_shape(sh, false, &d);
  if (st != SDM_OK) return st;
  if (dim < 1) return fail(SDM_ERR_INVALID_ARG, "dim must be >= 1");
  if (!sv || !gr) return fail(SDM_ERR_INVALID_ARG, "saved and grads are required");
  const int64_t ab = elem_bytes(sh->act_dtype), BT = sh->B * sh->T;
  const LayerBwdLayout L = layer_bwd_layout(sh, d, dim);
  const Range need[] = {{x, BT * dim * ab, "x"}, {w_qw, L.dq * dim * ab, "w_qw"}, {w_qr, L.dq * dim * ab, "w_qr"},
                        {w_v, L.dv * dim * ab, "w_v"}, {w_g, L.ng * dim * ab, "w_g"}, {w_o, dim * L.dv * ab, "w_o"},
                        {dout, BT * dim * ab, "dout"}, {sv->y, BT * L.dv * ab, "saved.y"},
                        {gr->dx, BT * dim * ab, "grads.dx"}, {gr->dw_qw, L.dq * dim * 4, "grads.dw_qw"},
                        {gr->dw_qr, L.dq * dim * 4, "grads.dw_qr"}, {gr->dw_v, L.dv * dim * 4, "grads.dw_v"},
                        {gr->dw_g, L.ng * dim * 4, "grads.dw_g"}, {gr->dw_o, dim * L.dv * 4, "grads.dw_o"}};
  for (const Range &r : need) {
    if (BT * sh->H > 0 && !r.p) return fail(SDM_ERR_INVALID_ARG, "%s is NULL", r.name);
    if (r.p && !aligned(r.p, 16)) return fail(SDM_ERR_INVALID_ARG, "%s is not 16-byte aligned", r.name);
  }
  if (gr->d_bank_init && !aligned(gr->d_bank_init, 16))
    return fail(SDM_ERR_INVALID_ARG, "grads.d_bank_init is not 16-byte aligned");
  if (!workspace) return fail(SDM_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(SDM_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if ((int64_t)workspace_bytes < L.total)
    return fail(SDM_ERR_WORKSPACE, "workspace has %zu bytes, needs %lld", workspace_bytes, (long long)L.total);
  // outputs written before the op's backward checks its own arguments: none may overlap
  // an input or each other
  const Range ins[] = {need[0], need[1], need[2], need[3], need[4], need[5], need[6], need[7],
                       {sv->q_w, BT * L.dq * ab, "saved.q_w"}, {sv->q_r, BT * L.dq * ab, "saved.q_r"},
                       {sv->k_val, BT * L.dv * ab, "saved.k_val"}, {sv->gates, BT * L.ng * 4, "saved.gates"}};
  const Range outs[] = {need[8], need[9], need[10], need[11], need[12], need[13],
                        {gr->d_bank_init, sh->H * d.N * sh->d_v * 4, "grads.d_bank_init"},
                        {gr->dbank, sh->B * sh->H * d.N * sh->d_v * 4, "grads.dbank"},
                        {workspace, (int64_t)workspace_bytes, "workspace"}};
  for (const Range &o : outs)
    for (const Range &i : ins)
      if (overlap(o, i)) return fail(SDM_ERR_ALIAS, "%s overlaps %s", o.name, i.name);
  for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i)
    for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
      if (overlap(outs[i], outs[j])) return fail(SDM_ERR_ALIAS, "%s overlaps %s", outs[i].name, outs[j].name);

  unsigned char *ws = static_cast<unsigned char *>(workspace);
  void *gws = ws + L.gemm;
  void *dY = ws + L.dY, *gcat = ws + L.gcat, *wcat = ws + L.wcat;
  float *d_qw = reinterpret_cast<float *>(ws + L.d_qw), *d_qr = reinterpret_cast<float *>(ws + L.d_qr);
  float *d_kv = reinterpret_cast<float *>(ws + L.d_kv), *d_g = reinterpret_cast<float *>(ws + L.d_g);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int adt = sh->act_dtype;
  int sms = 0;
  if ((st = sm_count(&sms)) != SDM_OK) return st;
  const size_t gwb = (size_t)kLayerGemmWorkspace;
  if (BT > 0) {
    // dY = dout w_o (the op's dy) and dw_o = dout^T Y
    if ((st = run_library(SDM_KERNEL_LAYER_GEMM, cs, "layer dY", [&] {
           return lt_gemm(false, false, L.dv, BT, dim, w_o, L.dv, dout, dim, dY, L.dv, adt, adt, false, gws, gwb, cs);
         })) != SDM_OK)
      return st;
    if ((st = run_library(SDM_KERNEL_LAYER_GEMM, cs, "layer dw_o", [&] {
           return lt_gemm(false, true, L.dv, dim, BT, sv->y, L.dv, dout, dim, gr->dw_o, L.dv, adt, SDM_F32, false,
                          gws, gwb, cs);
         })) != SDM_OK)
      return st;
  }
  // the op's backward (restores the bank, disarms the snapshot)
  if ((st = backward_impl(sh, sv->q_w, sv->q_r, sv->k_val, sv->gates, subkeys, sv->idx_w, sv->wt_w, sv->idx_r,
                          sv->wt_r, sv->snapshot, sv->snapshot_bytes, sv->snapshot_dtype, bank, dY, gr->dbank, d_kv,
                          d_g, d_qw, d_qr, gr->d_subkeys, ws + L.op_ws, (size_t)(L.dY - L.op_ws), stream)) != SDM_OK)
    return st;
  if (BT > 0) {
    // G = [d_q_w | d_q_r | d_k_val | dz], W = [w_qw; w_qr; w_v; w_g]
    if ((st = run_kernel(SDM_KERNEL_LAYER_GRAD, cs, "layer_grad_cat", [&] {
           return launch_layer_grad_cat(d_qw, d_qr, d_kv, d_g, sv->gates, gcat, BT, L.dq, L.dv, L.ng, L.Kp, adt, sms,
                                        cs);
         })) != SDM_OK)
      return st;
    const void *wsrc[] = {w_qw, w_qr, w_v, w_g};
    const int64_t wrows[] = {L.dq, L.dq, L.dv, L.ng};
    int64_t roff = 0;
    for (int i = 0; i < 4; ++i) {
      const cudaError_t ce = cudaMemcpyAsync(static_cast<unsigned char *>(wcat) + roff * dim * ab, wsrc[i],
                                             (size_t)(wrows[i] * dim * ab), cudaMemcpyDeviceToDevice, cs);
      if (ce != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaMemcpyAsync: %s", cudaGetErrorString(ce));
      roff += wrows[i];
    }
    if (L.Kp > L.K) {                                 // the padding rows of W are zero
      const cudaError_t ce = cudaMemsetAsync(static_cast<unsigned char *>(wcat) + L.K * dim * ab, 0,
                                             (size_t)((L.Kp - L.K) * dim * ab), cs);
      if (ce != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(ce));
    }
    // dx = G W
    if ((st = run_library(SDM_KERNEL_LAYER_GEMM, cs, "layer dx", [&] {
           return lt_gemm(false, false, dim, BT, L.Kp, wcat, dim, gcat, L.Kp, gr->dx, dim, adt, adt, false, gws, gwb,
                          cs);
         })) != SDM_OK)
      return st;
    // dw_* = G_*^T X, G_* the columns of G that belong to the weight
    float *dws[] = {gr->dw_qw, gr->dw_qr, gr->dw_v, gr->dw_g};
    int64_t coff = 0;
    for (int i = 0; i < 4; ++i) {
      const void *gi = static_cast<const unsigned char *>(gcat) + coff * ab;
      if ((st = run_library(SDM_KERNEL_LAYER_GEMM, cs, "layer dw", [&] {
             return lt_gemm(false, true, dim, wrows[i], BT, x, dim, gi, L.Kp, dws[i], dim, adt, SDM_F32, false, gws,
                            gwb, cs);
           })) != SDM_OK)
        return st;
      coff += wrows[i];
    }
  }
  if (gr->d_bank_init &&
      (st = run_kernel(SDM_KERNEL_LAYER_GRAD, cs, "batch_sum", [&] {
         return launch_batch_sum(gr->dbank, gr->d_bank_init, sh->B, sh->H * d.N * sh->d_v, sms, cs);
       })) != SDM_OK)
    return st;
  return ok();
}

}  // namespace

// =================================================================== C ABI

extern "C" {

sdm_status sdm_write_read_workspace_size(const sdm_shape *shape, size_t *bytes) {
  if (!bytes) return fail(SDM_ERR_INVALID_ARG, "bytes is NULL");
  Derived d;
  sdm_status st = check_shape(shape, false, &d);
  if (st != SDM_OK) return st;
  *bytes = (size_t)write_read_ws_bytes(shape);
  return ok();
}

sdm_status sdm_decode_workspace_size(const sdm_shape *shape, size_t *bytes) {
  if (!bytes) return fail(SDM_ERR_INVALID_ARG, "bytes is NULL");
  sdm_status st = check_shape(shape, true, nullptr);
  if (st != SDM_OK) return st;
  *bytes = (size_t)kHeaderBytes;
  return ok();
}

sdm_status sdm_write_read(const sdm_shape *sh, const void *q_w, const void *q_r, const void *k_val,
                          const float *gates, const void *subkeys, const void *bank_init, void *bank,
                          void *y, int32_t *idx_w, float *wt_w, int32_t *idx_r, float *wt_r,
                          void *workspace, size_t workspace_bytes, sdm_stream_t stream) {
  return write_read_impl(sh, q_w, q_r, k_val, gates, subkeys, bank_init, bank, y, idx_w, wt_w, idx_r, wt_r,
                         workspace, workspace_bytes, stream, true);
}

sdm_status sdm_snapshot_bytes(const sdm_shape *shape, int32_t snapshot_dtype, size_t *bytes) {
  if (!bytes) return fail(SDM_ERR_INVALID_ARG, "bytes is NULL");
  sdm_status st = check_shape(shape, false, nullptr);
  if (st != SDM_OK) return st;
  if ((st = check_snapshot_dtype(snapshot_dtype)) != SDM_OK) return st;
  *bytes = (size_t)snapshot_bytes_of(shape, snapshot_dtype);
  return ok();
}

sdm_status sdm_write_read_train(const sdm_shape *sh, const void *q_w, const void *q_r, const void *k_val,
                                const float *gates, const void *subkeys, const void *bank_init, void *bank,
                                void *y, int32_t *idx_w, float *wt_w, int32_t *idx_r, float *wt_r,
                                void *snapshot, size_t snapshot_bytes, int32_t snapshot_dtype, void *workspace,
                                size_t workspace_bytes, sdm_stream_t stream) {
  return train_forward_impl(sh, q_w, q_r, k_val, gates, subkeys, bank_init, bank, y, idx_w, wt_w, idx_r, wt_r,
                            snapshot, snapshot_bytes, snapshot_dtype, workspace, workspace_bytes, stream);
}

sdm_status sdm_write_read_backward_workspace_size(const sdm_shape *shape, size_t *bytes) {
  if (!bytes) return fail(SDM_ERR_INVALID_ARG, "bytes is NULL");
  Derived d;
  sdm_status st = check_shape(shape, false, &d);
  if (st != SDM_OK) return st;
  *bytes = (size_t)bwd_layout(shape, d).total;
  return ok();
}

sdm_status sdm_write_read_backward(const sdm_shape *sh, const void *q_w, const void *q_r, const void *k_val,
                                   const float *gates, const void *subkeys, const int32_t *idx_w, const float *wt_w,
                                   const int32_t *idx_r, const float *wt_r, void *snapshot, size_t snapshot_bytes,
                                   int32_t snapshot_dtype, void *bank, const void *dy, float *dbank, float *d_k_val,
                                   float *d_gates, float *d_q_w, float *d_q_r, float *d_subkeys, void *workspace,
                                   size_t workspace_bytes, sdm_stream_t stream) {
  return backward_impl(sh, q_w, q_r, k_val, gates, subkeys, idx_w, wt_w, idx_r, wt_r, snapshot, snapshot_bytes,
                       snapshot_dtype, bank, dy, dbank, d_k_val, d_gates, d_q_w, d_q_r, d_subkeys, workspace,
                       workspace_bytes, stream);
}

sdm_status sdm_layer_workspace_size(const sdm_shape *shape, int64_t dim, size_t *bytes) {
  if (!bytes) return fail(SDM_ERR_INVALID_ARG, "bytes is NULL");
  Derived d;
  sdm_status st = check_shape(shape, false, &d);
  if (st != SDM_OK) return st;
  if (dim < 1) return fail(SDM_ERR_INVALID_ARG, "dim must be >= 1");
  *bytes = (size_t)layer_layout(shape, d).total;
  return ok();
}

sdm_status sdm_layer_forward(const sdm_shape *sh, int64_t dim, const void *x, const void *w_qw, const void *w_qr,
                             const void *w_v, const void *w_g, const void *w_o, const void *subkeys,
                             const void *bank_init, void *bank, void *out, void *q_w, void *q_r, void *k_val,
                             float *gates, void *y, void *workspace, size_t workspace_bytes, sdm_stream_t stream) {
  return layer_impl(sh, dim, x, w_qw, w_qr, w_v, w_g, w_o, subkeys, bank_init, bank, out, q_w, q_r, k_val, gates,
                    y, workspace, workspace_bytes, stream);
}

sdm_status sdm_layer_forward_train(const sdm_shape *sh, int64_t dim, const void *x, const void *w_qw,
                                   const void *w_qr, const void *w_v, const void *w_g, const void *w_o,
                                   const void *subkeys, const void *bank_init, void *bank, void *out,
                                   const sdm_layer_saved *saved, void *workspace, size_t workspace_bytes,
                                   sdm_stream_t stream) {
  if (!saved) return fail(SDM_ERR_INVALID_ARG, "saved is NULL");
  return layer_impl(sh, dim, x, w_qw, w_qr, w_v, w_g, w_o, subkeys, bank_init, bank, out, saved->q_w, saved->q_r,
                    saved->k_val, saved->gates, saved->y, workspace, workspace_bytes, stream, saved);
}

sdm_status sdm_layer_backward_workspace_size(const sdm_shape *shape, int64_t dim, size_t *bytes) {
  if (!bytes) return fail(SDM_ERR_INVALID_ARG, "bytes is NULL");
  Derived d;
  sdm_status st = check_shape(shape, false, &d);
  if (st != SDM_OK) return st;
  if (dim < 1) return fail(SDM_ERR_INVALID_ARG, "dim must be >= 1");
  *bytes = (size_t)layer_bwd_layout(shape, d, dim).total;
  return ok();
}

sdm_status sdm_layer_backward(const sdm_shape *sh, int64_t dim, const void *x, const void *w_qw, const void *w_qr,
                              const void *w_v, const void *w_g, const void *w_o, const void *subkeys, void *bank,
                              const void *dout, const sdm_layer_saved *saved, const sdm_layer_grads *grads,
                              void *workspace, size_t workspace_bytes, sdm_stream_t stream) {
  return layer_backward_impl(sh, dim, x, w_qw, w_qr, w_v, w_g, w_o, subkeys, bank, dout, saved, grads, workspace,
                             workspace_bytes, stream);
}

sdm_status sdm_decode_step(const sdm_shape *sh, const void *q_w, const void *q_r, const void *k_val,
                           const float *gates, const void *subkeys, const void *bank_in, int bank_in_shared,
                           void *bank_out, int donate, void *y, int32_t *idx_w, float *wt_w, int32_t *idx_r,
                           float *wt_r, void *workspace, size_t workspace_bytes, sdm_stream_t stream) {
  Derived d;
  sdm_status st = check_shape(sh, true, &d);
  if (st != SDM_OK) return st;
  static thread_local CandidateList cl;
  if ((st = build_candidates(d, &cl)) != SDM_OK) return st;
  if (donate) {
    if (bank_in_shared) return fail(SDM_ERR_INVALID_ARG, "a shared (broadcast) bank cannot be donated");
    if (bank_out == nullptr) bank_out = const_cast<void *>(bank_in);
    if (bank_out != bank_in) return fail(SDM_ERR_ALIAS, "donate needs bank_out == bank_in");
  }
  const int64_t ab = elem_bytes(sh->act_dtype), sb = elem_bytes(sh->bank_dtype);
  const int64_t rows = sh->B * sh->H;
  const int64_t qbytes = rows * sh->F * sh->d_sub * ab;
  const Range r_qw{q_w, qbytes, "q_w"}, r_qr{q_r, qbytes, "q_r"}, r_kv{k_val, rows * sh->d_v * ab, "k_val"};
  const Range r_g{gates, rows * 2 * 4, "gates"}, r_sk{subkeys, sh->H * d.ntot * sh->d_sub * ab, "subkeys"};
  const int64_t table = d.N * sh->d_v * sb;
  const Range r_bi{bank_in, (bank_in_shared ? sh->H : rows) * table, "bank_in"};
  const Range r_bo{bank_out, rows * table, "bank_out"};
  const Range r_y{y, rows * sh->d_v * ab, "y"};
  const Range r_iw{idx_w, rows * sh->W * 4, "idx_w"}, r_ww{wt_w, rows * sh->W * 4, "wt_w"};
  const Range r_ir{idx_r, rows * sh->R * 4, "idx_r"}, r_wr{wt_r, rows * sh->R * 4, "wt_r"};
  const Range r_ws{workspace, (int64_t)workspace_bytes, "workspace"};
  if (rows > 0) {
    const Range req[] = {r_qw, r_qr, r_kv, r_g, r_sk, r_bi, r_bo, r_y};
    for (const Range &r : req)
      if (!r.p) return fail(SDM_ERR_INVALID_ARG, "%s is NULL", r.name);
  }
  const Range al16[] = {r_qw, r_qr, r_kv, r_sk, r_bi, r_bo, r_y};
  for (const Range &r : al16)
    if (r.p && !aligned(r.p, 16)) return fail(SDM_ERR_INVALID_ARG, "%s is not 16-byte aligned", r.name);
  if (gates && !aligned(gates, 8)) return fail(SDM_ERR_INVALID_ARG, "gates is not 8-byte aligned");
  const Range al4[] = {r_iw, r_ww, r_ir, r_wr};
  for (const Range &r : al4)
    if (r.p && !aligned(r.p, 4)) return fail(SDM_ERR_INVALID_ARG, "%s is not 4-byte aligned", r.name);
  if (!workspace) return fail(SDM_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 16)) return fail(SDM_ERR_WORKSPACE, "workspace is not 16-byte aligned");
  if ((int64_t)workspace_bytes < kHeaderBytes)
    return fail(SDM_ERR_WORKSPACE, "workspace has %zu bytes, needs %lld", workspace_bytes, (long long)kHeaderBytes);
  const Range ins[] = {r_qw, r_qr, r_kv, r_g, r_sk};
  const Range outs[] = {r_bo, r_y, r_iw, r_ww, r_ir, r_wr, r_ws};
  for (const Range &o : outs)
    for (const Range &i : ins)
      if (overlap(o, i)) return fail(SDM_ERR_ALIAS, "%s overlaps %s", o.name, i.name);
  for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i)
    for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
      if (overlap(outs[i], outs[j])) return fail(SDM_ERR_ALIAS, "%s overlaps %s", outs[i].name, outs[j].name);
  const Range bin_others[] = {r_y, r_iw, r_ww, r_ir, r_wr, r_ws};
  for (const Range &o : bin_others)
    if (overlap(o, r_bi)) return fail(SDM_ERR_ALIAS, "%s overlaps bank_in", o.name);
  if (!donate && overlap(r_bi, r_bo)) return fail(SDM_ERR_ALIAS, "bank_out overlaps bank_in (use donate)");

  const int64_t region = decode_region_bytes(sh->W, sh->R, !donate);
  const int64_t smem = region + (int64_t)2 * (sh->F * sh->d_sub + 1) * 4 + (int64_t)2 * d.ntot * 4 +
                       (int64_t)(cl.n[0] + cl.n[1]) * 4;
  if (smem > 200 * 1024) return fail(SDM_ERR_UNSUPPORTED, "decode needs %lld bytes of shared memory", (long long)smem);

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int32_t *err = static_cast<int32_t *>(workspace);
  cudaError_t ce = cudaMemsetAsync(err, 0, sizeof(int32_t), cs);
  if (ce != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(ce));
  if (rows == 0) return ok();

  int EF, EC;
  sort_widths(d, cl, &EF, &EC);
  DecodeArgs da{};
  da.q[0] = q_w;
  da.q[1] = q_r;
  da.k_val = k_val;
  da.gates = gates;
  da.subkeys = subkeys;
  da.bank_in = bank_in;
  da.bank_out = bank_out;
  da.y = y;
  da.idx[0] = idx_w;
  da.idx[1] = idx_r;
  da.wt[0] = wt_w;
  da.wt[1] = wt_r;
  da.err = err;
  da.B = sh->B;
  da.N = d.N;
  da.d_v = sh->d_v;
  da.H = (int32_t)sh->H;
  da.bank_in_shared = bank_in_shared ? 1 : 0;
  da.copy_rest = donate ? 0 : 1;
  da.region_bytes = region;
  da.test_stall_copy = g_test_stall_decode_copy.load();
  da.g = d.g;
  if ((st = run_kernel(SDM_KERNEL_DECODE, cs, "decode",
                       [&] { return launch_decode(da, cl, sh->act_dtype, sh->bank_dtype, EF, EC, smem, cs); })) != SDM_OK)
    return st;
  return ok();
}

sdm_status sdm_last_device_error(const void *workspace, size_t workspace_bytes, int32_t *code,
                                 sdm_stream_t stream) {
  if (!code) return fail(SDM_ERR_INVALID_ARG, "code is NULL");
  if (!workspace || workspace_bytes < sizeof(int32_t)) return fail(SDM_ERR_WORKSPACE, "workspace too small");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return fail(SDM_ERR_CUDA, "reading the device flag: %s", cudaGetErrorString(e));
  *code = v;
  if (v != 0) return fail(SDM_ERR_DEVICE, "kernel-side error code %d", v);
  return ok();
}

const char *sdm_status_string(sdm_status s) {
  switch (s) {
    case SDM_OK: return "ok";
    case SDM_ERR_INVALID_ARG: return "invalid argument";
    case SDM_ERR_UNSUPPORTED: return "unsupported configuration";
    case SDM_ERR_ALIAS: return "buffers overlap";
    case SDM_ERR_WORKSPACE: return "workspace missing or too small";
    case SDM_ERR_CUDA: return "CUDA error";
    case SDM_ERR_DEVICE: return "kernel-side error";
  }
  return "unknown status";
}

const char *sdm_last_error_message(void) { return g_msg; }

int32_t sdm_abi_version(void) { return SDM_ABI_VERSION; }

uint64_t sdm_launch_count(void) { return g_launches.load(); }

sdm_status sdm_test_stall_decode_copy(int on) {
  g_test_stall_decode_copy.store(on ? 1 : 0);
  return SDM_OK;
}

sdm_status sdm_test_force_write_read_layout(int slice_bytes, int stage_tokens) {
  if (!(slice_bytes == 0 || slice_bytes == 32 || slice_bytes == 128 || slice_bytes == 256) || stage_tokens < 0)
    return fail(SDM_ERR_INVALID_ARG, "slice_bytes must be 0, 32, 128 or 256 and stage_tokens >= 0");
  g_test_slice_bytes.store(slice_bytes);
  g_test_stage_tokens.store(stage_tokens);
  return ok();
}

sdm_status sdm_test_factor_scores(const sdm_shape *sh, const void *q_w, const void *q_r, const void *subkeys,
                                  float *scores, void *workspace, size_t workspace_bytes, sdm_stream_t stream) {
  Derived d;
  sdm_status st = check_shape(sh, false, &d);
  if (st != SDM_OK) return st;
  const int64_t ab = elem_bytes(sh->act_dtype);
  const int64_t rows = sh->B * sh->T * sh->H;
  const int64_t qbytes = rows * sh->F * sh->d_sub * ab;
  const Range r_qw{q_w, qbytes, "q_w"}, r_qr{q_r, qbytes, "q_r"};
  const Range r_sk{subkeys, sh->H * d.ntot * sh->d_sub * ab, "subkeys"};
  const Range r_s{scores, 2 * rows * d.ntot * 4, "scores"};
  const Range r_ws{workspace, (int64_t)workspace_bytes, "workspace"};
  if (rows == 0) return ok();
  for (const Range &r : {r_qw, r_qr, r_sk, r_s}) {
    if (!r.p) return fail(SDM_ERR_INVALID_ARG, "%s is NULL", r.name);
    if (!aligned(r.p, 16)) return fail(SDM_ERR_INVALID_ARG, "%s is not 16-byte aligned", r.name);
  }
  if (!workspace || !aligned(workspace, 16) || (int64_t)workspace_bytes < write_read_ws_bytes(sh))
    return fail(SDM_ERR_WORKSPACE, "workspace is NULL, misaligned or short");
  for (const Range &i : {r_qw, r_qr, r_sk})
    for (const Range &o : {r_s, r_ws})
      if (overlap(o, i)) return fail(SDM_ERR_ALIAS, "%s overlaps %s", o.name, i.name);
  if (overlap(r_s, r_ws)) return fail(SDM_ERR_ALIAS, "scores overlaps workspace");
  const WsLayout wl = ws_layout(sh, PlanLayout{});   // the split region does not depend on the plan
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  int32_t *err = reinterpret_cast<int32_t *>(ws);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t ce = cudaMemsetAsync(err, 0, sizeof(int32_t), cs);
  if (ce != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(ce));
  ScoreArgs sa{};
  sa.q[0] = q_w;
  sa.q[1] = q_r;
  sa.subkeys = subkeys;
  sa.scores = scores;
  sa.split = ws + wl.split;
  sa.err = err;
  sa.BT = sh->B * sh->T;
  sa.H = (int32_t)sh->H;
  sa.g = d.g;
  const bool tc = use_tensor_cores(d, sh);
  if ((st = run_kernel(SDM_KERNEL_SCORE, cs, tc ? "score_tc" : "score_simt", [&] {
         return tc ? launch_score_tc(sa, sh->act_dtype, cs) : launch_score_simt(sa, sh->act_dtype, cs);
       })) != SDM_OK)
    return st;
  return ok();
}

sdm_status sdm_test_force_simt_scorer(int on) {
  g_test_simt_scorer.store(on ? 1 : 0);
  return SDM_OK;
}

sdm_status sdm_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.created) {
    g_prof.start.resize(kProfSlots);
    g_prof.stop.resize(kProfSlots);
    g_prof.kind.resize(kProfSlots);
    for (int i = 0; i < kProfSlots; ++i) {
      if (cudaEventCreate(&g_prof.start[i]) != cudaSuccess || cudaEventCreate(&g_prof.stop[i]) != cudaSuccess)
        return fail(SDM_ERR_CUDA, "cudaEventCreate failed");
    }
    g_prof.created = true;
  }
  g_prof.used = 0;
  g_prof.active = true;
  return ok();
}

sdm_status sdm_profile_end(sdm_kernel_times *out) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!out) return fail(SDM_ERR_INVALID_ARG, "out is NULL");
  memset(out, 0, sizeof(*out));
  if (!g_prof.active) return fail(SDM_ERR_INVALID_ARG, "profiling was not started");
  g_prof.active = false;
  for (int i = 0; i < g_prof.used; ++i) {
    cudaError_t e = cudaEventSynchronize(g_prof.stop[i]);
    float ms = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, g_prof.start[i], g_prof.stop[i]);
    if (e != cudaSuccess) return fail(SDM_ERR_CUDA, "event timing: %s", cudaGetErrorString(e));
    const int k = g_prof.kind[i];
    out->launches[k] += 1;
    out->ms[k] += ms;
  }
  return ok();
}

const char *sdm_kernel_name(int32_t kind) {
  switch (kind) {
    case SDM_KERNEL_BANK_COPY: return "bank_copy";
    case SDM_KERNEL_SCORE: return "score";
    case SDM_KERNEL_SELECT: return "select";
    case SDM_KERNEL_PLAN_SORT: return "plan_sort";
    case SDM_KERNEL_PLAN_LINK: return "plan_link";
    case SDM_KERNEL_WRITE_READ: return "write_read";
    case SDM_KERNEL_DECODE: return "decode";
    case SDM_KERNEL_BWD_FLAGS: return "bwd_flags";
    case SDM_KERNEL_BWD_SWEEP: return "bwd_sweep";
    case SDM_KERNEL_BWD_REDUCE: return "bwd_reduce";
    case SDM_KERNEL_BWD_SUBKEY: return "bwd_subkeys";
    case SDM_KERNEL_LAYER_GATES: return "layer_gates";
    case SDM_KERNEL_LAYER_GEMM: return "layer_gemm";
    case SDM_KERNEL_LAYER_GRAD: return "layer_grad";
  }
  return "unknown";
}

}  // extern "C"

// ============================================== write/read with the library's own scratch

namespace {

// Scratch of sdm_write_read_static: one array per device, never allocated at run time.
static __device__ __align__(256) unsigned char g_static_scratch[SDM_STATIC_SCRATCH_BYTES];

std::mutex g_static_mu;
void *g_static_ptr[64] = {nullptr};

}  // namespace

extern "C" sdm_status sdm_write_read_static(const sdm_shape *shape, const void *q_w, const void *q_r,
                                            const void *k_val, const float *gates, const void *subkeys,
                                            const void *bank_init, void *bank, void *y, int32_t *idx_w,
                                            float *wt_w, int32_t *idx_r, float *wt_r, sdm_stream_t stream) {
  size_t need = 0;
  sdm_status st = sdm_write_read_workspace_size(shape, &need);
  if (st != SDM_OK) return st;
  if (need > SDM_STATIC_SCRATCH_BYTES)
    return fail(SDM_ERR_WORKSPACE, "shape needs %zu bytes of scratch; the static array holds %zu", need,
                (size_t)SDM_STATIC_SCRATCH_BYTES);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(SDM_ERR_UNSUPPORTED, "device ordinal %d is not supported", dev);
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
      e = cudaGetSymbolAddress(&scratch, g_static_scratch);
      if (e != cudaSuccess) return fail(SDM_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      g_static_ptr[dev] = scratch;
    }
    scratch = g_static_ptr[dev];
  }
  return write_read_impl(shape, q_w, q_r, k_val, gates, subkeys, bank_init, bank, y, idx_w, wt_w, idx_r, wt_r,
                         scratch, SDM_STATIC_SCRATCH_BYTES, stream, false);
}
