// The SDM layer around the op (sparse-delta-memory README, usage example: a layer of
// dim model width with num_heads heads, whose input projections give the write and read
// queries, the values and the gates, and whose output projection maps the read back to
// dim): the dense projections are plain GEMMs run by cuBLASLt, the gate projection and
// its sigmoid are one kernel of this library.
//
// cuBLASLt is loaded with dlopen when a layer call first needs it, so the op's own entry
// points never depend on it; a missing library makes the layer call return
// SDM_ERR_CUDA.  Its GEMMs run with the caller's workspace (no allocation) and with
// split-K reductions excluded, so that each product is computed the same way on every
// call (bitwise repeatable).
#include <dlfcn.h>

#include <mutex>

#include <cublasLt.h>

#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

// ---------------------------------------------------------------- gates

constexpr int kGateWarps = kThreads / 32;

// gates[r][j] = sigmoid(<x[r], w_g[j]>) for the 2H gate rows j = 2h + (0: alpha, 1: beta),
// float32: one warp per token row, the dim terms split over the lanes in a fixed order
// (lane-strided partial sums, then an xor butterfly).
template <typename ACT>
__global__ void __launch_bounds__(kThreads) layer_gates_kernel(const ACT *x, const ACT *w_g, float *gates,
                                                               int64_t rows, int64_t dim, int32_t n_gates) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t r = (int64_t)blockIdx.x * kGateWarps + warp; r < rows; r += (int64_t)gridDim.x * kGateWarps) {
    const ACT *xr = x + r * dim;
    for (int j = 0; j < n_gates; ++j) {
      const ACT *wj = w_g + (int64_t)j * dim;
      float acc = 0.0f;
      for (int64_t d = lane; d < dim; d += 32) acc = __fmaf_rn(to_f32(xr[d]), to_f32(wj[d]), acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
      if (lane == 0) gates[r * n_gates + j] = 1.0f / (1.0f + expf(-acc));
    }
  }
}

// ---------------------------------------------------------------- cuBLASLt, loaded on demand

struct Lt {
  bool tried = false, ok = false;
  decltype(&cublasLtCreate) create = nullptr;
  decltype(&cublasLtMatmulDescCreate) desc_create = nullptr;
  decltype(&cublasLtMatmulDescDestroy) desc_destroy = nullptr;
  decltype(&cublasLtMatmulDescSetAttribute) desc_set = nullptr;
  decltype(&cublasLtMatrixLayoutCreate) layout_create = nullptr;
  decltype(&cublasLtMatrixLayoutDestroy) layout_destroy = nullptr;
  decltype(&cublasLtMatmulPreferenceCreate) pref_create = nullptr;
  decltype(&cublasLtMatmulPreferenceDestroy) pref_destroy = nullptr;
  decltype(&cublasLtMatmulPreferenceSetAttribute) pref_set = nullptr;
  decltype(&cublasLtMatmulAlgoGetHeuristic) heuristic = nullptr;
  decltype(&cublasLtMatmul) matmul = nullptr;
  cublasLtHandle_t handle[64] = {};
};
Lt g_lt;
std::mutex g_lt_mu;

template <class F>
bool sym(void *lib, const char *name, F *out) {
  *out = reinterpret_cast<F>(dlsym(lib, name));
  return *out != nullptr;
}

// The process's cuBLASLt and a handle for the current device; nullptr if unavailable.
cublasLtHandle_t lt_handle(const char **why) {
  std::lock_guard<std::mutex> lock(g_lt_mu);
  if (!g_lt.tried) {
    g_lt.tried = true;
    void *lib = dlopen("libcublasLt.so.13", RTLD_NOW | RTLD_GLOBAL);
    if (!lib) lib = dlopen("libcublasLt.so", RTLD_NOW | RTLD_GLOBAL);
    g_lt.ok = lib && sym(lib, "cublasLtCreate", &g_lt.create) &&
              sym(lib, "cublasLtMatmulDescCreate", &g_lt.desc_create) &&
              sym(lib, "cublasLtMatmulDescDestroy", &g_lt.desc_destroy) &&
              sym(lib, "cublasLtMatmulDescSetAttribute", &g_lt.desc_set) &&
              sym(lib, "cublasLtMatrixLayoutCreate", &g_lt.layout_create) &&
              sym(lib, "cublasLtMatrixLayoutDestroy", &g_lt.layout_destroy) &&
              sym(lib, "cublasLtMatmulPreferenceCreate", &g_lt.pref_create) &&
              sym(lib, "cublasLtMatmulPreferenceDestroy", &g_lt.pref_destroy) &&
              sym(lib, "cublasLtMatmulPreferenceSetAttribute", &g_lt.pref_set) &&
              sym(lib, "cublasLtMatmulAlgoGetHeuristic", &g_lt.heuristic) &&
              sym(lib, "cublasLtMatmul", &g_lt.matmul);
  }
  if (!g_lt.ok) {
    *why = "libcublasLt could not be loaded";
    return nullptr;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *why = "no current CUDA device";
    return nullptr;
  }
  if (!g_lt.handle[dev] && g_lt.create(&g_lt.handle[dev]) != CUBLAS_STATUS_SUCCESS) {
    g_lt.handle[dev] = nullptr;
    *why = "cublasLtCreate failed";
    return nullptr;
  }
  return g_lt.handle[dev];
}

}  // namespace

// out[n][m] = sum_k a[m][k] * b[n][k] for row-major a [m, k] (weights, out x in) and b
// [n, k] (activations): the column-major product op(A) = a (transposed) times b.
const char *layer_gemm(const void *a, const void *b, void *out, int64_t m, int64_t n, int64_t k, int act_dtype,
                       void *ws, size_t ws_bytes, cudaStream_t st) {
  if (m == 0 || n == 0) return nullptr;
  const char *why = nullptr;
  cublasLtHandle_t h = lt_handle(&why);
  if (!h) return why;
  const cudaDataType_t t = act_dtype == SDM_BF16 ? CUDA_R_16BF : CUDA_R_32F;
  cublasLtMatmulDesc_t desc = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  const char *err = nullptr;
  const cublasOperation_t tr = CUBLAS_OP_T, nt = CUBLAS_OP_N;
  const uint32_t no_split_k = CUBLASLT_REDUCTION_SCHEME_NONE;
  cublasLtMatmulHeuristicResult_t res{};
  int found = 0;
  const float one = 1.0f, zero = 0.0f;
  if (g_lt.desc_create(&desc, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS ||
      g_lt.desc_set(desc, CUBLASLT_MATMUL_DESC_TRANSA, &tr, sizeof(tr)) != CUBLAS_STATUS_SUCCESS ||
      g_lt.desc_set(desc, CUBLASLT_MATMUL_DESC_TRANSB, &nt, sizeof(nt)) != CUBLAS_STATUS_SUCCESS ||
      g_lt.layout_create(&la, t, (uint64_t)k, (uint64_t)m, k) != CUBLAS_STATUS_SUCCESS ||
      g_lt.layout_create(&lb, t, (uint64_t)k, (uint64_t)n, k) != CUBLAS_STATUS_SUCCESS ||
      g_lt.layout_create(&lc, t, (uint64_t)m, (uint64_t)n, m) != CUBLAS_STATUS_SUCCESS ||
      g_lt.pref_create(&pref) != CUBLAS_STATUS_SUCCESS ||
      g_lt.pref_set(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes, sizeof(ws_bytes)) !=
          CUBLAS_STATUS_SUCCESS ||
      g_lt.pref_set(pref, CUBLASLT_MATMUL_PREF_REDUCTION_SCHEME_MASK, &no_split_k, sizeof(no_split_k)) !=
          CUBLAS_STATUS_SUCCESS) {
    err = "cuBLASLt descriptor set-up failed";
  } else if (g_lt.heuristic(h, desc, la, lb, lc, lc, pref, 1, &res, &found) != CUBLAS_STATUS_SUCCESS ||
             found < 1) {
    err = "cuBLASLt found no algorithm for the projection";
  } else if (g_lt.matmul(h, desc, &one, a, la, b, lb, &zero, out, lc, out, lc, &res.algo, ws, ws_bytes, st) !=
             CUBLAS_STATUS_SUCCESS) {
    err = "cublasLtMatmul failed";
  }
  if (pref) g_lt.pref_destroy(pref);
  if (lc) g_lt.layout_destroy(lc);
  if (lb) g_lt.layout_destroy(lb);
  if (la) g_lt.layout_destroy(la);
  if (desc) g_lt.desc_destroy(desc);
  return err;
}

cudaError_t launch_layer_gates(const void *x, const void *w_g, float *gates, int64_t rows, int64_t dim,
                               int32_t n_gates, int act_dtype, int sm_count, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  int64_t blocks = (rows + kGateWarps - 1) / kGateWarps;
  if (blocks > (int64_t)sm_count * 16) blocks = (int64_t)sm_count * 16;
  if (act_dtype == SDM_BF16)
    layer_gates_kernel<__nv_bfloat16><<<(unsigned)blocks, kThreads, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(w_g), gates, rows, dim, n_gates);
  else
    layer_gates_kernel<float><<<(unsigned)blocks, kThreads, 0, st>>>(static_cast<const float *>(x),
                                                                     static_cast<const float *>(w_g), gates, rows,
                                                                     dim, n_gates);
  return cudaGetLastError();
}

}  // namespace sdm
