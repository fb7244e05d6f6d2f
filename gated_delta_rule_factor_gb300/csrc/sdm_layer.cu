// The SDM layer around the op (sparse-delta-memory README, usage example: a layer of
// dim model width with num_heads heads, whose input projections give the write and read
// queries, the values and the gates, and whose output projection maps the read back to
// dim): the dense projections are plain GEMMs run by cuBLASLt, the gate projection and
// its sigmoid are one kernel of this library.
//
// cuBLASLt is loaded with dlopen when a layer call first needs it, so the op's own entry
// points never depend on it; a missing library makes the layer call return
// SDM_ERR_CUDA.  Its GEMMs run with the caller's workspace (no allocation); split-K is
// allowed only with the partial products reduced in the workspace by a separate step, so
// that each product is computed the same way on every call (bitwise repeatable).
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

// The layer backward's concatenated input gradient, one token row r at a time:
//   gcat[r] = [d_q_w[r] | d_q_r[r] | d_k_val[r] | dz[r] | 0 ...]  (activation type, row
//   stride K: the zero padding keeps the rows 16-byte aligned for the products)
// with dz[r][j] = d_gates[r][j] * g (1 - g), g = gates[r][j] (the sigmoid's derivative).
template <typename ACT>
__global__ void __launch_bounds__(kThreads) layer_grad_cat_kernel(const float *d_qw, const float *d_qr,
                                                                  const float *d_kv, const float *d_g,
                                                                  const float *gates, ACT *gcat, int64_t rows,
                                                                  int64_t dq, int64_t dv, int64_t ng, int64_t K) {
  const int64_t K0 = 2 * dq + dv + ng;               // K >= K0: the row stride, zero-padded
  // one CTA per token row at a time: the row's four pieces, each with contiguous loads
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    ACT *out = gcat + r * K;
    for (int64_t c = threadIdx.x; c < dq; c += kThreads) out[c] = from_f32<ACT>(d_qw[r * dq + c]);
    for (int64_t c = threadIdx.x; c < dq; c += kThreads) out[dq + c] = from_f32<ACT>(d_qr[r * dq + c]);
    for (int64_t c = threadIdx.x; c < dv; c += kThreads) out[2 * dq + c] = from_f32<ACT>(d_kv[r * dv + c]);
    for (int64_t j = threadIdx.x; j < ng; j += kThreads) {
      const float g = gates[r * ng + j];
      out[2 * dq + dv + j] = from_f32<ACT>(__fmul_rn(d_g[r * ng + j], __fmul_rn(g, __fsub_rn(1.0f, g))));
    }
    for (int64_t c = K0 + threadIdx.x; c < K; c += kThreads) out[c] = from_f32<ACT>(0.0f);
  }
}

// out[i] = sum over b = 0 .. B-1, in that order, of in[b * n + i] (the learned table's
// gradient: the streams' bank gradients summed over the batch).
__global__ void __launch_bounds__(kThreads) batch_sum_kernel(const float *in, float *out, int64_t B, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads) {
    float acc = 0.0f;
    for (int64_t b = 0; b < B; ++b) acc = __fadd_rn(acc, in[b * n + i]);
    out[i] = acc;
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

cudaError_t launch_layer_grad_cat(const float *d_qw, const float *d_qr, const float *d_kv, const float *d_g,
                                  const float *gates, void *gcat, int64_t rows, int64_t dq, int64_t dv, int64_t ng,
                                  int64_t K, int act_dtype, int sm_count, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  int64_t blocks = rows;
  if (blocks > (int64_t)sm_count * 16) blocks = (int64_t)sm_count * 16;
  if (act_dtype == SDM_BF16)
    layer_grad_cat_kernel<__nv_bfloat16><<<(unsigned)blocks, kThreads, 0, st>>>(
        d_qw, d_qr, d_kv, d_g, gates, static_cast<__nv_bfloat16 *>(gcat), rows, dq, dv, ng, K);
  else
    layer_grad_cat_kernel<float><<<(unsigned)blocks, kThreads, 0, st>>>(d_qw, d_qr, d_kv, d_g, gates,
                                                                        static_cast<float *>(gcat), rows, dq, dv, ng, K);
  return cudaGetLastError();
}

cudaError_t launch_batch_sum(const float *in, float *out, int64_t B, int64_t n, int sm_count, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + kThreads - 1) / kThreads;
  if (blocks > (int64_t)sm_count * 32) blocks = (int64_t)sm_count * 32;
  batch_sum_kernel<<<(unsigned)blocks, kThreads, 0, st>>>(in, out, B, n);
  return cudaGetLastError();
}

// D = op(A) op(B) (+ D when accumulate), column-major (cuBLASLt's convention): op(A) is
// m x k, op(B) is k x n, D is m x n with leading dimension ldd.  A and B have the type ab
// (bfloat16 or float32 activations), D the type dd; float32 accumulation.
const char *lt_gemm(bool ta, bool tb, int64_t m, int64_t n, int64_t k, const void *A, int64_t lda, const void *B,
                    int64_t ldb, void *D, int64_t ldd, int ab, int dd, bool accumulate, void *ws, size_t ws_bytes,
                    cudaStream_t st) {
  if (m == 0 || n == 0) return nullptr;
  const char *why = nullptr;
  cublasLtHandle_t h = lt_handle(&why);
  if (!h) return why;
  const cudaDataType_t tab = ab == SDM_BF16 ? CUDA_R_16BF : CUDA_R_32F;
  const cudaDataType_t tdd = dd == SDM_BF16 ? CUDA_R_16BF : CUDA_R_32F;
  cublasLtMatmulDesc_t desc = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  const char *err = nullptr;
  const cublasOperation_t opa = ta ? CUBLAS_OP_T : CUBLAS_OP_N, opb = tb ? CUBLAS_OP_T : CUBLAS_OP_N;
  // split-K only through a workspace and a separate reduction step (a fixed order); not
  // the in-place scheme
  const uint32_t no_split_k =
      CUBLASLT_REDUCTION_SCHEME_NONE | CUBLASLT_REDUCTION_SCHEME_COMPUTE_TYPE | CUBLASLT_REDUCTION_SCHEME_OUTPUT_TYPE;
  cublasLtMatmulHeuristicResult_t res{};
  int found = 0;
  const float one = 1.0f, beta = accumulate ? 1.0f : 0.0f;
  // the operands' actual alignments (an operand may start inside a larger matrix)
  auto align_of = [](const void *p) -> uint32_t {
    const uintptr_t a = (uintptr_t)p;
    const uintptr_t low = a & (~a + 1);
    return (uint32_t)(low == 0 || low > 256 ? 256 : low);
  };
  const uint32_t al_a = align_of(A), al_b = align_of(B), al_d = align_of(D);
  if (g_lt.desc_create(&desc, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS ||
      g_lt.desc_set(desc, CUBLASLT_MATMUL_DESC_TRANSA, &opa, sizeof(opa)) != CUBLAS_STATUS_SUCCESS ||
      g_lt.desc_set(desc, CUBLASLT_MATMUL_DESC_TRANSB, &opb, sizeof(opb)) != CUBLAS_STATUS_SUCCESS ||
      g_lt.layout_create(&la, tab, (uint64_t)(ta ? k : m), (uint64_t)(ta ? m : k), lda) != CUBLAS_STATUS_SUCCESS ||
      g_lt.layout_create(&lb, tab, (uint64_t)(tb ? n : k), (uint64_t)(tb ? k : n), ldb) != CUBLAS_STATUS_SUCCESS ||
      g_lt.layout_create(&lc, tdd, (uint64_t)m, (uint64_t)n, ldd) != CUBLAS_STATUS_SUCCESS ||
      g_lt.pref_create(&pref) != CUBLAS_STATUS_SUCCESS ||
      g_lt.pref_set(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes, sizeof(ws_bytes)) !=
          CUBLAS_STATUS_SUCCESS ||
      g_lt.pref_set(pref, CUBLASLT_MATMUL_PREF_REDUCTION_SCHEME_MASK, &no_split_k, sizeof(no_split_k)) !=
          CUBLAS_STATUS_SUCCESS ||
      g_lt.pref_set(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_A_BYTES, &al_a, sizeof(al_a)) != CUBLAS_STATUS_SUCCESS ||
      g_lt.pref_set(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_B_BYTES, &al_b, sizeof(al_b)) != CUBLAS_STATUS_SUCCESS ||
      g_lt.pref_set(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_C_BYTES, &al_d, sizeof(al_d)) != CUBLAS_STATUS_SUCCESS ||
      g_lt.pref_set(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_D_BYTES, &al_d, sizeof(al_d)) != CUBLAS_STATUS_SUCCESS) {
    err = "cuBLASLt descriptor set-up failed";
  } else if (g_lt.heuristic(h, desc, la, lb, lc, lc, pref, 1, &res, &found) != CUBLAS_STATUS_SUCCESS ||
             found < 1) {
    err = "cuBLASLt found no algorithm for the product";
  } else if (g_lt.matmul(h, desc, &one, A, la, B, lb, &beta, D, lc, D, lc, &res.algo, ws, ws_bytes, st) !=
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

// out[n][m] = sum_k a[m][k] * b[n][k] for row-major a [m, k] (weights, out x in) and b
// [n, k] (activations): the column-major product op(A) = a (transposed) times b.
const char *layer_gemm(const void *a, const void *b, void *out, int64_t m, int64_t n, int64_t k, int act_dtype,
                       void *ws, size_t ws_bytes, cudaStream_t st) {
  return lt_gemm(true, false, m, n, k, a, k, b, k, out, m, act_dtype, act_dtype, false, ws, ws_bytes, st);
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
