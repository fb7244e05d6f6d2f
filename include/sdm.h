/*
 * sdm.h - C ABI of the GB300 (sm_103a) Sparse Delta Memory hot path.
 *
 * Sparse Delta Memory (SDM) is a sequence mixer that reads from and writes to a
 * large memory bank addressed by product keys, with gated (forget/input)
 * delta-rule updates (sparse-delta-memory README, introduction).  This library
 * runs its data-parallel hot path on one GPU:
 *
 *   sdm_write_read   the chunked write/read op over a sequence
 *                    (CHANGELOG 2.0.0 > Removed: sdm_write_read is the one op;
 *                     reads happen inside the write/read call)
 *   sdm_decode_step  the single-token decode step, copying or in place
 *                    (CHANGELOG 2.0.0 > New: a single-token decode kernel;
 *                     lumen PR #29 > Donating is a permission)
 *
 * What one token of one stream (batch element b, head h) computes, in token order:
 *   1. factor scores  s_f[a] = <q[f*d_sub:(f+1)*d_sub], K_f[a]>  for q in {q_w, q_r}
 *      (product-key memory, README > prior ideas);
 *   2. the exact top-k slots (k = W for q_w, R for q_r) over all factor
 *      combinations: slot score = the float32 sum of the factor scores, ties to the
 *      larger rank sum, then the larger first rank, then the second, ...
 *      (CHANGELOG 2.0.0 > Upgrading from v1; "rank" is a factor's ascending score
 *      rank, equal factor scores ordered by index);  slot id = mixed radix of the
 *      factor indices, first factor most significant;
 *   3. weights w_j = softmax over the selected slot scores (the same for reads, r_j);
 *   4. gated delta-rule write of the W selected rows of the stream's bank M:
 *        m_j = alpha M[i_j];  p = sum_j w_j m_j;  M[i_j] <- m_j + beta w_j (v - p)
 *      with (alpha, beta) = gates[b,t,h] and v = k_val[b,t,h];  the row is rounded to
 *      the bank type after every token;
 *   5. the read after the write: y[b,t,h] = sum_j r_j M[i^r_j].
 * Results do not depend on chunk_size at all (bitwise), which the CHANGELOG allows
 * ("the chunk size changes outputs only through floating-point rounding").
 * Outputs, the final bank and the selections are bitwise identical across runs.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, row-major and contiguous, with the
 *     shapes given below, and 16-byte aligned unless marked otherwise.
 *   - The caller owns every buffer.  The library allocates no device memory and
 *     never synchronises the stream, except sdm_last_device_error (it reads back a
 *     flag) and sdm_profile_end.  All work is enqueued on `stream`.
 *   - Every argument check runs on the host before any work is enqueued; a call that
 *     returns an error has enqueued nothing.  sdm_last_error_message() then gives
 *     the reason.
 *   - Kernel-side anomalies (a corrupt plan, an out-of-range slot) never fault: the
 *     kernel skips the access and records a code in the workspace, read back with
 *     sdm_last_device_error.
 */
#ifndef SDM_GB300_H
#define SDM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SDM_ABI_VERSION 4

/* Compiled limits.  Shapes beyond them are refused with SDM_ERR_UNSUPPORTED. */
#define SDM_MAX_FACTORS 4          /* product-key factors F                          */
#define SDM_MAX_FACTOR_DIM 1024    /* sub-keys per factor n_f                        */
#define SDM_MAX_K 128              /* writes W and reads R per token                 */
#define SDM_MAX_CANDIDATES 1024    /* position tuples with prod(p_f+1) <= k          */
#define SDM_MAX_CHUNK 256          /* chunk_size                                     */
#define SDM_MAX_HEAD_DIM (1 << 20) /* d_v (CHANGELOG 2.0.0 > Behavior changes)       */
#define SDM_MAX_SUBKEY_DIM 4096    /* d_sub                                          */

typedef struct CUstream_st *sdm_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  SDM_OK = 0,
  SDM_ERR_INVALID_ARG = 1, /* malformed shape, NULL/misaligned pointer, W or R > N     */
  SDM_ERR_UNSUPPORTED = 2, /* float16, or a shape beyond the compiled limits           */
  SDM_ERR_ALIAS = 3,       /* an output overlaps an input it must not overlap          */
  SDM_ERR_WORKSPACE = 4,   /* workspace NULL, misaligned or smaller than required      */
  SDM_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed                     */
  SDM_ERR_DEVICE = 6       /* sdm_last_device_error found a kernel-side error code     */
} sdm_status;

typedef enum { SDM_F32 = 0, SDM_BF16 = 1, SDM_F16 = 2 /* always refused */ } sdm_dtype;

/* Kernel-side codes written to the workspace flag (see sdm_last_device_error). */
#define SDM_DEVERR_NONE 0
#define SDM_DEVERR_SLOT_RANGE 1    /* a selected slot id outside [0, N)                */
#define SDM_DEVERR_PLAN 2          /* a chunk plan count or row index out of range     */
#define SDM_DEVERR_TIMEOUT 3       /* a bounded wait inside a kernel gave up             */
#define SDM_DEVERR_SNAPSHOT 4      /* a backward found no armed snapshot (second backward) */

/*
 * Shape of one call.  Tensors (row-major, contiguous):
 *   q_w, q_r  [B, T, H, F*d_sub]   act_dtype   write / read queries
 *   k_val     [B, T, H, d_v]       act_dtype   values
 *   gates     [B, T, H, 2]         float32     (alpha = forget, beta = input), in [0, 1]
 *   subkeys   [H, sum_f n_f, d_sub] act_dtype  factor f at row offset sum_{g<f} n_g
 *   bank      [B, H, N, d_v]       bank_dtype  N = prod_f n_f slots per head
 *   y         [B, T, H, d_v]       act_dtype
 *   idx_w/wt_w [B, T, H, W] int32 / float32, idx_r/wt_r [B, T, H, R]: selected slot
 *             ids (best first) and their softmax weights.
 * Field order avoids padding: five int64 then ten int32 (80 bytes).
 */
typedef struct {
  int64_t B, T, H;       /* streams = B*H; T tokens per stream (decode: T == 1)      */
  int64_t d_sub, d_v;    /* sub-key dim, head (value) dim; d_v % 8 == 0              */
  int32_t F;             /* number of product-key factors, 1..SDM_MAX_FACTORS         */
  int32_t factor_dims[SDM_MAX_FACTORS]; /* n_f; entries >= F ignored                 */
  int32_t W, R;          /* writes / reads per token, 1..min(N, SDM_MAX_K)            */
  int32_t chunk_size;    /* 1..SDM_MAX_CHUNK; caps the tokens planned together         */
  int32_t act_dtype;     /* sdm_dtype of q_w, q_r, k_val, subkeys, y                  */
  int32_t bank_dtype;    /* sdm_dtype of the bank                                     */
} sdm_shape;

/* Device bytes of workspace sdm_write_read needs for `shape` (16-byte aligned buffer).
 * Depends only on the shape.  Errors as for sdm_write_read's shape checks. */
sdm_status sdm_write_read_workspace_size(const sdm_shape *shape, size_t *bytes);

/* Device bytes of workspace sdm_decode_step needs (a few hundred bytes). */
sdm_status sdm_decode_workspace_size(const sdm_shape *shape, size_t *bytes);

/*
 * The chunked write/read op (CHANGELOG 2.0.0 > Removed: sdm_write_read), all B*H
 * streams, T tokens each, in token order.  The bank advances in place
 * (README usage example: "the bank advances in place").
 *   bank_init  NULL, or a learned initial table [H, N, d_v] (bank_dtype) that is first
 *              copied into every stream's bank (the per-call bank copy of a layer
 *              call, CHANGELOG 2.0.0 > Behavior changes).  Must not overlap `bank`.
 *   bank       [B, H, N, d_v] in/out.
 *   y          [B, T, H, d_v] out; must not overlap any input or the bank.
 *   idx_w, wt_w, idx_r, wt_r  outputs, each NULL or a buffer of the shape above (4-byte
 *              aligned); NULL ones are kept in the workspace instead.
 *   workspace  device scratch of >= sdm_write_read_workspace_size bytes; its contents
 *              need not be initialised and are overwritten.  Calls sharing one
 *              workspace must be ordered on one stream.
 * Refusals (nothing enqueued): float16 (UNSUPPORTED; CHANGELOG > Behavior changes);
 * W or R > N (INVALID); d_v > 2^20 (UNSUPPORTED); limits above (UNSUPPORTED);
 * NULL/misaligned pointers (INVALID); overlaps (ALIAS); short workspace (WORKSPACE).
 */
sdm_status sdm_write_read(const sdm_shape *shape, const void *q_w, const void *q_r,
                          const void *k_val, const float *gates, const void *subkeys,
                          const void *bank_init, void *bank, void *y, int32_t *idx_w,
                          float *wt_w, int32_t *idx_r, float *wt_r, void *workspace,
                          size_t workspace_bytes, sdm_stream_t stream);

/*
 * sdm_write_read without a caller-provided workspace.  The method itself has no
 * counterpart to this: it exists for callers that cannot allocate device memory, such
 * as a C host that links this library without any allocator, or a framework whose
 * allocator has reserved the device's memory up front and grants no buffer to a
 * library call.  Arguments and results are those of sdm_write_read, and so are the
 * kernels it enqueues; this entry allocates nothing (no cudaMalloc, cudaFree or
 * allocating routine of any library).
 *   scratch    a fixed device array of SDM_STATIC_SCRATCH_BYTES (16 MiB) that this
 *              library defines; shapes whose sdm_write_read_workspace_size exceeds it
 *              are refused with SDM_ERR_WORKSPACE, nothing enqueued.  Nothing in it
 *              has to start at zero: the one word the kernels read before writing (the
 *              device error code) is cleared on `stream` at the start of every call.
 *   set-up     the first call on a device, with that device current, looks up the
 *              array's address (cudaGetSymbolAddress) and keeps it for the life of the
 *              process; make that first call before any stream capture begins.  A
 *              failed lookup returns SDM_ERR_CUDA.  A device reset (cudaDeviceReset, or a
 *              framework that destroys and recreates the primary context) invalidates the
 *              kept address: do not use this entry after one.
 *   races      every call on a device shares the one array: calls whose work may
 *              overlap on the device (other streams, other host threads) corrupt each
 *              other's scratch.  Order them on one stream.
 *   errors     kernel-side codes (SDM_DEVERR_*) land in the array and are not readable
 *              through sdm_last_device_error; use sdm_write_read to read them.
 */
#define SDM_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
sdm_status sdm_write_read_static(const sdm_shape *shape, const void *q_w, const void *q_r,
                                 const void *k_val, const float *gates, const void *subkeys,
                                 const void *bank_init, void *bank, void *y, int32_t *idx_w,
                                 float *wt_w, int32_t *idx_r, float *wt_r, sdm_stream_t stream);

/*
 * Training: the forward with a snapshot, then the deterministic sparse backward
 * (CHANGELOG 2.0.0 > New: "exact product-key top-k with a deterministic sparse
 * backward"; > Deterministic: every gradient is bitwise repeatable; > Package: training
 * saves a snapshot of the rows each step overwrites, float32 by default or bf16 at half
 * the size; > Behavior changes: the first backward restores the bank in place and a
 * second backward through the same forward is refused).
 *
 * The gradient is the chain rule through the forward above, per stream, from the last
 * token to the first.  With X_j the token's W rows before its write, m_j = alpha X_j,
 * u = v - sum_j w_j m_j, G = dL/d(bank after the token) and dy = dL/dy[b,t,h]:
 *   read:    dr_j = <dy, M[i^r_j]> (the rows after the write);  G[i^r_j] += r_j dy
 *   write:   dv = beta sum_j w_j G[i_j];  dm_j = G[i_j] - w_j dv;
 *            dw_j = beta <G[i_j], u> - <dv, m_j>;  dbeta = sum_j w_j <G[i_j], u>;
 *            dalpha = sum_j <dm_j, X_j>;  G[i_j] <- alpha dm_j;  M[i_j] <- X_j
 *   weights: dS_j = w_j (dw_j - sum_k w_k dw_k) (and the same for the read weights);
 *   scores:  the slot score is the sum of the factor scores, so dS_j flows to each
 *            factor's score of the slot, and from s_f[a] = <q_f, K_f[a]> to the query
 *            and the sub-key.
 * Readings where the pages are silent: the selected slot ids are piecewise constant
 * (no gradient flows through the choice); float32 roundings of scores, stored rows and
 * outputs pass the gradient unchanged; the gate gradients are with respect to the
 * post-sigmoid (alpha, beta) the op takes.
 */

/* Bytes of a snapshot buffer for `shape` (snapshot_dtype SDM_F32, exact, or SDM_BF16,
 * rows rounded to bfloat16; on a bfloat16 bank both are exact).  The buffer holds a
 * 256-byte header and, per stream and token, the W rows the token overwrites, in a
 * layout private to the library. */
sdm_status sdm_snapshot_bytes(const sdm_shape *shape, int32_t snapshot_dtype, size_t *bytes);

/* sdm_write_read that also fills `snapshot` (>= sdm_snapshot_bytes bytes, 16-byte
 * aligned) and arms it for one backward.  idx_w, wt_w, idx_r, wt_r are required here
 * (16-byte aligned): the backward reads the selections from them.  y, the bank and
 * the selections are bitwise those of sdm_write_read, whatever the snapshot type.
 * Takes sdm_write_read's workspace. */
sdm_status sdm_write_read_train(const sdm_shape *shape, const void *q_w, const void *q_r,
                                const void *k_val, const float *gates, const void *subkeys,
                                const void *bank_init, void *bank, void *y, int32_t *idx_w,
                                float *wt_w, int32_t *idx_r, float *wt_r, void *snapshot,
                                size_t snapshot_bytes, int32_t snapshot_dtype, void *workspace,
                                size_t workspace_bytes, sdm_stream_t stream);

/* Device bytes of workspace sdm_write_read_backward needs for `shape` (depends only on
 * the shape). */
sdm_status sdm_write_read_backward_workspace_size(const sdm_shape *shape, size_t *bytes);

/*
 * The backward of one sdm_write_read_train call.
 *   q_w ... subkeys, idx_*, wt_*  the forward's inputs and selections, unchanged since;
 *   snapshot   the forward's snapshot and its type; the backward disarms it.  A
 *              snapshot that is not armed (never filled, or already used) makes the
 *              call touch neither the bank nor dbank, record SDM_DEVERR_SNAPSHOT and
 *              leave the other outputs unspecified;
 *   bank       [B,H,N,d_v] in: the bank the forward left; out: the bank before the
 *              forward (the rows the forward wrote are restored from the snapshot, so
 *              with a bfloat16 snapshot of a float32 bank they come back rounded);
 *   dy         [B,T,H,d_v] act_dtype: dL/dy;
 *   dbank      [B,H,N,d_v] float32 in: dL/d(bank after the forward); out: dL/d(bank
 *              before it) (zeros in: y is the only output that matters);
 *   d_k_val    [B,T,H,d_v], d_gates [B,T,H,2], d_q_w / d_q_r [B,T,H,F*d_sub],
 *   d_subkeys  [H, sum_f n_f, d_sub]: float32 outputs (sub-key gradients summed over
 *              the batch).
 * Every pointer is 16-byte aligned and non-NULL (when B*T*H > 0).  Outputs must not
 * overlap inputs or each other.  Gradients are bitwise repeatable: every sum runs in a
 * fixed order (no float atomics) that depends only on the shape.
 */
sdm_status sdm_write_read_backward(const sdm_shape *shape, const void *q_w, const void *q_r,
                                   const void *k_val, const float *gates, const void *subkeys,
                                   const int32_t *idx_w, const float *wt_w, const int32_t *idx_r,
                                   const float *wt_r, void *snapshot, size_t snapshot_bytes,
                                   int32_t snapshot_dtype, void *bank, const void *dy, float *dbank,
                                   float *d_k_val, float *d_gates, float *d_q_w, float *d_q_r,
                                   float *d_subkeys, void *workspace, size_t workspace_bytes,
                                   sdm_stream_t stream);

/*
 * The SDM layer forward around the op (sparse-delta-memory README, usage example: a layer
 * of model width dim with num_heads heads, slots_per_head slots, num_writes / num_reads and
 * chunk_size; y = layer(x) with the bank advancing in place).  With X = x as [B*T, dim] and
 * row-major weights [out, in]:
 *   q_w = X w_qw^T, q_r = X w_qr^T   [B,T,H,F*d_sub]   w_qw, w_qr: [H*F*d_sub, dim]
 *   k_val = X w_v^T                  [B,T,H,d_v]       w_v: [H*d_v, dim]
 *   gates = sigmoid(X w_g^T)         [B,T,H,2] float32 w_g: [2H, dim], row 2h = alpha of
 *                                                      head h, row 2h+1 = beta
 *   y = the write/read op (sdm_write_read) on them, bank_init copied into bank first
 *   out = Y w_o^T                    [B,T,dim]         w_o: [dim, H*d_v]
 * x, the weights, subkeys, the intermediates and out are in the activation dtype (the
 * gates float32); products accumulate in float32.  The dense projections are cuBLASLt
 * GEMMs (loaded on first use; unavailable -> SDM_ERR_CUDA) run on the caller's workspace
 * with split-K reductions excluded; the gate projection and its sigmoid are a kernel of
 * this library.  Results are bitwise repeatable on one device.
 *   q_w, q_r, k_val, gates, y  NULL, or buffers that receive those intermediates (else
 *              they live in the workspace).
 * Every pointer is 16-byte aligned.  Refusals as for sdm_write_read, plus dim < 1
 * (INVALID).  Training through the layer: sdm_layer_forward_train / sdm_layer_backward.
 */
sdm_status sdm_layer_workspace_size(const sdm_shape *shape, int64_t dim, size_t *bytes);
sdm_status sdm_layer_forward(const sdm_shape *shape, int64_t dim, const void *x, const void *w_qw,
                             const void *w_qr, const void *w_v, const void *w_g, const void *w_o,
                             const void *subkeys, const void *bank_init, void *bank, void *out,
                             void *q_w, void *q_r, void *k_val, float *gates, void *y,
                             void *workspace, size_t workspace_bytes, sdm_stream_t stream);

/*
 * Training through the layer (README > usage example: the layer's output goes into a loss
 * and backward() runs through it with deterministic kernels).  sdm_layer_forward_train is
 * sdm_layer_forward that keeps what the backward needs in `saved` (every pointer required:
 * the intermediates as in sdm_layer_forward, the selections [B,T,H,W|R], the snapshot as
 * for sdm_write_read_train); sdm_layer_backward then gives, for a loss gradient dout
 * [B,T,dim] (activation dtype):
 *   dY = dout w_o;  dw_o = dout^T Y                      (cuBLASLt)
 *   the op's backward (sdm_write_read_backward) on the saved intermediates, which
 *   restores the bank in place and disarms the snapshot;
 *   dz = d_gates * g (1 - g) for the gate logits (the sigmoid's derivative);
 *   G = [d_q_w | d_q_r | d_k_val | dz] rounded to the activation dtype, then
 *   dx = G [w_qw; w_qr; w_v; w_g] and dw_* = G_*^T X        (cuBLASLt)
 *   d_bank_init = the sum over the batch, in increasing b, of the streams' bank gradients.
 * Weight gradients and d_subkeys are float32; dx has the activation dtype.  dbank is the
 * float32 gradient table of the op's backward: dL/d(final bank) in (zeros when only the
 * layer's output enters the loss), dL/d(bank after the learned-table copy) out.
 */
typedef struct {
  void *q_w, *q_r, *k_val;   /* [B,T,H,F*d_sub] x2, [B,T,H,d_v]              */
  float *gates;              /* [B,T,H,2]                                     */
  void *y;                   /* [B,T,H,d_v]: the op's read                    */
  int32_t *idx_w;            /* [B,T,H,W] */
  float *wt_w;
  int32_t *idx_r;            /* [B,T,H,R] */
  float *wt_r;
  void *snapshot;            /* sdm_snapshot_bytes(shape, snapshot_dtype) bytes */
  size_t snapshot_bytes;
  int32_t snapshot_dtype;
} sdm_layer_saved;

typedef struct {
  void *dx;                  /* [B,T,dim], activation dtype                   */
  float *dw_qw, *dw_qr;      /* [H*F*d_sub, dim]                              */
  float *dw_v;               /* [H*d_v, dim]                                  */
  float *dw_g;               /* [2H, dim]                                     */
  float *dw_o;               /* [dim, H*d_v]                                  */
  float *d_subkeys;          /* [H, sum_f n_f, d_sub]                         */
  float *dbank;              /* [B,H,N,d_v] in/out (above)                    */
  float *d_bank_init;        /* [H,N,d_v], or NULL                            */
} sdm_layer_grads;

sdm_status sdm_layer_forward_train(const sdm_shape *shape, int64_t dim, const void *x, const void *w_qw,
                                   const void *w_qr, const void *w_v, const void *w_g, const void *w_o,
                                   const void *subkeys, const void *bank_init, void *bank, void *out,
                                   const sdm_layer_saved *saved, void *workspace, size_t workspace_bytes,
                                   sdm_stream_t stream);
sdm_status sdm_layer_backward_workspace_size(const sdm_shape *shape, int64_t dim, size_t *bytes);
sdm_status sdm_layer_backward(const sdm_shape *shape, int64_t dim, const void *x, const void *w_qw,
                              const void *w_qr, const void *w_v, const void *w_g, const void *w_o,
                              const void *subkeys, void *bank, const void *dout, const sdm_layer_saved *saved,
                              const sdm_layer_grads *grads, void *workspace, size_t workspace_bytes,
                              sdm_stream_t stream);

/*
 * One decode step (shape->T must be 1; chunk_size is ignored) for all B*H streams.
 * Tensors as above with T = 1.
 *   bank_in         the state's tables: [B, H, N, d_v], or, with bank_in_shared != 0,
 *                   one [H, N, d_v] table every stream starts from (a learned initial
 *                   table; only with donate == 0).
 *   bank_out        [B, H, N, d_v], receives the successor tables.
 *   donate != 0     in place: bank_out must equal bank_in (or be NULL); only the W
 *                   written rows are touched (lumen PR #29 > Donating is a permission).
 *   donate == 0     copy: bank_out must not overlap bank_in; every row is written
 *                   (the unselected ones copied).  Both forms run the same arithmetic
 *                   and give bit-identical y and successor tables.
 * A decode bank smaller than the configured slots cannot be expressed here: N is
 * derived from factor_dims (CHANGELOG 2.0.0 > Behavior changes: decoding with a
 * smaller bank raises).
 */
sdm_status sdm_decode_step(const sdm_shape *shape, const void *q_w, const void *q_r,
                           const void *k_val, const float *gates, const void *subkeys,
                           const void *bank_in, int bank_in_shared, void *bank_out,
                           int donate, void *y, int32_t *idx_w, float *wt_w, int32_t *idx_r,
                           float *wt_r, void *workspace, size_t workspace_bytes,
                           sdm_stream_t stream);

/* Synchronises `stream`, reads the kernel-side error code of the last call that used
 * `workspace` into *code (SDM_DEVERR_*), and returns SDM_ERR_DEVICE if it is nonzero. */
sdm_status sdm_last_device_error(const void *workspace, size_t workspace_bytes,
                                 int32_t *code, sdm_stream_t stream);

/* Static English name of a status. */
const char *sdm_status_string(sdm_status status);

/* Reason for the last non-OK status returned on this host thread ("" if none). */
const char *sdm_last_error_message(void);

/* SDM_ABI_VERSION of the loaded library. */
int32_t sdm_abi_version(void);

/* Number of kernels this library has launched in this process (monotonic). */
uint64_t sdm_launch_count(void);

/* Per-kernel timing with CUDA events recorded on the launch stream around each of
 * this library's launches between sdm_profile_begin and sdm_profile_end.  begin
 * creates its events on first use (not inside a CUDA-graph capture); end synchronises
 * the recorded events and returns, per kernel kind, the number of launches and the
 * summed milliseconds.  Up to 4096 launches are recorded per session. */
enum {
  SDM_KERNEL_BANK_COPY = 0,
  SDM_KERNEL_SCORE = 1,      /* factor scores (tensor cores, or CUDA cores)             */
  SDM_KERNEL_SELECT = 2,     /* exact product-key top-k and weights                   */
  SDM_KERNEL_PLAN_SORT = 3,
  SDM_KERNEL_PLAN_LINK = 4,
  SDM_KERNEL_WRITE_READ = 5,
  SDM_KERNEL_DECODE = 6,
  SDM_KERNEL_BWD_FLAGS = 7,   /* backward: tokens that read a row they write            */
  SDM_KERNEL_BWD_SWEEP = 8,   /* backward: reverse sweep over the rows, bank restored   */
  SDM_KERNEL_BWD_REDUCE = 9,  /* backward: column sums, softmax backward, dq            */
  SDM_KERNEL_BWD_SUBKEY = 10, /* backward: sub-key gradient tiles and their sum         */
  SDM_KERNEL_LAYER_GATES = 11, /* layer: gate projection + sigmoid                      */
  SDM_KERNEL_LAYER_GEMM = 12,  /* layer: the cuBLASLt products (library kernels, not     */
                               /* counted by sdm_launch_count)                            */
  SDM_KERNEL_LAYER_GRAD = 13,  /* layer backward: gradient concatenation, batch sum       */
  SDM_NUM_KERNEL_KINDS = 14
};
typedef struct {
  int64_t launches[SDM_NUM_KERNEL_KINDS];
  double ms[SDM_NUM_KERNEL_KINDS];
} sdm_kernel_times;
sdm_status sdm_profile_begin(void);
sdm_status sdm_profile_end(sdm_kernel_times *out);

/* Name of a kernel kind ("write_read", ...). */
const char *sdm_kernel_name(int32_t kind);

/* Test hook of the device-side failure path; not for production use.  While `on` is
 * nonzero, the copying form of sdm_decode_step (donate == 0) makes its copy thread wait
 * on an mbarrier that nothing arrives at, instead of streaming the table: the bounded
 * wait gives up after its limit (2 s), issues no copy, records SDM_DEVERR_TIMEOUT in
 * the workspace flag and the step completes with an unspecified bank_out.  The GPU
 * context stays usable.  Process-wide; returns SDM_OK. */
sdm_status sdm_test_stall_decode_copy(int on);

/* Test hooks of the write/read launch choice; not for production use.  Results are
 * bitwise the same for every choice (the per-element arithmetic and its order depend on
 * W and R only); only speed changes.  Process-wide; 0 restores the automatic choice.
 *   sdm_test_force_write_read_layout  slice_bytes: bytes of every row one CTA owns (32,
 *       128 or 256, i.e. 1, 4 or 8 compute warps of 32 bytes each); stage_tokens: an
 *       upper bound on the tokens staged together (>= 1).  SDM_ERR_INVALID_ARG for
 *       other values.  Applies to calls made after it.
 *   sdm_test_force_simt_scorer  on != 0: score on the CUDA-core scorer (compensated
 *       float32 sums) instead of the tensor cores.  The tensor cores score bfloat16 inputs
 *       directly and float32 inputs through an exact three-way bfloat16 split of every
 *       value, of which the six part products above 2^-24 relative are kept; the scores of
 *       the two scorers may differ in the last bits. */
sdm_status sdm_test_force_write_read_layout(int slice_bytes, int stage_tokens);
sdm_status sdm_test_force_simt_scorer(int on);

/* Test hook of step 1 (the factor scores, product-key memory as cited at the top of this
 * file); not for production use.  Scores the queries of `shape` with the scorer that
 * sdm_write_read would use and writes scores [2][B*T*H][sum n_f] float32: the q_w rows,
 * then the q_r rows, row (b*T + t)*H + h, factor f's scores at column offset
 * sum_{g<f} n_g.  q_w, q_r, subkeys and scores are device pointers, 16-byte aligned, as in
 * sdm_write_read; workspace as for sdm_write_read (sdm_write_read_workspace_size bytes).
 * Refusals (INVALID_ARG, WORKSPACE, ALIAS) are decided on the host before any launch. */
sdm_status sdm_test_factor_scores(const sdm_shape *shape, const void *q_w, const void *q_r,
                                  const void *subkeys, float *scores, void *workspace,
                                  size_t workspace_bytes, sdm_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SDM_GB300_H */
