// Host <-> kernel interface of the SDM library (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sdm.h"

namespace sdm {

constexpr int kThreads = 256;

// Decode kernel geometry.  Its dynamic shared memory starts with one region that serves,
// in turn, as the sub-key tile of the scoring, the ring through which the copying form
// streams the table, and the rows of the write and the read; the queries, factor scores
// and candidate tuples follow it.
constexpr int kDecodeNCG = 8;                               // 16-byte column groups per warp
constexpr int64_t kDecodeRowSlice = kDecodeNCG * 16;        // bytes of a row a warp stages
constexpr int kDecodeScoreRows = kThreads / 2;              // sub-key rows per scoring tile
constexpr int kDecodeScoreCols = 32;                        // sub-key columns per scoring tile
constexpr int64_t kDecodeCopyRingBytes = 3 * 16384;
inline int64_t decode_region_bytes(int64_t W, int64_t R, bool copy) {
  int64_t b = (int64_t)(kThreads / 32) * (W > R ? W : R) * kDecodeRowSlice;
  const int64_t tile = (int64_t)kDecodeScoreRows * (kDecodeScoreCols + 1) * 4;
  if (tile > b) b = tile;
  if (copy && kDecodeCopyRingBytes > b) b = kDecodeCopyRingBytes;
  return (b + 127) / 128 * 128;
}

// Position tuples (p_1..p_F), p_f < min(k, n_f), with prod(p_f + 1) <= k, in
// lexicographic order; byte f of an entry holds p_f.  Index 0 = write query (k = W),
// 1 = read query (k = R).  Passed to kernels by value.
struct CandidateList {
  int32_t n[2];
  uint32_t tup[2][SDM_MAX_CANDIDATES];
  // Boxes {p_f < a_f for every f} holding at least k tuples, by their corner (a_f - 1 in
  // byte f): every slot of such a box scores at least the corner's slot, so the k-th
  // best slot score is at least the best corner score (the selection's pruning bound).
  int32_t nbox[2];
  uint32_t box[2][32];
};

// Geometry of the product keys, shared by the top-k and decode kernels.
struct KeyGeometry {
  int32_t F, d_sub, ntot;            // factors, sub-key dim, sum of n_f
  int32_t nf[SDM_MAX_FACTORS];       // n_f
  int32_t off[SDM_MAX_FACTORS];      // row offset of factor f in the sub-key table
  int32_t k[2];                      // W, R
  int32_t kf[2][SDM_MAX_FACTORS];    // min(k, n_f)
};

// Factor scores of every query row: scores[qsel][(b*T + t)*H + h][ntot] (float32).
struct ScoreArgs {
  const void *q[2];      // q_w, q_r [BT, H, F*d_sub]
  const void *subkeys;   // [H, ntot, d_sub]
  float *scores;         // [2, BT*H, ntot]
  void *split;           // tensor-core scoring of float32 inputs: score_split_bytes of workspace
  int32_t *err;
  int64_t BT;            // B*T tokens
  int32_t H;
  KeyGeometry g;
};

// Exact top-k of every query row from its factor scores.
struct SelectArgs {
  const float *scores;   // [2, rows, ntot]
  int32_t *idx[2];       // [rows, k]
  float *wt[2];
  int32_t *err;
  int64_t rows;          // B*T*H rows per query kind
  KeyGeometry g;
};

struct BankCopyArgs {
  const void *src;       // [H, N, d_v]
  void *dst;             // [B, H, N, d_v]
  int64_t B;
  int64_t head_bytes;    // N * d_v * elem bytes (multiple of 16)
  int64_t H;
};

// Chunk plan (per stream s = b*H + h and stage g of G tokens, L = G*(W+R) refs).
// The write/read kernel keeps a stage's distinct rows in one of three shared-memory
// row buffers; row u of a stage lives at byte offset o(u) = u*RB + (color << 5) of its
// buffer, where RB is the CTA's row slice in bytes and `color` (0..3, masked by cmask)
// rotates which 32-byte piece of the slot each compute warp uses, so that the four
// rows a quarter-warp reads at once sit in four different bank groups.  Every offset
// the kernel uses is such an o (a u16: L*RB <= 65536).
//   uniq[s][g][u]    sorted unique slot ids of the stage        (int32, L per stage)
//   nuniq[s][g]      number of unique rows
//   uo[s][g][u]      o(u)                                        (uint16, L per stage)
//   written[s][g][u] 1 if a write ref of the stage hits row u   (uint8, L per stage)
//   lrec[s][g]       the stage's row lists, fetched three stages ahead:
//     int32 n_u, n_load, n_out1, n_out2, n_wb, 3 x pad           (32 bytes)
//     uint2 ent[L]     the n_load bank rows fetched, {row offset, o}, the row offset
//                      being slot * (d_v * elem / 16) in 16-byte units from the
//                      stream's table
//     uint2 out[L]     n_out1 rows this stage hands to stage g+1, then n_out2 rows it
//                      hands to stage g+2 (rows g+1 does not hold), {o_dst | o_src << 16,
//                      0}: the compute warps copy them out of this stage's buffer at its
//                      end (the bank may be stale for them)
//     uint2 wb[L]      rows written back after the stage, {row offset, o}: dirty ones
//                      (written, or carried in) that neither of the next two stages holds
//   crec[s][g]       the compute warps' per-stage data, one contiguous copy:
//     uint16 refmap[L]    o of ref (t_local*(W+R) + j)
//     uint8  tokflag[G]   1 if the token reads a row it also writes
//     float  wts[L]       the weights of ref (t_local*(W+R) + j): W write, then R read
//     float  gates[G][2]  (alpha, beta) of each token
struct PlanLayout {
  int32_t G;             // tokens per stage
  int32_t L;             // refs per full stage = G*(W+R)
  int32_t n_stages;      // ceil(T / G)
  int32_t RB;            // row slice bytes of one CTA (row slot stride)
  int32_t cmask;         // color bits usable in o (3 when RB >= 128, else 0)
  int64_t lrec_bytes;    // bytes per row-list record (multiple of 16)
  int64_t off_ent, off_out, off_wb;
  int64_t crec_bytes;    // bytes per compute record (multiple of 16)
  int64_t off_refmap, off_tokflag, off_wts, off_gates;
};

struct PlanArgs {
  const int32_t *idx[2];  // idx_w [B,T,H,W], idx_r [B,T,H,R]
  const float *wt[2];     // their weights
  const float *gates;     // [B,T,H,2]
  uint32_t pitch16;       // a bank row in 16-byte units (d_v * elem / 16)
  int32_t *uniq;
  int32_t *nuniq;
  uint16_t *uo;
  uint8_t *written;
  unsigned char *lrecs;
  unsigned char *crecs;
  int32_t *err;
  int64_t T;
  int32_t H, W, R;
  int64_t N;
  PlanLayout lay;
};

struct WriteReadArgs {
  const void *k_val;      // [B,T,H,d_v]
  const unsigned char *lrecs;
  const unsigned char *crecs;
  void *bank;             // [B,H,N,d_v]
  void *y;                // [B,T,H,d_v]
  int32_t *err;
  int64_t T, N, d_v;
  int32_t H, W, R;
  int32_t slices;         // ceil(row bytes / RB)
  int32_t row_bytes;      // d_v * bank element bytes (the last slice may be partial)
  PlanLayout lay;
  // Snapshot of the rows each token overwrites, taken before its write (NULL: none).
  // Layout [B*H, T, P, W, PC] of the snapshot type, P = ceil(row_bytes / 32) 32-byte
  // pieces of a bank row and PC = 32 / bank element bytes columns per piece: the rows a
  // compute warp holds for one token are contiguous.
  unsigned char *snap;
  int32_t snap_bf16;      // snapshot rounded to bfloat16 (else float32, exact)
  int32_t pieces;         // P
};

struct DecodeArgs {
  const void *q[2];       // [B, H, F*d_sub]
  const void *k_val;      // [B, H, d_v]
  const float *gates;     // [B, H, 2]
  const void *subkeys;
  const void *bank_in;    // [B,H,N,d_v] or [H,N,d_v] when shared
  void *bank_out;
  void *y;
  int32_t *idx[2];        // nullable
  float *wt[2];           // nullable
  int32_t *err;
  int64_t B, N, d_v;
  int32_t H;
  int32_t bank_in_shared; // bank_in is one [H,N,d_v] table for all streams
  int32_t copy_rest;      // copy the table bank_in -> bank_out (then write its written rows)
  int64_t region_bytes;   // decode_region_bytes(W, R, copy_rest)
  int32_t test_stall_copy;  // test hook: the copy waits on a barrier nothing arrives at
  KeyGeometry g;
};

// The backward of the write/read op (sdm_backward.cu).  Stream s = b*H + h; row r of
// a token = (b*T + t)*H + h.
//   sweep: one warp per (stream, 32-byte piece p of every bank row) runs the tokens from
//          last to first on its piece, with the bank (restored from the snapshot) and
//          the gradient table G (float32) in global memory, and writes per-piece partial
//          sums of the per-token scalars: part[s][t][p][PS], PS = align4(W + R + 2):
//          dw_j (j < W), dr_j (W + j), dalpha (W + R), dbeta (W + R + 1).
//   reduce: one warp per token row: sums the partials over p in increasing p, the
//          softmax backward, the gate gradients, the dense factor-score gradients
//          ds[h][kind][b*T + t][ntot] and the query gradients.
//   subkey_grad: split-K tiles of dK_f = sum_k ds_f[k]^T q_f[k], then their sum in
//          split order.
struct BackwardArgs {
  const int32_t *idx[2];  // idx_w [B,T,H,W], idx_r [B,T,H,R]
  const float *wt[2];
  const float *gates;     // [B,T,H,2]
  const void *q[2];       // q_w, q_r [B,T,H,F*d_sub] (act)
  const void *k_val;      // [B,T,H,d_v] (act)
  const void *dy;         // [B,T,H,d_v] (act)
  const void *subkeys;    // [H, ntot, d_sub] (act)
  const unsigned char *snap;  // snapshot data (layout as WriteReadArgs::snap)
  const int32_t *snap_hdr;    // the snapshot's header word (armed by the forward)
  uint8_t *flags;         // [B*H*T] 1 if the token reads a row it writes
  void *bank;             // [B,H,N,d_v] (bank type): final bank in, restored out
  float *grad;            // [B,H,N,d_v]: dL/d(final bank) in, dL/d(initial bank) out
  float *d_kv;            // [B,T,H,d_v]
  float *d_gates;         // [B,T,H,2]
  float *d_q[2];          // [B,T,H,F*d_sub]
  float *d_subkeys;       // [H, ntot, d_sub]
  float *part;            // [B*H, T, P, PS]
  float *ds;              // [H, 2, B*T, ntot]
  float *dk_part;         // [KS, H, ntot, d_sub]
  int32_t *err;
  int64_t B, T, N, d_v;
  int32_t H, W, R, P, PS;  // P: partial records per token; PS: their stride (floats)
  int32_t Pw;             // column pieces of the sweep (one warp each)
  int32_t P32;            // 32-byte pieces of a row (the snapshot's layout)
  int32_t act_bf16, snap_bf16;
  int32_t KS;             // split of the sub-key gradient's K = 2*B*T rows
  int64_t k_chunk;        // rows per split (multiple of 16)
  KeyGeometry g;
};
constexpr int32_t kSnapshotArmed = 0x5a5a5a5a;   // header word of a snapshot a backward may use
constexpr int64_t kSnapshotHeaderBytes = 256;
cudaError_t launch_bwd_flags(const BackwardArgs &a, cudaStream_t st);
cudaError_t launch_bwd_sweep(const BackwardArgs &a, int bank_dtype, cudaStream_t st);
cudaError_t launch_bwd_reduce(const BackwardArgs &a, cudaStream_t st);
cudaError_t launch_bwd_subkeys(const BackwardArgs &a, cudaStream_t st);
inline int32_t bwd_part_stride(int W, int R) { return (W + R + 2 + 3) & ~3; }
// 16-byte column groups per warp of the backward's reverse sweep (the piece is
// 16 * kSweepCG bytes of every bank row), warps per sweep CTA, and whether a CTA's warps
// store one combined record of partial column sums per token (else one each).
constexpr int kSweepCG = 2;
constexpr int kSweepCtaWarps = 2;
constexpr bool kSweepCtaRecord = true;

// The layer around the op (sdm_layer.cu).  layer_gemm: out[n][m] = sum_k a[m][k] b[n][k]
// (row-major weights a [m, k], activations b [n, k]) by cuBLASLt, loaded on first use;
// returns nullptr or the reason it failed.
const char *layer_gemm(const void *a, const void *b, void *out, int64_t m, int64_t n, int64_t k, int act_dtype,
                       void *ws, size_t ws_bytes, cudaStream_t st);
cudaError_t launch_layer_gates(const void *x, const void *w_g, float *gates, int64_t rows, int64_t dim,
                               int32_t n_gates, int act_dtype, int sm_count, cudaStream_t st);
// The general column-major product D (m x n, ldd) = op(A) op(B) (+ D), A/B of type ab, D
// of type dd, float32 accumulation; nullptr or the reason it failed.
const char *lt_gemm(bool ta, bool tb, int64_t m, int64_t n, int64_t k, const void *A, int64_t lda, const void *B,
                    int64_t ldb, void *D, int64_t ldd, int ab, int dd, bool accumulate, void *ws, size_t ws_bytes,
                    cudaStream_t st);
cudaError_t launch_layer_grad_cat(const float *d_qw, const float *d_qr, const float *d_kv, const float *d_g,
                                  const float *gates, void *gcat, int64_t rows, int64_t dq, int64_t dv, int64_t ng,
                                  int64_t K, int act_dtype, int sm_count, cudaStream_t st);
cudaError_t launch_batch_sum(const float *in, float *out, int64_t B, int64_t n, int sm_count, cudaStream_t st);
constexpr int64_t kLayerGemmWorkspace = (int64_t)32 << 20;   // cuBLASLt's share of a layer workspace

// Raises a kernel's dynamic shared-memory limit to at least `smem` bytes on the current
// device, once per (kernel, device, larger size): the attribute call is not repeated per
// launch, so steady-state calls make only stream-ordered CUDA calls (graph capture).
cudaError_t raise_smem_limit(const void *kernel, int64_t smem);

// Launchers, defined next to their kernels.  Each returns the launch error.
cudaError_t launch_score_simt(const ScoreArgs &a, int act_dtype, cudaStream_t st);
// Tensor-core scoring: bf16 inputs directly, float32 inputs through an exact three-way
// bf16 split kept in ScoreArgs::split (score_split_bytes bytes, 16-byte aligned).
cudaError_t launch_score_tc(const ScoreArgs &a, int act_dtype, cudaStream_t st);
bool score_tc_supported(const KeyGeometry &g, int64_t H, int act_dtype);
int64_t score_split_bytes(const KeyGeometry &g, int64_t BT, int64_t H, int act_dtype);
cudaError_t launch_select(const SelectArgs &a, const CandidateList &cl, int EF, int EC,
                          int sm_count, cudaStream_t st);
cudaError_t launch_bank_copy(const BankCopyArgs &a, int sm_count, cudaStream_t st);
cudaError_t launch_plan_sort(const PlanArgs &a, int64_t streams, int sort_pow2,
                             cudaStream_t st);
cudaError_t launch_plan_link(const PlanArgs &a, int64_t streams, cudaStream_t st);
// Write/read launch: NCW compute warps (RB = 32*NCW bytes of every row per CTA), LW
// loader warps, grid (slices, streams).
struct WriteReadLaunch {
  int32_t NCW;            // 1, 4 or 8
  int32_t LW;             // 4 or 8
  int64_t smem_bytes;
};
cudaError_t launch_write_read(const WriteReadArgs &a, int64_t streams, int bank_dtype,
                              int act_dtype, const WriteReadLaunch &l, cudaStream_t st);
// The instances of one (bank, activation) type pair, from sdm_write_read_<bank>_<act>.cu.
cudaError_t launch_write_read_f32_f32(const WriteReadArgs &a, int64_t streams, const WriteReadLaunch &l, cudaStream_t st);
cudaError_t launch_write_read_f32_bf16(const WriteReadArgs &a, int64_t streams, const WriteReadLaunch &l, cudaStream_t st);
cudaError_t launch_write_read_bf16_f32(const WriteReadArgs &a, int64_t streams, const WriteReadLaunch &l, cudaStream_t st);
cudaError_t launch_write_read_bf16_bf16(const WriteReadArgs &a, int64_t streams, const WriteReadLaunch &l,
                                        cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs &a, const CandidateList &cl, int act_dtype,
                          int bank_dtype, int EF, int EC, int64_t smem_bytes,
                          cudaStream_t st);

// Dynamic shared memory of the write/read kernel for a plan layout (RB, G, records) and
// the activation element size.
int64_t write_read_smem_bytes(const PlanLayout &lay, int bank_elem, int act_elem);

}  // namespace sdm
