// Exact product-key top-k of every query row from its factor scores: one warp per row
// (row_topk in sdm_topk.cuh), CTAs looping over rows so that the candidate lists and
// pruning boxes are staged into shared memory once per CTA.
#include "sdm_common.cuh"
#include "sdm_internal.h"
#include "sdm_topk.cuh"

namespace sdm {

namespace {

template <int EF, int EC>
__global__ void __launch_bounds__(kThreads, 3)
    select_kernel(const __grid_constant__ SelectArgs a, const __grid_constant__ CandidateList cl) {
  __shared__ uint32_t cand[2 * SDM_MAX_CANDIDATES];
  __shared__ uint32_t boxes[2][32];
  __shared__ RowScratch rs[kThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < cl.n[0]; i += kThreads) cand[i] = cl.tup[0][i];
  for (int i = tid; i < cl.n[1]; i += kThreads) cand[cl.n[0] + i] = cl.tup[1][i];
  if (tid < 64) boxes[tid >> 5][tid & 31] = cl.box[tid >> 5][tid & 31];
  __syncthreads();
  const KeyGeometry &g = a.g;
  const int64_t total = 2 * a.rows;
  for (int64_t r = (int64_t)blockIdx.x * (kThreads / 32) + warp; r < total;
       r += (int64_t)gridDim.x * (kThreads / 32)) {
    const int qsel = r >= a.rows ? 1 : 0;
    const int64_t row = r - qsel * a.rows;
    const int k = g.k[qsel];
    row_topk<EF, EC>(a.scores + r * g.ntot, g, qsel, cand + (qsel ? cl.n[0] : 0), cl.n[qsel], boxes[qsel],
                     cl.nbox[qsel], rs[warp], a.idx[qsel] + row * k, a.wt[qsel] + row * k);
  }
}

template <int EF, int EC>
cudaError_t launch_select_t(const SelectArgs &a, const CandidateList &cl, int sm_count, cudaStream_t st) {
  const int64_t warps_needed = 2 * a.rows;
  int64_t blocks = (warps_needed + kThreads / 32 - 1) / (kThreads / 32);
  // one wave of resident CTAs, each warp looping over rows
  static int per_sm = 0;
  if (per_sm == 0 &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, select_kernel<EF, EC>, kThreads, 0) != cudaSuccess)
    per_sm = 0;
  const int64_t cap = (int64_t)sm_count * (per_sm > 0 ? per_sm : 2);
  if (blocks > cap) blocks = cap;
  select_kernel<EF, EC><<<(unsigned)blocks, kThreads, 0, st>>>(a, cl);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select(const SelectArgs &a, const CandidateList &cl, int EF, int EC, int sm_count,
                          cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  if (EF == 2 && EC == 2) return launch_select_t<2, 2>(a, cl, sm_count, st);
  if (EF == 4 && EC == 4) return launch_select_t<4, 4>(a, cl, sm_count, st);
  return cudaErrorInvalidValue;
}

}  // namespace sdm
