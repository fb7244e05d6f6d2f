// Instances of the write/read kernel on 128-byte row slices with the block-ordered
// token step (sdm_delta.cuh token_blocks2): two compute warps per slice splitting the
// rows, JB = the most rows a lane holds (4, 8 or 16: W and R up to 32, 64 or 128), and
// W = R = 64 with the row counts fixed at compile time.
#include "sdm_wr_kernel.cuh"

namespace sdm {

namespace {

template <typename BANK, typename ACT>
cudaError_t launch_blocks_t(const WriteReadArgs &a, int64_t streams, int64_t smem, cudaStream_t st) {
  constexpr int CW = 128 / (int)sizeof(BANK);
  dim3 grid((unsigned)a.slices, (unsigned)streams);
  auto go = [&](auto kern, int threads) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, threads, smem, st>>>(a);
    return cudaGetLastError();
  };
  // rows per lane: one block of ceil(n / 8) rows for the larger of W and R
  const int n = a.W > a.R ? a.W : a.R;
  const int per_lane = (n + 7) / 8;
  if (a.W == 64 && a.R == 64)
    return go(wr::write_read_kernel<BANK, ACT, CW, 8, true>, wr::WrGeometry<BANK, CW, 8>::NTHR);
  if (per_lane <= 4) return go(wr::write_read_kernel<BANK, ACT, CW, 4>, wr::WrGeometry<BANK, CW, 4>::NTHR);
  if (per_lane <= 8) return go(wr::write_read_kernel<BANK, ACT, CW, 8>, wr::WrGeometry<BANK, CW, 8>::NTHR);
  if (per_lane <= 16) return go(wr::write_read_kernel<BANK, ACT, CW, 16>, wr::WrGeometry<BANK, CW, 16>::NTHR);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_write_read_blocks(const WriteReadArgs &a, int64_t streams, int bank_dtype, int act_dtype,
                                     int64_t smem, cudaStream_t st) {
  if (bank_dtype == SDM_F32) {
    if (act_dtype == SDM_F32) return launch_blocks_t<float, float>(a, streams, smem, st);
    return launch_blocks_t<float, __nv_bfloat16>(a, streams, smem, st);
  }
  if (act_dtype == SDM_F32) return launch_blocks_t<__nv_bfloat16, float>(a, streams, smem, st);
  return launch_blocks_t<__nv_bfloat16, __nv_bfloat16>(a, streams, smem, st);
}

}  // namespace sdm
