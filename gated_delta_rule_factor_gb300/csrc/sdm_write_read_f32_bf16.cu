// Write/read kernel instances: f32 bank, bf16 activations, every column slice width.
#include "sdm_wr_kernel.cuh"

namespace sdm {

cudaError_t launch_write_read_f32_bf16(const WriteReadArgs &a, int64_t streams, int CW, int64_t smem,
                                    cudaStream_t st) {
  switch (CW) {
    case 8: return wr::launch_cw<float, __nv_bfloat16, 8>(a, streams, smem, st);
    case 16: return wr::launch_cw<float, __nv_bfloat16, 16>(a, streams, smem, st);
    case 32: return wr::launch_cw<float, __nv_bfloat16, 32>(a, streams, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sdm
