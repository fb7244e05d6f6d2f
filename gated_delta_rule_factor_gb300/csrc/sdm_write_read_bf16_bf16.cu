// Write/read kernel instances: bf16 bank, bf16 activations, every launch geometry.
#include "sdm_wr_kernel.cuh"

namespace sdm {

cudaError_t launch_write_read_bf16_bf16(const WriteReadArgs &a, int64_t streams, const WriteReadLaunch &l,
                                      cudaStream_t st) {
  return wr::launch_types<__nv_bfloat16, __nv_bfloat16>(a, streams, l, st);
}

}  // namespace sdm
