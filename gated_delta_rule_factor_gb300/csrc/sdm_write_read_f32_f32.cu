// Write/read kernel instances: f32 bank, f32 activations, every launch geometry.
#include "sdm_wr_kernel.cuh"

namespace sdm {

cudaError_t launch_write_read_f32_f32(const WriteReadArgs &a, int64_t streams, const WriteReadLaunch &l,
                                      cudaStream_t st) {
  return wr::launch_types<float, float>(a, streams, l, st);
}

}  // namespace sdm
