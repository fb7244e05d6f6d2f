// Decode kernel instances: f32 activations, f32 bank.
#include "sdm_decode.cuh"

namespace sdm {
namespace dec {

cudaError_t launch_decode_f32_f32(const DecodeArgs &a, const CandidateList &cl, int EF, int EC, int64_t smem,
                                 cudaStream_t st) {
  return launch_decode_dt<float, float>(a, cl, EF, EC, smem, st);
}

}  // namespace dec
}  // namespace sdm
