// Decode kernel instances: f32 activations, bf16 bank.
#include "sdm_decode.cuh"

namespace sdm {
namespace dec {

cudaError_t launch_decode_f32_bf16(const DecodeArgs &a, const CandidateList &cl, int EF, int EC, int64_t smem,
                                 cudaStream_t st) {
  return launch_decode_dt<float, __nv_bfloat16>(a, cl, EF, EC, smem, st);
}

}  // namespace dec
}  // namespace sdm
