// Dispatch of the single-token decode kernel (sdm_decode.cuh) by activation and bank
// type; each (activation, bank) pair is compiled in its own translation unit.
#include "sdm_decode.cuh"

namespace sdm {

cudaError_t launch_decode(const DecodeArgs &a, const CandidateList &cl, int act_dtype,
                          int bank_dtype, int EF, int EC, int64_t smem, cudaStream_t st) {
  if (a.B == 0 || a.H == 0) return cudaSuccess;
  if (act_dtype == SDM_BF16) {
    if (bank_dtype == SDM_BF16) return dec::launch_decode_bf16_bf16(a, cl, EF, EC, smem, st);
    return dec::launch_decode_bf16_f32(a, cl, EF, EC, smem, st);
  }
  if (bank_dtype == SDM_BF16) return dec::launch_decode_f32_bf16(a, cl, EF, EC, smem, st);
  return dec::launch_decode_f32_f32(a, cl, EF, EC, smem, st);
}

}  // namespace sdm
