// Launch dispatch of the fused gather / gated delta-rule update / read kernel of
// sdm_write_read (kernel in sdm_wr_kernel.cuh, instances per type pair in
// sdm_write_read_<bank>_<act>.cu), its shared-memory size, and the per-call bank copy
// (learned table -> per-stream banks).
#include "sdm_wr_kernel.cuh"

namespace sdm {

namespace {

// Learned table [H, N, d_v] -> every stream's bank [B, H, N, d_v]: each 16-byte chunk
// of the source is read once and written B times.
__global__ void __launch_bounds__(kThreads) bank_copy_kernel(const __grid_constant__ BankCopyArgs a) {
  const int64_t chunks_per_head = a.head_bytes / 16;
  const int64_t total = chunks_per_head * a.H;
  const uint4 *src = static_cast<const uint4 *>(a.src);
  uint4 *dst = static_cast<uint4 *>(a.dst);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const uint4 v = src[i];
    const int64_t h = i / chunks_per_head, c = i % chunks_per_head;
    for (int64_t bb = 0; bb < a.B; ++bb) dst[(bb * a.H + h) * chunks_per_head + c] = v;
  }
}

}  // namespace

int64_t write_read_smem_bytes(const PlanLayout &lay, int bank_elem, int act_elem) {
  return wr::smem_layout(lay, bank_elem, act_elem).bytes;
}

cudaError_t launch_write_read(const WriteReadArgs &a, int64_t streams, int bank_dtype, int act_dtype,
                              const WriteReadLaunch &l, cudaStream_t st) {
  if (streams == 0 || a.slices == 0) return cudaSuccess;
  if (bank_dtype == SDM_F32) {
    if (act_dtype == SDM_F32) return launch_write_read_f32_f32(a, streams, l, st);
    return launch_write_read_f32_bf16(a, streams, l, st);
  }
  if (act_dtype == SDM_F32) return launch_write_read_bf16_f32(a, streams, l, st);
  return launch_write_read_bf16_bf16(a, streams, l, st);
}

cudaError_t launch_bank_copy(const BankCopyArgs &a, int sm_count, cudaStream_t st) {
  if (a.B == 0 || a.H == 0 || a.head_bytes == 0) return cudaSuccess;
  const int64_t total = a.head_bytes / 16 * a.H;
  int64_t blocks = (total + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)sm_count * 8;
  if (blocks > cap) blocks = cap;
  bank_copy_kernel<<<(unsigned)blocks, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sdm
