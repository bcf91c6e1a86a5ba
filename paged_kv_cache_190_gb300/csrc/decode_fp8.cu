// float8 e4m3 cache instantiations of the persistent paged-decode kernel
// (head_dim 128: one 128-byte row per token; q and out bf16).
#include "decode_instances.cuh"

namespace pa {
cudaError_t run_decode_fp8(int head_dim, int group, const DecodeKernelParams& kp, int grid,
                           int device, cudaStream_t stream) {
  if (head_dim != 128) return cudaErrorInvalidValue;
  switch (group) {
    case 1: return run_decode_kernel<true, 128, 1, true>(kp, grid, device, stream);
    case 2: return run_decode_kernel<true, 128, 2, true>(kp, grid, device, stream);
    case 4: return run_decode_kernel<true, 128, 4, true>(kp, grid, device, stream);
    case 8: return run_decode_kernel<true, 128, 8, true>(kp, grid, device, stream);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace pa
