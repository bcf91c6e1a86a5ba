// fp32 instantiations of the persistent paged-decode kernel.
#include "decode_instances.cuh"

namespace pa {
cudaError_t run_decode_f32(int head_dim, int group, const DecodeKernelParams& kp, int grid,
                           int device, cudaStream_t stream) {
  return run_decode_dispatch<false>(head_dim, group, kp, grid, device, stream);
}
}  // namespace pa
