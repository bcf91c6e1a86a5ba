// Launch of one instantiation of the persistent decode kernel.  Each cache
// element type gets its own translation unit (decode_bf16.cu, decode_f32.cu,
// decode_fp8.cu) so the instantiations compile in parallel.
#pragma once

#include <atomic>

#include "paged_decode.cuh"

namespace pa {

template <bool BF16, int D, int G, bool KV8 = false>
cudaError_t run_decode_kernel(const DecodeKernelParams& kp, int grid, int device,
                              cudaStream_t stream) {
  using Tr = DecodeTraits<BF16, D, G, KV8>;
  // the opt-in to more than 48 KiB of dynamic shared memory is per device
  static std::atomic<uint64_t> configured{0};
  const uint64_t bit = 1ull << (device & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    const cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<BF16, D, G, KV8>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               Tr::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  // programmatic dependent launch: the CTAs become resident while the plan
  // kernel finishes and wait for it on the device
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(Tr::THREADS);
  cfg.dynamicSmemBytes = Tr::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_decode_kernel<BF16, D, G, KV8>, kp);
}

template <bool BF16>
cudaError_t run_decode_dispatch(int head_dim, int group, const DecodeKernelParams& kp, int grid,
                                int device, cudaStream_t stream) {
#define PA_CASE(D_, G_) \
  if (head_dim == D_ && group == G_) return run_decode_kernel<BF16, D_, G_>(kp, grid, device, stream);
  PA_CASE(64, 1) PA_CASE(64, 2) PA_CASE(64, 4) PA_CASE(64, 8)
  PA_CASE(128, 1) PA_CASE(128, 2) PA_CASE(128, 4) PA_CASE(128, 8)
#undef PA_CASE
  return cudaErrorInvalidValue;
}

cudaError_t run_decode_bf16(int head_dim, int group, const DecodeKernelParams& kp, int grid,
                            int device, cudaStream_t stream);
cudaError_t run_decode_f32(int head_dim, int group, const DecodeKernelParams& kp, int grid,
                           int device, cudaStream_t stream);
cudaError_t run_decode_fp8(int head_dim, int group, const DecodeKernelParams& kp, int grid,
                           int device, cudaStream_t stream);
// A tensor map of bf16 elements with 128-byte swizzle: `rank` dimensions
// (innermost first), the byte strides of dimensions 1.. and the box.
cudaError_t make_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides, const uint32_t* box);
cudaError_t launch_cascade_prefix(const DecodeArgs& a, const DecodeKernelParams& kp, int device,
                                  cudaStream_t stream);
cudaError_t launch_cascade_merge(const DecodeArgs& a, const DecodeKernelParams& kp,
                                 cudaStream_t stream);

}  // namespace pa
