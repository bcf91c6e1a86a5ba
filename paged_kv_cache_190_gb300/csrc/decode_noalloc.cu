// pa_decode_noalloc: paged decode for callers that cannot allocate device
// memory themselves -- code running where no allocator is reachable (a plugin
// inside another runtime that owns all device memory, a process whose memory
// pool is fixed up front, or a caller that must not call cudaMalloc between
// steps).  Instead of a caller-provided workspace, it uses a fixed-size
// scratch array that is part of this library's device code.
//
// The array is a file-scope __device__ variable: it is allocated when the
// library's device code is loaded on a GPU and held until the process exits.
// In host code `g_decode_scratch` is only a host-side stand-in for the symbol,
// not a device address, so the device address is looked up once per device
// with cudaGetSymbolAddress (with that device current) and cached.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/pa.h"

namespace {

constexpr size_t kScratchBytes = PA_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_address[kMaxDevices];

// Device address of g_decode_scratch on the current device.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  void* p = g_scratch_address[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return PA_ERR_CUDA;
    g_scratch_address[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_noalloc(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 const int32_t* context_lens, float scale, int num_kv_heads,
                                 int num_seqs, int num_q_heads, int head_dim, int block_size,
                                 int num_blocks, int max_blocks_per_seq, int max_context_len,
                                 pa_dtype dtype, int chunk_tokens, int32_t* device_errors,
                                 void* stream) {
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != PA_OK) return rc;
  if (num_seqs > 0) {
    const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 block_size, max_context_len, chunk_tokens);
    if (need > kScratchBytes) return PA_ERR_WORKSPACE;  // larger than the static scratch
  }
  // Everything the kernels need zeroed (the work counter) or rewritten (the
  // work list, chunk offsets, partials) is reset by the call itself, so the
  // previous call's leftovers in the array do not matter.
  return pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                   num_seqs, num_q_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
                   max_context_len, dtype, chunk_tokens, scratch, kScratchBytes, device_errors,
                   stream);
}
