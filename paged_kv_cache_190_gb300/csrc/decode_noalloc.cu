// pa_decode_noalloc: paged decode for callers that cannot allocate device
// memory themselves -- code running where no allocator is reachable (a plugin
// inside another runtime that owns all device memory, a process whose memory
// pool is fixed up front, or a caller that must not call cudaMalloc between
// steps).  Instead of a caller-provided workspace, it uses a fixed-size
// scratch array that is part of this library's device code.
//
// The array is a file-scope __device__ variable.  Under CUDA's default lazy
// module loading it is reserved on a device when its address is first looked
// up there (the first call in that CUDA context), and held until the process
// exits.  In host code `g_decode_scratch` is only a host-side stand-in for the
// symbol, not a device address, so the device address is looked up with
// cudaGetSymbolAddress, with the caller's device and context current, and
// cached.  The cache is keyed by the context's unique id (cuCtxGetId), not by
// the device ordinal: a symbol's address belongs to a context, so a caller in
// a non-primary context, or a primary context created again after
// cudaDeviceReset, gets a lookup of its own rather than another context's
// address.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "../../include/pa.h"

namespace {

constexpr size_t kScratchBytes = PA_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Driver calls through the runtime's entry-point query (no libcuda link).
struct CtxCalls {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxCalls& ctx_calls() {
  static const CtxCalls calls = [] {
    CtxCalls c;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      c.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      c.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    return c;
  }();
  return calls;
}

// Unique id of the current context (0 when there is none yet).
int current_context_id(unsigned long long* id) {
  const CtxCalls& c = ctx_calls();
  if (!c.get_current || !c.get_id) return PA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (c.get_current(&ctx) != CUDA_SUCCESS) return PA_ERR_CUDA;
  *id = 0;
  if (ctx != nullptr && c.get_id(ctx, id) != CUDA_SUCCESS) return PA_ERR_CUDA;
  return PA_OK;
}

constexpr int kCacheEntries = 16;
struct Entry {
  unsigned long long context_id;
  void* address;
};
std::mutex g_cache_lock;
Entry g_cache[kCacheEntries];
int g_cache_used = 0;

// Device address of g_decode_scratch in the current context.
int scratch_address(void** out) {
  unsigned long long id = 0;
  int rc = current_context_id(&id);
  if (rc != PA_OK) return rc;
  if (id != 0) {
    std::lock_guard<std::mutex> g(g_cache_lock);
    for (int i = 0; i < g_cache_used; ++i)
      if (g_cache[i].context_id == id) {
        *out = g_cache[i].address;
        return PA_OK;
      }
  }
  // First call in this context: the lookup loads this file's module on the
  // device (reserving the array) and, when no context was current yet, makes
  // the runtime's primary context current.
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
    return PA_ERR_CUDA;
  if (id == 0 && (rc = current_context_id(&id)) != PA_OK) return rc;
  {
    std::lock_guard<std::mutex> g(g_cache_lock);
    if (id != 0 && g_cache_used < kCacheEntries) g_cache[g_cache_used++] = Entry{id, p};
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
