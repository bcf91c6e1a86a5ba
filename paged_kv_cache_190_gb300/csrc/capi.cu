// C ABI entry points: argument checks on the host, then the launchers.
// Nothing here synchronises except pa_read_device_errors.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bound on each decode pipeline wait, in polls (< 0: the kernels' default).
std::atomic<int64_t> g_wait_limit{-1};

bool supported_shape(int head_dim, int block_size) {
  return (head_dim == 64 || head_dim == 128) && (block_size == 16 || block_size == 32);
}

int elt_size(pa_dtype dt) { return dt == PA_BF16 ? 2 : (dt == PA_F32 ? 4 : 0); }

// SM count of the current device (cached per device id).
int current_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Split size: halve 512 until the (sequence, kv head, chunk) items give every
// SM a few, but never below 64 tokens; at most 32 pages per chunk.
int choose_chunk(int num_seqs, int num_kv_heads, int block_size, int max_context_len, int sms,
                 bool kv8 = false) {
  int c = (kv8 ? pa::kItemPages : pa::kAutoChunkPages) * block_size;
  const int64_t units = static_cast<int64_t>(num_seqs) * num_kv_heads;
  const int64_t target = 4 * static_cast<int64_t>(sms > 0 ? sms : 1);
  while (c > 64 && units * ((static_cast<int64_t>(max_context_len) + c - 1) / c) < target) c /= 2;
  return c;
}

bool valid_chunk(int chunk, int block_size) {
  return chunk >= 16 && chunk % 16 == 0 && chunk % block_size == 0 &&
         chunk <= pa::kItemPages * block_size;
}

}  // namespace

extern "C" {

const char* pa_get_error_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument (null, out-of-range size or misaligned buffer)";
    case PA_ERR_UNSUPPORTED: return "unsupported dtype, head_dim, block_size or head grouping";
    case PA_ERR_OUT_OF_BLOCKS: return "out of blocks: the free list is empty";
    case PA_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case PA_ERR_NOT_FOUND: return "unknown sequence id";
    case PA_ERR_EXISTS: return "sequence id already in use";
    case PA_ERR_WORKSPACE: return "decode workspace missing, misaligned or too small";
    case PA_ERR_SWAPPED: return "the sequence is swapped out to host memory";
    default: return "unknown status";
  }
}

int pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                         int32_t* device_errors, void* stream) {
  const int elt = elt_size(dtype);
  if (!elt || !supported_shape(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const cudaError_t e = pa::launch_reshape_and_cache(
      k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim * elt, block_size,
      num_blocks, device_errors, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst_pairs, int num_pairs,
                   size_t block_bytes, int num_blocks, int32_t* device_errors, void* stream) {
  if (num_pairs < 0 || num_blocks <= 0 || block_bytes == 0 || block_bytes % 16 != 0)
    return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !src_dst_pairs || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const cudaError_t e =
      pa::launch_copy_blocks(k_cache, v_cache, src_dst_pairs, num_pairs, block_bytes, num_blocks,
                             device_errors, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                   const int64_t* src_dst_pairs, int num_pairs, size_t block_bytes,
                   int num_src_blocks, int num_dst_blocks, int32_t* device_errors, void* stream) {
  if (num_pairs < 0 || num_src_blocks <= 0 || num_dst_blocks <= 0 || block_bytes == 0 ||
      block_bytes % 16 != 0)
    return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!src_k || !src_v || !dst_k || !dst_v || !src_dst_pairs || !aligned16(src_k) ||
      !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v))
    return PA_ERR_INVALID_ARG;
  const cudaError_t e = pa::launch_swap_blocks(src_k, src_v, dst_k, dst_v, src_dst_pairs,
                                               num_pairs, block_bytes, num_src_blocks,
                                               num_dst_blocks, device_errors,
                                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_decode_chunk_tokens(int num_seqs, int num_kv_heads, int block_size, int max_context_len) {
  if (num_seqs < 0 || num_kv_heads <= 0 || max_context_len < 0) return PA_ERR_INVALID_ARG;
  if (block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
  const int sms = current_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  return choose_chunk(num_seqs, num_kv_heads, block_size, max_context_len, sms);
}

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int max_context_len, int chunk_tokens) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_context_len < 0) return 0;
  if (!supported_shape(head_dim, block_size)) return 0;
  int chunk = chunk_tokens;
  if (chunk == 0) {
    const int sms = current_sm_count();
    if (sms <= 0) return 0;
    chunk = choose_chunk(num_seqs, num_kv_heads, block_size, max_context_len, sms);
  } else if (!valid_chunk(chunk, block_size)) {
    return 0;
  }
  return pa::decode_workspace_layout(num_seqs, num_q_heads, head_dim, max_context_len, chunk).total;
}

size_t pa_decode_cascade_workspace_size(int num_seqs, int num_groups, int num_q_heads,
                                         int num_kv_heads, int head_dim, int block_size,
                                         int max_context_len, int chunk_tokens) {
  if (num_seqs < 0 || num_groups < 1 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      max_context_len < 0)
    return 0;
  if (!supported_shape(head_dim, block_size)) return 0;
  int chunk = chunk_tokens;
  if (chunk == 0) {
    const int sms = current_sm_count();
    if (sms <= 0) return 0;
    chunk = choose_chunk(num_seqs, num_kv_heads, block_size, max_context_len, sms);
  } else if (!valid_chunk(chunk, block_size)) {
    return 0;
  }
  return pa::decode_workspace_layout(num_seqs, num_q_heads, head_dim, max_context_len, chunk,
                                     num_groups).total;
}

}  // extern "C"

namespace {

// Shared body of pa_decode and pa_decode_fp8 (kv8: e4m3 caches, bf16 q / out).
int decode_common(void* out, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, float scale,
                  int num_kv_heads, int num_seqs, int num_q_heads, int head_dim, int block_size,
                  int num_blocks, int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                  bool kv8, const float* k_scale, const float* v_scale, int q_len,
                  int chunk_tokens, void* workspace, size_t workspace_bytes,
                  int32_t* device_errors, void* stream, const int32_t* group_start = nullptr,
                  const int32_t* shared_lens = nullptr, int num_groups = 0) {
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_seqs < 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0 || max_context_len < 0)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  const int group = num_q_heads / num_kv_heads;
  if (q_len < 1) return PA_ERR_INVALID_ARG;
  // an item holds the q_len new tokens of one kv head's group: 1, 2, 4 or 8 rows
  const int rows = q_len * group;
  if (rows != 1 && rows != 2 && rows != 4 && rows != 8) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if (kv8 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int sms = current_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  int chunk = chunk_tokens;
  if (chunk == 0)
    chunk = choose_chunk(num_seqs, num_kv_heads, block_size, max_context_len, sms, kv8);
  else if (!valid_chunk(chunk, block_size))
    return PA_ERR_INVALID_ARG;
  const pa::WorkspaceLayout lay = pa::decode_workspace_layout(
      num_seqs, q_len * num_q_heads, head_dim, max_context_len, chunk, num_groups);
  if (lay.max_chunks >= (int64_t{1} << 30)) return PA_ERR_INVALID_ARG;   // chunk ids keep 30 bits
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < lay.total)
    return PA_ERR_WORKSPACE;

  char* ws = static_cast<char*>(workspace);
  pa::DecodeArgs a;
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.scale = scale;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_context_len = max_context_len;
  a.chunk_tokens = chunk;
  a.q_len = q_len;
  a.bf16 = dtype == PA_BF16;
  a.kv8 = kv8 ? 1 : 0;
  a.k_scale = kv8 ? k_scale : nullptr;
  a.v_scale = kv8 ? v_scale : nullptr;
  a.ws.header = reinterpret_cast<int32_t*>(ws);
  a.ws.chunk_base = reinterpret_cast<int32_t*>(ws + lay.chunk_base);
  a.ws.work = reinterpret_cast<int4*>(ws + lay.work);
  a.ws.part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
  a.ws.part_out = reinterpret_cast<float*>(ws + lay.part_out);
  a.ws.q8 = reinterpret_cast<unsigned char*>(ws + lay.q8);
  a.ws.prefix_parts = reinterpret_cast<int32_t*>(ws + lay.prefix_parts);
  a.ws.prefix_items = reinterpret_cast<int4*>(ws + lay.prefix_items);
  a.ws.inline_start = reinterpret_cast<int32_t*>(ws + lay.inline_start);
  a.group_start = group_start;
  a.shared_lens = shared_lens;
  a.num_groups = num_groups;
  a.ws.max_chunks = lay.max_chunks;
  a.device_errors = device_errors;
  a.num_sms = sms;
  a.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  const cudaError_t e = pa::launch_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens, float scale,
              int num_kv_heads, int num_seqs, int num_q_heads, int head_dim, int block_size,
              int num_blocks, int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
              int chunk_tokens, void* workspace, size_t workspace_bytes,
              int32_t* device_errors, void* stream) {
  if (!elt_size(dtype) || !supported_shape(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
  return decode_common(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                       num_seqs, num_q_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, dtype, false, nullptr, nullptr, 1,
                       chunk_tokens, workspace, workspace_bytes, device_errors, stream);
}

int pa_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, float scale,
                  const float* k_scale, const float* v_scale, int num_kv_heads, int num_seqs,
                  int num_q_heads, int head_dim, int block_size, int num_blocks,
                  int max_blocks_per_seq, int max_context_len, int chunk_tokens, void* workspace,
                  size_t workspace_bytes, int32_t* device_errors, void* stream) {
  if (head_dim != 128 || !supported_shape(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
  return decode_common(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                       num_seqs, num_q_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, PA_BF16, true, k_scale, v_scale, 1,
                       chunk_tokens, workspace, workspace_bytes, device_errors, stream);
}

int pa_decode_multi(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens, float scale,
                    int num_kv_heads, int num_seqs, int num_q_heads, int q_len, int head_dim,
                    int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len,
                    pa_dtype dtype, int chunk_tokens, void* workspace, size_t workspace_bytes,
                    int32_t* device_errors, void* stream) {
  if (!elt_size(dtype) || !supported_shape(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
  return decode_common(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                       num_seqs, num_q_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, dtype, false, nullptr, nullptr, q_len,
                       chunk_tokens, workspace, workspace_bytes, device_errors, stream);
}

int pa_decode_cascade(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens,
                      const int32_t* group_start, const int32_t* shared_lens, int num_groups,
                      float scale, int num_kv_heads, int num_seqs, int num_q_heads, int head_dim,
                      int block_size, int num_blocks, int max_blocks_per_seq,
                      int max_context_len, int chunk_tokens, void* workspace,
                      size_t workspace_bytes, int32_t* device_errors, void* stream) {
  if (!supported_shape(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
  if (num_seqs > 0 && (num_groups < 1 || num_groups > num_seqs || !group_start || !shared_lens))
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  return decode_common(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                       num_seqs, num_q_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, PA_BF16, false, nullptr, nullptr, 1,
                       chunk_tokens, workspace, workspace_bytes, device_errors, stream,
                       group_start, shared_lens, num_groups);
}

int pa_reshape_and_cache_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, const float* k_scale,
                             const float* v_scale, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks,
                             int32_t* device_errors, void* stream) {
  if (head_dim != 128 || !supported_shape(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping || !k_scale || !v_scale)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const cudaError_t e = pa::launch_reshape_and_cache_fp8(
      k, v, k_cache, v_cache, slot_mapping, k_scale, v_scale, num_tokens, num_kv_heads, head_dim,
      block_size, num_blocks, device_errors, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_debug_set_wait_limit(int polls) {
  g_wait_limit.store(polls < 0 ? -1 : polls, std::memory_order_relaxed);
  return PA_OK;
}

int pa_read_device_errors(int32_t* device_errors, int32_t* host_flags, int clear, void* stream) {
  if (!device_errors || !host_flags) return PA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemcpy(host_flags, device_errors, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PA_ERR_CUDA;
  if (clear && cudaMemset(device_errors, 0, sizeof(int32_t)) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

}  // extern "C"
