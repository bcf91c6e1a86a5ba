// Internal launcher interface between the C ABI (capi.cu) and the kernels.
// Every launcher only enqueues on `stream` and returns a cudaError_t.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace pa {

// Tokens of a group's shared prefix per item of the cascade prefix kernel.
// Shared-prefix decode: tokens per pipeline stage of the prefix kernel, most
// prefix partials (pieces) per row, and the longest own suffix a sequence may
// have for the merge kernel to attend to it directly.
constexpr int kPrefixStageTokens = 64;
// Pages of one decode work item (its slice of the block table, staged in shared
// memory): a chunk holds at most kItemPages * block_size tokens.  The automatic
// chunk starts from kAutoChunkPages pages for bf16 / fp32 pools and from
// kItemPages for float8 pools, whose pages carry half the bytes, so that an
// item's fixed costs weigh double (measured on the 128K workload: 0.89 -> 0.91
// of the peak; on bf16 pools longer items cost the shared-prefix batch its L2
// reuse).
constexpr int kItemPages = 128;
constexpr int kAutoChunkPages = 64;
constexpr int kMaxPrefixPieces = 32;
constexpr int kInlineSuffixTokens = 32;

// Workspace of one pa_decode call, carved from the caller's buffer.
struct DecodeWorkspace {
  int32_t* header;       // [0] work counter, [1] total chunks, rest reserved
  int32_t* chunk_base;   // [num_seqs + 1] first global chunk of each sequence
  int4* work;            // [max_chunks] {b, first token, length, global chunk | single flag}
  float* part_lse;       // [max_chunks][num_q_heads] base-2 log-sum-exp of a chunk
  float* part_out;       // [max_chunks][num_q_heads][head_dim] chunk output, normalised
  unsigned char* q8;     // fp8 caches: [num_seqs * num_q_heads][2 * head_dim + 16] prepared q
  int32_t* prefix_parts; // cascade: [num_seqs] prefix partials of each sequence
  int4* prefix_items;    // cascade: {shared length, leader, members | piece << 24,
                         //           row set | stages per piece << 16}
  int32_t* inline_start; // cascade: [num_seqs] first own token the merge attends to, or -1
  int64_t max_chunks;
};

struct WorkspaceLayout {
  size_t chunk_base, work, part_lse, part_out, q8, prefix_parts, prefix_items, inline_start, total;
  int64_t max_chunks;
};

// num_groups > 0: the cascade layout (partials for each sequence's prefix
// chunks too, the prefix item list).
WorkspaceLayout decode_workspace_layout(int num_seqs, int num_q_heads, int head_dim,
                                        int max_context_len, int chunk_tokens,
                                        int num_groups = 0);

struct DecodeArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float scale;
  int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks;
  int max_blocks_per_seq, max_context_len, chunk_tokens;
  int q_len;  // new tokens per sequence (q and out are [num_seqs][q_len][num_q_heads][head_dim])
  // cascade (num_groups > 0): sequences group_start[f] .. group_start[f+1]-1 share
  // their first shared_lens[f] tokens (device arrays)
  const int32_t* group_start = nullptr;
  const int32_t* shared_lens = nullptr;
  int num_groups = 0;
  int bf16;  // q / out element type: 1 bf16, 0 f32 (and the caches' unless kv8)
  int kv8;   // caches hold float8 e4m3 codes (q / out bf16)
  const float* k_scale;  // kv8: dequantisation scale per kv head, device memory
  const float* v_scale;
  DecodeWorkspace ws;
  int32_t* device_errors;
  int num_sms;
  int64_t wait_limit;  // polls before a pipeline wait gives up; < 0: the default bound
};

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_cascade_plan(const DecodeArgs& a, cudaStream_t stream);
int prefix_grid(int num_sms);   // CTAs of the shared-prefix kernel

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int num_tokens,
                                     int num_kv_heads, int row_bytes, int block_size,
                                     int num_blocks, int32_t* device_errors, cudaStream_t stream);

cudaError_t launch_reshape_and_cache_fp8(const void* k, const void* v, void* k_cache,
                                         void* v_cache, const int64_t* slot_mapping,
                                         const float* k_scale, const float* v_scale,
                                         int num_tokens, int num_kv_heads, int head_dim,
                                         int block_size, int num_blocks, int32_t* device_errors,
                                         cudaStream_t stream);

cudaError_t launch_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                               const int64_t* pairs, int num_pairs, size_t block_bytes,
                               int num_src_blocks, int num_dst_blocks, int32_t* device_errors,
                               cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int num_pairs,
                               size_t block_bytes, int num_blocks, int32_t* device_errors,
                               cudaStream_t stream);

}  // namespace pa
