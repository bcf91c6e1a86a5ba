/*
 * pa.h -- C ABI of libpagedattn: paged-KV-cache decode for NVIDIA GB300 (sm_103a).
 *
 * The operations follow the statement of the problem on the pages this library
 * is built from:
 *   - "PagedAttention原理" (ch. 3 of a vLLM long-sequence inference memory guide),
 *     §3.2 (the KV cache is cut into fixed-size pages; logically contiguous tokens
 *     live in scattered physical pages reached through a page table), §3.3.1
 *     (page size 16 or 32 tokens), §3.3.2 (pages are taken on demand and returned
 *     when a request ends), §3.3.3 (pages shared between requests carry reference
 *     counts), §3.3.4 (teaching allocator: a LIFO free list, out-of-memory when it
 *     is empty), §3.4 (paging leaves the attention mathematics unchanged);
 *   - "PagedAttentionMetal", sections "块表管理" (the block table maps logical to
 *     physical pages) and "注意力计算优化" (the kernel looks the physical page up,
 *     loads the K/V block into shared memory, and batches variable-length
 *     sequences without padding);
 *   - "mlx-paged-attention", feature 2 (shared prefixes with copy-on-write).
 *
 * Conventions for every call:
 *   - Device pointers are raw CUDA device addresses owned by the caller; the
 *     library allocates no device memory and keeps no pointer after returning.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Every device call only enqueues work on that stream and never
 *     synchronises; results are ready when the caller's stream work is.
 *   - Each call returns an int status: PA_OK (0) or a negative PA_ERR_*.  All
 *     argument checks happen on the host before anything is enqueued; a failing
 *     check enqueues nothing.
 *   - `device_errors` (nullable) is a caller-owned device int32 into which the
 *     kernels OR PA_DEVERR_* bits when they meet data they refuse (an
 *     out-of-range block id or slot, a length outside the table); the kernels
 *     skip that work instead of faulting.  Read it with pa_read_device_errors.
 *   - Layouts are row-major and contiguous:
 *       k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *       q, out           : [num_seqs][num_q_heads][head_dim]
 *       k, v (new tokens): [num_tokens][num_kv_heads][head_dim]
 *       block_tables     : int32 [num_seqs][max_blocks_per_seq]
 *     Element type: PA_F32 (IEEE binary32) or PA_BF16 (bfloat16); all float
 *     tensors of one call share it.  Supported: head_dim 64 or 128, block_size 16
 *     or 32, num_q_heads / num_kv_heads in {1, 2, 4, 8}.  Device buffers must be
 *     16-byte aligned.
 */
#ifndef PAGEDATTN_PA_H
#define PAGEDATTN_PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_dtype { PA_F32 = 0, PA_BF16 = 1 } pa_dtype;

/* Status codes. */
#define PA_OK 0
#define PA_ERR_INVALID_ARG (-1)   /* null pointer, bad size, misaligned buffer   */
#define PA_ERR_UNSUPPORTED (-2)   /* dtype / head_dim / block_size / group size  */
#define PA_ERR_OUT_OF_BLOCKS (-3) /* block manager: the free list is empty       */
#define PA_ERR_CUDA (-4)          /* a CUDA runtime call or launch failed        */
#define PA_ERR_NOT_FOUND (-5)     /* block manager: unknown sequence id          */
#define PA_ERR_EXISTS (-6)        /* block manager: sequence id already in use   */
#define PA_ERR_WORKSPACE (-7)     /* decode workspace missing or too small       */
#define PA_ERR_SWAPPED (-8)       /* block manager: the sequence is swapped out   */

/* Bits the kernels OR into *device_errors. */
#define PA_DEVERR_BAD_BLOCK 1     /* block id outside [0, num_blocks)            */
#define PA_DEVERR_BAD_LENGTH 2    /* context length < 0 or beyond its table      */
#define PA_DEVERR_BAD_SLOT 4      /* slot outside the pool                       */
#define PA_DEVERR_TIMEOUT 8       /* a bounded pipeline wait expired             */

/* Human-readable text of a status code (static storage, never NULL). */
const char* pa_get_error_string(int status);

/*
 * Cache write ("PagedAttention原理" §3.3.4, append_token: a new token's K/V goes
 * into the next position of its sequence's last page).  For every token t with
 * slot = slot_mapping[t] >= 0:
 *     k_cache[slot / block_size][h][slot % block_size][:] = k[t][h][:]   (all h)
 * and the same for v.  Negative slots are padding and write nothing; a slot at
 * or beyond num_blocks * block_size sets PA_DEVERR_BAD_SLOT and writes nothing.
 * slot_mapping is a device int64 array of num_tokens entries.  Bytes are copied
 * exactly.  Slots must be distinct (two tokens to one slot race).
 */
int pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                         int32_t* device_errors, void* stream);

/*
 * Copy-on-write page copy ("mlx-paged-attention", feature 2).  For each pair
 * (src, dst) in src_dst_pairs (device int64 [num_pairs][2]):
 *     k_cache[dst] = k_cache[src]; v_cache[dst] = v_cache[src]
 * where one "block" is block_bytes bytes (num_kv_heads * block_size * head_dim *
 * element size, a multiple of 16).  Destinations must be distinct and must not
 * also be sources.  Ids outside [0, num_blocks) set PA_DEVERR_BAD_BLOCK and that
 * pair is skipped.
 */
int pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst_pairs, int num_pairs,
                   size_t block_bytes, int num_blocks, int32_t* device_errors, void* stream);

/*
 * Page copy between two pools, for swapping pages to host memory and back
 * ("PagedAttention MLX：为Apple Silicon打造的高吞吐量LLM推理引擎": dynamic
 * scheduling swaps the caches of inactive requests out to CPU memory; the
 * physical KV pool supports swapping out).  For each pair (src, dst) in
 * src_dst_pairs (device int64 [num_pairs][2]):
 *     dst_k[dst] = src_k[src]; dst_v[dst] = src_v[src]
 * where one block is block_bytes bytes (a multiple of 16).  Either pool may be
 * device memory or pinned host memory the GPU can address (cudaHostAlloc /
 * cudaHostRegister, or a pinned torch tensor), e.g. device -> host with the
 * pairs of pa_bm_swap_out and host -> device with those of pa_bm_swap_in.  The
 * copy runs as one kernel (all pages at once over the host link).  Ids outside
 * [0, num_src_blocks) or [0, num_dst_blocks) set PA_DEVERR_BAD_BLOCK and that
 * pair is skipped.  Destinations must be distinct; the two pools must not
 * overlap.
 */
int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                   const int64_t* src_dst_pairs, int num_pairs, size_t block_bytes,
                   int num_src_blocks, int num_dst_blocks, int32_t* device_errors, void* stream);

/*
 * Split size (in tokens) pa_decode uses when chunk_tokens == 0: the work of each
 * (sequence, kv head) is cut into chunks of this many tokens, chosen from the
 * batch, the longest context and the current device's SM count (at most 64
 * pages; pa_decode_fp8 starts from 128 pages, see there).
 */
int pa_decode_chunk_tokens(int num_seqs, int num_kv_heads, int block_size, int max_context_len);

/* Bytes of workspace pa_decode needs for these arguments on the current device. */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int max_context_len, int chunk_tokens);

/*
 * Single-token paged decode attention ("PagedAttentionMetal", "注意力计算优化";
 * "PagedAttention原理" §3.4: the mathematics is ordinary softmax attention).
 * For sequence b, query head i, kv head h = i / (num_q_heads / num_kv_heads),
 * length L = context_lens[b] (it counts the token just written), tokens
 * t = 0 .. L-1 at page block_tables[b][t / block_size], offset t % block_size:
 *     s_t = scale * <q[b][i], K_t>,  p = softmax(s),  out[b][i] = sum_t p_t V_t.
 * Rows with L == 0 are written as zeros.  Accumulation is fp32; out has the
 * input element type.  Table entries past a sequence's pages are not read.
 *
 * max_context_len must be >= every context_lens[b] and <= max_blocks_per_seq *
 * block_size (it sizes the launch and the workspace); a length outside
 * [0, max_context_len] sets PA_DEVERR_BAD_LENGTH and is clamped.
 * chunk_tokens: 0 chooses automatically (pa_decode_chunk_tokens); otherwise a
 * multiple of 16 and of block_size, at most 128 * block_size.  Contexts longer
 * than one chunk are split and merged by a second kernel (log-sum-exp).
 * workspace: caller-owned device scratch of at least pa_decode_workspace_size()
 * bytes with the same arguments, 256-byte aligned; it carries no state between
 * calls, but two calls in flight at once must not share it.
 */
int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens, float scale,
              int num_kv_heads, int num_seqs, int num_q_heads, int head_dim, int block_size,
              int num_blocks, int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
              int chunk_tokens, void* workspace, size_t workspace_bytes,
              int32_t* device_errors, void* stream);

/*
 * Allocation-free decode.  The pages this library is built from have no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory (code embedded in a runtime that owns every device allocation, a
 * process with a fixed memory pool, a decode loop that must not call cudaMalloc
 * between steps), so they cannot provide pa_decode's workspace.
 *
 * Same arguments and result as pa_decode, minus the workspace: the scratch is a
 * static device array of PA_NOALLOC_SCRATCH_BYTES (96 MiB) inside the library,
 * held until the process exits on every GPU where it has been used.  The call
 * itself allocates nothing (no cudaMalloc, no allocating library routine).
 * Problems whose workspace (pa_decode_workspace_size with the same arguments)
 * exceeds PA_NOALLOC_SCRATCH_BYTES are rejected with PA_ERR_WORKSPACE before
 * anything is enqueued.
 *
 * Set-up: the first call in a CUDA context looks the array's device address
 * up (cudaGetSymbolAddress, with the caller's device and context current) and
 * caches it under the context's unique id, so a non-primary context, or a
 * primary context created again after cudaDeviceReset, gets its own lookup.
 * Under CUDA's default lazy module loading that first lookup is also when the
 * driver loads this part of the library onto the device and reserves the
 * 96 MiB: make the first call at set-up time, before any stream capture and
 * before a fixed memory pool takes the device's free memory.  All calls share
 * the one array: calls that may overlap on the GPU (different streams, or host
 * threads enqueueing concurrently) race on it and must be serialised by the
 * caller.  Each call resets what must start at zero, so the previous call's
 * contents do no harm.
 */
#define PA_NOALLOC_SCRATCH_BYTES ((size_t)96 << 20)
int pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens, float scale,
                      int num_kv_heads, int num_seqs, int num_q_heads, int head_dim,
                      int block_size, int num_blocks, int max_blocks_per_seq,
                      int max_context_len, pa_dtype dtype, int chunk_tokens,
                      int32_t* device_errors, void* stream);

/*
 * Paged attention for q_len new tokens per sequence, causal among them -- the
 * verify step of speculative decoding ("mlx-paged-attention", future plans:
 * "speculative decoding"), or a short chunked extend.  q and out are
 * [num_seqs][q_len][num_q_heads][head_dim] (token-major), in the pool's element
 * type.  context_lens[b] counts all q_len new tokens (written beforehand with
 * pa_reshape_and_cache, q_len slots per sequence); new token j of sequence b
 * sits at position L_b - q_len + j and attends to positions 0 .. L_b - q_len + j:
 *     out[b][j][i] = softmax_t<=L_b-q_len+j (scale q[b][j][i] . K_t) V_t.
 * One pass over each (sequence, kv head)'s pages serves all q_len x group query
 * rows; q_len * (num_q_heads / num_kv_heads) must be 1, 2, 4 or 8
 * (PA_ERR_UNSUPPORTED otherwise).  A length below q_len sets
 * PA_DEVERR_BAD_LENGTH (the rows with no visible key are zero).  Workspace:
 * pa_decode_workspace_size(num_seqs, q_len * num_q_heads, ...).  Other
 * arguments and rules as pa_decode; q_len = 1 is pa_decode.
 */
int pa_decode_multi(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens, float scale,
                    int num_kv_heads, int num_seqs, int num_q_heads, int q_len, int head_dim,
                    int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len,
                    pa_dtype dtype, int chunk_tokens, void* workspace, size_t workspace_bytes,
                    int32_t* device_errors, void* stream);

/*
 * Shared-prefix ("cascade") decode.  "mlx-paged-attention" (feature 2, memory
 * sharing) and "PagedAttention原理" §3.3.3 let several sequences hold the same
 * physical pages for a common prefix; this call reads those pages once per
 * group instead of once per sequence.  The result is pa_decode's (softmax
 * attention of each sequence's q over its whole context, same tolerance).
 *
 * Groups: sequences group_start[f] .. group_start[f + 1] - 1 form group f
 * (group_start: device int32 [num_groups + 1], group_start[0] = 0, increasing,
 * group_start[num_groups] = num_seqs).  shared_lens: device int32 [num_groups],
 * the number of leading tokens every member of group f shares: a whole number
 * of pages, 0 <= shared_lens[f] < context_lens[b] for every member b (0: no
 * sharing), and every member's block table holds the group leader's
 * (group_start[f]'s) pages for them.  Device-side checks: a shared length that
 * is not a whole number of pages or not below a member's length sets
 * PA_DEVERR_BAD_LENGTH (that member, or the group, is then decoded without the
 * sharing); a member whose table differs from the leader's over the prefix sets
 * PA_DEVERR_BAD_BLOCK (its rows use the leader's pages).
 *
 * bf16 only; q_len 1; num_q_heads / num_kv_heads in {1, 2, 4, 8}; other
 * arguments as pa_decode.  Workspace: pa_decode_cascade_workspace_size (0 for
 * unsupported sizes).  Host errors: PA_ERR_INVALID_ARG when num_groups is not
 * in 1 .. num_seqs or a group array is null.
 */
int pa_decode_cascade(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens,
                      const int32_t* group_start, const int32_t* shared_lens, int num_groups,
                      float scale, int num_kv_heads, int num_seqs, int num_q_heads, int head_dim,
                      int block_size, int num_blocks, int max_blocks_per_seq,
                      int max_context_len, int chunk_tokens, void* workspace,
                      size_t workspace_bytes, int32_t* device_errors, void* stream);
size_t pa_decode_cascade_workspace_size(int num_seqs, int num_groups, int num_q_heads,
                                         int num_kv_heads, int head_dim, int block_size,
                                         int max_context_len, int chunk_tokens);

/*
 * Groups for pa_decode_cascade, from HOST copies of the block tables
 * [num_seqs][max_blocks_per_seq] and context lengths [num_seqs].  A run of
 * consecutive sequences with the same first page forms a group; its shared
 * length is the number of leading pages all members hold in common, times
 * block_size, cut to whole pages below the shortest member's length.
 * Sequences that share no page with a neighbour are gathered into groups with
 * shared length 0.  Outputs (host, caller-owned): group_start [num_seqs + 1],
 * shared_lens [num_seqs], *num_groups.  PA_ERR_INVALID_ARG on null pointers,
 * non-positive sizes or a negative length.
 */
int pa_cascade_groups(const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                      int max_blocks_per_seq, int block_size, int32_t* group_start,
                      int32_t* shared_lens, int* num_groups);

/*
 * float8 e4m3 KV pools.  "mlx-paged-attention" (future plans) names
 * quantization as the next optimisation; the pages give no format, so this is
 * the plainest one: the pools hold one-byte e4m3 codes (1 sign, 4 exponent bits
 * with bias 7, 3 fraction bits, no infinities, 0x7F/0xFF NaN) and every kv head
 * h has a fixed dequantisation scale, so the stored K element is
 * code * k_scale[h] (and V: code * v_scale[h]).  Only head_dim 128 (one
 * 128-byte row per token) is supported; q, k, v and out are bf16.
 * k_scale, v_scale: device float32 [num_kv_heads], positive and finite.
 *
 * pa_reshape_and_cache_fp8: the cache write of pa_reshape_and_cache, where each
 * element x of kv head h is stored as e4m3(x / scale[h]): IEEE float32
 * division, round to nearest (ties to the even code), magnitudes above 448
 * (and infinities) saturate to +-448, NaN stores a NaN code.
 *
 * pa_decode_fp8: pa_decode over such pools, with the same arguments and
 * workspace (pa_decode_workspace_size with the same sizes: enough, since with
 * chunk_tokens == 0 its chunks start from 128 pages rather than 64 -- a page
 * of codes is half the bytes -- and longer chunks need fewer partials).  The kernel uses
 * the codes as they are (e4m3 tensor-core products, fp32 accumulation) and
 * applies K's scale to the logits and V's to the output.  The other operand of
 * each product is carried as two e4m3 parts: q scaled per row by a power of
 * two and split into hi + lo codes, and the probabilities (times 2^8) split
 * the same way, so the result carries about the precision of bf16 operands.
 */
int pa_reshape_and_cache_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, const float* k_scale,
                             const float* v_scale, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks,
                             int32_t* device_errors, void* stream);
int pa_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, float scale,
                  const float* k_scale, const float* v_scale, int num_kv_heads, int num_seqs,
                  int num_q_heads, int head_dim, int block_size, int num_blocks,
                  int max_blocks_per_seq, int max_context_len, int chunk_tokens, void* workspace,
                  size_t workspace_bytes, int32_t* device_errors, void* stream);

/*
 * Test hook for the failure path.  Every pipeline wait of the decode kernels
 * enqueued after this call gives up after `polls` polls (0: at once) and
 * reports PA_DEVERR_TIMEOUT; the kernel then waits for its own copies in flight
 * (with the normal bound) and returns, leaving the context usable.  polls < 0
 * restores the normal bound (well over a second).  Process-wide; meant for
 * tests, not for concurrent use.
 */
int pa_debug_set_wait_limit(int polls);

/* Synchronise `stream`, copy *device_errors to *host_flags, and zero it on the
 * device when `clear` is non-zero.  This is the one call that waits. */
int pa_read_device_errors(int32_t* device_errors, int32_t* host_flags, int clear, void* stream);

/* ---------------------------------------------------------------------------
 * Host block manager ("PagedAttention原理" §3.3.2-§3.3.4, "mlx-paged-attention"
 * feature 2).  Host memory only, no CUDA.  Not thread-safe: one owner at a time.
 *   - The free list starts as initial_free_order (or 0..num_blocks-1 when NULL);
 *     pages are taken from its END and returned to its end (LIFO), in page-table
 *     order when a sequence is freed.
 *   - add_seq gives a new sequence its first page at once (length 0).
 *   - append_slot reserves the slot of the sequence's next token: a new page when
 *     the last one is full; a copy when the target page is shared (refcount > 1):
 *     a fresh page replaces it in this sequence's table, the old page loses one
 *     reference, and (*cow_src, *cow_dst) name the copy the caller must run with
 *     pa_copy_blocks before writing the token.  Otherwise *cow_src = *cow_dst = -1.
 *     slot = physical_page * block_size + offset.
 *   - fork gives `child` the parent's table and length, one more reference each.
 *   - free drops one reference per page; pages at zero return to the free list.
 *   - PA_ERR_OUT_OF_BLOCKS leaves every piece of state unchanged.
 *   - Swapping (after pa_bm_enable_swap): pa_bm_swap_out moves a whole sequence
 *     to host blocks -- each of its pages in table order takes a host block
 *     from the end of the host free list, pairs[i] = (device page, host block);
 *     then each page drops one reference (pages at zero return to the device
 *     free list in table order).  pa_bm_swap_in takes a device page for each
 *     host block in table order, pairs[i] = (host block, device page), and
 *     returns the host blocks in table order.  The caller runs pa_swap_blocks
 *     with the pairs before anything else writes the freed pages.  A swapped
 *     sequence keeps its length; append_slot, fork and block_table refuse it
 *     with PA_ERR_SWAPPED; free returns its host blocks.  A page still shared
 *     with a resident sequence stays with that holder; the swapped copy is
 *     private from then on.  cap < the sequence's pages is PA_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------- */
typedef struct pa_bm pa_bm;

int pa_bm_create(int num_blocks, int block_size, const int32_t* initial_free_order, pa_bm** out);
void pa_bm_destroy(pa_bm* bm);
int pa_bm_add_seq(pa_bm* bm, int64_t seq_id);
int pa_bm_append_slot(pa_bm* bm, int64_t seq_id, int64_t* slot, int64_t* cow_src, int64_t* cow_dst);
int pa_bm_fork(pa_bm* bm, int64_t parent, int64_t child);
int pa_bm_free(pa_bm* bm, int64_t seq_id);
/* Copy up to `cap` page ids of seq_id's table to out; *num_pages and *length
 * receive its page count and token count. */
int pa_bm_block_table(const pa_bm* bm, int64_t seq_id, int32_t* out, int cap, int* num_pages,
                      int* length);
/* Reference count of a page (>= 0), or PA_ERR_INVALID_ARG. */
int pa_bm_refcount(const pa_bm* bm, int32_t block);
int pa_bm_num_free(const pa_bm* bm);
/* Copy the free list, bottom to top (the next page taken is the last), up to cap. */
int pa_bm_free_list(const pa_bm* bm, int32_t* out, int cap);
/* out4 = {pages in use, free pages, pages shared (refcount > 1),
 *         unused token slots summed over each sequence's pages}. */
int pa_bm_stats(const pa_bm* bm, int64_t* out4);
/* One decode step for n sequences, in the given order: append_slot for each,
 * slots[j] its slot, and each copy needed appended to cow_pairs ([n][2] capacity)
 * with *num_cow their count.  On PA_ERR_OUT_OF_BLOCKS, *num_done sequences were
 * served (their effects stay) and the rest untouched. */
int pa_bm_append_slots(pa_bm* bm, const int64_t* seq_ids, int n, int64_t* slots,
                       int64_t* cow_pairs, int* num_cow, int* num_done);
/* Fill tables [n][max_blocks] (padded with -1) and context_lens [n] for seq_ids. */
int pa_bm_build_block_tables(const pa_bm* bm, const int64_t* seq_ids, int n, int32_t* tables,
                             int max_blocks, int32_t* context_lens);
/* Give the manager a host pool of num_host_blocks blocks (free list as for the
 * device pool: initial_host_order or 0..num_host_blocks-1).  Once per manager. */
int pa_bm_enable_swap(pa_bm* bm, int num_host_blocks, const int32_t* initial_host_order);
/* Swap a resident sequence out / a swapped one in; pairs [cap][2] as above,
 * *num_pairs = the sequence's page count. */
int pa_bm_swap_out(pa_bm* bm, int64_t seq_id, int64_t* pairs, int cap, int* num_pairs);
int pa_bm_swap_in(pa_bm* bm, int64_t seq_id, int64_t* pairs, int cap, int* num_pairs);
int pa_bm_num_free_host(const pa_bm* bm);
/* Copy the host free list, bottom to top, up to cap; returns its length. */
int pa_bm_host_free_list(const pa_bm* bm, int32_t* out, int cap);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDATTN_PA_H */
