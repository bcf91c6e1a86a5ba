// Shared-prefix ("cascade") decode: the sequences of a group share their first
// pages (a common prompt, forked children, beams), so the attention over those
// pages is computed once for all of the group's query rows, and each sequence
// only walks its own pages afterwards.
//
// "mlx-paged-attention", feature 2 (memory sharing: sequences with a common
// prefix share its pages) and "PagedAttention原理" §3.3.3 (pages shared by
// several requests) -- the pages say the memory is shared; reading it once is
// this library's use of that.  The result is exactly pa_decode's (softmax
// attention over each sequence's whole context); only the work is split:
//   * plan: per group, the prefix items (row set x piece of the shared tokens);
//     per sequence, its prefix partials, then its own ("suffix") tokens: a short
//     suffix is left to the merge, a long one becomes decode-kernel chunks;
//   * the decode kernel over the long suffixes (chunks, as pa_decode);
//   * prefix kernel: per (item, kv head) the shared K/V pages stream through
//     shared memory once (TMA, a 3-stage pipeline) while every row of the group
//     (members x query heads of the kv head) attends to them on the tensor
//     cores; one partial per row and piece;
//   * merge: per row, the partials (log-sum-exp) and, for a short suffix, the
//     attention over its few tokens, computed in the same pass.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "decode_instances.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kCascadePlanThreads = 1024;               // the plan's largest block
constexpr int kPlanGroupCache = 2048;                   // groups the plan keeps in shared memory
constexpr int kPrefixSoftmaxWarps = 4;                  // one TMEM lane quadrant each
// softmax warps, as many epilogue warps, two producer warps (K, V) and two MMA
// warps (one issues the scores, one the value products)
constexpr int kPrefixThreads = (2 * kPrefixSoftmaxWarps + 4) * 32;
constexpr int kPrefixRows = 64;                         // query rows of one item (a row set)
constexpr int kMmaRows = 128;                           // the MMA's M: every row twice
constexpr int kPrefixKStages = 3;                       // K ring of the prefix kernel
constexpr int kPrefixVStages = 4;                       // V ring
constexpr int kPrefixMetaSlots = 4;                     // item descriptions in flight
constexpr int kPrefixCtasPerSm = 1;
// Longest piece (in stages) the plan considers, and the fixed cost of an item
// of the prefix kernel (q rows, first scores, last products, hand-over) in
// stage times, as measured on the kernel's timeline.
constexpr int kMaxPieceSpan = 32;
constexpr int kPieceOverheadStages = 3;
static_assert(kMaxPieceSpan == 32, "the plan scores one candidate span per lane of a warp");

// Tensor maps of the prefix kernel: the K and V pools as 2-D {head_dim, rows}
// with 16-row x 128-byte boxes, and q as 4-D {head_dim, group, kv heads,
// sequences} with boxes of one kv head's 128 / group members.
struct PrefixMaps {
  CUtensorMap k, v, q;
};
static_assert(kInlineSuffixTokens <= 32, "the merge attends to a short suffix one token per lane");

// Group of sequence b: the last f with group_start[f] <= b.
__device__ __forceinline__ int group_of(const int32_t* group_start, int num_groups, int b) {
  int lo = 0, hi = num_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (group_start[mid] <= b) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Block-wide exclusive scan of one value per thread (THREADS of them); the
// total lands in *total.
template <int THREADS>
__device__ __forceinline__ int block_scan(int x, int* warp_sums, int* total) {
  constexpr int NW = THREADS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NW ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NW) warp_sums[lane] = w;
  }
  __syncthreads();
  const int excl = incl - x + (warp > 0 ? warp_sums[warp - 1] : 0);
  if (threadIdx.x == THREADS - 1) *total = excl + x;
  __syncthreads();
  return excl;
}

// A group's shared length when it is usable (whole pages inside the tables and
// the longest context), else 0.
__device__ __forceinline__ int usable_shared(const int32_t* shared_lens, int f, int block_size,
                                             int max_blocks_per_seq, int max_len) {
  const int sl = shared_lens[f];
  return (sl > 0 && sl % block_size == 0 && sl <= max_blocks_per_seq * block_size &&
          sl <= max_len)
             ? sl
             : 0;
}

// Members of group f, clamped to the batch.
__device__ __forceinline__ int2 members_of(const int32_t* group_start, int f, int num_seqs) {
  const int gs = min(max(group_start[f], 0), num_seqs);
  const int ge = min(max(group_start[f + 1], gs), num_seqs);
  return make_int2(gs, ge);
}

struct PrefixShape {
  int stages, rowsets, span, pieces;
};

// Stages (kPrefixStageTokens each), row sets and pieces of group f; `span` is
// the stages of one piece: the plan-wide choice, raised so that no group has
// more than kMaxPrefixPieces pieces.
__device__ __forceinline__ PrefixShape prefix_shape(int sl, int members, int group, int span) {
  PrefixShape s;
  s.stages = (sl + kPrefixStageTokens - 1) / kPrefixStageTokens;
  s.rowsets = (members * group + kPrefixRows - 1) / kPrefixRows;
  s.span = max(span, (s.stages + kMaxPrefixPieces - 1) / kMaxPrefixPieces);
  s.pieces = s.stages > 0 ? (s.stages + s.span - 1) / s.span : 0;
  return s;
}

// One block.
//  1. Groups: the prefix work (stages x row sets x kv heads) is cut into pieces
//     of `span` stages, span chosen so that the busiest prefix CTA's stages
//     (with a per-item overhead) are fewest; an item holds the group's shared
//     length, leader and member count, and its piece, row set and span.
//  2. Sequences: b has p_b prefix partials (its group's pieces when its shared
//     length is valid for it, else 0) and then its own tokens [start_b, L_b):
//     up to kInlineSuffixTokens of them are left to the merge (inline_start[b]
//     = start_b), more become decode work entries of chunk_tokens each, never
//     single-chunk (every row goes through the merge).  chunk_base[b] = first
//     partial of b.  Checks: a shared length that is not whole pages or not
//     below a member's length sets PA_DEVERR_BAD_LENGTH, and that member is
//     decoded without the sharing.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) cascade_plan_kernel(
    const int32_t* __restrict__ context_lens, const int32_t* group_start,
    const int32_t* shared_lens, int num_groups, int num_seqs, int chunk_tokens,
    int max_len, int block_size, int max_blocks_per_seq, int group, int num_kv_heads,
    int prefix_ctas, int32_t* __restrict__ header, int32_t* __restrict__ chunk_base,
    int32_t* __restrict__ prefix_parts, int32_t* __restrict__ inline_start,
    int4* __restrict__ work, int4* __restrict__ prefix_items, uint4* __restrict__ out,
    int64_t row_chunks, int32_t* device_errors) {
  __shared__ int warp_sums[THREADS / 32];
  __shared__ int total_s;
  __shared__ int carry_parts, carry_work, carry_items, units_s;
  __shared__ unsigned span_items[kMaxPieceSpan + 1];
  __shared__ int32_t gs_cache[kPlanGroupCache + 1], sl_cache[kPlanGroupCache];
  allow_next_grid();                      // the next kernel may start its prologue
  // the first sequences' lengths, loaded now: they are needed last
  const int len_first = threadIdx.x < num_seqs ? context_lens[threadIdx.x] : 0;
  if (threadIdx.x == 0) carry_parts = carry_work = carry_items = units_s = 0;
  // the group arrays are read many times (a binary search per sequence): keep
  // them in shared memory when they fit
  const bool cached = num_groups <= kPlanGroupCache;
  if (cached) {
    for (int i = threadIdx.x; i <= num_groups; i += THREADS) gs_cache[i] = group_start[i];
    for (int i = threadIdx.x; i < num_groups; i += THREADS) sl_cache[i] = shared_lens[i];
    group_start = gs_cache;
    shared_lens = sl_cache;
  }
  __syncthreads();
  // ---- 1a. the piece length: for every candidate span (stages per piece) the
  // items it makes, then the span whose busiest CTA (items per CTA x (span +
  // the per-item overhead, in stages)) finishes first
  for (int i = threadIdx.x; i <= kMaxPieceSpan; i += THREADS) span_items[i] = 0;
  __syncthreads();
  {
    // warp w takes groups w, w + (warps), ...; lane c - 1 counts candidate c's items
    const int c = (threadIdx.x & 31) + 1;
    unsigned acc = 0;
    for (int f = threadIdx.x >> 5; f < num_groups; f += THREADS / 32) {
      const int sl = usable_shared(shared_lens, f, block_size, max_blocks_per_seq, max_len);
      const int2 m = members_of(group_start, f, num_seqs);
      const PrefixShape s1 = prefix_shape(sl, m.y - m.x, group, 1);
      if (s1.stages > 0) {
        // the pieces prefix_shape makes with span c (raised so that a group
        // has at most kMaxPrefixPieces pieces)
        const int span_c = max(c, (s1.stages + kMaxPrefixPieces - 1) / kMaxPrefixPieces);
        acc += static_cast<unsigned>(s1.rowsets * ((s1.stages + span_c - 1) / span_c));
      }
    }
    if (acc) atomicAdd(&span_items[c], acc);
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    // lane c - 1 scores candidate c; the warp keeps the cheapest (shortest on ties)
    const int c = threadIdx.x + 1;
    const int64_t ctas = prefix_ctas > 0 ? prefix_ctas : 1;
    const int64_t items_c = static_cast<int64_t>(span_items[c]) * num_kv_heads;
    int64_t cost = (items_c + ctas - 1) / ctas * (c + kPieceOverheadStages);
    int best = c;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const int64_t oc = __shfl_xor_sync(0xffffffffu, cost, o);
      const int ob = __shfl_xor_sync(0xffffffffu, best, o);
      if (oc < cost || (oc == cost && ob < best)) {
        cost = oc;
        best = ob;
      }
    }
    if (threadIdx.x == 0) units_s = best;
  }
  __syncthreads();
  const int span = units_s;
  // ---- 1b. the item list
  for (int base = 0; base < num_groups; base += THREADS) {
    const int f = base + threadIdx.x;
    PrefixShape s{0, 0, 1, 0};
    int sl = 0;
    int2 m = make_int2(0, 0);
    if (f < num_groups) {
      sl = usable_shared(shared_lens, f, block_size, max_blocks_per_seq, max_len);
      m = members_of(group_start, f, num_seqs);
      s = prefix_shape(sl, m.y - m.x, group, span);
    }
    const int n = s.rowsets * s.pieces;
    const int first = block_scan<THREADS>(n, warp_sums, &total_s);
    const int tot = total_s;
    // an item carries what its producer needs, so that it starts with one load:
    // {shared length, leader, members | piece << 24, row set | span << 16}
    for (int i = 0; i < n; ++i)
      prefix_items[carry_items + first + i] =
          make_int4(sl, m.x, (m.y - m.x) | ((i % s.pieces) << 24), (i / s.pieces) | (s.span << 16));
    __syncthreads();
    if (threadIdx.x == 0) carry_items += tot;
    __syncthreads();
  }
  // ---- 2. sequences
  for (int base = 0; base < num_seqs; base += THREADS) {
    const int b = base + threadIdx.x;
    int L = 0, start = 0, pb = 0, nb = 0;
    bool inl = false;
    if (b < num_seqs) {
      L = base == 0 ? len_first : context_lens[b];
      if (L < 0 || L > max_len) {
        report(device_errors, PA_DEVERR_BAD_LENGTH);
        L = L < 0 ? 0 : max_len;
      }
      const int f = group_of(group_start, num_groups, b);
      const int raw = shared_lens[f];
      const int sl = usable_shared(shared_lens, f, block_size, max_blocks_per_seq, max_len);
      start = sl;
      if (raw != sl || (sl > 0 && sl >= L)) {
        report(device_errors, PA_DEVERR_BAD_LENGTH);
        start = 0;                                   // the prefix kernel writes nothing for b
      }
      if (group_start[f] < 0 || group_start[f] > b) {   // sorted, from 0
        report(device_errors, PA_DEVERR_BAD_LENGTH);
        start = 0;
      }
      if (start > 0) {
        const int2 m = members_of(group_start, f, num_seqs);
        pb = prefix_shape(sl, m.y - m.x, group, span).pieces;
      }
      if (L > 0) {
        inl = L - start <= kInlineSuffixTokens;
        nb = inl ? 0 : (L - start + chunk_tokens - 1) / chunk_tokens;
      }
    }
    const int parts = block_scan<THREADS>(pb + nb, warp_sums, &total_s);
    const int tparts = total_s;
    const int wk = block_scan<THREADS>(nb, warp_sums, &total_s);
    const int twork = total_s;
    if (b < num_seqs) {
      const int first = carry_parts + parts;
      chunk_base[b] = first;
      prefix_parts[b] = pb;                          // the prefix kernel writes only these
      inline_start[b] = inl ? start : -1;
      for (int k = 0; k < nb; ++k)
        work[carry_work + wk + k] = make_int4(b, start + k * chunk_tokens, L, first + pb + k);
      if (L == 0)
        for (int64_t k = 0; k < row_chunks; ++k) out[b * row_chunks + k] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      carry_parts += tparts;
      carry_work += twork;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    chunk_base[num_seqs] = carry_parts;
    header[0] = 0;
    header[1] = carry_work;
    header[2] = carry_items;
  }
}

// ------------------------------------------------------------ prefix kernel
// Item = (group f, row set rs, piece) x kv head h: the piece's stages of the
// group's shared tokens (kPrefixStageTokens = 64 each, read through the group
// leader's block table) for the row set's kPrefixRows = 64 query rows
// rr = (member, query head of h), member = rr / group.  The products run on the
// fifth-generation tensor cores (tcgen05.mma, M = 128): every row is in the
// MMA twice, rows 32 quadrant + i and 32 quadrant + 16 + i for rr = 16 quadrant
// + i, so that the four TMEM lane quadrants (one per softmax warp) hold 16 rows
// each and a row's 64 scores of a stage split over two threads.  Warp roles:
//   * items producer: per item, its description into a shared ring and the
//     row set's q rows into one of two Q buffers (tensor-map boxes of 16 rows x
//     128 bytes, straight from q viewed as [member][kv head][group][head_dim]);
//     per stage, the K pages into a ring (one 16-row box per page and 128-byte
//     column slab: a tile is [slab][64 tokens][128 bytes], 128-byte swizzle);
//   * V producer: the V pages the same way into a ring of their own;
//   * scores (one thread): per stage, S = Q K^T with one tcgen05.mma per 16
//     columns of head_dim (N = the stage's tokens, bf16 operands in shared
//     memory, fp32 accumulator in tensor memory, two S buffers); a K slot is
//     released as soon as its product completes (tcgen05.commit on mbarriers);
//   * values (one thread): once a stage's probabilities are in shared memory,
//     O += P V with one product per 16 tokens (N = head_dim, V read in its
//     stored layout as an MN-major operand), into one of two O buffers;
//   * softmax (four warps): read the row's scores, keep its reference maximum
//     (moved only when a score passes it by more than 8 in base 2; then the
//     thread rescales the copy of the row's O in its own TMEM lane) and sum,
//     write the probabilities as bf16 into both copies of the row in P; at the
//     item's end hand (max, sum) over;
//   * epilogue (four warps): read the item's O rows from tensor memory (a
//     lane: one copy of a row, half of head_dim) and write each row's partial
//     (output divided by its sum, base-2 log-sum-exp) at chunk_base[member] +
//     piece, when the plan gave the member that many prefix partials; items of
//     kv head 0 also check that the members hold the leader's pages
//     (PA_DEVERR_BAD_BLOCK).
// S, P, Q and O are double-buffered, so the next stage's scores, and the next
// item's first stages, run while a stage is in softmax and an item in its
// epilogue.
template <int D>
struct PrefixLayout {
  static constexpr int SLABS = D / 64;                       // 128-byte column slabs of a row
  static constexpr int SLAB_TILE = kPrefixStageTokens * 128; // one slab of a stage's tile
  static constexpr int TILE_BYTES = SLABS * SLAB_TILE;       // K (or V) of one stage
  static constexpr int OFF_V = kPrefixKStages * TILE_BYTES;
  static constexpr int Q_SLAB = kMmaRows * 128;              // Q: [slab][128 rows][128 B]
  static constexpr int Q_BYTES = SLABS * Q_SLAB;
  static constexpr int P_BYTES = kMmaRows * 128;             // P: [128 rows][64 tokens bf16]
  static constexpr int OFF_Q = OFF_V + kPrefixVStages * TILE_BYTES;
  static constexpr int OFF_P = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_ML = OFF_P + 2 * P_BYTES;         // (max, sum) of every row, 2 items
  static constexpr int OFF_META = OFF_ML + 2 * kPrefixRows * 8;
  static constexpr int OFF_BARS = OFF_META + kPrefixMetaSlots * 32;
  // k_full/k_empty[NK], v_full/v_empty[NV], s_full/s_free/p_full/p_free[2],
  // q_full/q_empty/o_full/o_free/ml_full[2], meta_full/meta_empty[slots], mma_done
  static constexpr int NUM_BARS =
      2 * (kPrefixKStages + kPrefixVStages) + 18 + 2 * kPrefixMetaSlots + 1;
  static constexpr int SMEM = OFF_BARS + NUM_BARS * 8 + 16 + 1024;   // + room to align to 1 KiB
  static constexpr int KS = D / 16;                          // k-steps of S
  static_assert(kPrefixStageTokens == 64, "a P row is one 128-byte swizzle row of 64 tokens");
  static_assert(SMEM <= 227 * 1024, "shared memory over budget");
};

// Tensor memory: O of two items in columns [0, 128) and [128, 256), the two S
// buffers of 64 columns at 256 and 320; 512 columns are allocated.
constexpr uint32_t kPrefixTmemCols = 512;
constexpr uint32_t kPrefixTmemO = 128;       // column stride of the O buffers
constexpr uint32_t kPrefixTmemS = 256;

// Shared-memory matrix descriptor of a tcgen05 operand in the 128-byte swizzled
// layout: start address, leading-dimension byte offset (between 128-byte column
// slabs, for an MN-major operand wider than one slab), stride byte offset (between
// groups of 8 rows), descriptor version 1, swizzle mode 2 (128 bytes).
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of a kind::f16 tcgen05.mma: fp32 accumulator, bf16 A
// and B, A K-major, B K-major or MN-major, N and M.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
      : "memory");
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-wide swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + (((c ^ r) & 7) << 4));
}

// Tokens (multiple of 16) of stage st of a shared prefix of sl tokens.
__device__ __forceinline__ int stage_tokens(int st, int sl) {
  return min(kPrefixStageTokens, sl - st * kPrefixStageTokens);
}

// One item as the producer hands it to the other roles.
struct PrefixMeta {
  int sl;         // the group's shared tokens
  int st01;       // first stage | (stages after the last) << 16
  int rows;       // rows of this row set (<= kPrefixRows)
  int base;       // first row of the set within the group | kv head << 24
  int leader;     // the group's first sequence (its table holds the shared pages)
  int members;    // one past the group's last sequence
  int piece;
  int pad;
};

template <int D>
__global__ void __launch_bounds__(kPrefixThreads, 1) prefix_attention_kernel(
    const __grid_constant__ DecodeKernelParams p, const __grid_constant__ PrefixMaps maps,
    const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ prefix_parts,
    const int4* __restrict__ items) {
  using Ly = PrefixLayout<D>;
  constexpr int NK = kPrefixKStages, NV = kPrefixVStages;
  constexpr int NM = kPrefixMetaSlots;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::OFF_BARS);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* p_free = p_full + 2;
  uint64_t* q_full = p_free + 2;
  uint64_t* q_empty = q_full + 2;
  uint64_t* o_full = q_empty + 2;
  uint64_t* o_free = o_full + 2;
  uint64_t* ml_full = o_free + 2;
  uint64_t* meta_full = ml_full + 2;
  uint64_t* meta_empty = meta_full + NM;
  uint64_t* mma_done = meta_empty + NM;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Ly::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  PrefixMeta* meta = reinterpret_cast<PrefixMeta*>(smem + Ly::OFF_META);
  float2* ml = reinterpret_cast<float2*>(smem + Ly::OFF_ML);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = p.num_kv_heads, G = p.group, bs = p.block_size;
  constexpr int kEpiWarp0 = kPrefixSoftmaxWarps;
  constexpr int kProducerWarp = 2 * kPrefixSoftmaxWarps;    // items, q rows and K
  constexpr int kMmaWarp = kProducerWarp + 1;                 // scores (and TMEM)
  constexpr int kVProducerWarp = kMmaWarp + 2;                // V (kMmaWarp + 1: values)
  if (threadIdx.x == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], kPrefixSoftmaxWarps);
      mbar_init(&p_full[i], kPrefixSoftmaxWarps);
      mbar_init(&p_free[i], 1);
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], kPrefixSoftmaxWarps);
      mbar_init(&ml_full[i], kPrefixSoftmaxWarps);
    }
    for (int i = 0; i < NM; ++i) {
      mbar_init(&meta_full[i], 1);
      // released by the two MMA threads, the softmax warps, the epilogue warps
      // and the V producer
      mbar_init(&meta_empty[i], 3 + 2 * kPrefixSoftmaxWarps);
    }
    mbar_init(mma_done, 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    // one CTA per SM (its shared memory), so the columns are always free
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kPrefixTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = *tmem_slot;
  wait_prior_grids();                     // the plan's item list and partial offsets
  allow_next_grid();                      // the merge may start its independent loads
  const int n_items = p.header[2] * Hkv;
  auto fail = [&]() {
    if (!*abort_flag) {
      report(p.device_errors, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
  };
  // the item's description from the ring slot (every role but the producer)
  auto take_meta = [&](uint32_t ic, PrefixMeta& mt) -> bool {
    if (*abort_flag || !mbar_wait(&meta_full[ic % NM], (ic / NM) & 1, p.wait_limit)) return false;
    mt = meta[ic % NM];
    return true;
  };

  // Copies of one pool's pages of a stage into ring slot `dst`: lane (page j,
  // slab) takes 16 tokens x 128 bytes, the pages of the piece's first 32
  // 16-token groups fetched once per item (`pre_page`, one per lane).
  auto stage_copies = [&](const CUtensorMap* map, unsigned char* dst, uint64_t* full, int st,
                          int st0, int sl, int h, const int32_t* table, int pre_page) {
    const int t0 = st * kPrefixStageTokens;
    const int ngrp = stage_tokens(st, sl) / 16;
    if (lane == 0) mbar_arrive_expect_tx(full, ngrp * Ly::SLABS * 16 * 128);
    const int j = lane / Ly::SLABS, sl_ = lane % Ly::SLABS;
    const int gi = (st - st0) * (kPrefixStageTokens / 16) + j;    // page within the piece
    int page = __shfl_sync(kFull, pre_page, gi < 32 ? gi : 31);
    if (j < ngrp) {
      const int t = t0 + 16 * j;
      if (gi >= 32) {                        // past the prefetched pages
        page = table[t / bs];
        if (page < 0 || page >= p.num_blocks) {
          report(p.device_errors, PA_DEVERR_BAD_BLOCK);
          page = -1;
        }
      }
      const int row = (page * Hkv + h) * bs + t % bs;
      tma_load_2d(dst + sl_ * Ly::SLAB_TILE + j * 16 * 128, map, 64 * sl_, row, full);
    }
  };
  auto prefetch_pages = [&](const int32_t* table, int st0, int st1, int sl) {
    const int ngi = (min(st1 * kPrefixStageTokens, sl) - st0 * kPrefixStageTokens) / 16;
    int pre_page = -1;
    if (lane < ngi) {
      pre_page = table[(st0 * kPrefixStageTokens + 16 * lane) / bs];
      if (pre_page < 0 || pre_page >= p.num_blocks) {
        report(p.device_errors, PA_DEVERR_BAD_BLOCK);
        pre_page = -1;                         // a row outside the pool: the box reads zeros
      }
    }
    return pre_page;
  };

  if (warp == kProducerWarp) {
    // ---------------- producer: items, q rows, K pages
    uint32_t k = 0, ic = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++ic) {
      const int4 item = items[it / Hkv];
      const int h = it % Hkv;
      const int sl = item.x;
      const int2 mem = make_int2(item.y, item.y + (item.z & 0xFFFFFF));
      const int piece = item.z >> 24, rowset = item.w & 0xFFFF, span = item.w >> 16;
      const int32_t* table = p.block_tables + static_cast<int64_t>(mem.x) * p.max_blocks_per_seq;
      const int stages = (sl + kPrefixStageTokens - 1) / kPrefixStageTokens;
      const int st0 = piece * span, st1 = min(st0 + span, stages);
      // the item's description, then its q rows
      bool waited = true;
      if (lane == 0) {
        waited = !*abort_flag && mbar_wait(&meta_empty[ic % NM], ((ic / NM) & 1) ^ 1, p.wait_limit) &&
                 mbar_wait(&q_empty[ic & 1], ((ic >> 1) & 1) ^ 1, p.wait_limit);
        if (waited) {
          PrefixMeta mt;
          mt.sl = sl;
          mt.st01 = st0 | (st1 << 16);
          mt.rows = min((mem.y - mem.x) * G - rowset * kPrefixRows, kPrefixRows);
          mt.base = rowset * kPrefixRows | (h << 24);
          mt.leader = mem.x;
          mt.members = mem.y;
          mt.piece = piece;
          mt.pad = 0;
          meta[ic % NM] = mt;
          mbar_arrive(&meta_full[ic % NM]);
          uint64_t* qb = &q_full[ic & 1];
          mbar_arrive_expect_tx(qb, Ly::Q_BYTES);
          unsigned char* qdst = smem + Ly::OFF_Q + (ic & 1) * Ly::Q_BYTES;
          const int m0 = mem.x + rowset * kPrefixRows / G;
          // row set row rr = 16 quadrant + i lands in MMA rows 32 quadrant + i
          // and 32 quadrant + 16 + i: each a box of the quadrant's 16 / group
          // members (16 rows x 128 bytes)
#pragma unroll
          for (int s = 0; s < Ly::SLABS; ++s)
#pragma unroll
            for (int qd = 0; qd < 4; ++qd)
#pragma unroll
              for (int c = 0; c < 2; ++c)
                tma_load_4d(qdst + s * Ly::Q_SLAB + (32 * qd + 16 * c) * 128, &maps.q, 64 * s, 0,
                            h, m0 + 16 * qd / G, qb);
        }
      }
      if (!__shfl_sync(kFull, waited, 0)) {
        if (lane == 0) fail();
        ok = false;
        break;
      }
      const int pre_page = prefetch_pages(table, st0, st1, sl);
      for (int st = st0; st < st1; ++st, ++k) {
        const int slot = static_cast<int>(k % NK);
        bool w = false;
        if (lane == 0 && !*abort_flag)
          w = mbar_wait(&k_empty[slot], ((k / NK) & 1) ^ 1, p.wait_limit);
        if (!__shfl_sync(kFull, w, 0)) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        stage_copies(&maps.k, smem + slot * Ly::TILE_BYTES, &k_full[slot], st, st0, sl, h, table,
                     pre_page);
      }
    }
    // the copies still in flight must land before the shared memory is released
    if (lane == 0) {
      for (uint32_t j = k > NK ? k - NK : 0; j < k; ++j) mbar_wait(&k_full[j % NK], (j / NK) & 1);
      for (uint32_t j = ic > 2 ? ic - 2 : 0; j < ic; ++j) mbar_wait(&q_full[j & 1], (j >> 1) & 1);
    }
  } else if (warp == kVProducerWarp) {
    // ---------------- producer: V pages
    uint32_t k = 0, ic = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++ic) {
      PrefixMeta mt;
      bool got = take_meta(ic, mt);
      if (!__all_sync(kFull, got)) {
        if (lane == 0) fail();
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&meta_empty[ic % NM]);
      const int st0 = mt.st01 & 0xFFFF, st1 = mt.st01 >> 16, sl = mt.sl, h = mt.base >> 24;
      const int32_t* table = p.block_tables + static_cast<int64_t>(mt.leader) * p.max_blocks_per_seq;
      const int pre_page = prefetch_pages(table, st0, st1, sl);
      for (int st = st0; st < st1; ++st, ++k) {
        const int slot = static_cast<int>(k % NV);
        bool w = false;
        if (lane == 0 && !*abort_flag)
          w = mbar_wait(&v_empty[slot], ((k / NV) & 1) ^ 1, p.wait_limit);
        if (!__shfl_sync(kFull, w, 0)) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        stage_copies(&maps.v, smem + Ly::OFF_V + slot * Ly::TILE_BYTES, &v_full[slot], st, st0, sl,
                     h, table, pre_page);
      }
    }
    if (lane == 0)
      for (uint32_t j = k > NV ? k - NV : 0; j < k; ++j) mbar_wait(&v_full[j % NV], (j / NV) & 1);
  } else if (warp == kMmaWarp) {
    // ---------------- S = Q K^T issue: one thread
    if (lane == 0) {
      const uint32_t q_base = smem_addr(smem + Ly::OFF_Q);
      const uint32_t stage_base = smem_addr(smem);
      uint32_t k = 0, ic = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++ic) {
        PrefixMeta mt;
        if (!take_meta(ic, mt)) { ok = false; break; }
        mbar_arrive(&meta_empty[ic % NM]);
        const int st0 = mt.st01 & 0xFFFF, st1 = mt.st01 >> 16, sl = mt.sl;
        if (*abort_flag || !mbar_wait(&q_full[ic & 1], (ic >> 1) & 1, p.wait_limit)) {
          ok = false;
          break;
        }
        // descriptors advance by (byte offset >> 4) in their address field
        const uint64_t qd0 = umma_desc(q_base + (ic & 1) * Ly::Q_BYTES, 16, 1024);
        for (int st = st0; st < st1 && ok; ++st, ++k) {
          const int slot = static_cast<int>(k % NK), sb = k & 1;
          if (*abort_flag || !mbar_wait(&k_full[slot], (k / NK) & 1, p.wait_limit) ||
              !mbar_wait(&s_free[sb], ((k >> 1) & 1) ^ 1, p.wait_limit)) {
            ok = false;
            break;
          }
          tmem_fence_after();
          const int tokens = stage_tokens(st, sl);
          const uint32_t id_s = umma_idesc_bf16(kMmaRows, tokens, false);
          const uint64_t kd = umma_desc(stage_base + slot * Ly::TILE_BYTES, 16, 1024);
#pragma unroll
          for (int ks = 0; ks < Ly::KS; ++ks)
            umma_bf16(tmem + kPrefixTmemS + 64 * sb,
                      qd0 + (((ks >> 2) * Ly::Q_SLAB + (ks & 3) * 32) >> 4),
                      kd + (((ks >> 2) * Ly::SLAB_TILE + (ks & 3) * 32) >> 4), id_s,
                      ks > 0 ? 1u : 0u);
          umma_commit(&s_full[sb]);
          umma_commit(&k_empty[slot]);          // the K slot may be refilled
          if (st + 1 == st1) umma_commit(&q_empty[ic & 1]);   // the item's q rows are read
        }
      }
      if (!ok) fail();
      // nothing may be in flight when the columns are released
      umma_commit(mma_done);
      mbar_wait(mma_done, 0);
    }
    __syncwarp();
  } else if (warp == kMmaWarp + 1) {
    // ---------------- O += P V issue: one thread
    if (lane == 0) {
      constexpr uint32_t kIdPV = umma_idesc_bf16(kMmaRows, D, true);
      const uint32_t p_base = smem_addr(smem + Ly::OFF_P);
      const uint32_t stage_base = smem_addr(smem);
      uint32_t k = 0, ic = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++ic) {
        PrefixMeta mt;
        if (!take_meta(ic, mt)) { ok = false; break; }
        mbar_arrive(&meta_empty[ic % NM]);
        const int st0 = mt.st01 & 0xFFFF, st1 = mt.st01 >> 16, sl = mt.sl;
        const uint32_t o_col = tmem + (ic & 1) * kPrefixTmemO;
        for (int st = st0; st < st1 && ok; ++st, ++k) {
          const int pb = k & 1, slot = static_cast<int>(k % NV);
          const bool first = st == st0;
          if (*abort_flag || !mbar_wait(&p_full[pb], (k >> 1) & 1, p.wait_limit) ||
              !mbar_wait(&v_full[slot], (k / NV) & 1, p.wait_limit) ||
              (first && !mbar_wait(&o_free[ic & 1], ((ic >> 1) & 1) ^ 1, p.wait_limit))) {
            ok = false;
            break;
          }
          tmem_fence_after();
          const int tokens = stage_tokens(st, sl);
          const uint64_t pd = umma_desc(p_base + pb * Ly::P_BYTES, 16, 1024);
          const uint64_t vd =
              umma_desc(stage_base + Ly::OFF_V + slot * Ly::TILE_BYTES, Ly::SLAB_TILE, 1024);
          for (int g = 0; g < tokens / 16; ++g)
            umma_bf16(o_col, pd + 2 * g, vd + 128 * g, kIdPV, (first && g == 0) ? 0u : 1u);
          umma_commit(&v_empty[slot]);         // the V slot may be refilled
          umma_commit(&p_free[pb]);            // the P buffer may be rewritten
        }
        if (ok) umma_commit(&o_full[ic & 1]);
      }
      if (!ok) fail();
      umma_commit(mma_done);
      mbar_wait(mma_done, 0);
    }
    __syncwarp();
  } else if (warp < kPrefixSoftmaxWarps) {
    // ---------------- softmax warps.  Thread (warp qd, lane l) holds MMA row
    // 32 qd + l, i.e. row set row rr = 16 qd + l % 16 (every row is in the MMA
    // twice, rows 32 qd + i and 32 qd + 16 + i), and half h = l / 16 of the
    // stage's 64 columns; the two halves of a row meet through one shuffle.
    // Each thread writes its half of the probabilities into both copies of the
    // row in P, so O holds every row twice as well and each thread rescales the
    // copy in its own TMEM lane.
    const int rr = 16 * warp + (lane & 15);
    const int half = lane >> 4;
    const int r0 = 32 * warp + (lane & 15);          // the row's two MMA rows: r0, r0 + 16
    const uint32_t lane_tmem = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float sc = p.scale_log2;
    unsigned char* ps = smem + Ly::OFF_P;
    uint32_t k = 0, ic = 0;
    bool live = true;
    for (int it = blockIdx.x; it < n_items && live; it += gridDim.x, ++ic) {
      PrefixMeta mt;
      bool got = take_meta(ic, mt);
      got = __all_sync(kFull, got);
      if (!got) {
        if (lane == 0) fail();
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&meta_empty[ic % NM]);
      const int st0 = mt.st01 & 0xFFFF, st1 = mt.st01 >> 16, sl = mt.sl;
      const uint32_t o_col = (ic & 1) * kPrefixTmemO;
      float m = kNoScore, l = 0.f;                   // l: this half's columns
      for (int st = st0; st < st1; ++st, ++k) {
        const int sb = k & 1;
        bool waited = !*abort_flag && mbar_wait(&s_full[sb], (k >> 1) & 1, p.wait_limit);
        waited = __all_sync(kFull, waited);
        if (!waited) {
          if (lane == 0) fail();
          live = false;
          break;
        }
        tmem_fence_after();
        const int tokens = stage_tokens(st, sl);
        // a TMEM load takes one address for the whole warp: every lane reads
        // the 64 columns of its row and keeps its half
        float s[32], t[32];
        tmem_ld16(lane_tmem + kPrefixTmemS + 64 * sb, s);
        tmem_ld16(lane_tmem + kPrefixTmemS + 64 * sb + 16, s + 16);
        tmem_ld16(lane_tmem + kPrefixTmemS + 64 * sb + 32, t);
        tmem_ld16(lane_tmem + kPrefixTmemS + 64 * sb + 48, t + 16);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) s[c] = half ? t[c] : s[c];
        tmem_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[sb]);      // the S buffer may be rewritten
        if (tokens < kPrefixStageTokens) {            // the piece's last, partial stage
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (32 * half + c >= tokens) s[c] = -INFINITY;
        }
        float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
        for (int c = 4; c < 32; ++c) mx[c & 3] = fmaxf(mx[c & 3], s[c]);
        float x = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        x = fmaxf(x, __shfl_xor_sync(kFull, x, 16)) * sc;
        // The reference maximum moves only when a score passes it by more than
        // 8 (every probability stays <= 2^8, exact in fp32 and bf16); then the
        // row's O, complete up to the previous stage, is rescaled in place.
        float alpha = 1.f;
        const bool grow = x > m + 8.f;
        if (grow) {
          alpha = fast_exp2(m - x);
          m = x;
        }
        l *= alpha;
        if (st > st0 && __any_sync(kFull, grow)) {
          const uint32_t kp = k - 1;
          bool ok = mbar_wait(&p_free[kp & 1], (kp >> 1) & 1, p.wait_limit);   // PV(kp) done
          ok = __all_sync(kFull, ok);
          if (!ok) {
            if (lane == 0) fail();
            live = false;
            break;
          }
          tmem_fence_after();
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            float o[16];
            tmem_ld16(lane_tmem + o_col + 16 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= alpha;
            tmem_st16(lane_tmem + o_col + 16 * c, o);
          }
          tmem_wait_st();
        }
        // ---- probabilities into the P buffer of this stage (this half's four
        // 16-byte chunks of both copies of the row), once the products of two
        // stages ago have read it
        bool ok = mbar_wait(&p_free[sb], ((k >> 1) & 1) ^ 1, p.wait_limit);
        ok = __all_sync(kFull, ok);
        if (!ok) {
          if (lane == 0) fail();
          live = false;
          break;
        }
        float sum[4] = {0.f, 0.f, 0.f, 0.f};
        unsigned char* prow = ps + sb * Ly::P_BYTES;
        const float nm = -m;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float e[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            e[i] = fast_exp2(fmaf(s[8 * c + i], sc, nm));
            sum[i & 3] += e[i];
          }
          uint4 w;
          w.x = pack_bf16x2(e[0], e[1]);
          w.y = pack_bf16x2(e[2], e[3]);
          w.z = pack_bf16x2(e[4], e[5]);
          w.w = pack_bf16x2(e[6], e[7]);
          *reinterpret_cast<uint4*>(prow + sw128(r0, 4 * half + c)) = w;
          *reinterpret_cast<uint4*>(prow + sw128(r0 + 16, 4 * half + c)) = w;
        }
        l += (sum[0] + sum[1]) + (sum[2] + sum[3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tmem_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
      }
      if (!live) break;
      // ---- hand the row's (max, sum) to the epilogue, once the epilogue of two
      // items ago has read this buffer
      l += __shfl_xor_sync(kFull, l, 16);
      bool freed = mbar_wait(&o_free[ic & 1], ((ic >> 1) & 1) ^ 1, p.wait_limit);
      freed = __all_sync(kFull, freed);
      if (!freed) {
        if (lane == 0) fail();
        break;
      }
      if (half == 0) ml[(ic & 1) * kPrefixRows + rr] = make_float2(m, l);
      __syncwarp();
      if (lane == 0) mbar_arrive(&ml_full[ic & 1]);
    }
  } else {
    // ---------------- epilogue warps: the lane quadrant of warp % 4
    const int qd = warp - kEpiWarp0;
    const int r = qd * 32 + lane;                    // thread index of the epilogue warps
    const uint32_t lane_tmem = tmem + (static_cast<uint32_t>(qd * 32) << 16);
    uint32_t ic = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++ic) {
      PrefixMeta mt;
      bool got = take_meta(ic, mt);
      got = __all_sync(kFull, got);
      if (!got) {
        if (lane == 0) fail();
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&meta_empty[ic % NM]);
      const int h = mt.base >> 24, rs0 = mt.base & 0xFFFFFF;
      const int2 mem = make_int2(mt.leader, mt.members);
      const int piece = mt.piece;
      if (h == 0) {
        // members of this row set that use this piece hold the leader's pages
        const int st0 = mt.st01 & 0xFFFF, st1 = mt.st01 >> 16;
        const int m_lo = mem.x + rs0 / G;
        const int m_hi = min(mem.y, mem.x + (rs0 + kPrefixRows) / G);
        const int pg0 = st0 * kPrefixStageTokens / bs;
        const int np = min(st1 * kPrefixStageTokens, mt.sl) / bs - pg0;
        const int32_t* lead = p.block_tables + static_cast<int64_t>(mem.x) * p.max_blocks_per_seq;
        for (int i = r; i < (m_hi - m_lo) * np; i += kPrefixSoftmaxWarps * 32) {
          const int m = m_lo + i / np, pg = pg0 + i % np;
          if (piece < prefix_parts[m] &&
              p.block_tables[static_cast<int64_t>(m) * p.max_blocks_per_seq + pg] != lead[pg])
            report(p.device_errors, PA_DEVERR_BAD_BLOCK);
        }
      }
      // lane l: row set row rr = 16 qd + l % 16 (its copy in TMEM lane 32 qd + l)
      // and half l / 16 of head_dim
      const int rr = 16 * qd + (lane & 15), half = lane >> 4;
      const bool active = 16 * qd < mt.rows;
      const bool has_row = rr < mt.rows;
      const int gr = rs0 + rr;                       // row within the group
      const int b = has_row ? mem.x + gr / G : mem.x;
      const bool write = has_row && piece < prefix_parts[b];
      const int qh = h * G + gr % G;
      const int64_t prow =
          write ? static_cast<int64_t>(chunk_base[b] + piece) * p.num_q_heads + qh : 0;
      bool done = !*abort_flag && mbar_wait(&o_full[ic & 1], (ic >> 1) & 1, p.wait_limit) &&
                  mbar_wait(&ml_full[ic & 1], (ic >> 1) & 1, p.wait_limit);
      done = __all_sync(kFull, done);
      if (!done) {
        if (lane == 0) fail();
        break;
      }
      tmem_fence_after();
      if (active) {
        const float2 st = ml[(ic & 1) * kPrefixRows + rr];
        const float inv = st.y > 0.f ? 1.f / st.y : 0.f;
        const uint32_t o_col = (ic & 1) * kPrefixTmemO;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          float o[16];
          tmem_ld16(lane_tmem + o_col + 16 * c, o);     // one address for the warp
          tmem_wait_ld();
          if (write && (c >= D / 32) == (half != 0)) {
            float4* dst = reinterpret_cast<float4*>(p.part_out + prow * D + 16 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                   o[4 * i + 3] * inv);
          }
        }
        if (write && half == 0) p.part_lse[prow] = st.y > 0.f ? st.x + __log2f(st.y) : -INFINITY;
      }
      tmem_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[ic & 1]);
    }
  }
  tmem_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tmem_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kPrefixTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------ merge
// One warp per (sequence b, kv head h): the G = group query rows of h, each
// lane owning CPL = head_dim / 32 columns of every row.  Every row keeps a
// running base-2 softmax state (maximum M, weight sum S, weighted sum acc) into
// which terms enter as (log-sum-exp, normalised value):
//   out = sum_c 2^(lse_c - M) o_c / sum_c 2^(lse_c - M),  M = max_c lse_c.
// Blocks are small (two warps) and registers few (at most 80 a thread up to 4
// rows, no shared memory), so that the whole grid finds room on the SMs beside
// the prefix kernel's blocks and waits there for it; everything that does not
// depend on the prefix kernel is done before that wait: the attention over a
// short own suffix [inline_start[b], L_b) (at most 32 tokens), token by token,
// each a term of its own (lse = its score, o = its V row), its score summed
// across the warp from each lane's columns.  After the wait the row's partials
// c (the prefix pieces, then any decode-kernel chunks of its own tokens) join.
// Rows with neither (L_b = 0) were zeroed by the plan.
constexpr int kCascadeMergeWarps = 2;          // warps per block
template <int CPL, int G>
__global__ void __launch_bounds__(kCascadeMergeWarps * 32, G <= 4 ? 12 : 8) cascade_merge_kernel(
    const __grid_constant__ DecodeKernelParams p, const int32_t* __restrict__ chunk_base,
    const int32_t* __restrict__ inline_start, const int32_t* __restrict__ context_lens,
    int max_len, int num_seqs) {
  using Cols = typename std::conditional<CPL == 4, uint2, uint32_t>::type;   // CPL bf16
  constexpr int D = CPL * 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int Hq = p.num_q_heads, Hkv = p.num_kv_heads;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kCascadeMergeWarps + warp;
  if (item >= static_cast<int64_t>(num_seqs) * Hkv) {
    wait_prior_grids();
    return;
  }
  const int b = static_cast<int>(item / Hkv);
  const int h = static_cast<int>(item - static_cast<int64_t>(b) * Hkv);
  const int c0 = chunk_base[b];
  const int n = chunk_base[b + 1] - c0;
  const int s0 = inline_start[b];
  if (n <= 0 && s0 < 0) {                       // uniform over the warp
    wait_prior_grids();
    return;
  }
  const int bs = p.block_size;
  const int L = s0 >= 0 ? min(max(context_lens[b], 0), max_len) : 0;
  const int nsuf = s0 >= 0 ? min(L - s0, 32) : 0;
  const int64_t row0 = static_cast<int64_t>(b) * Hq + h * G;   // first output row
  float M[G], S[G], acc[G][CPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    M[g] = kNoScore;
    S[g] = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) acc[g][k] = 0.f;
  }
  // one more term (lse, v) of row g
  auto add = [&](int g, float lse, const float* v) {
    const float Mn = fmaxf(M[g], lse);
    const float sc = fast_exp2(M[g] - Mn);
    const float w = fast_exp2(lse - Mn);
    S[g] = fmaf(S[g], sc, w);
#pragma unroll
    for (int k = 0; k < CPL; ++k) acc[g][k] = fmaf(acc[g][k], sc, w * v[k]);
    M[g] = Mn;
  };
  auto unpack = [](Cols c, float* f) {
    if constexpr (CPL == 4) {
      f[0] = bf16_lo(c.x); f[1] = bf16_hi(c.x); f[2] = bf16_lo(c.y); f[3] = bf16_hi(c.y);
    } else {
      f[0] = bf16_lo(c); f[1] = bf16_hi(c);
    }
  };
  if (nsuf > 0) {
    Cols qc[G];                                 // this lane's columns of the G q rows
#pragma unroll
    for (int g = 0; g < G; ++g)
      qc[g] = *reinterpret_cast<const Cols*>(p.q + ((row0 + g) * D + lane * CPL) * 2);
    // lane j: the pool row of suffix token j (-1: its page is unreadable)
    int64_t kv_row = -1;
    if (lane < nsuf) {
      const int t = s0 + lane;
      const int page = p.block_tables[static_cast<int64_t>(b) * p.max_blocks_per_seq + t / bs];
      if (page < 0 || page >= p.num_blocks)
        report(p.device_errors, PA_DEVERR_BAD_BLOCK);
      else
        kv_row = ((static_cast<int64_t>(page) * Hkv + h) * bs + t % bs) * D;
    }
    // token by token, the loads of two tokens issued together
    for (int t0 = 0; t0 < nsuf; t0 += 2) {
      Cols kc[2], vc[2];
      int64_t rr[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        rr[j] = __shfl_sync(kFull, kv_row, min(t0 + j, 31));
        if (t0 + j >= nsuf) rr[j] = -1;
        kc[j] = rr[j] >= 0 ? *reinterpret_cast<const Cols*>(p.k_cache + (rr[j] + lane * CPL) * 2)
                           : Cols{};
        vc[j] = rr[j] >= 0 ? *reinterpret_cast<const Cols*>(p.v_cache + (rr[j] + lane * CPL) * 2)
                           : Cols{};
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (rr[j] < 0) continue;                // uniform over the warp
        float kf[CPL], vf[CPL], d[G];
        unpack(kc[j], kf);
        unpack(vc[j], vf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float qf[CPL];
          unpack(qc[g], qf);
          d[g] = 0.f;
#pragma unroll
          for (int k = 0; k < CPL; ++k) d[g] = fmaf(qf[k], kf[k], d[g]);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) d[g] += __shfl_xor_sync(kFull, d[g], o2);
#pragma unroll
        for (int g = 0; g < G; ++g) add(g, d[g] * p.scale_log2, vf);
      }
    }
  }
  wait_prior_grids();                           // every partial is written
  // ---- the partials, each (lse, normalised rows) a term of its row
#pragma unroll 2
  for (int cc = 0; cc < n; ++cc) {
    const int64_t prow = (static_cast<int64_t>(c0) + cc) * Hq + h * G;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float* src = p.part_out + (prow + g) * D + lane * CPL;
      float v[CPL];
      if constexpr (CPL == 4) {
        const float4 t4 = *reinterpret_cast<const float4*>(src);
        v[0] = t4.x; v[1] = t4.y; v[2] = t4.z; v[3] = t4.w;
      } else {
        const float2 t2 = *reinterpret_cast<const float2*>(src);
        v[0] = t2.x; v[1] = t2.y;
      }
      add(g, p.part_lse[prow + g], v);          // -inf (an empty partial): weight 0
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float inv = S[g] > 0.f ? 1.f / S[g] : 0.f;   // 0: the row saw no token
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + (row0 + g) * D + lane * CPL;
#pragma unroll
    for (int k = 0; k < CPL; k += 2)
      *reinterpret_cast<uint32_t*>(dst + k) =
          f32_to_bf16_bits(acc[g][k] * inv) | (f32_to_bf16_bits(acc[g][k + 1] * inv) << 16);
  }
}

// Launch as a programmatic dependent of the kernel before it on the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned blocks, unsigned threads, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int D>
cudaError_t run_prefix(const DecodeArgs& a, const DecodeKernelParams& kp, int device,
                       cudaStream_t stream) {
  using Ly = PrefixLayout<D>;
  static std::atomic<uint64_t> configured{0};
  const uint64_t bit = 1ull << (device & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    const cudaError_t e = cudaFuncSetAttribute(
        prefix_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const int group = a.num_q_heads / a.num_kv_heads;
  PrefixMaps maps;
  const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * a.num_kv_heads * a.block_size;
  const uint64_t pool_dims[2] = {static_cast<uint64_t>(D), rows};
  const uint64_t pool_strides[1] = {static_cast<uint64_t>(D) * 2};
  const uint32_t pool_box[2] = {64, 16};
  cudaError_t e = make_bf16_map(&maps.k, a.k_cache, 2, pool_dims, pool_strides, pool_box);
  if (e == cudaSuccess) e = make_bf16_map(&maps.v, a.v_cache, 2, pool_dims, pool_strides, pool_box);
  const uint64_t q_dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(group),
                              static_cast<uint64_t>(a.num_kv_heads),
                              static_cast<uint64_t>(a.num_seqs)};
  const uint64_t q_strides[3] = {static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(group) * D * 2,
                                 static_cast<uint64_t>(a.num_q_heads) * D * 2};
  const uint32_t q_box[4] = {64, static_cast<uint32_t>(group), 1,
                             static_cast<uint32_t>(16 / group)};
  if (e == cudaSuccess) e = make_bf16_map(&maps.q, a.q, 4, q_dims, q_strides, q_box);
  if (e != cudaSuccess) return e;
  // a dependent of the decode kernel (itself one of the plan kernel): its
  // blocks wait on the device for both, i.e. for the item list
  return launch_pdl(prefix_attention_kernel<D>, static_cast<unsigned>(prefix_grid(a.num_sms)),
                    kPrefixThreads, Ly::SMEM, stream, kp, maps,
                    static_cast<const int32_t*>(a.ws.chunk_base),
                    static_cast<const int32_t*>(a.ws.prefix_parts),
                    static_cast<const int4*>(a.ws.prefix_items));
}

}  // namespace

int prefix_grid(int num_sms) { return (num_sms > 0 ? num_sms : 1) * kPrefixCtasPerSm; }

cudaError_t launch_cascade_plan(const DecodeArgs& a, cudaStream_t stream) {
  // the item fields are packed: a group's members < 2^24 and row sets < 2^16,
  // a piece's stages < 2^16
  if (a.num_seqs >= (1 << 19) || a.max_context_len >= (1 << 27)) return cudaErrorInvalidValue;
  const int64_t row_chunks = static_cast<int64_t>(a.num_q_heads) * a.head_dim * 2 / 16;
  // the smallest block that takes every sequence and group in one pass (its
  // block-wide scans and barriers cost less with fewer warps)
  const int n = a.num_seqs > a.num_groups ? a.num_seqs : a.num_groups;
  auto run = [&](auto kernel, int threads) {
    kernel<<<1, threads, 0, stream>>>(
        a.context_lens, a.group_start, a.shared_lens, a.num_groups, a.num_seqs, a.chunk_tokens,
        a.max_context_len, a.block_size, a.max_blocks_per_seq, a.num_q_heads / a.num_kv_heads,
        a.num_kv_heads, prefix_grid(a.num_sms), a.ws.header, a.ws.chunk_base, a.ws.prefix_parts,
        a.ws.inline_start, a.ws.work, a.ws.prefix_items, static_cast<uint4*>(a.out), row_chunks,
        a.device_errors);
  };
  if (n <= 128) run(cascade_plan_kernel<128>, 128);
  else if (n <= 256) run(cascade_plan_kernel<256>, 256);
  else if (n <= 512) run(cascade_plan_kernel<512>, 512);
  else run(cascade_plan_kernel<kCascadePlanThreads>, kCascadePlanThreads);
  return cudaGetLastError();
}

cudaError_t launch_cascade_prefix(const DecodeArgs& a, const DecodeKernelParams& kp, int device,
                                  cudaStream_t stream) {
  if (a.head_dim == 128) return run_prefix<128>(a, kp, device, stream);
  if (a.head_dim == 64) return run_prefix<64>(a, kp, device, stream);
  return cudaErrorInvalidValue;
}

template <int CPL, int G>
cudaError_t launch_merge_instance(const DecodeArgs& a, const DecodeKernelParams& kp,
                                  unsigned blocks, cudaStream_t stream) {
  return launch_pdl(cascade_merge_kernel<CPL, G>, blocks, kCascadeMergeWarps * 32, 0, stream, kp,
                    static_cast<const int32_t*>(a.ws.chunk_base),
                    static_cast<const int32_t*>(a.ws.inline_start), a.context_lens,
                    a.max_context_len, a.num_seqs);
}

cudaError_t launch_cascade_merge(const DecodeArgs& a, const DecodeKernelParams& kp,
                                 cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads;
  const unsigned blocks =
      static_cast<unsigned>((items + kCascadeMergeWarps - 1) / kCascadeMergeWarps);
  const int group = a.num_q_heads / a.num_kv_heads;
#define PA_MERGE(CPL_, G_)                                    \
  if (a.head_dim == CPL_ * 32 && group == G_)                \
    return launch_merge_instance<CPL_, G_>(a, kp, blocks, stream);
  PA_MERGE(4, 1) PA_MERGE(4, 2) PA_MERGE(4, 4) PA_MERGE(4, 8)
  PA_MERGE(2, 1) PA_MERGE(2, 2) PA_MERGE(2, 4) PA_MERGE(2, 8)
#undef PA_MERGE
  return cudaErrorInvalidValue;
}

}  // namespace pa
