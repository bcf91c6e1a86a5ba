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

constexpr int kCascadePlanThreads = 1024;
constexpr int kPlanGroupCache = 2048;                   // groups the plan keeps in shared memory
constexpr int kPrefixConsumerWarps = 4;                 // one 16-row tile each
constexpr int kPrefixThreads = (kPrefixConsumerWarps + 1) * 32;   // + the producer warp
constexpr int kPrefixRows = 16 * kPrefixConsumerWarps;  // rows of one item (a row set)
constexpr int kPrefixStages = 3;
constexpr int kPrefixCtasPerSm = 2;
constexpr int kCascadeMergeWarps = 8;
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

// Block-wide exclusive scan of one value per thread (kCascadePlanThreads); the
// total lands in *total.
__device__ __forceinline__ int block_scan(int x, int* warp_sums, int* total) {
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
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int excl = incl - x + (warp > 0 ? warp_sums[warp - 1] : 0);
  if (threadIdx.x == kCascadePlanThreads - 1) *total = excl + x;
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
//     of `span` stages, span chosen so that the prefix kernel's CTAs get about
//     two items each; the item list holds (group, row set, piece, span).
//  2. Sequences: b has p_b prefix partials (its group's pieces when its shared
//     length is valid for it, else 0) and then its own tokens [start_b, L_b):
//     up to kInlineSuffixTokens of them are left to the merge (inline_start[b]
//     = start_b), more become decode work entries of chunk_tokens each, never
//     single-chunk (every row goes through the merge).  chunk_base[b] = first
//     partial of b.  Checks: a shared length that is not whole pages or not
//     below a member's length sets PA_DEVERR_BAD_LENGTH, and that member is
//     decoded without the sharing.
__global__ void __launch_bounds__(kCascadePlanThreads) cascade_plan_kernel(
    const int32_t* __restrict__ context_lens, const int32_t* group_start,
    const int32_t* shared_lens, int num_groups, int num_seqs, int chunk_tokens,
    int max_len, int block_size, int max_blocks_per_seq, int group, int num_kv_heads,
    int prefix_ctas, int32_t* __restrict__ header, int32_t* __restrict__ chunk_base,
    int32_t* __restrict__ prefix_parts, int32_t* __restrict__ inline_start,
    int4* __restrict__ work, int4* __restrict__ prefix_items, uint4* __restrict__ out,
    int64_t row_chunks, int32_t* device_errors) {
  __shared__ int warp_sums[kCascadePlanThreads / 32];
  __shared__ int total_s;
  __shared__ int carry_parts, carry_work, carry_items, units_s;
  __shared__ int32_t gs_cache[kPlanGroupCache + 1], sl_cache[kPlanGroupCache];
  allow_next_grid();                      // the next kernel may start its prologue
  if (threadIdx.x == 0) carry_parts = carry_work = carry_items = units_s = 0;
  // the group arrays are read many times (a binary search per sequence): keep
  // them in shared memory when they fit
  const bool cached = num_groups <= kPlanGroupCache;
  if (cached) {
    for (int i = threadIdx.x; i <= num_groups; i += kCascadePlanThreads) gs_cache[i] = group_start[i];
    for (int i = threadIdx.x; i < num_groups; i += kCascadePlanThreads) sl_cache[i] = shared_lens[i];
    group_start = gs_cache;
    shared_lens = sl_cache;
  }
  __syncthreads();
  // ---- 1a. total prefix work in stages (x kv heads)
  for (int base = 0; base < num_groups; base += kCascadePlanThreads) {
    const int f = base + threadIdx.x;
    int units = 0;
    if (f < num_groups) {
      const int sl = usable_shared(shared_lens, f, block_size, max_blocks_per_seq, max_len);
      const int2 m = members_of(group_start, f, num_seqs);
      const PrefixShape s = prefix_shape(sl, m.y - m.x, group, 1);
      units = s.stages * s.rowsets;
    }
    block_scan(units, warp_sums, &total_s);
    if (threadIdx.x == 0) units_s += total_s;
    __syncthreads();
  }
  const int64_t total_units = static_cast<int64_t>(units_s) * num_kv_heads;
  const int64_t target = 2 * static_cast<int64_t>(prefix_ctas > 0 ? prefix_ctas : 1);
  const int64_t want = (total_units + target - 1) / target;
  const int span = static_cast<int>(want > 1 ? want : 1);
  // ---- 1b. the item list
  for (int base = 0; base < num_groups; base += kCascadePlanThreads) {
    const int f = base + threadIdx.x;
    PrefixShape s{0, 0, 1, 0};
    if (f < num_groups) {
      const int sl = usable_shared(shared_lens, f, block_size, max_blocks_per_seq, max_len);
      const int2 m = members_of(group_start, f, num_seqs);
      s = prefix_shape(sl, m.y - m.x, group, span);
    }
    const int n = s.rowsets * s.pieces;
    const int first = block_scan(n, warp_sums, &total_s);
    const int tot = total_s;
    for (int i = 0; i < n; ++i)
      prefix_items[carry_items + first + i] = make_int4(f, i / s.pieces, i % s.pieces, s.span);
    __syncthreads();
    if (threadIdx.x == 0) carry_items += tot;
    __syncthreads();
  }
  // ---- 2. sequences
  for (int base = 0; base < num_seqs; base += kCascadePlanThreads) {
    const int b = base + threadIdx.x;
    int L = 0, start = 0, pb = 0, nb = 0;
    bool inl = false;
    if (b < num_seqs) {
      L = context_lens[b];
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
    const int parts = block_scan(pb + nb, warp_sums, &total_s);
    const int tparts = total_s;
    const int wk = block_scan(nb, warp_sums, &total_s);
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
// group's shared tokens (kPrefixStageTokens each, read through the group
// leader's block table) and the row set's 64 rows r = (member, query head of h),
// member = r / group.  One producer warp streams each stage's K and V into a
// 3-slot ring (one tensor-map box per 16 tokens and pool, the decode kernel's
// swizzled layout); four consumer warps own 16 rows each and keep q, the running
// maximum and sum, and the output in registers for the whole piece:
//   S = Q K^T per 16 tokens (mma.sync m16n8k16, bf16, fp32 accumulation; Q rows
//   as A, K via ldmatrix), online softmax per row in base 2, O += P V (P re-packed
//   from the S fragments as A, V via ldmatrix.trans).
// Each row's piece ends as one partial (output divided by its sum, base-2
// log-sum-exp) at chunk_base[member] + piece, written only when the plan gave
// the member that many prefix partials.  Items of kv head 0 also check that the
// members hold the leader's pages (PA_DEVERR_BAD_BLOCK).
template <int D>
struct PrefixLayout {
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int GROUP_BYTES = 16 * ROW_BYTES;         // 16 tokens, all slabs
  static constexpr int GROUPS = kPrefixStageTokens / 16;
  static constexpr int TILE_BYTES = GROUPS * GROUP_BYTES;    // K (or V) of one stage
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int SMEM = kPrefixStages * STAGE_BYTES + 1024 + 64;  // + alignment, barriers
  static constexpr int KS = D / 16;                          // k-steps of S
  static constexpr int NT = D / 8;                           // n-tiles of O
};

// Byte offset of 16-byte chunk `chunk` of token row `row` (0..15) in a 16-token
// group: slabs of 16 rows x 128 bytes, 128-byte swizzle.
__device__ __forceinline__ uint32_t prefix_swz(int row, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// NG (1 or 2) consecutive 16-token groups of a stage, for one warp's 16 rows
// (g and g + 8 of lane g * 4 + c): the scores of all 16 NG tokens first (2 NG
// independent accumulation chains over head_dim), one online-softmax update
// of the rows' reference maximum and sum (base 2), then O += P V with NG k-steps.
template <int D, int NG>
__device__ __forceinline__ void prefix_step(uint32_t kg, uint32_t vg,
                                            const uint32_t (&qa)[D / 16][4],
                                            float (&o)[D / 8][4], float& m0, float& m1,
                                            float& l0, float& l1, float sc, int lane) {
  constexpr int KS = D / 16, NT = D / 8, GB = 16 * D * 2;
  const int mi = lane >> 3, r8 = lane & 7;
  float s[2 * NG][4];
#pragma unroll
  for (int t = 0; t < 2 * NG; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
  // ---- S = Q K^T: n-tiles 2 gi (tokens 0-7 of group gi) and 2 gi + 1 (8-15)
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      uint32_t b00, b01, b10, b11;
      ldsm_x4(kg + gi * GB + prefix_swz((mi >> 1) * 8 + r8, 2 * ks + (mi & 1)), b00, b01, b10,
              b11);
      mma_bf16_full(s[2 * gi], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b00, b01);
      mma_bf16_full(s[2 * gi + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b10, b11);
    }
  }
  // ---- online softmax: row g holds elements 0, 1 of each tile, row g + 8 elements 2, 3
  float x0 = fmaxf(s[0][0], s[0][1]), x1 = fmaxf(s[0][2], s[0][3]);
#pragma unroll
  for (int t = 1; t < 2 * NG; ++t) {
    x0 = fmaxf(x0, fmaxf(s[t][0], s[t][1]));
    x1 = fmaxf(x1, fmaxf(s[t][2], s[t][3]));
  }
  x0 *= sc;
  x1 *= sc;
  x0 = fmaxf(x0, __shfl_xor_sync(kFull, x0, 1));
  x0 = fmaxf(x0, __shfl_xor_sync(kFull, x0, 2));
  x1 = fmaxf(x1, __shfl_xor_sync(kFull, x1, 1));
  x1 = fmaxf(x1, __shfl_xor_sync(kFull, x1, 2));
  // The reference maximum of a row only moves when a score exceeds it by more
  // than 8 (every probability stays <= 2^8, exact in fp32 and bf16), and then
  // for the whole warp: most steps rescale nothing.
  const bool grow = x0 > m0 + 8.f || x1 > m1 + 8.f;
  const bool rescale = __any_sync(kFull, grow);
  float a0 = 1.f, a1 = 1.f;
  if (rescale) {
    const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
    a0 = fast_exp2(m0 - n0);
    a1 = fast_exp2(m1 - n1);
    m0 = n0;
    m1 = n1;
  }
  const float n0 = m0, n1 = m1;
  float sum0 = 0.f, sum1 = 0.f;
  uint32_t pa[NG][4];
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) {
    float pr[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      pr[u][0] = fast_exp2(s[2 * gi + u][0] * sc - n0);
      pr[u][1] = fast_exp2(s[2 * gi + u][1] * sc - n0);
      pr[u][2] = fast_exp2(s[2 * gi + u][2] * sc - n1);
      pr[u][3] = fast_exp2(s[2 * gi + u][3] * sc - n1);
      sum0 += pr[u][0] + pr[u][1];
      sum1 += pr[u][2] + pr[u][3];
    }
    // P as the A operand (rows g / g + 8; tokens 2c, 2c + 1 / 8 + 2c, 9 + 2c)
    pa[gi][0] = pack_bf16x2(pr[0][0], pr[0][1]);
    pa[gi][1] = pack_bf16x2(pr[0][2], pr[0][3]);
    pa[gi][2] = pack_bf16x2(pr[1][0], pr[1][1]);
    pa[gi][3] = pack_bf16x2(pr[1][2], pr[1][3]);
  }
  l0 = l0 * a0 + sum0;
  l1 = l1 * a1 + sum1;
  if (rescale) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      o[t][0] *= a0;
      o[t][1] *= a0;
      o[t][2] *= a1;
      o[t][3] *= a1;
    }
  }
  // ---- O = O + P V; V^T fragments for n-tiles 2j, 2j + 1
#pragma unroll
  for (int j = 0; j < NT / 2; ++j) {
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      uint32_t v00, v01, v10, v11;
      ldsm_x4_trans(vg + gi * GB + prefix_swz((mi & 1) * 8 + r8, 2 * j + (mi >> 1)), v00, v01,
                    v10, v11);
      mma_bf16_full(o[2 * j], pa[gi][0], pa[gi][1], pa[gi][2], pa[gi][3], v00, v01);
      mma_bf16_full(o[2 * j + 1], pa[gi][0], pa[gi][1], pa[gi][2], pa[gi][3], v10, v11);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kPrefixThreads) prefix_attention_kernel(
    const __grid_constant__ DecodeKernelParams p, const int32_t* __restrict__ group_start,
    const int32_t* __restrict__ shared_lens, const int32_t* __restrict__ chunk_base,
    const int32_t* __restrict__ prefix_parts, const int4* __restrict__ items, int num_seqs) {
  using Ly = PrefixLayout<D>;
  constexpr int NST = kPrefixStages;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * Ly::STAGE_BYTES);
  uint64_t* empty = full + NST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + NST);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = p.num_kv_heads, G = p.group, bs = p.block_size;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kPrefixConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  wait_prior_grids();                     // the plan's item list and partial offsets
  const int n_items = p.header[2] * Hkv;

  if (warp == kPrefixConsumerWarps) {
    // ---------------- producer: lane 2j (2j + 1) copies K (V) of 16-token group j
    uint32_t k = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const int4 item = items[it / Hkv];
      const int h = it % Hkv;
      const int sl = shared_lens[item.x];
      const int leader = members_of(group_start, item.x, num_seqs).x;
      const int32_t* table = p.block_tables + static_cast<int64_t>(leader) * p.max_blocks_per_seq;
      const int stages = (sl + kPrefixStageTokens - 1) / kPrefixStageTokens;
      const int st0 = item.z * item.w, st1 = min(st0 + item.w, stages);
      // the pages of the piece's first 32 16-token groups, one per lane, fetched
      // while the first slot is awaited
      const int ngi = (min(st1 * kPrefixStageTokens, sl) - st0 * kPrefixStageTokens) / 16;
      int pre_page = -1;
      if (lane < ngi) {
        pre_page = table[(st0 * kPrefixStageTokens + 16 * lane) / bs];
        if (pre_page < 0 || pre_page >= p.num_blocks) {
          report(p.device_errors, PA_DEVERR_BAD_BLOCK);
          pre_page = -1;                       // a row outside the pool: the box reads zeros
        }
      }
      for (int st = st0; st < st1; ++st, ++k) {
        const int slot = static_cast<int>(k % NST);
        bool waited = false;
        if (lane == 0 && !*abort_flag)
          waited = mbar_wait(&empty[slot], ((k / NST) & 1) ^ 1, p.wait_limit);
        waited = __shfl_sync(kFull, waited, 0);
        if (!waited) {
          if (lane == 0 && !*abort_flag) {
            report(p.device_errors, PA_DEVERR_TIMEOUT);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
        const int t0 = st * kPrefixStageTokens;
        const int ngrp = min(kPrefixStageTokens, sl - t0) / 16;
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], ngrp * 2 * Ly::GROUP_BYTES);
        const int gi = (st - st0) * Ly::GROUPS + (lane >> 1);   // group within the piece
        int page = __shfl_sync(kFull, pre_page, gi < 32 ? gi : 31);
        if (lane < 2 * ngrp) {
          const int j = lane >> 1;
          const int t = t0 + 16 * j;
          if (gi >= 32) {                        // past the prefetched pages
            page = table[t / bs];
            if (page < 0 || page >= p.num_blocks) {
              report(p.device_errors, PA_DEVERR_BAD_BLOCK);
              page = -1;
            }
          }
          const int row = (page * Hkv + h) * bs + t % bs;
          const bool is_v = lane & 1;
          unsigned char* dst = smem + slot * Ly::STAGE_BYTES + (is_v ? Ly::TILE_BYTES : 0) +
                               j * Ly::GROUP_BYTES;
          if constexpr (Ly::ROW_BYTES == 128)
            tma_load_2d(dst, is_v ? &p.tmap_v : &p.tmap_k, 0, row, &full[slot]);
          else
            tma_load_3d(dst, is_v ? &p.tmap_v : &p.tmap_k, 0, row, 0, &full[slot]);
        }
      }
    }
    // the copies of the last stages must land before the shared memory is released
    if (lane == 0)
      for (uint32_t j = k > NST ? k - NST : 0; j < k; ++j) mbar_wait(&full[j % NST], (j / NST) & 1);
    return;
  }

  // ---------------- consumers
  const int g = lane >> 2, c = lane & 3;
  uint32_t k = 0;
  bool live = true;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int4 item = items[it / Hkv];
    const int h = it % Hkv;
    const int sl = shared_lens[item.x];
    const int2 mem = members_of(group_start, item.x, num_seqs);
    const int rows = (mem.y - mem.x) * G;
    const int stages = (sl + kPrefixStageTokens - 1) / kPrefixStageTokens;
    const int piece = item.z;
    const int st0 = piece * item.w, st1 = min(st0 + item.w, stages);
    const int row0 = item.y * kPrefixRows + 16 * warp;      // this warp's first row
    if (h == 0) {
      // members of this row set that use this piece hold the leader's pages
      const int m_lo = mem.x + item.y * kPrefixRows / G;
      const int m_hi = min(mem.y, mem.x + (item.y + 1) * kPrefixRows / G);
      const int pg0 = st0 * kPrefixStageTokens / bs;
      const int np = min(st1 * kPrefixStageTokens, sl) / bs - pg0;
      const int32_t* lead = p.block_tables + static_cast<int64_t>(mem.x) * p.max_blocks_per_seq;
      for (int i = threadIdx.x; i < (m_hi - m_lo) * np; i += kPrefixConsumerWarps * 32) {
        const int m = m_lo + i / np, pg = pg0 + i % np;
        if (piece < prefix_parts[m] &&
            p.block_tables[static_cast<int64_t>(m) * p.max_blocks_per_seq + pg] != lead[pg])
          report(p.device_errors, PA_DEVERR_BAD_BLOCK);
      }
    }
    // ---- q of rows ra = row0 + g and rb = ra + 8: member r / G, head h G + r % G
    const int ra = row0 + g, rb = ra + 8;
    const char* qra = ra < rows ? p.q + ((static_cast<int64_t>(mem.x + ra / G) * p.num_q_heads +
                                          h * G + ra % G) * D) * 2
                                : nullptr;
    const char* qrb = rb < rows ? p.q + ((static_cast<int64_t>(mem.x + rb / G) * p.num_q_heads +
                                          h * G + rb % G) * D) * 2
                                : nullptr;
    uint32_t qa[Ly::KS][4];
#pragma unroll
    for (int ks = 0; ks < Ly::KS; ++ks) {
      const int col = 16 * ks + 2 * c;
      qa[ks][0] = qra ? *reinterpret_cast<const uint32_t*>(qra + col * 2) : 0u;
      qa[ks][1] = qrb ? *reinterpret_cast<const uint32_t*>(qrb + col * 2) : 0u;
      qa[ks][2] = qra ? *reinterpret_cast<const uint32_t*>(qra + (col + 8) * 2) : 0u;
      qa[ks][3] = qrb ? *reinterpret_cast<const uint32_t*>(qrb + (col + 8) * 2) : 0u;
    }
    float o[Ly::NT][4];
#pragma unroll
    for (int n = 0; n < Ly::NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = kNoScore, m1 = kNoScore, l0 = 0.f, l1 = 0.f;   // rows g, g + 8
    const bool has_rows = row0 < rows;
    for (int st = st0; st < st1; ++st, ++k) {
      const int slot = static_cast<int>(k % NST);
      if (live) {
        bool waited = !*abort_flag && mbar_wait(&full[slot], (k / NST) & 1, p.wait_limit);
        waited = __all_sync(kFull, waited);
        if (!waited) {
          if (lane == 0 && !*abort_flag) {
            report(p.device_errors, PA_DEVERR_TIMEOUT);
            *abort_flag = 1;
          }
          live = false;
        }
      }
      if (live && has_rows) {
        const uint32_t kb = smem_addr(smem + slot * Ly::STAGE_BYTES);
        const uint32_t vb = kb + Ly::TILE_BYTES;
        const int ngrp = min(kPrefixStageTokens, sl - st * kPrefixStageTokens) / 16;
        const float sc = p.scale_log2;
        int grp = 0;
        for (; grp + 2 <= ngrp; grp += 2)
          prefix_step<D, 2>(kb + grp * Ly::GROUP_BYTES, vb + grp * Ly::GROUP_BYTES, qa, o, m0, m1,
                            l0, l1, sc, lane);
        if (grp < ngrp)
          prefix_step<D, 1>(kb + grp * Ly::GROUP_BYTES, vb + grp * Ly::GROUP_BYTES, qa, o, m0, m1,
                            l0, l1, sc, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);   // the slot may be refilled
    }
    if (!live || !has_rows) continue;
    // ---- partials of rows g and g + 8
    l0 += __shfl_xor_sync(kFull, l0, 1);
    l0 += __shfl_xor_sync(kFull, l0, 2);
    l1 += __shfl_xor_sync(kFull, l1, 1);
    l1 += __shfl_xor_sync(kFull, l1, 2);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = half ? rb : ra;
      if (r >= rows) continue;
      const int b = mem.x + r / G;
      if (piece >= prefix_parts[b]) continue;      // the plan gave this member no such partial
      const int qh = h * G + r % G;
      const int64_t prow = static_cast<int64_t>(chunk_base[b] + piece) * p.num_q_heads + qh;
      const float l = half ? l1 : l0;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int n = 0; n < Ly::NT; ++n) {
        const float2 v = half ? make_float2(o[n][2] * inv, o[n][3] * inv)
                              : make_float2(o[n][0] * inv, o[n][1] * inv);
        *reinterpret_cast<float2*>(p.part_out + prow * D + 8 * n + 2 * c) = v;
      }
      if (c == 0) p.part_lse[prow] = l > 0.f ? (half ? m1 : m0) + __log2f(l) : -INFINITY;
    }
  }
}

// ------------------------------------------------------------ merge
// One warp per (sequence b, kv head h): the G = group query rows of h.  Each
// row's partials c (the prefix pieces, then any decode-kernel chunks of its own
// tokens) combine as
//   out = sum_c 2^(lse_c - M) o_c / sum_c 2^(lse_c - M),  M = max_c lse_c,
// each lane owning CPL = head_dim / 32 columns.  A short own suffix
// [inline_start[b], L_b) (at most 32 tokens) is one more term per row, computed
// here: the suffix's tokens share the warp, LPT = 32 / (its length rounded up to
// a power of two) lanes each (at most one 16-byte piece of the row per lane
// and token fewer), every lane forming the G partial scores of its part of its
// token's K row (q rows as fp32 in shared memory), summed over the token's
// lanes; the base-2 softmax of each row runs over the tokens; the weighted sum
// of V uses every token's V columns of this lane, all loaded up front.  Every load of the warp (pages,
// then K, V and the partials) is issued before the arithmetic that needs it.
// Rows with neither (L_b = 0) were zeroed by the plan.
template <int CPL, int G>
__global__ void __launch_bounds__(kCascadeMergeWarps * 32) cascade_merge_kernel(
    const __grid_constant__ DecodeKernelParams p, const int32_t* __restrict__ chunk_base,
    const int32_t* __restrict__ inline_start, const int32_t* __restrict__ context_lens,
    int max_len, int num_seqs) {
  constexpr int D = CPL * 32;
  constexpr int KV = D / 8;                     // 16-byte pieces of a row
  __shared__ __align__(16) float q_s[kCascadeMergeWarps][G * D];
  wait_prior_grids();                           // every partial is written
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int Hq = p.num_q_heads, Hkv = p.num_kv_heads;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kCascadeMergeWarps + warp;
  if (item >= static_cast<int64_t>(num_seqs) * Hkv) return;
  const int b = static_cast<int>(item / Hkv);
  const int h = static_cast<int>(item - static_cast<int64_t>(b) * Hkv);
  const int c0 = chunk_base[b];
  const int n = chunk_base[b + 1] - c0;
  const int s0 = inline_start[b];
  if (n <= 0 && s0 < 0) return;                 // uniform over the warp
  const int bs = p.block_size;
  const int L = s0 >= 0 ? min(max(context_lens[b], 0), max_len) : 0;
  const int nsuf = s0 >= 0 ? min(L - s0, 32) : 0;
  const int64_t row0 = static_cast<int64_t>(b) * Hq + h * G;   // first output row
  // ---- the G q rows -> shared memory as fp32
  if (nsuf > 0) {
    const uint4* qsrc = reinterpret_cast<const uint4*>(p.q) + row0 * KV;
    float4* qdst = reinterpret_cast<float4*>(q_s[warp]);
    for (int e = lane; e < G * KV; e += 32) {
      const uint4 w = qsrc[e];
      qdst[2 * e] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
      qdst[2 * e + 1] = make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
    }
  }
  // ---- this lane's token (LPT lanes per token), its page and its part of the K row
  int p2 = 1;
  while (p2 < nsuf) p2 <<= 1;
  const int lpt = min(32 / p2, KV);              // lanes per token
  const int per = KV / lpt;                      // 16-byte pieces per lane
  const int tok = lane / lpt, part = lane - tok * lpt;
  int page = -1;
  if (tok < nsuf) {
    const int t = s0 + tok;
    page = p.block_tables[static_cast<int64_t>(b) * p.max_blocks_per_seq + t / bs];
    if (page < 0 || page >= p.num_blocks) {
      if (part == 0) report(p.device_errors, PA_DEVERR_BAD_BLOCK);
      page = -1;
    }
  }
  const int64_t kv_row =
      page >= 0 ? ((static_cast<int64_t>(page) * Hkv + h) * bs + (s0 + tok) % bs) * D : 0;
  uint4 kr[KV];
#pragma unroll
  for (int e = 0; e < KV; ++e)
    kr[e] = page >= 0 && e < per
                ? reinterpret_cast<const uint4*>(p.k_cache + kv_row * 2)[part * per + e]
                : make_uint4(0, 0, 0, 0);
  // ---- this lane's V columns of every token (token j's row from its first lane)
  using VCols = typename std::conditional<CPL == 4, uint2, uint32_t>::type;
  VCols vr[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int64_t rj = __shfl_sync(kFull, kv_row, j < nsuf ? j * lpt : 0);
    vr[j] = j < nsuf ? *reinterpret_cast<const VCols*>(p.v_cache + (rj + lane * CPL) * 2)
                     : VCols{};
  }
  // ---- the partials of the G rows
  float M[G], S[G], acc[G][CPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    M[g] = kNoScore;
    S[g] = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) acc[g][k] = 0.f;
  }
  auto add = [&](int g, float lse, const float* v) {
    const float Mn = fmaxf(M[g], lse);
    const float sc = fast_exp2(M[g] - Mn);
    const float w = fast_exp2(lse - Mn);
    S[g] = fmaf(S[g], sc, w);
#pragma unroll
    for (int k = 0; k < CPL; ++k) acc[g][k] = fmaf(acc[g][k], sc, w * v[k]);
    M[g] = Mn;
  };
  // Each row's largest log-sum-exp first (lane i takes the (partial, row)
  // entries i, i + 32, ...: row i % G, as 32 is a multiple of G), so that the
  // weighted sum below has no chain from one partial to the next.
  if (n > 0) {
    float mloc = kNoScore;
    for (int i = lane; i < n * G; i += 32)
      mloc = fmaxf(mloc, p.part_lse[(static_cast<int64_t>(c0) + i / G) * Hq + h * G + i % G]);
    for (int o2 = 16; o2 >= G; o2 >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, o2));
#pragma unroll
    for (int g = 0; g < G; ++g) M[g] = __shfl_sync(kFull, mloc, g);   // lane g holds row g's
#pragma unroll 4
    for (int cc = 0; cc < n; ++cc) {
      const int64_t prow = (static_cast<int64_t>(c0) + cc) * Hq + h * G;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float* src = p.part_out + (prow + g) * D + lane * CPL;
        const float w = fast_exp2(p.part_lse[prow + g] - M[g]);   // 0 for an empty partial
        float v[CPL];
        if constexpr (CPL == 4) {
          const float4 t4 = *reinterpret_cast<const float4*>(src);
          v[0] = t4.x; v[1] = t4.y; v[2] = t4.z; v[3] = t4.w;
        } else {
          const float2 t2 = *reinterpret_cast<const float2*>(src);
          v[0] = t2.x; v[1] = t2.y;
        }
        S[g] += w;
#pragma unroll
        for (int k = 0; k < CPL; ++k) acc[g][k] = fmaf(w, v[k], acc[g][k]);
      }
    }
  }
  // ---- the suffix term of each row
  if (nsuf > 0) {
    __syncwarp();
    float s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = 0.f;
    const float4* qv = reinterpret_cast<const float4*>(q_s[warp]);
#pragma unroll
    for (int e = 0; e < KV; ++e) {
      if (e < per) {                              // uniform over the warp
        const uint4 kk = kr[e];
        const float k0 = bf16_lo(kk.x), k1 = bf16_hi(kk.x), k2 = bf16_lo(kk.y), k3 = bf16_hi(kk.y);
        const float k4 = bf16_lo(kk.z), k5 = bf16_hi(kk.z), k6 = bf16_lo(kk.w), k7 = bf16_hi(kk.w);
        const int ci = part * per + e;            // 16-byte piece of the row: 8 columns
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = qv[(g * D) / 4 + 2 * ci], qb = qv[(g * D) / 4 + 2 * ci + 1];
          float d = s[g];
          d = fmaf(qa.x, k0, d);
          d = fmaf(qa.y, k1, d);
          d = fmaf(qa.z, k2, d);
          d = fmaf(qa.w, k3, d);
          d = fmaf(qb.x, k4, d);
          d = fmaf(qb.y, k5, d);
          d = fmaf(qb.z, k6, d);
          d = fmaf(qb.w, k7, d);
          s[g] = d;
        }
      }
    }
    // the token's score: the sum over its lanes
    for (int o2 = 1; o2 < lpt; o2 <<= 1)
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] += __shfl_xor_sync(kFull, s[g], o2);
    float pj[G], mx[G], l[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float sg = page >= 0 ? s[g] * p.scale_log2 : -INFINITY;
      float m = sg;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o2));
      mx[g] = m;
      pj[g] = m > -INFINITY ? fast_exp2(sg - m) : 0.f;
      float t = part == 0 ? pj[g] : 0.f;          // each token once
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) t += __shfl_xor_sync(kFull, t, o2);
      l[g] = t;
    }
    float o[G][CPL];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int k = 0; k < CPL; ++k) o[g][k] = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < nsuf) {                           // uniform over the warp
        float v[CPL];
        if constexpr (CPL == 4) {
          v[0] = bf16_lo(vr[j].x); v[1] = bf16_hi(vr[j].x);
          v[2] = bf16_lo(vr[j].y); v[3] = bf16_hi(vr[j].y);
        } else {
          v[0] = bf16_lo(vr[j]); v[1] = bf16_hi(vr[j]);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float w = __shfl_sync(kFull, pj[g], j * lpt);   // 0 for an unreadable token
#pragma unroll
          for (int k = 0; k < CPL; ++k) o[g][k] = fmaf(w, w != 0.f ? v[k] : 0.f, o[g][k]);
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (l[g] > 0.f) {
        const float inv = 1.f / l[g];
#pragma unroll
        for (int k = 0; k < CPL; ++k) o[g][k] *= inv;
        add(g, mx[g] + __log2f(l[g]), o[g]);
      }
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
  // a dependent of the decode kernel (itself one of the plan kernel): its
  // blocks wait on the device for both, i.e. for the item list
  return launch_pdl(prefix_attention_kernel<D>, static_cast<unsigned>(prefix_grid(a.num_sms)),
                    kPrefixThreads, Ly::SMEM, stream, kp,
                    static_cast<const int32_t*>(a.group_start),
                    static_cast<const int32_t*>(a.shared_lens),
                    static_cast<const int32_t*>(a.ws.chunk_base),
                    static_cast<const int32_t*>(a.ws.prefix_parts),
                    static_cast<const int4*>(a.ws.prefix_items), a.num_seqs);
}

}  // namespace

int prefix_grid(int num_sms) { return (num_sms > 0 ? num_sms : 1) * kPrefixCtasPerSm; }

cudaError_t launch_cascade_plan(const DecodeArgs& a, cudaStream_t stream) {
  const int64_t row_chunks = static_cast<int64_t>(a.num_q_heads) * a.head_dim * 2 / 16;
  cascade_plan_kernel<<<1, kCascadePlanThreads, 0, stream>>>(
      a.context_lens, a.group_start, a.shared_lens, a.num_groups, a.num_seqs, a.chunk_tokens,
      a.max_context_len, a.block_size, a.max_blocks_per_seq, a.num_q_heads / a.num_kv_heads,
      a.num_kv_heads, prefix_grid(a.num_sms), a.ws.header, a.ws.chunk_base, a.ws.prefix_parts,
      a.ws.inline_start, a.ws.work, a.ws.prefix_items, static_cast<uint4*>(a.out), row_chunks,
      a.device_errors);
  return cudaGetLastError();
}

cudaError_t launch_cascade_prefix(const DecodeArgs& a, const DecodeKernelParams& kp, int device,
                                  cudaStream_t stream) {
  if (a.head_dim == 128) return run_prefix<128>(a, kp, device, stream);
  if (a.head_dim == 64) return run_prefix<64>(a, kp, device, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_cascade_merge(const DecodeArgs& a, const DecodeKernelParams& kp,
                                 cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads;
  const unsigned blocks =
      static_cast<unsigned>((items + kCascadeMergeWarps - 1) / kCascadeMergeWarps);
  const int group = a.num_q_heads / a.num_kv_heads;
#define PA_MERGE(CPL_, G_)                                                                   \
  if (a.head_dim == CPL_ * 32 && group == G_)                                               \
    return launch_pdl(cascade_merge_kernel<CPL_, G_>, blocks, kCascadeMergeWarps * 32, 0, stream, \
                      kp, static_cast<const int32_t*>(a.ws.chunk_base),                     \
                      static_cast<const int32_t*>(a.ws.inline_start), a.context_lens,        \
                      a.max_context_len, a.num_seqs);
  PA_MERGE(4, 1) PA_MERGE(4, 2) PA_MERGE(4, 4) PA_MERGE(4, 8)
  PA_MERGE(2, 1) PA_MERGE(2, 2) PA_MERGE(2, 4) PA_MERGE(2, 8)
#undef PA_MERGE
  return cudaErrorInvalidValue;
}

}  // namespace pa
