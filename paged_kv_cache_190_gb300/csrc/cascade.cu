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
//   * plan: per sequence, the prefix chunks (kPrefixChunk tokens of the group's
//     shared pages) and its own suffix chunks, in one partial list;
//   * prefix kernel: per (group, kv head, prefix chunk) the K/V pages are
//     loaded once and all rows of the group (members x query heads of the kv
//     head) attend to them on the tensor cores, writing one partial per row;
//   * the decode kernel over every sequence's own tokens (suffix chunks);
//   * the merge kernel combines each row's partials (log-sum-exp).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "decode_instances.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kCascadePlanThreads = 1024;
constexpr int kPrefixWarps = 4;
constexpr int kPrefixCtasPerSm = 3;

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

// One block.  Sequences: prefix partials p_b = ceil(start_b / kPrefixChunk)
// (start_b = its group's shared length) followed by suffix chunks over
// [start_b, L_b); chunk_base[b] = first partial of b; suffix work entries never
// take the single-chunk shortcut (every row goes through the merge).  Groups:
// the list of (group, prefix chunk) items.  Checks: shared lengths are whole
// pages below every member's length (else PA_DEVERR_BAD_LENGTH, and the member
// is decoded without the sharing).
__global__ void __launch_bounds__(kCascadePlanThreads) cascade_plan_kernel(
    const int32_t* __restrict__ context_lens, const int32_t* __restrict__ group_start, const int32_t* __restrict__ shared_lens,
    int num_groups, int num_seqs, int chunk_tokens, int max_len, int block_size,
    int max_blocks_per_seq, int32_t* __restrict__ header, int32_t* __restrict__ chunk_base,
    int32_t* __restrict__ prefix_parts, int4* __restrict__ work, int2* __restrict__ prefix_items,
    uint4* __restrict__ out, int64_t row_chunks, int32_t* device_errors) {
  __shared__ int warp_sums[kCascadePlanThreads / 32];
  __shared__ int total_s;
  __shared__ int carry_parts, carry_work, carry_items;
  if (threadIdx.x == 0) carry_parts = carry_work = carry_items = 0;
  __syncthreads();
  for (int base = 0; base < num_seqs; base += kCascadePlanThreads) {
    const int b = base + threadIdx.x;
    int L = 0, start = 0, pb = 0, nb = 0;
    if (b < num_seqs) {
      L = context_lens[b];
      if (L < 0 || L > max_len) {
        report(device_errors, PA_DEVERR_BAD_LENGTH);
        L = L < 0 ? 0 : max_len;
      }
      const int f = group_of(group_start, num_groups, b);
      start = shared_lens[f];
      if (start < 0 || start % block_size != 0 || (start > 0 && start >= L) ||
          start > max_blocks_per_seq * block_size) {
        report(device_errors, PA_DEVERR_BAD_LENGTH);
        start = 0;                                   // the prefix kernel still runs for the group
      }
      const int leader = group_start[f];
      if (leader < 0 || leader > b) {                // group_start must be sorted, from 0
        report(device_errors, PA_DEVERR_BAD_LENGTH);
        start = 0;
      }
      // (that the member holds the leader's pages is checked by the prefix kernel,
      // page by page, where the pages are read)
      pb = (start + kPrefixChunk - 1) / kPrefixChunk;
      nb = L > start ? (L - start + chunk_tokens - 1) / chunk_tokens : 0;
    }
    const int parts = block_scan(pb + nb, warp_sums, &total_s);
    const int tparts = total_s;
    const int wk = block_scan(nb, warp_sums, &total_s);
    const int twork = total_s;
    if (b < num_seqs) {
      const int first = carry_parts + parts;
      chunk_base[b] = first;
      prefix_parts[b] = pb;                          // the prefix kernel writes only these
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
  for (int base = 0; base < num_groups; base += kCascadePlanThreads) {
    const int f = base + threadIdx.x;
    int nc = 0;
    if (f < num_groups) {
      const int sl = shared_lens[f];
      const bool ok = sl > 0 && sl % block_size == 0 && sl <= max_blocks_per_seq * block_size &&
                      sl <= max_len;
      nc = ok ? (sl + kPrefixChunk - 1) / kPrefixChunk : 0;
    }
    const int first = block_scan(nc, warp_sums, &total_s);
    const int tot = total_s;
    if (f < num_groups)
      for (int c = 0; c < nc; ++c) prefix_items[carry_items + first + c] = make_int2(f, c);
    __syncthreads();
    if (threadIdx.x == 0) carry_items += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    chunk_base[num_seqs] = carry_parts;
    header[0] = 0;
    header[1] = carry_work;
    header[2] = carry_items;
  }
}

// Prefix attention.  Item = (group f, prefix chunk c) x kv head h: the chunk's
// tokens [c kPrefixChunk, ...) of the group's shared pages (read through the
// leader's block table) are copied into shared memory once -- one tensor-map
// box per 16 rows and pool, the decode kernel's swizzled layout -- and every
// row of the group attends to them: rows r = (member m, head g) of kv head h,
// 16 rows per warp at a time (mma.sync m16n8k16, bf16, fp32 accumulation):
//   S = Q K^T (Q rows as A, K via ldmatrix), online softmax per row in base 2,
//   O += P V (P re-packed from the S fragments as A, V via ldmatrix.trans).
// Each row's result is one partial (output divided by its sum, base-2
// log-sum-exp) at chunk_base[member] + c, written only when the plan gave the
// member that many prefix partials.
template <int D>
struct PrefixLayout {
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int GROUP_BYTES = 16 * ROW_BYTES;         // 16 tokens, all slabs
  static constexpr int TILE_BYTES = kPrefixChunk * ROW_BYTES;
  static constexpr int SMEM = 2 * TILE_BYTES + 1024 + 64;    // K, V, alignment, barrier
  static constexpr int KS = D / 16;                          // k-steps of S
  static constexpr int NT = D / 8;                           // n-tiles of O
};

template <int D>
__device__ __forceinline__ uint32_t prefix_swz(int row, int chunk) {
  // token row (0..15 within a 16-token group), 16-byte chunk of the row
  return static_cast<uint32_t>((chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kPrefixWarps * 32) prefix_attention_kernel(
    const __grid_constant__ DecodeKernelParams p, const int32_t* __restrict__ group_start,
    const int32_t* __restrict__ shared_lens, const int32_t* __restrict__ chunk_base,
    const int32_t* __restrict__ prefix_parts, const int2* __restrict__ items, int num_groups,
    int num_seqs) {
  using Ly = PrefixLayout<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  char* ktile = reinterpret_cast<char*>(smem);
  char* vtile = ktile + Ly::TILE_BYTES;
  uint64_t* bar = reinterpret_cast<uint64_t*>(vtile + Ly::TILE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3, mi = lane >> 3, r8 = lane & 7;
  const int Hkv = p.num_kv_heads, G = p.group, bs = p.block_size;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int n_items = p.header[2] * Hkv;
  uint32_t phase = 0;
  bool ok = true;
  for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, phase ^= 1) {
    const int2 fc = items[it / Hkv];
    const int h = it % Hkv;
    const int f = fc.x, chunk = fc.y;
    const int gs = min(max(group_start[f], 0), num_seqs);
    const int ge = min(max(group_start[f + 1], gs), num_seqs);
    const int t0 = chunk * kPrefixChunk;
    const int ntok = min(kPrefixChunk, shared_lens[f] - t0);   // a multiple of 16
    const int ngrp = ntok / 16;
    // ---- copy the chunk's K and V: lane j < ngrp of warp 0 takes 16-token group j
    if (warp == 0) {
      if (lane == 0) mbar_arrive_expect_tx(bar, ngrp * Ly::GROUP_BYTES * 2);
      __syncwarp();
      if (lane < 2 * ngrp) {
        const int j = lane >> 1;
        const int t = t0 + 16 * j;
        int page = p.block_tables[static_cast<int64_t>(gs) * p.max_blocks_per_seq + t / bs];
        if (page < 0 || page >= p.num_blocks) {
          report(p.device_errors, PA_DEVERR_BAD_BLOCK);
          page = -1;                         // a row outside the pool: the box reads zeros
        }
        const int row = (page * Hkv + h) * bs + t % bs;
        const bool is_v = lane & 1;
        char* dst = (is_v ? vtile : ktile) + j * Ly::GROUP_BYTES;
        if constexpr (Ly::ROW_BYTES == 128)
          tma_load_2d(dst, is_v ? &p.tmap_v : &p.tmap_k, 0, row, bar);
        else
          tma_load_3d(dst, is_v ? &p.tmap_v : &p.tmap_k, 0, row, 0, bar);
      }
    }
    // every member that uses this chunk must hold the leader's pages for it
    {
      const int np = ntok / bs, pg0 = t0 / bs;
      const int32_t* lead = p.block_tables + static_cast<int64_t>(gs) * p.max_blocks_per_seq;
      for (int i = threadIdx.x; i < (ge - gs) * np; i += kPrefixWarps * 32) {
        const int m = gs + i / np, pg = pg0 + i % np;
        if (chunk < prefix_parts[m] &&
            p.block_tables[static_cast<int64_t>(m) * p.max_blocks_per_seq + pg] != lead[pg])
          report(p.device_errors, PA_DEVERR_BAD_BLOCK);
      }
    }
    // the decision to give up is taken by the whole block, so that no warp is
    // left at the barrier below
    const bool waited = mbar_wait(bar, phase, p.wait_limit);
    if (__syncthreads_or(!waited)) {
      if (threadIdx.x == 0) report(p.device_errors, PA_DEVERR_TIMEOUT);
      ok = false;
      // wait (bounded) for the copies before the shared memory is released
      mbar_wait(bar, phase);
      break;
    }
    const uint32_t kb = smem_addr(ktile), vb = smem_addr(vtile);
    const int rows = (ge - gs) * G;
    for (int rt = warp * 16; rt < rows; rt += kPrefixWarps * 16) {
      // ---- q of rows rt + g and rt + g + 8: member (r / G), head h G + r % G
      uint32_t qa[Ly::KS][4];
      const int ra = rt + g, rb = rt + g + 8;
      const char* qra = ra < rows ? p.q + ((static_cast<int64_t>(gs + ra / G) * p.num_q_heads +
                                           h * G + ra % G) * D) * 2 : nullptr;
      const char* qrb = rb < rows ? p.q + ((static_cast<int64_t>(gs + rb / G) * p.num_q_heads +
                                           h * G + rb % G) * D) * 2 : nullptr;
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
      for (int grp = 0; grp < ngrp; ++grp) {
        const uint32_t kg = kb + grp * Ly::GROUP_BYTES, vg = vb + grp * Ly::GROUP_BYTES;
        // ---- S for 16 tokens: n-tile 0 (tokens 0-7), 1 (8-15)
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < Ly::KS; ++ks) {
          uint32_t b00, b01, b10, b11;
          ldsm_x4(kg + prefix_swz<D>((mi >> 1) * 8 + r8, 2 * ks + (mi & 1)), b00, b01, b10, b11);
          mma_bf16_full(s0, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b00, b01);
          mma_bf16_full(s1, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b10, b11);
        }
        // ---- online softmax, rows g (c0, c1) and g + 8 (c2, c3)
        const float sc = p.scale_log2;
        float x0 = fmaxf(fmaxf(s0[0], s0[1]), fmaxf(s1[0], s1[1])) * sc;
        float x1 = fmaxf(fmaxf(s0[2], s0[3]), fmaxf(s1[2], s1[3])) * sc;
        x0 = fmaxf(x0, __shfl_xor_sync(kFull, x0, 1));
        x0 = fmaxf(x0, __shfl_xor_sync(kFull, x0, 2));
        x1 = fmaxf(x1, __shfl_xor_sync(kFull, x1, 1));
        x1 = fmaxf(x1, __shfl_xor_sync(kFull, x1, 2));
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float a0 = fast_exp2(m0 - n0), a1 = fast_exp2(m1 - n1);
        m0 = n0;
        m1 = n1;
        const float p00 = fast_exp2(s0[0] * sc - n0), p01 = fast_exp2(s0[1] * sc - n0);
        const float p02 = fast_exp2(s0[2] * sc - n1), p03 = fast_exp2(s0[3] * sc - n1);
        const float p10 = fast_exp2(s1[0] * sc - n0), p11 = fast_exp2(s1[1] * sc - n0);
        const float p12 = fast_exp2(s1[2] * sc - n1), p13 = fast_exp2(s1[3] * sc - n1);
        l0 = l0 * a0 + ((p00 + p01) + (p10 + p11));
        l1 = l1 * a1 + ((p02 + p03) + (p12 + p13));
        // P as the A operand (rows g / g + 8; tokens 2c, 2c + 1 / 8 + 2c, 9 + 2c)
        const uint32_t pa0 = pack_bf16x2(p00, p01), pa1 = pack_bf16x2(p02, p03);
        const uint32_t pa2 = pack_bf16x2(p10, p11), pa3 = pack_bf16x2(p12, p13);
        // ---- O = O alpha + P V; V^T fragments for n-tiles 2j, 2j + 1
#pragma unroll
        for (int j = 0; j < Ly::NT / 2; ++j) {
          uint32_t v00, v01, v10, v11;
          ldsm_x4_trans(vg + prefix_swz<D>((mi & 1) * 8 + r8, 2 * j + (mi >> 1)), v00, v01, v10, v11);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float(&od)[4] = o[2 * j + e];
            od[0] *= a0;
            od[1] *= a0;
            od[2] *= a1;
            od[3] *= a1;
          }
          mma_bf16_full(o[2 * j], pa0, pa1, pa2, pa3, v00, v01);
          mma_bf16_full(o[2 * j + 1], pa0, pa1, pa2, pa3, v10, v11);
        }
      }
      // ---- partials of rows g and g + 8
      l0 += __shfl_xor_sync(kFull, l0, 1);
      l0 += __shfl_xor_sync(kFull, l0, 2);
      l1 += __shfl_xor_sync(kFull, l1, 1);
      l1 += __shfl_xor_sync(kFull, l1, 2);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = half ? rb : ra;
        if (r >= rows) continue;
        const int b = gs + r / G;
        if (chunk >= prefix_parts[b]) continue;    // the plan gave this member no such partial
        const int qh = h * G + r % G;
        const int64_t prow = static_cast<int64_t>(chunk_base[b] + chunk) * p.num_q_heads + qh;
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
    // every warp is done with the chunk before the next copy overwrites it
    __syncthreads();
  }
}

cudaError_t cascade_plan_launch(const DecodeArgs& a, cudaStream_t stream) {
  const int64_t row_chunks = static_cast<int64_t>(a.num_q_heads) * a.head_dim * 2 / 16;
  cascade_plan_kernel<<<1, kCascadePlanThreads, 0, stream>>>(
      a.context_lens, a.group_start, a.shared_lens, a.num_groups, a.num_seqs,
      a.chunk_tokens, a.max_context_len, a.block_size, a.max_blocks_per_seq, a.ws.header,
      a.ws.chunk_base, a.ws.prefix_parts, a.ws.work, a.ws.prefix_items,
      static_cast<uint4*>(a.out), row_chunks, a.device_errors);
  return cudaGetLastError();
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
  const int grid = a.num_sms * kPrefixCtasPerSm;
  // an ordinary launch: it starts after the plan kernel has finished (the item
  // list), and the decode kernel, launched as its dependent, after it
  prefix_attention_kernel<D><<<grid, kPrefixWarps * 32, Ly::SMEM, stream>>>(
      kp, a.group_start, a.shared_lens, a.ws.chunk_base, a.ws.prefix_parts, a.ws.prefix_items,
      a.num_groups, a.num_seqs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cascade_prefix(const DecodeArgs& a, const DecodeKernelParams& kp, int device,
                                  cudaStream_t stream) {
  if (a.head_dim == 128) return run_prefix<128>(a, kp, device, stream);
  if (a.head_dim == 64) return run_prefix<64>(a, kp, device, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_cascade_plan(const DecodeArgs& a, cudaStream_t stream) {
  return cascade_plan_launch(a, stream);
}

}  // namespace pa
