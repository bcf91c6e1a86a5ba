// Orchestration of one pa_decode call: plan kernel -> persistent decode kernel
// -> split-K merge kernel, all on the caller's stream.
#include <cuda_runtime.h>

#include <cstdint>

#include "decode_instances.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kPlanThreads = 1024;

// Lists every (sequence, chunk) pair in sequence order, records where each
// sequence's chunks start, resets the work counter and writes zero rows for
// empty sequences.  One block; sequences are scanned 1024 at a time.
__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(
    const int32_t* __restrict__ context_lens, int num_seqs, int chunk_tokens, int max_len,
    int32_t* __restrict__ header, int32_t* __restrict__ chunk_base, int4* __restrict__ work,
    uint4* __restrict__ out, int64_t row_chunks, int32_t* device_errors) {
  __shared__ int warp_sums[kPlanThreads / 32];
  __shared__ int carry_s;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < num_seqs; base += kPlanThreads) {
    const int b = base + threadIdx.x;
    int L = 0, n = 0;
    if (b < num_seqs) {
      L = context_lens[b];
      if (L < 0 || L > max_len) {
        report(device_errors, PA_DEVERR_BAD_LENGTH);
        L = L < 0 ? 0 : max_len;
      }
      n = (L + chunk_tokens - 1) / chunk_tokens;
    }
    int x = n;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
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
    const int excl = x - n + (warp > 0 ? warp_sums[warp - 1] : 0);
    const int carry = carry_s;
    if (b < num_seqs) {
      const int first = carry + excl;
      chunk_base[b] = first;
      for (int c = 0; c < n; ++c) work[first + c] = make_int4(b, c, L, first + c);
      if (L == 0)
        for (int64_t k = 0; k < row_chunks; ++k) out[b * row_chunks + k] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    if (threadIdx.x == kPlanThreads - 1) carry_s = carry + excl + n;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    chunk_base[num_seqs] = carry_s;
    header[0] = 0;
    header[1] = carry_s;
  }
}

__device__ __forceinline__ float block_reduce_128(float v, bool is_max, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float y = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, y) : v + y;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < 4; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  __syncthreads();
  return r;
}

// Split-K merge (log-sum-exp): for sequence b, query head i with n >= 2 chunks,
//   M = max_c lse_c,  w_c = 2^(lse_c - M),  out = sum_c w_c o_c / sum_c w_c,
// where o_c is chunk c's normalised output and lse_c its base-2 log-sum-exp.
template <bool BF16>
__global__ void __launch_bounds__(128) decode_merge_kernel(const int32_t* __restrict__ chunk_base,
                                                           const float* __restrict__ part_lse,
                                                           const float* __restrict__ part_out,
                                                           void* __restrict__ out,
                                                           int num_q_heads, int head_dim) {
  __shared__ float red[4];
  const int64_t row = blockIdx.x;                 // b * num_q_heads + i
  const int b = static_cast<int>(row / num_q_heads);
  const int i = static_cast<int>(row - static_cast<int64_t>(b) * num_q_heads);
  const int c0 = chunk_base[b];
  const int n = chunk_base[b + 1] - c0;
  if (n < 2) return;
  float M = -INFINITY;
  for (int c = threadIdx.x; c < n; c += blockDim.x)
    M = fmaxf(M, part_lse[static_cast<int64_t>(c0 + c) * num_q_heads + i]);
  M = block_reduce_128(M, true, red);
  float S = 0.f;
  for (int c = threadIdx.x; c < n; c += blockDim.x)
    S += fast_exp2(part_lse[static_cast<int64_t>(c0 + c) * num_q_heads + i] - M);
  S = block_reduce_128(S, false, red);
  const float inv = 1.f / S;
  for (int d = threadIdx.x; d < head_dim; d += blockDim.x) {
    float a = 0.f;
#pragma unroll 8
    for (int c = 0; c < n; ++c) {
      const int64_t prow = static_cast<int64_t>(c0 + c) * num_q_heads + i;
      a = fmaf(fast_exp2(part_lse[prow] - M), part_out[prow * head_dim + d], a);
    }
    a *= inv;
    const int64_t o = row * head_dim + d;
    if constexpr (BF16) {
      reinterpret_cast<uint16_t*>(out)[o] = static_cast<uint16_t>(f32_to_bf16_bits(a));
    } else {
      reinterpret_cast<float*>(out)[o] = a;
    }
  }
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

WorkspaceLayout decode_workspace_layout(int num_seqs, int num_q_heads, int head_dim,
                                        int max_context_len, int chunk_tokens) {
  WorkspaceLayout w{};
  const int64_t per_seq =
      max_context_len > 0 ? (static_cast<int64_t>(max_context_len) + chunk_tokens - 1) / chunk_tokens
                          : 0;
  w.max_chunks = static_cast<int64_t>(num_seqs) * per_seq;
  size_t off = 256;  // header
  w.chunk_base = off;
  off += align256(static_cast<size_t>(num_seqs + 1) * 4);
  w.work = off;
  off += align256(static_cast<size_t>(w.max_chunks) * 16);
  w.part_lse = off;
  off += align256(static_cast<size_t>(w.max_chunks) * num_q_heads * 4);
  w.part_out = off;
  off += align256(static_cast<size_t>(w.max_chunks) * num_q_heads * head_dim * 4);
  w.total = off;
  return w;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  const int elt = a.bf16 ? 2 : 4;
  const int64_t row_chunks = static_cast<int64_t>(a.num_q_heads) * a.head_dim * elt / 16;
  decode_plan_kernel<<<1, kPlanThreads, 0, stream>>>(
      a.context_lens, a.num_seqs, a.chunk_tokens, a.max_context_len, a.ws.header,
      a.ws.chunk_base, a.ws.work, static_cast<uint4*>(a.out), row_chunks, a.device_errors);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.ws.max_chunks == 0) return cudaSuccess;  // every length is zero

  DecodeKernelParams kp;
  kp.out = a.out;
  kp.q = static_cast<const char*>(a.q);
  kp.k_cache = static_cast<const char*>(a.k_cache);
  kp.v_cache = static_cast<const char*>(a.v_cache);
  kp.block_tables = a.block_tables;
  kp.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  kp.num_q_heads = a.num_q_heads;
  kp.num_kv_heads = a.num_kv_heads;
  kp.block_size = a.block_size;
  kp.num_blocks = a.num_blocks;
  kp.max_blocks_per_seq = a.max_blocks_per_seq;
  kp.chunk_tokens = a.chunk_tokens;
  kp.header = a.ws.header;
  kp.work = a.ws.work;
  kp.part_lse = a.ws.part_lse;
  kp.part_out = a.ws.part_out;
  kp.device_errors = a.device_errors;
  const int64_t items_upper = a.ws.max_chunks * a.num_kv_heads;
  const int grid = static_cast<int>(items_upper < a.num_sms ? items_upper : a.num_sms);
  int device = 0;
  e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  const int group = a.num_q_heads / a.num_kv_heads;
  e = a.bf16 ? run_decode_bf16(a.head_dim, group, kp, grid, device, stream)
             : run_decode_f32(a.head_dim, group, kp, grid, device, stream);
  if (e != cudaSuccess) return e;
  if (a.max_context_len > a.chunk_tokens) {
    const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
    if (a.bf16)
      decode_merge_kernel<true><<<static_cast<unsigned>(rows), 128, 0, stream>>>(
          a.ws.chunk_base, a.ws.part_lse, a.ws.part_out, a.out, a.num_q_heads, a.head_dim);
    else
      decode_merge_kernel<false><<<static_cast<unsigned>(rows), 128, 0, stream>>>(
          a.ws.chunk_base, a.ws.part_lse, a.ws.part_out, a.out, a.num_q_heads, a.head_dim);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace pa
