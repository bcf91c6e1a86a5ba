// Cache write (new tokens' K/V scattered into their slots) and copy-on-write
// page copy.  Both are byte moves in 16-byte vectors: one thread per 16-byte
// chunk of a head row, consecutive threads on consecutive chunks so every warp
// moves contiguous 512-byte runs.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// "PagedAttention原理" §3.3.4 (append_token): token t's row for kv head h goes to
// page slot / block_size, position slot % block_size of that page.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, int num_tokens,
    int num_kv_heads, int chunks_per_row, int block_size, int64_t num_slots,
    int32_t* device_errors) {
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * chunks_per_row;
  const int64_t total = per_token * num_tokens;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / per_token;
    const int64_t rem = i - t * per_token;        // h * chunks_per_row + c
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;                       // padding token
    if (slot >= num_slots) {
      if (rem == 0) report(device_errors, PA_DEVERR_BAD_SLOT);
      continue;
    }
    const int64_t page = slot / block_size;
    const int64_t offset = slot - page * block_size;
    const int64_t h = rem / chunks_per_row;
    const int64_t c = rem - h * chunks_per_row;
    const int64_t dst = ((page * num_kv_heads + h) * block_size + offset) * chunks_per_row + c;
    k_cache[dst] = k[i];
    v_cache[dst] = v[i];
  }
}

// Two quotients x / s (IEEE division) -> two e4m3 codes, round to nearest even,
// magnitudes past 448 (and infinities) saturated to 448.
__device__ __forceinline__ uint32_t e4m3x2_div(uint32_t two_bf16, float s) {
  const float2 f = make_float2(__fdiv_rn(bf16_lo(two_bf16), s), __fdiv_rn(bf16_hi(two_bf16), s));
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3));
}

// The cache write for float8 e4m3 pools: token t's bf16 row for kv head h is
// divided by that head's scale and stored as e4m3 codes in the same slot as the
// bf16 write.  One thread per 8 elements (16 bytes in, 8 bytes out).
__global__ void __launch_bounds__(256) reshape_and_cache_fp8_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, uint2* __restrict__ k_cache,
    uint2* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping,
    const float* __restrict__ k_scale, const float* __restrict__ v_scale, int num_tokens,
    int num_kv_heads, int groups_per_row, int block_size, int64_t num_slots,
    int32_t* device_errors) {
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * groups_per_row;
  const int64_t total = per_token * num_tokens;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / per_token;
    const int64_t rem = i - t * per_token;        // h * groups_per_row + c
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;                       // padding token
    if (slot >= num_slots) {
      if (rem == 0) report(device_errors, PA_DEVERR_BAD_SLOT);
      continue;
    }
    const int64_t page = slot / block_size;
    const int64_t offset = slot - page * block_size;
    const int64_t h = rem / groups_per_row;
    const int64_t c = rem - h * groups_per_row;
    const int64_t dst = ((page * num_kv_heads + h) * block_size + offset) * groups_per_row + c;
    const float ks = k_scale[h], vs = v_scale[h];
    const uint4 a = k[i], b = v[i];
    k_cache[dst] = make_uint2(e4m3x2_div(a.x, ks) | (e4m3x2_div(a.y, ks) << 16),
                              e4m3x2_div(a.z, ks) | (e4m3x2_div(a.w, ks) << 16));
    v_cache[dst] = make_uint2(e4m3x2_div(b.x, vs) | (e4m3x2_div(b.y, vs) << 16),
                              e4m3x2_div(b.z, vs) | (e4m3x2_div(b.w, vs) << 16));
  }
}

// "mlx-paged-attention", feature 2: the page a writer shares is copied first.
// Block (pair, part): `part` walks a strided share of the page's 16-byte chunks.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ k_cache,
                                                          uint4* __restrict__ v_cache,
                                                          const int64_t* __restrict__ pairs,
                                                          int64_t chunks_per_block,
                                                          int num_blocks, int32_t* device_errors) {
  const int64_t src = pairs[2 * blockIdx.x];
  const int64_t dst = pairs[2 * blockIdx.x + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) report(device_errors, PA_DEVERR_BAD_BLOCK);
    return;
  }
  const uint4* ks = k_cache + src * chunks_per_block;
  const uint4* vs = v_cache + src * chunks_per_block;
  uint4* kd = k_cache + dst * chunks_per_block;
  uint4* vd = v_cache + dst * chunks_per_block;
  for (int64_t i = blockIdx.y * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       i < chunks_per_block; i += static_cast<int64_t>(gridDim.y) * blockDim.x) {
    const uint4 a = ks[i];
    const uint4 b = vs[i];
    kd[i] = a;
    vd[i] = b;
  }
}

// Page copy between two pools (device <-> pinned host memory for swapping).
// Block (pair, part); each thread keeps four 16-byte loads of K and four of V in
// flight before storing, because a load over the host link takes microseconds.
__global__ void __launch_bounds__(256) swap_pages_kernel(
    const uint4* __restrict__ src_k, const uint4* __restrict__ src_v, uint4* __restrict__ dst_k,
    uint4* __restrict__ dst_v, const int64_t* __restrict__ pairs, int64_t chunks_per_block,
    int num_src_blocks, int num_dst_blocks, int32_t* device_errors) {
  constexpr int kU = 4;
  const int64_t src = pairs[2 * blockIdx.x];
  const int64_t dst = pairs[2 * blockIdx.x + 1];
  if (src < 0 || src >= num_src_blocks || dst < 0 || dst >= num_dst_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) report(device_errors, PA_DEVERR_BAD_BLOCK);
    return;
  }
  const uint4* ks = src_k + src * chunks_per_block;
  const uint4* vs = src_v + src * chunks_per_block;
  uint4* kd = dst_k + dst * chunks_per_block;
  uint4* vd = dst_v + dst * chunks_per_block;
  const int64_t step = static_cast<int64_t>(gridDim.y) * blockDim.x;
  for (int64_t i0 = blockIdx.y * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       i0 < chunks_per_block; i0 += kU * step) {
    uint4 a[kU], b[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = i0 + u * step;
      if (i < chunks_per_block) {
        a[u] = ks[i];
        b[u] = vs[i];
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = i0 + u * step;
      if (i < chunks_per_block) {
        kd[i] = a[u];
        vd[i] = b[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                               const int64_t* pairs, int num_pairs, size_t block_bytes,
                               int num_src_blocks, int num_dst_blocks, int32_t* device_errors,
                               cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t chunks = static_cast<int64_t>(block_bytes / 16);
  const int threads = 256;
  // parts per pair: about four chunks per thread per part
  int64_t parts = (chunks + 4 * threads - 1) / (4 * threads);
  if (parts < 1) parts = 1;
  if (parts > 64) parts = 64;
  dim3 grid(static_cast<unsigned>(num_pairs), static_cast<unsigned>(parts));
  swap_pages_kernel<<<grid, threads, 0, stream>>>(
      static_cast<const uint4*>(src_k), static_cast<const uint4*>(src_v),
      static_cast<uint4*>(dst_k), static_cast<uint4*>(dst_v), pairs, chunks, num_src_blocks,
      num_dst_blocks, device_errors);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int num_tokens,
                                     int num_kv_heads, int row_bytes, int block_size,
                                     int num_blocks, int32_t* device_errors,
                                     cudaStream_t stream) {
  const int chunks_per_row = row_bytes / 16;
  const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * chunks_per_row;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 65535) blocks = 65535;
  reshape_and_cache_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), slot_mapping, num_tokens, num_kv_heads, chunks_per_row,
      block_size, static_cast<int64_t>(num_blocks) * block_size, device_errors);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache_fp8(const void* k, const void* v, void* k_cache,
                                         void* v_cache, const int64_t* slot_mapping,
                                         const float* k_scale, const float* v_scale,
                                         int num_tokens, int num_kv_heads, int head_dim,
                                         int block_size, int num_blocks, int32_t* device_errors,
                                         cudaStream_t stream) {
  const int groups_per_row = head_dim / 8;
  const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * groups_per_row;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 65535) blocks = 65535;
  reshape_and_cache_fp8_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint2*>(k_cache),
      static_cast<uint2*>(v_cache), slot_mapping, k_scale, v_scale, num_tokens, num_kv_heads,
      groups_per_row, block_size, static_cast<int64_t>(num_blocks) * block_size, device_errors);
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int num_pairs,
                               size_t block_bytes, int num_blocks, int32_t* device_errors,
                               cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t chunks = static_cast<int64_t>(block_bytes / 16);
  const int threads = 256;
  // enough parts per pair that a page moves in one or two passes of the block
  int64_t parts = (chunks + 2 * threads - 1) / (2 * threads);
  if (parts < 1) parts = 1;
  if (parts > 64) parts = 64;
  dim3 grid(static_cast<unsigned>(num_pairs), static_cast<unsigned>(parts));
  copy_blocks_kernel<<<grid, threads, 0, stream>>>(static_cast<uint4*>(k_cache),
                                                   static_cast<uint4*>(v_cache), pairs, chunks,
                                                   num_blocks, device_errors);
  return cudaGetLastError();
}

}  // namespace pa
