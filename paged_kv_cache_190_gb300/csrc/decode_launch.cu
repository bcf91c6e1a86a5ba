// Orchestration of one pa_decode call: plan kernel -> persistent decode kernel
// -> split-K merge kernel, all on the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>

#include "decode_instances.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kPlanThreads = 1024;          // the plan's largest block
constexpr int kQPrepWarps = 8;

// q preparation of the fp8-cache decode (head_dim 128): each bf16 row q[b][i]
// is scaled by the power of two 2^e that brings its largest magnitude into
// [128, 256) and split into e4m3 hi = e4m3(x 2^e) and lo = e4m3(x 2^e - hi)
// (nearest, saturating).  Output row (272 bytes): hi codes [128], lo codes
// [128], 2^-e as float32, 12 bytes of padding.  One warp per row, four
// columns per lane.
__global__ void __launch_bounds__(kQPrepWarps * 32) q_prep_fp8_kernel(
    const uint2* __restrict__ q, unsigned char* __restrict__ q8, int64_t rows) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kQPrepWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const uint2 w = q[row * 32 + lane];
  float x[4] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y)};
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu);
  const int se = min(max(134 - e, -126), 126);            // amax 2^se in [128, 256)
  const float up = __uint_as_float(static_cast<uint32_t>(se + 127) << 23);
  uint32_t hi = 0, lo = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float2 v = make_float2(x[2 * j] * up, x[2 * j + 1] * up);
    const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
    const float2 back = __half22float2(static_cast<__half2>(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3)));
    const float2 r = make_float2(v.x - back.x, v.y - back.y);
    const __nv_fp8x2_storage_t l = __nv_cvt_float2_to_fp8x2(r, __NV_SATFINITE, __NV_E4M3);
    hi |= static_cast<uint32_t>(h) << (16 * j);
    lo |= static_cast<uint32_t>(l) << (16 * j);
  }
  unsigned char* dst = q8 + row * 272;
  reinterpret_cast<uint32_t*>(dst)[lane] = hi;
  reinterpret_cast<uint32_t*>(dst + 128)[lane] = lo;
  if (lane < 4)
    reinterpret_cast<float*>(dst + 256)[lane] =
        lane == 0 ? __uint_as_float(static_cast<uint32_t>(127 - se) << 23) : 0.f;
}

// Lists every (sequence, chunk) pair in sequence order, records where each
// sequence's chunks start, resets the work counter and writes zero rows for
// empty sequences.  One block of THREADS (the smallest of 128 .. 1024 that
// covers the batch: its barriers and scans cost less with fewer warps);
// sequences are taken THREADS at a time: a block scan gives each sequence's
// first chunk, then all threads fill the tile's entries together (entry ->
// sequence by binary search over the tile's offsets).
template <int THREADS>
__global__ void __launch_bounds__(THREADS) decode_plan_kernel(
    const int32_t* __restrict__ context_lens, int num_seqs, int chunk_tokens, int max_len,
    int q_len, int32_t* __restrict__ header, int32_t* __restrict__ chunk_base,
    int4* __restrict__ work, uint4* __restrict__ out, int64_t row_chunks,
    int32_t* device_errors) {
  constexpr int NW = THREADS / 32;
  __shared__ int warp_sums[NW];
  __shared__ int first_s[THREADS + 1];          // tile-local exclusive offsets (+ total)
  __shared__ int len_s[THREADS];
  __shared__ int carry_s;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  allow_next_grid();                      // the decode kernel may start its prologue
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < num_seqs; base += THREADS) {
    const int b = base + threadIdx.x;
    int L = 0, n = 0;
    if (b < num_seqs) {
      L = context_lens[b];
      if (L < 0 || L > max_len) {
        report(device_errors, PA_DEVERR_BAD_LENGTH);
        L = L < 0 ? 0 : max_len;
      }
      // fewer tokens than new tokens: the first new tokens see no key (zero rows)
      if (L > 0 && L < q_len) report(device_errors, PA_DEVERR_BAD_LENGTH);
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
      int w = lane < NW ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < NW) warp_sums[lane] = w;
    }
    __syncthreads();
    const int excl = x - n + (warp > 0 ? warp_sums[warp - 1] : 0);
    const int carry = carry_s;
    first_s[threadIdx.x] = excl;
    len_s[threadIdx.x] = L;
    if (threadIdx.x == THREADS - 1) first_s[THREADS] = excl + n;
    if (b < num_seqs) {
      chunk_base[b] = carry + excl;
      if (L == 0)
        for (int64_t k = 0; k < row_chunks; ++k) out[b * row_chunks + k] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    const int tile_total = first_s[THREADS];
    for (int e = threadIdx.x; e < tile_total; e += THREADS) {
      int lo = 0, hi = THREADS - 1;          // last t with first_s[t] <= e
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (first_s[mid] <= e) lo = mid; else hi = mid - 1;
      }
      const int single = len_s[lo] <= chunk_tokens ? kSingleChunk : 0;
      work[carry + e] =
          make_int4(base + lo, (e - first_s[lo]) * chunk_tokens, len_s[lo], (carry + e) | single);
    }
    __syncthreads();
    if (threadIdx.x == 0) carry_s = carry + tile_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    chunk_base[num_seqs] = carry_s;
    header[0] = 0;
    header[1] = carry_s;
  }
}

constexpr int kMergeWarps = 8;

// Partials a sequence can have: its chunks, plus (cascade) its prefix chunks.
int64_t cascade_parts_per_seq(int max_context_len, int chunk_tokens, bool cascade) {
  if (max_context_len <= 0) return 0;
  const int64_t L = max_context_len;
  return (L + chunk_tokens - 1) / chunk_tokens + (cascade ? kMaxPrefixPieces : 0);
}
constexpr int kWideMergeWarps = 16;

// Running log-sum-exp state of one output row over some chunks (base 2):
//   M = max lse_c, S = sum 2^(lse_c - M), acc = sum 2^(lse_c - M) o_c.
template <int CPL>
struct LseAcc {
  // M starts finite and below any real log-sum-exp, so that a chunk in which
  // the row saw no token (lse = -inf) adds weight 2^-inf = 0 instead of NaN
  float M = -3.0e38f, S = 0.f, acc[CPL] = {};

  __device__ __forceinline__ void add(float lse, const float* v) {
    const float Mn = fmaxf(M, lse);
    const float sc = fast_exp2(M - Mn);     // 0 on the first real chunk
    const float w = fast_exp2(lse - Mn);
    S = fmaf(S, sc, w);
#pragma unroll
    for (int k = 0; k < CPL; ++k) acc[k] = fmaf(acc[k], sc, w * v[k]);
    M = Mn;
  }
};

template <int CPL>
__device__ __forceinline__ void load_cols(const float* p, float* v) {
  if constexpr (CPL == 4) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x; v[1] = t.y;
  }
}

template <bool BF16, int CPL>
__device__ __forceinline__ void store_row(void* out, int64_t o, const float* r) {
  if constexpr (BF16) {
    const uint32_t w0 = f32_to_bf16_bits(r[0]) | (f32_to_bf16_bits(r[1]) << 16);
    if constexpr (CPL == 4) {
      const uint32_t w1 = f32_to_bf16_bits(r[2]) | (f32_to_bf16_bits(r[3]) << 16);
      *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(out) + o) = make_uint2(w0, w1);
    } else {
      *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(out) + o) = w0;
    }
  } else {
    float* dst = reinterpret_cast<float*>(out) + o;
#pragma unroll
    for (int k = 0; k < CPL; ++k) dst[k] = r[k];
  }
}

// Split-K merge (log-sum-exp): for sequence b, query head i with n >= 2 chunks,
//   out = sum_c 2^(lse_c - M) o_c / sum_c 2^(lse_c - M),  M = max_c lse_c,
// where o_c is chunk c's normalised output and lse_c its base-2 log-sum-exp.
// One warp per (b, i) row, each lane owning head_dim / 32 columns; one pass with
// a running maximum, so every chunk's loads can be in flight together.
template <bool BF16, int CPL>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(
    const int32_t* __restrict__ chunk_base, const float* __restrict__ part_lse,
    const float* __restrict__ part_out, void* __restrict__ out, int num_q_heads, int64_t rows) {
  constexpr int D = CPL * 32;
  wait_prior_grids();                     // the decode kernel's partials
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int b = static_cast<int>(row / num_q_heads);
  const int i = static_cast<int>(row - static_cast<int64_t>(b) * num_q_heads);
  const int c0 = chunk_base[b];
  const int n = chunk_base[b + 1] - c0;
  if (n < 2) return;                      // one chunk: the decode kernel wrote the row
  const int64_t prow0 = static_cast<int64_t>(c0) * num_q_heads + i;
  LseAcc<CPL> st;
#pragma unroll 8
  for (int c = 0; c < n; ++c) {
    const int64_t prow = prow0 + static_cast<int64_t>(c) * num_q_heads;
    float v[CPL];
    load_cols<CPL>(part_out + prow * D + lane * CPL, v);
    st.add(part_lse[prow], v);
  }
  float r[CPL];
  const float inv = st.S > 0.f ? 1.f / st.S : 0.f;   // 0: the row saw no token
#pragma unroll
  for (int k = 0; k < CPL; ++k) r[k] = st.acc[k] * inv;
  store_row<BF16, CPL>(out, row * D + lane * CPL, r);
}

// The same merge for long chunk lists: one block per (b, i) row; its 16 warps
// take chunks c = warp, warp + 16, ... and their states are combined in
// shared memory.
template <bool BF16, int CPL>
__global__ void __launch_bounds__(kWideMergeWarps * 32) decode_merge_wide_kernel(
    const int32_t* __restrict__ chunk_base, const float* __restrict__ part_lse,
    const float* __restrict__ part_out, void* __restrict__ out, int num_q_heads) {
  constexpr int D = CPL * 32;
  __shared__ float sM[kWideMergeWarps], sS[kWideMergeWarps];
  __shared__ float sacc[kWideMergeWarps][D];
  wait_prior_grids();                     // the decode kernel's partials
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t row = blockIdx.x;
  const int b = static_cast<int>(row / num_q_heads);
  const int i = static_cast<int>(row - static_cast<int64_t>(b) * num_q_heads);
  const int c0 = chunk_base[b];
  const int n = chunk_base[b + 1] - c0;
  if (n < 2) return;                      // uniform over the block
  const int64_t prow0 = static_cast<int64_t>(c0) * num_q_heads + i;
  LseAcc<CPL> st;
#pragma unroll 8
  for (int c = warp; c < n; c += kWideMergeWarps) {
    const int64_t prow = prow0 + static_cast<int64_t>(c) * num_q_heads;
    float v[CPL];
    load_cols<CPL>(part_out + prow * D + lane * CPL, v);
    st.add(part_lse[prow], v);
  }
#pragma unroll
  for (int k = 0; k < CPL; ++k) sacc[warp][lane * CPL + k] = st.acc[k];
  if (lane == 0) {
    sM[warp] = st.M;
    sS[warp] = st.S;
  }
  __syncthreads();
  if (warp != 0) return;
  float M = -3.0e38f;
#pragma unroll
  for (int w = 0; w < kWideMergeWarps; ++w) M = fmaxf(M, sM[w]);
  float S = 0.f, r[CPL] = {};
#pragma unroll
  for (int w = 0; w < kWideMergeWarps; ++w) {
    const float f = fast_exp2(sM[w] - M);   // warps without chunks: S = 0, acc = 0
    S = fmaf(f, sS[w], S);
#pragma unroll
    for (int k = 0; k < CPL; ++k) r[k] = fmaf(f, sacc[w][lane * CPL + k], r[k]);
  }
  const float inv = S > 0.f ? 1.f / S : 0.f;
#pragma unroll
  for (int k = 0; k < CPL; ++k) r[k] *= inv;
  store_row<BF16, CPL>(out, row * D + lane * CPL, r);
}

// Launch as a programmatic dependent of the decode kernel (its blocks wait for
// the decode kernel on the device), which hides the launch gap.
template <typename... Args>
cudaError_t launch_dependent(void (*kernel)(Args...), unsigned blocks, unsigned threads,
                             cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <bool BF16, int CPL>
cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t stream) {
  const int rows_q = a.q_len * a.num_q_heads;         // query rows per sequence
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * rows_q;
  const int64_t max_chunks_per_seq = cascade_parts_per_seq(a.max_context_len, a.chunk_tokens,
                                                           false);
  if (max_chunks_per_seq >= 32)
    return launch_dependent(decode_merge_wide_kernel<BF16, CPL>, static_cast<unsigned>(rows),
                            kWideMergeWarps * 32, stream,
                            static_cast<const int32_t*>(a.ws.chunk_base),
                            static_cast<const float*>(a.ws.part_lse),
                            static_cast<const float*>(a.ws.part_out), a.out, rows_q);
  const unsigned blocks = static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps);
  return launch_dependent(decode_merge_kernel<BF16, CPL>, blocks, kMergeWarps * 32, stream,
                          static_cast<const int32_t*>(a.ws.chunk_base),
                          static_cast<const float*>(a.ws.part_lse),
                          static_cast<const float*>(a.ws.part_out), a.out, rows_q, rows);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// View of a K or V pool (rows = blocks * kv heads * block size, bf16 or byte
// (e4m3) elements) for copies of box_rows whole rows with 128-byte swizzle: 2-D
// {128 bytes, rows} when a row is 128 bytes; otherwise 3-D {128 bytes, rows,
// 128-byte slabs of a row}, so that one box takes every slab of the rows and
// lands them slab after slab (the layout the consumers read).
cudaError_t make_pool_map(CUtensorMap* map, const void* pool, int head_dim, int64_t rows,
                          int elt, int box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  if (rows <= 0 || rows > INT_MAX) return cudaErrorInvalidValue;
  const int row_bytes = head_dim * elt;
  if (row_bytes % 128 != 0) return cudaErrorInvalidValue;
  const cuuint32_t slabs = static_cast<cuuint32_t>(row_bytes / 128);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(128 / elt), static_cast<cuuint64_t>(rows), slabs};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), 128};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elt), static_cast<cuuint32_t>(box_rows), slabs};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUtensorMapDataType type =
      elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUresult r = encode(map, type, slabs == 1 ? 2 : 3, const_cast<void*>(pool), dims,
                            strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t make_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides, const uint32_t* box) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  if (rank < 1 || rank > 5) return cudaErrorInvalidValue;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                            const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

WorkspaceLayout decode_workspace_layout(int num_seqs, int num_q_heads, int head_dim,
                                        int max_context_len, int chunk_tokens, int num_groups) {
  WorkspaceLayout w{};
  const int64_t per_seq = cascade_parts_per_seq(max_context_len, chunk_tokens, num_groups > 0);
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
  w.q8 = off;                             // the fp8-cache path's prepared q rows
  off += align256(static_cast<size_t>(num_seqs) * num_q_heads * (2 * head_dim + 16));
  w.prefix_parts = off;                   // the cascade's per-sequence prefix partials
  w.prefix_items = off;
  w.inline_start = off;
  if (num_groups > 0) {
    off += align256(static_cast<size_t>(num_seqs) * 4);
    w.prefix_items = off;                 // (group, row set, piece, span) items
    // row sets: one per group plus one per 64 rows (8 query heads per kv head at most)
    const int64_t rowsets = num_groups + (static_cast<int64_t>(num_seqs) * 8 + 63) / 64;
    off += align256(static_cast<size_t>(rowsets) * kMaxPrefixPieces * 16);
    w.inline_start = off;
    off += align256(static_cast<size_t>(num_seqs) * 4);
  }
  w.total = off;
  return w;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  const int elt = a.bf16 ? 2 : 4;
  const int rows_q = a.q_len * a.num_q_heads;         // query rows per sequence
  if (a.kv8) {
    const int64_t rows = static_cast<int64_t>(a.num_seqs) * rows_q;
    q_prep_fp8_kernel<<<static_cast<unsigned>((rows + kQPrepWarps - 1) / kQPrepWarps),
                        kQPrepWarps * 32, 0, stream>>>(static_cast<const uint2*>(a.q), a.ws.q8,
                                                       rows);
    const cudaError_t qe = cudaGetLastError();
    if (qe != cudaSuccess) return qe;
  }
  const bool cascade = a.num_groups > 0;
  const int64_t row_chunks = static_cast<int64_t>(rows_q) * a.head_dim * elt / 16;
  cudaError_t e;
  if (cascade) {
    e = launch_cascade_plan(a, stream);
  } else {
    auto run = [&](auto kernel, int threads) {
      kernel<<<1, threads, 0, stream>>>(a.context_lens, a.num_seqs, a.chunk_tokens,
                                        a.max_context_len, a.q_len, a.ws.header, a.ws.chunk_base,
                                        a.ws.work, static_cast<uint4*>(a.out), row_chunks,
                                        a.device_errors);
    };
    if (a.num_seqs <= 128) run(decode_plan_kernel<128>, 128);
    else if (a.num_seqs <= 256) run(decode_plan_kernel<256>, 256);
    else if (a.num_seqs <= 512) run(decode_plan_kernel<512>, 512);
    else run(decode_plan_kernel<kPlanThreads>, kPlanThreads);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  if (a.ws.max_chunks == 0) return cudaSuccess;  // every length is zero

  DecodeKernelParams kp;
  std::memset(&kp, 0, sizeof(kp));
  const int group = a.num_q_heads / a.num_kv_heads;
  // fp8 pools with 16-token pages: items over kv-head pairs, so that one copy
  // takes both heads' rows of a page (4 KiB instead of two of 2 KiB)
  const bool paired = a.kv8 && a.block_size == 16 && a.q_len == 1 && a.num_kv_heads % 2 == 0 &&
                      group <= 4;
  const int rows = (paired ? 2 : 1) * a.q_len * group;   // rows per item
  // the kernel instance is chosen by the rows of an item, and so is its consumer
  // (the cascade's prefix kernel reads through the maps too)
  if (a.kv8 || cascade || decode_uses_tensor_cores(a.bf16 != 0, rows)) {
    const int64_t rows = static_cast<int64_t>(a.num_blocks) * a.num_kv_heads * a.block_size;
    const int kv_elt = a.kv8 ? 1 : 2;
    // one box per page a unit touches: min(page, unit) rows
    const int unit_tokens =
        a.kv8 ? DecodeTraits<true, 128, 4, true>::UT : DecodeTraits<true, 128, 4, false>::UT;
    const int box_rows = paired ? 2 * a.block_size
                                : (a.block_size < unit_tokens ? a.block_size : unit_tokens);
    e = make_pool_map(&kp.tmap_k, a.k_cache, a.head_dim, rows, kv_elt, box_rows);
    if (e == cudaSuccess)
      e = make_pool_map(&kp.tmap_v, a.v_cache, a.head_dim, rows, kv_elt, box_rows);
    if (e != cudaSuccess) return e;
  }
  kp.out = a.out;
  kp.q = a.kv8 ? reinterpret_cast<const char*>(a.ws.q8) : static_cast<const char*>(a.q);
  kp.k_cache = static_cast<const char*>(a.k_cache);
  kp.v_cache = static_cast<const char*>(a.v_cache);
  kp.block_tables = a.block_tables;
  kp.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  kp.num_q_heads = a.num_q_heads;
  kp.num_kv_heads = paired ? a.num_kv_heads / 2 : a.num_kv_heads;   // item heads
  kp.pool_heads = a.num_kv_heads;
  kp.head_pairs = paired ? 1 : 0;
  kp.pair_shift = group >= 4 ? 2 : (group >= 2 ? 1 : 0);
  kp.block_size = a.block_size;
  kp.num_blocks = a.num_blocks;
  kp.max_blocks_per_seq = a.max_blocks_per_seq;
  kp.chunk_tokens = a.chunk_tokens;
  kp.header = a.ws.header;
  kp.work = a.ws.work;
  kp.part_lse = a.ws.part_lse;
  kp.part_out = a.ws.part_out;
  kp.device_errors = a.device_errors;
  kp.wait_limit = a.wait_limit < 0 ? kMaxPolls : static_cast<uint32_t>(a.wait_limit);
  kp.k_scale = a.k_scale;
  kp.v_scale = a.v_scale;
  kp.q_len = a.q_len;
  const int item_group = paired ? 2 * group : group;   // query heads of an item
  kp.group = item_group;
  kp.group_log2 = item_group >= 8 ? 3 : (item_group >= 4 ? 2 : (item_group >= 2 ? 1 : 0));
  const int64_t items_upper = a.ws.max_chunks * kp.num_kv_heads;
  const int grid = static_cast<int>(items_upper < a.num_sms ? items_upper : a.num_sms);
  int device = 0;
  e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  e = a.kv8    ? run_decode_fp8(a.head_dim, rows, kp, grid, device, stream)
      : a.bf16 ? run_decode_bf16(a.head_dim, rows, kp, grid, device, stream)
               : run_decode_f32(a.head_dim, rows, kp, grid, device, stream);
  if (e != cudaSuccess) return e;
  if (cascade) {
    // after the decode kernel over the sequences' long own suffixes (often none,
    // and then it ends right after the plan) come the shared prefixes and the
    // merge, which also attends to the short suffixes; each launch is a
    // programmatic dependent of the one before
    e = launch_cascade_prefix(a, kp, device, stream);
    if (e != cudaSuccess) return e;
    return launch_cascade_merge(a, kp, stream);
  }
  if (a.max_context_len > a.chunk_tokens) {
    if (a.bf16 && a.head_dim == 128) e = launch_merge<true, 4>(a, stream);
    else if (a.bf16) e = launch_merge<true, 2>(a, stream);
    else if (a.head_dim == 128) e = launch_merge<false, 4>(a, stream);
    else e = launch_merge<false, 2>(a, stream);
  }
  return e;
}

}  // namespace pa
