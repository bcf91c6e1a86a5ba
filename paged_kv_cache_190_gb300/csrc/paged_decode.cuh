// Paged decode attention for sm_103a: a persistent, warp-specialised kernel.
//
// What it computes ("PagedAttention原理" §3.4: paging leaves the attention
// mathematics unchanged; "PagedAttentionMetal", "注意力计算优化": look the
// physical page up in the block table, stage the K/V block in shared memory,
// batch variable lengths without padding): for each sequence b and query head
// i, softmax(scale * q K^T) V over the sequence's L_b tokens, read page by page
// through block_tables[b].
//
// How (GB300 design, not a translation of any page's kernel):
//   * Work item = (sequence, kv head, chunk of `chunk_tokens` tokens).  A tiny
//     plan kernel lists the (sequence, chunk) pairs; items are handed out by an
//     atomic counter, so lognormal lengths balance across SMs.
//   * One CTA per SM, persistent.  Behind the consumer warps come the producer,
//     the scheduler and the merger.  The scheduler claims items and
//     resolves them (work entry, block-table slice) into shared item slots and
//     starts the copy of each item's q rows.  The producer warp: lane
//     w streams the K and V tiles of consumer warp w's units into that warp's
//     ring of stages (mbarrier-guarded), with blocking waits of its own, so the
//     lanes advance independently and several copies are in issue at once (a
//     single issuing thread cannot keep HBM busy).  Tiles move with
//     cp.async.bulk (one contiguous run per tile) for the CUDA-core consumer,
//     or with cp.async.bulk.tensor through a tensor map with 128-byte swizzle
//     (so that ldmatrix reads them without bank conflicts) for the tensor-core
//     consumers: one box per page touched and pool, taking every 128-byte slab
//     of its rows (a 3-D box when a row is wider than 128 bytes) -- the number
//     of copies per byte, not their size, limits one issuing warp.
//   * The other warps consume.  Unit u (16 tokens; 32 for e4m3 pools) of item i
//     goes to warp (u + i) % CW, through that warp's own ring of S / CW stages
//     (stage w + CW k).  The split of an item between warps is therefore a
//     function of the item alone, which makes the result bit-reproducible
//     whatever CTA runs it.  Each warp keeps an online-softmax state (running
//     max m, sum l, accumulator) in fp32 registers for every query head of the
//     GQA group -- one K/V read serves the whole group.  Three consumers:
//       - CUDA cores (fp32 inputs, and bf16 with one query head per kv head):
//         QK with 8 lanes per token and a butterfly reduction, PV with each
//         lane owning head_dim / 32 output columns;
//       - tensor cores, bf16 (2..8 query heads per kv head): mma.sync
//         m16n8k16 with the group's q rows as the A operand (rows past the
//         group are zero), K through ldmatrix, P re-packed from the score
//         fragments as the next B operand, V through ldmatrix.trans;
//       - tensor cores, float8 e4m3 pools (any group): mma.sync m16n8k32 with
//         e4m3 operands, so the stored codes enter the products unconverted
//         (see Fp8TensorConsumer).
//   * At the end of an item the consumer warps hand their partial states to
//     the merge warp through shared memory and go on with their next item; it
//     merges them (log-sum-exp) and writes the item's rows either straight to
//     `out` (single-chunk sequence) or as a normalised partial plus its base-2
//     log-sum-exp for the split-K merge kernel.
//   * Every wait is bounded; on expiry the kernel reports PA_DEVERR_TIMEOUT,
//     drains its own copies in flight and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kConsumerWarps = 8;    // consumer warps (the bf16 8-row kernel: 6)
constexpr int kItemSlots = 8;        // items the producer may run ahead
constexpr int kUnitsAhead = 32;      // claimed-but-unissued units a CTA may hold
constexpr int kSmemBudget = 227 * 1024;
constexpr unsigned kFull = 0xffffffffu;
// Start of every running maximum: finite, below any real logit, so that a row
// with no visible token yet (the first new tokens of a step, in a chunk past
// them) keeps alpha = 2^0 and probabilities 2^-inf = 0 instead of NaN.
constexpr float kNoScore = -3.0e38f;

struct ItemDesc {
  int b, h, tok0, len, gchunk, n_units, n_tokens, single, rot;
};

// Work entry of a (sequence, chunk): {sequence, first token of the chunk, sequence
// length, global chunk index | kSingleChunk when the sequence is this one chunk
// (its rows go straight to `out`)}.
constexpr int kSingleChunk = 1 << 30;

// Tensor-core consumer: bf16 with a group of 2..8 query heads per kv head.
constexpr bool decode_uses_tensor_cores(bool bf16, int group) { return bf16 && group >= 2; }

// BF16: q, out (and the caches unless KV8) are bf16, else fp32.  KV8: the
// caches hold float8 e4m3 codes with a scale per kv head (q and out bf16).
template <bool BF16, int D, int G, bool KV8 = false>
struct DecodeTraits {
  static_assert(!KV8 || BF16, "fp8 caches pair with bf16 q and out");
  static constexpr int D_ = D;
  static constexpr int G_ = G;
  static constexpr bool KV8_ = KV8;
  static constexpr bool TC = KV8 || decode_uses_tensor_cores(BF16, G);
  // Consumer warps: 8, which with the producer, the scheduler and the merger
  // puts three warps on three of the SM's four sub-partitions and so caps a
  // thread at 168 registers; every consumer fits that without spilling (the fp8 one too:
  // 8 warps against 6 measured 206 -> 187 us on the 128K workload, 212 -> 193
  // on MHA).  The 8-row kernels have 7: their per-warp merge buffers (rows x
  // head_dim floats each) are half their shared memory's fixed part, and with
  // 7 warps 21 stages fit instead of 16 (GQA fp8 162.6 -> 160.0 us; 2 draft
  // tokens x GQA-4 248.0 -> 244.7 us against 6 warps and 18 stages).  The fp32
  // one keeps 6 (its q rows take 128 registers).
  static constexpr int CW = G == 8 ? (BF16 ? 7 : 6) : kConsumerWarps;
  // + producer + scheduler + merger
  static constexpr int THREADS = (CW + 3) * 32;
  static constexpr int ELT = KV8 ? 1 : (BF16 ? 2 : 4);         // cache element bytes
  static constexpr int QELT = BF16 ? 2 : 4;                    // q element bytes
  static constexpr int ROW_BYTES = D * ELT;                    // one cache row
  // one q row; fp8 caches: the row prepared as e4m3 hi and lo parts plus its
  // inverse scale (see Fp8TensorConsumer)
  static constexpr int QROW_BYTES = KV8 ? 2 * D + 16 : D * QELT;
  static constexpr int BOX_COLS = 128 / ELT;                   // elements per 128-byte box row
  static constexpr int UT = KV8 ? 32 : (ROW_BYTES >= 512 ? 8 : 16);   // tokens per stage
  static constexpr int BOXES = ROW_BYTES / 128;                // 128-byte tensor-map boxes per row
  static constexpr int BOX_BYTES = UT * 128;
  static constexpr int TILE_BYTES = UT * ROW_BYTES;            // K (or V) of one stage
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int Q_BYTES = G * QROW_BYTES;
  static constexpr int CE = 16 / ELT;                          // elements per 16-byte chunk
  static constexpr int CPR = ROW_BYTES / 16;                   // chunks per row
  static constexpr int NCH = CPR / 8;                          // chunks per lane in QK
  static constexpr int EPL = NCH * CE;                         // elements per lane in QK
  static constexpr int CPL = D / 32;                           // PV columns per lane
  static constexpr int P = UT / 4;                             // QK passes per stage
  static constexpr int N = P * G;                              // dot products per lane
  static constexpr int RC = N >= 8 ? N / 8 : 1;                // sums per lane after reduction
  // butterfly levels that split the values (the rest only add): lane bits
  // below 3 - LV hold duplicates
  static constexpr int LV = N >= 8 ? 3 : (N >= 4 ? 2 : 1);
  static constexpr int DUP_MASK_END = 1 << (3 - LV);
  static_assert(CPR % 8 == 0, "head row must split into 8 lanes of 16-byte chunks");
  static_assert(D % 32 == 0, "head_dim must split over 32 lanes");

  // shared memory carve-up (bytes)
  static constexpr int MERGE_ACC = CW * G * D * 4;
  static constexpr int MERGE_ML = CW * G * 2 * 4;
  static constexpr int PS = TC ? 0 : CW * UT * G * 4;   // CUDA-core probabilities
  static constexpr int QBUF = kItemSlots * Q_BYTES;
  static constexpr int DESC = kItemSlots * static_cast<int>(sizeof(ItemDesc));
  static constexpr int TBL = kItemSlots * kItemPages * 4;      // block-table slice per item
  static constexpr int FIXED = MERGE_ACC + MERGE_ML + PS + QBUF + DESC + TBL + 64 /*flags*/ +
                               (3 * kItemSlots + 4) * 8 + 1024 /*alignment slack*/;
  static constexpr int S_RAW = (kSmemBudget - FIXED) / (STAGE_BYTES + 2 * 8 + 4);
  static constexpr int S_CAP_MAX = STAGE_BYTES <= 4096 ? 48 : 32;
  static constexpr int S_CAP = S_RAW > S_CAP_MAX ? S_CAP_MAX : S_RAW;
  static constexpr int S = (S_CAP / CW) * CW;
  static_assert(!TC || (UT % 16 == 0 && STAGE_BYTES % 1024 == 0),
                "swizzled stages need 1 KiB alignment");
  static constexpr int SPW = S / CW;               // stages per consumer warp
  static_assert(S >= CW, "at least one stage per consumer warp");

  static constexpr int OFF_STAGES = 0;
  static constexpr int OFF_QBUF = OFF_STAGES + S * STAGE_BYTES;
  static constexpr int OFF_MACC = OFF_QBUF + QBUF;
  static constexpr int OFF_MML = OFF_MACC + MERGE_ACC;
  static constexpr int OFF_PS = OFF_MML + MERGE_ML;
  static constexpr int OFF_DESC = OFF_PS + PS;
  static constexpr int OFF_TBL = OFF_DESC + DESC;
  static constexpr int OFF_SFLAG = OFF_TBL + TBL;
  // abort flag, a spare word, units issued per producer lane [8]
  static constexpr int OFF_ABORT = OFF_SFLAG + S * 4;
  static constexpr int OFF_BARS = ((OFF_ABORT + 8 + 4 * kConsumerWarps + 7) / 8) * 8;
  // barriers: full[S], empty[S], item_full[NI], item_empty[NI], sched_full[NI], merge_free,
  // merge_full
  static constexpr int NUM_BARS = 2 * S + 3 * kItemSlots + 2;
  static constexpr int SMEM_BYTES = OFF_BARS + NUM_BARS * 8;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;        // room to align the base to 1 KiB
  static_assert(SMEM_ALLOC <= kSmemBudget, "shared memory over budget");
};

struct DecodeKernelParams {
  CUtensorMap tmap_k;               // 2-D views [rows = NB*Hkv*bs][head_dim] of the pools
  CUtensorMap tmap_v;               // (tensor-core consumer only)
  void* out;
  const char* q;
  const char* k_cache;
  const char* v_cache;
  const int32_t* block_tables;
  float scale_log2;                 // scale * log2(e): logits are kept in base 2
  int num_q_heads, num_kv_heads, block_size, num_blocks, max_blocks_per_seq, chunk_tokens;
  int32_t* header;                  // [0] item counter, [1] total chunks
  const int4* work;
  float* part_lse;
  float* part_out;
  int32_t* device_errors;
  uint32_t wait_limit;              // polls before a pipeline wait gives up (drains use kMaxPolls)
  const float* k_scale;             // fp8 caches: dequantisation scale per kv head
  const float* v_scale;
  // new tokens per sequence (causal among themselves) and the query heads per kv
  // head (a power of two, as log2): an item's G rows are (token j, head g) =
  // row j * group + g
  int q_len, group, group_log2;
  // fp8 pools with 16-token pages: items over kv-head pairs (head_pairs = 1).
  // num_kv_heads and group then count pairs and the pair's query rows; a stage
  // holds 16 positions of both heads (one 32-row box per pool: the two heads'
  // rows of a page are adjacent), and row g belongs to head 2 h + (g >> pair_shift).
  int head_pairs, pair_shift;
  int pool_heads;                   // kv heads of the pools (the row stride of a page)
};

// Butterfly step over lane bit `mask` (within 8-lane groups): lanes with the
// bit set keep the upper half of the values, the others the lower half, and each
// adds its partner's copy of the half it keeps.
template <int COUNT>
__device__ __forceinline__ void butterfly_level(float* v, int lane, int mask) {
  if constexpr (COUNT >= 2) {
    constexpr int H = COUNT / 2;
    const bool upper = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < H; ++i) {
      const float send = upper ? v[i] : v[i + H];
      const float keep = upper ? v[i + H] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, mask);
    }
  } else {
    v[0] += __shfl_xor_sync(kFull, v[0], mask);
  }
}

template <typename Tr>
__device__ __forceinline__ void unpack_chunk(const uint4& c, float* dst) {
  if constexpr (Tr::ELT == 2) {
    dst[0] = bf16_lo(c.x); dst[1] = bf16_hi(c.x);
    dst[2] = bf16_lo(c.y); dst[3] = bf16_hi(c.y);
    dst[4] = bf16_lo(c.z); dst[5] = bf16_hi(c.z);
    dst[6] = bf16_lo(c.w); dst[7] = bf16_hi(c.w);
  } else {
    dst[0] = __uint_as_float(c.x); dst[1] = __uint_as_float(c.y);
    dst[2] = __uint_as_float(c.z); dst[3] = __uint_as_float(c.w);
  }
}

// Load this lane's CPL value columns of row `t` as floats.
template <typename Tr>
__device__ __forceinline__ void load_v_cols(const char* vt, int t, int lane, float* v) {
  const char* row = vt + t * Tr::ROW_BYTES + lane * Tr::CPL * Tr::ELT;
  if constexpr (Tr::ELT == 2) {
    if constexpr (Tr::CPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(row);
      v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(row);
      v[0] = bf16_lo(w); v[1] = bf16_hi(w);
    }
  } else {
    if constexpr (Tr::CPL == 4) {
      const float4 w = *reinterpret_cast<const float4*>(row);
      v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
    } else {
      const float2 w = *reinterpret_cast<const float2*>(row);
      v[0] = w.x; v[1] = w.y;
    }
  }
}

// ------------------------------------------------------------------ tensor-core helpers

// 2-D tensor-map copy of one box (rows y.., columns x..) into shared memory.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// Rows [row, row + rows) of a K or V pool into a stage tile: one tensor-map box
// of every 128-byte column slab of the rows (a 3-D box {128 B, rows, slabs}
// when a row is wider than 128 bytes: one copy lands all slabs, slab b at
// b * UT * 128 bytes).
template <typename Tr>
__device__ __forceinline__ void tma_rows(void* smem_dst, const CUtensorMap* map, int row,
                                         uint64_t* bar) {
  if constexpr (Tr::BOXES == 1)
    tma_load_2d(smem_dst, map, 0, row, bar);
  else
    tma_load_3d(smem_dst, map, 0, row, 0, bar);
}

// Byte offset of (row, 16-byte chunk) inside a tile stored as 128-byte-wide boxes
// with the tensor map's 128-byte swizzle: chunk index XOR (row mod 8).
template <typename Tr>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * Tr::BOX_BYTES + row * 128 +
                               (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A * B + D for one m16n8k16 bf16 tile with fp32 accumulation.  A rows 8..15
// (a1, a3) are zero here: the group has at most 8 query heads.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// D = A * B + D for one m16n8k16 bf16 tile, all four A registers given.
__device__ __forceinline__ void mma_bf16_full(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// ------------------------------------------------------------------ consumers
// Both consumers hold one warp's online-softmax state for the item in flight:
//   begin(q rows)  -> reset the state, load the group's q
//   unit(K, V, nt) -> fold 16 tokens (nt valid) into the state
//   store(...)     -> hand (m, l, unnormalised accumulator) to the merge

// CUDA-core consumer.  QK: 8 lanes per token (16-byte chunks contiguous within a
// quarter warp), 4 tokens per pass, butterfly reduction; PV: each lane owns
// head_dim / 32 output columns of every head.
template <typename Tr>
struct CoreConsumer {
  static constexpr int G = Tr::G_, D = Tr::D_;
  float qf[G][Tr::EPL];
  float m[G], acc[G][Tr::CPL];
  float lsum;                       // this lane's share of l[g_lane]
  int lane, j4, r, base, g_lane;
  float* ps;                        // this warp's probabilities [UT][G]

  __device__ __forceinline__ void init(int lane_, float* ps_) {
    lane = lane_;
    j4 = lane >> 3;
    r = lane & 7;
    // after the butterfly this lane holds the sums of indices base .. base+RC-1
    // (index = head * P + pass) -- all for one head, g_lane
    base = ((r >> 2) & 1) * (Tr::N / 2) + (Tr::N >= 4 ? ((r >> 1) & 1) * (Tr::N / 4) : 0) +
           (Tr::N >= 8 ? (r & 1) * (Tr::N / 8) : 0);
    g_lane = base / Tr::P;
    ps = ps_;
  }

  // new-token index of this lane's row (rows are token-major: j * group + head)
  __device__ __forceinline__ int row_token(int group_log2) const { return g_lane >> group_log2; }

  __device__ __forceinline__ void begin(const char* qs, float scale_log2, float) {
    // q scaled so that logits come out in base 2
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int c = 0; c < Tr::NCH; ++c) {
        const uint4 raw =
            *reinterpret_cast<const uint4*>(qs + g * Tr::QROW_BYTES + (r + 8 * c) * 16);
        unpack_chunk<Tr>(raw, &qf[g][c * Tr::CE]);
#pragma unroll
        for (int e = 0; e < Tr::CE; ++e) qf[g][c * Tr::CE + e] *= scale_log2;
      }
    lsum = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = kNoScore;
#pragma unroll
      for (int c = 0; c < Tr::CPL; ++c) acc[g][c] = 0.f;
    }
  }

  // qlim: the last of the unit's tokens this lane's row may see (causal among
  // the new tokens; with one new token it is never below nt - 1)
  template <typename Release>
  __device__ __forceinline__ void unit(const char* kt, const char* vt, int nt, int qlim, float,
                                       Release release) {
    // ---- scores: 8 lanes per token, 4 tokens per pass
    float part[Tr::N];
#pragma unroll
    for (int pi = 0; pi < Tr::P; ++pi) {
      const int t = 4 * pi + j4;
      float kf[Tr::EPL];
#pragma unroll
      for (int c = 0; c < Tr::NCH; ++c) {
        const uint4 raw =
            *reinterpret_cast<const uint4*>(kt + t * Tr::ROW_BYTES + (r + 8 * c) * 16);
        unpack_chunk<Tr>(raw, &kf[c * Tr::CE]);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < Tr::EPL; ++e) dot = fmaf(qf[g][e], kf[e], dot);
        part[g * Tr::P + pi] = dot;
      }
    }
    butterfly_level<Tr::N>(part, lane, 4);
    butterfly_level<(Tr::N >= 4 ? Tr::N / 2 : 1)>(part, lane, 2);
    butterfly_level<(Tr::N >= 8 ? Tr::N / 4 : 1)>(part, lane, 1);
    // part[e], e < RC: score of head g_lane, token 4 * ((base % P) + e) + j4
    float umax = -INFINITY;
    const int lim = min(nt - 1, qlim);          // last token this lane's row sees
#pragma unroll
    for (int e = 0; e < Tr::RC; ++e) {
      const int t = 4 * ((base % Tr::P) + e) + j4;
      if (t > lim) part[e] = -INFINITY;
      umax = fmaxf(umax, part[e]);
    }
    // max over the lanes that hold the same head
#pragma unroll
    for (int mask = 1; mask < 8 / G; mask <<= 1)
      umax = fmaxf(umax, __shfl_xor_sync(kFull, umax, mask));
    umax = fmaxf(umax, __shfl_xor_sync(kFull, umax, 8));
    umax = fmaxf(umax, __shfl_xor_sync(kFull, umax, 16));
    float alpha[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mu = __shfl_sync(kFull, umax, g * (8 / G));
      const float mn = fmaxf(m[g], mu);
      alpha[g] = fast_exp2(m[g] - mn);
      m[g] = mn;
    }
    float m_lane = m[0];
    float a_lane = alpha[0];
#pragma unroll
    for (int g = 1; g < G; ++g)
      if (g_lane == g) { m_lane = m[g]; a_lane = alpha[g]; }
    float psum = 0.f;
#pragma unroll
    for (int e = 0; e < Tr::RC; ++e) {
      const int t = 4 * ((base % Tr::P) + e) + j4;
      const float pr = fast_exp2(part[e] - m_lane);
      psum += pr;
      ps[t * G + g_lane] = pr;       // duplicate lanes (G == 1) store equal values
    }
    lsum = lsum * a_lane + psum;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int c = 0; c < Tr::CPL; ++c) acc[g][c] *= alpha[g];
    __syncwarp();
    // ---- values: each lane owns CPL columns of every head
    auto pv_row = [&](int t) {
      float pv[G];
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int g4 = 0; g4 < G; g4 += 4) {
          const float4 w4 = *reinterpret_cast<const float4*>(ps + t * G + g4);
          pv[g4] = w4.x; pv[g4 + 1] = w4.y; pv[g4 + 2] = w4.z; pv[g4 + 3] = w4.w;
        }
      } else if constexpr (G == 2) {
        const float2 w2 = *reinterpret_cast<const float2*>(ps + t * 2);
        pv[0] = w2.x; pv[1] = w2.y;
      } else {
        pv[0] = ps[t];
      }
      float vv[Tr::CPL];
      load_v_cols<Tr>(vt, t, lane, vv);
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int c = 0; c < Tr::CPL; ++c) acc[g][c] = fmaf(pv[g], vv[c], acc[g][c]);
    };
    if (nt == Tr::UT) {
#pragma unroll
      for (int t = 0; t < Tr::UT; ++t) pv_row(t);
    } else {
      for (int t = 0; t < nt; ++t) pv_row(t);
    }
    release();
  }

  // macc_w: this warp's [G][D] accumulator slot; mml_w: its [G][2] (m, l) slot.
  __device__ __forceinline__ void store(float* macc_w, float* mml_w) {
    // whole l for the lane's head: sum over the lanes sharing it, leaving out
    // the low lane bits that only hold duplicates
#pragma unroll
    for (int mask = Tr::DUP_MASK_END; mask < 8 / G; mask <<= 1)
      lsum += __shfl_xor_sync(kFull, lsum, mask);
    lsum += __shfl_xor_sync(kFull, lsum, 8);
    lsum += __shfl_xor_sync(kFull, lsum, 16);
    if (j4 == 0 && (r % (8 / G)) == 0) {
      float mlane = m[0];
#pragma unroll
      for (int g = 1; g < G; ++g)
        if (g_lane == g) mlane = m[g];
      mml_w[g_lane * 2 + 0] = mlane;
      mml_w[g_lane * 2 + 1] = lsum;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float* dst = macc_w + g * D + lane * Tr::CPL;
      if constexpr (Tr::CPL == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
      } else {
        *reinterpret_cast<float2*>(dst) = make_float2(acc[g][0], acc[g][1]);
      }
    }
  }
};

// Tensor-core consumer (bf16, G in 2..8), mma.sync m16n8k16 with fp32 accumulation.
//   Scores  S = Q K^T : rows = the group's query heads (rows >= G carry zero q),
//                       columns = 8 tokens per n-tile, k = head_dim.
//   Values  O^T = V^T P^T : rows = 16 head_dim columns per m-tile, columns = the
//                       heads (8 per tile; heads >= G are never stored), k = tokens.
// The score fragment of lane t (head t / 4, tokens 2 (t % 4) + {0, 1, 8, 9}) is
// exactly the B fragment P^T needs, so P never leaves registers.  The whole
// stage is read into registers first (K via ldmatrix, V^T via ldmatrix.trans)
// and handed back to the producer before the arithmetic starts.
template <typename Tr>
struct TensorConsumer {
  static constexpr int G = Tr::G_, D = Tr::D_;
  static constexpr int KS = D / 16;     // k-steps over head_dim (scores)
  static constexpr int MT = D / 16;     // m-tiles of O^T (16 head_dim columns each)
  uint32_t qa[KS][2];                   // A fragments of q (row t/4, k lo / k hi)
  float o[MT][4];                       // O^T fragments: d = 16 mt + t/4 (+8), heads 2(t%4) + {0,1}
  float m, l;                           // head t/4: running max (base 2) and this lane's sum share
  int lane;

  __device__ __forceinline__ void init(int lane_, float*) { lane = lane_; }

  __device__ __forceinline__ int row_token(int group_log2) const {
    return (lane >> 2) >> group_log2;
  }

  __device__ __forceinline__ void begin(const char* qs, float, float) {
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = 0u;
      qa[ks][1] = 0u;
      if (g < G) {
        qa[ks][0] = *reinterpret_cast<const uint32_t*>(qs + g * Tr::QROW_BYTES + (16 * ks + 2 * c) * 2);
        qa[ks][1] =
            *reinterpret_cast<const uint32_t*>(qs + g * Tr::QROW_BYTES + (16 * ks + 8 + 2 * c) * 2);
      }
    }
    m = kNoScore;
    l = 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  }

  template <typename Release>
  __device__ __forceinline__ void unit(const char* kt, const char* vt, int nt, int qlim,
                                       float scale_log2, Release release) {
    const uint32_t kb = smem_addr(kt), vb = smem_addr(vt);
    const int mi = lane >> 3, r8 = lane & 7, c = lane & 3;
    const int frow = (mi >> 1) * 8 + r8;          // token row this lane addresses
    uint32_t kf[KS][4], vf[MT][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
      ldsm_x4(kb + swz<Tr>(frow, 2 * ks + (mi & 1)), kf[ks][0], kf[ks][1], kf[ks][2], kf[ks][3]);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
      ldsm_x4_trans(vb + swz<Tr>(frow, 2 * mt + (mi & 1)), vf[mt][0], vf[mt][1], vf[mt][2],
                    vf[mt][3]);
    release();                                    // the stage's bytes are all in registers
    // ---- scores, two 8-token n-tiles
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      mma_bf16(s0, qa[ks][0], qa[ks][1], kf[ks][0], kf[ks][1]);
      mma_bf16(s1, qa[ks][0], qa[ks][1], kf[ks][2], kf[ks][3]);
    }
    // this lane's scores: head t/4, tokens 2c, 2c+1 (n-tile 0) and 8+2c, 9+2c (n-tile 1)
    float sv[4] = {s0[0], s0[1], s1[0], s1[1]};
    const int tk[4] = {2 * c, 2 * c + 1, 8 + 2 * c, 9 + 2 * c};
    const int lim = min(nt - 1, qlim);            // last token this lane's row sees
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sv[e] = tk[e] <= lim ? sv[e] * scale_log2 : -INFINITY;
      mx = fmaxf(mx, sv[e]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
    const float mn = fmaxf(m, mx);
    const float alpha = fast_exp2(m - mn);
    m = mn;
    float pr[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) pr[e] = fast_exp2(sv[e] - mn);
    l = l * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
    // P^T as the B operand: k = tokens 2c, 2c+1 (b0) and 8+2c, 9+2c (b1), n = head t/4
    const uint32_t pb0 = pack_bf16x2(pr[0], pr[1]);
    const uint32_t pb1 = pack_bf16x2(pr[2], pr[3]);
    // rescale: this lane's O^T columns are heads 2c and 2c+1 (alpha lives in lanes 4h..4h+3)
    const float a_even = __shfl_sync(kFull, alpha, 8 * c);
    const float a_odd = __shfl_sync(kFull, alpha, 8 * c + 4);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      o[mt][0] *= a_even;
      o[mt][1] *= a_odd;
      o[mt][2] *= a_even;
      o[mt][3] *= a_odd;
      mma_bf16_full(o[mt], vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3], pb0, pb1);
    }
  }

  __device__ __forceinline__ void store(float* macc_w, float* mml_w) {
    float lt = l + __shfl_xor_sync(kFull, l, 1);
    lt += __shfl_xor_sync(kFull, lt, 2);
    const int g = lane >> 2, c = lane & 3;
    if (g < G && c == 0) {
      mml_w[g * 2 + 0] = m;
      mml_w[g * 2 + 1] = lt;
    }
    const int h0 = 2 * c, h1 = 2 * c + 1;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int d0 = 16 * mt + g, d1 = d0 + 8;
      if (h0 < G) {
        macc_w[h0 * D + d0] = o[mt][0];
        macc_w[h0 * D + d1] = o[mt][2];
      }
      if (h1 < G) {
        macc_w[h1 * D + d0] = o[mt][1];
        macc_w[h1 * D + d1] = o[mt][3];
      }
    }
  }
};

// ------------------------------------------------------------ fp8 consumer
// e4m3 operands of one m16n8k32 tile, fp32 accumulation.  A: row-major 16 x 32
// (a0: row r, columns 4c..4c+3; a1: row r + 8; a2, a3: columns + 16), B:
// column-major 32 x 8 (b0: rows 4c..4c+3 of column r; b1: rows + 16), where
// r = lane / 4 and c = lane % 4; bytes in increasing column (row) order.
__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Two non-negative floats x0, x1 (< 448) as e4m3 hi + lo parts: hi = e4m3(x),
// lo = e4m3(x - hi).  hi + lo is within 2^-8 relative of x (for x above the
// subnormal range).  Returned as two codes each, x0's in the low byte.
__device__ __forceinline__ void split_e4m3x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 x = __floats2half2_rn(x0, x1);
  const __nv_fp8x2_storage_t h =
      __nv_cvt_halfraw2_to_fp8x2(static_cast<__half2_raw>(x), __NV_SATFINITE, __NV_E4M3);
  const __half2 back = static_cast<__half2>(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3));
  const __half2 r = __hsub2(x, back);
  hi = h;
  lo = __nv_cvt_halfraw2_to_fp8x2(static_cast<__half2_raw>(r), __NV_SATFINITE, __NV_E4M3);
}

// Tensor-core consumer for float8 e4m3 pools (any group 1..8), 32-token units,
// with e4m3 operands on both sides so that the stored codes enter the products
// without conversion (an e4m3 -> f16 conversion costs about ten issue slots;
// an m16n8k32 e4m3 MMA about four).  The other operand of each product is
// split into two e4m3 parts, hi + lo, and both are multiplied:
//   * q: prepared once per step by the q-preparation kernel (row scaled by a
//     power of two 2^e so that its largest element lies in [128, 256); hi, lo
//     and 2^-e stored side by side).  Scores use q' K^T * 2^-e * scale * k_scale.
//   * P: the probabilities scaled by 2^8 are split per unit; the output is
//     multiplied by v_scale / 2^8 at the end.
// The split keeps 2^-8 relative precision per element, against 2^-9 for a bf16
// operand.  The lo parts ride in MMA rows / columns the group leaves empty, so
// they cost no extra MMA: q' lo in A row g + 8 under q' hi in row g (any
// group), P lo in B columns 4..7 beside P hi in columns 0..3 (groups <= 4).
//   Scores S = q' K^T: the q rows are A (rows past the group are zero), K rows
//   are B: ldmatrix gives lane t the codes 4 (t % 4) .. + 3 of a 16-byte chunk
//   of token t / 4's row, which is exactly b0 (first 16 columns of a 32-column
//   step) or b1 (last 16).
//   Values O^T = V^T P^T: ldmatrix.trans on code pairs gives lane t, for
//   tokens 2 (t % 4), +1 of an 8-token block, the codes of columns 2 (t / 4) and
//   2 (t / 4) + 1 of a 16-byte chunk; a byte permutation of two such registers
//   (blocks 0-7 and 8-15) forms a0 / a1 (columns 2 (t / 4) and 2 (t / 4) + 1,
//   tokens 2c, 2c + 1, 2c + 8, 2c + 9), and blocks 16-31 form a2 / a3.  The
//   same token order is what each lane holds of P after the scores, so the
//   B operand of P is built from the lane's own probabilities.  An m-tile
//   covers one 16-byte chunk of V with its rows in the order 0, 2, .., 14,
//   1, 3, .., 15.
template <typename Tr>
struct Fp8TensorConsumer {
  static constexpr int G = Tr::G_, D = Tr::D_;
  static constexpr int KS = D / 32;     // score k-steps (32 columns: two 16-byte chunks)
  static constexpr int MT = D / 16;     // O^T m-tiles (one 16-byte chunk of a V row)
  static constexpr int NT = 4;          // score n-tiles (8 tokens) of a 32-token block
  static constexpr int NB = Tr::UT / 32;  // 32-token blocks per unit
  static_assert(Tr::UT % 32 == 0, "the fp8 consumer takes units of 32-token blocks");
  static constexpr float kPScale = 256.f;
  // a group of at most 4 leaves columns 4..7 of the PV product free for the lo
  // parts of P: one MMA per m-tile instead of two
  static constexpr bool kPackPV = G <= 4;
  uint32_t qaddr;                       // shared address of this lane's q' hi codes
  bool qrow;                            // lane / 4 is a row of the group
  float o[MT][4];
  float m, l, sc, vscale;
  int lane;
  // head pair (pshift >= 0): row g belongs to head g >> pshift of the pair, and
  // tokens 0-15 / 16-31 of a block are the 16 positions of head 0 / head 1
  int pshift = -1, rsub = 0;
  float sc1 = 0.f, vscale1 = 0.f;

  __device__ __forceinline__ void init(int lane_, float*) { lane = lane_; }

  __device__ __forceinline__ int row_token(int group_log2) const {
    return (lane >> 2) >> group_log2;
  }

  // The second head's scales when the items are head pairs (shift >= 0).
  __device__ __forceinline__ void set_pair(int shift, float score_scale1, float v_scale1) {
    pshift = shift;
    sc1 = score_scale1;
    vscale1 = v_scale1 * (1.f / kPScale);
  }

  __device__ __forceinline__ void begin(const char* qs, float score_scale, float v_scale) {
    const int g = lane >> 2, c = lane & 3;
    float qinv = 0.f;
    qrow = g < G;
    rsub = pshift >= 0 ? (g >> pshift) & 1 : 0;
    if (rsub) score_scale = sc1;
    // the q' fragments are read from shared memory in every unit (the slot
    // stays valid for the whole item), which keeps 16 registers free
    qaddr = smem_addr(qs + (qrow ? g : 0) * Tr::QROW_BYTES + 4 * c);
    if (qrow) qinv = *reinterpret_cast<const float*>(qs + g * Tr::QROW_BYTES + 2 * D);
    sc = score_scale * qinv;
    vscale = v_scale * (1.f / kPScale);
    m = kNoScore;
    l = 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  }

  // A unit is NB blocks of 32 tokens (block b: rows 32 b .. 32 b + 31 of the K
  // and V tiles, 4 KiB apart, which keeps the 128-byte swizzle phase); the
  // stage is released after the last block has been read.
  template <typename Release>
  __device__ __forceinline__ void unit(const char* kt, const char* vt, int nt, int qlim, float,
                                       Release release) {
#pragma unroll 1
    for (int b = 0; b < NB && 32 * b < nt; ++b)
      block32(smem_addr(kt) + 4096 * b, smem_addr(vt) + 4096 * b, nt - 32 * b, qlim - 32 * b);
    release();
  }

  __device__ __forceinline__ void block32(uint32_t kb, uint32_t vb, int nt, int qlim) {
    const int mi = lane >> 3, r8 = lane & 7, c = lane & 3;
    // ---- scores: per step ks, kr[n][0 / 1] = b0 / b1 of n-tile n.  The A rows
    // past the group are free, so q' lo sits in row g + 8 under q' hi in row g:
    // one MMA gives both products (c0, c1: hi; c2, c3: lo)
    float sh[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) sh[n][0] = sh[n][1] = sh[n][2] = sh[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t qh0 = 0u, qh1 = 0u, ql0 = 0u, ql1 = 0u;
      if (qrow) {
        qh0 = lds_u32(qaddr + 32 * ks);
        qh1 = lds_u32(qaddr + 32 * ks + 16);
        ql0 = lds_u32(qaddr + D + 32 * ks);
        ql1 = lds_u32(qaddr + D + 32 * ks + 16);
      }
      uint32_t kr[NT][2];
#pragma unroll
      for (int hb = 0; hb < NT / 2; ++hb)   // tokens 16 hb + (0-7 | 8-15) x chunks 2ks, 2ks+1
        ldsm_x4(kb + swz<Tr>(16 * hb + (mi >> 1) * 8 + r8, 2 * ks + (mi & 1)),
                kr[2 * hb][0], kr[2 * hb][1], kr[2 * hb + 1][0], kr[2 * hb + 1][1]);
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        mma_e4m3(sh[n], qh0, ql0, qh1, ql1, kr[n][0], kr[n][1]);
      }
    }
    // ---- online softmax over the unit's tokens 8 n + 2c, 8 n + 2c + 1 (row lane / 4)
    float sv[2 * NT];
    float mx = -INFINITY;
    const int lim = min(nt - 1, qlim);            // last token this lane's row sees
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tk = 8 * n + 2 * c + e;
        // a head pair: this row sees only its own head's half, positions tk % 16
        const bool seen = pshift < 0 ? tk <= lim : ((tk >> 4) == rsub && (tk & 15) <= lim);
        const float v = (sh[n][e] + sh[n][e + 2]) * sc;
        sv[2 * n + e] = seen ? v : -INFINITY;
        mx = fmaxf(mx, sv[2 * n + e]);
      }
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
    const float mn = fmaxf(m, mx);
    const float alpha = fast_exp2(m - mn);
    m = mn;
    float psum = 0.f;
#pragma unroll
    for (int e = 0; e < 2 * NT; ++e) {
      sv[e] = fast_exp2(sv[e] - mn);
      psum += sv[e];
    }
    l = l * alpha + psum;
    // P^T operand: b0 = tokens (2c, 2c+1, 2c+8, 2c+9), b1 = the same + 16
    uint32_t ph[NT], pl[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) split_e4m3x2(sv[2 * n] * kPScale, sv[2 * n + 1] * kPScale, ph[n], pl[n]);
    uint32_t bh0 = ph[0] | (ph[1] << 16), bh1 = ph[2] | (ph[3] << 16);
    const uint32_t bl0 = pl[0] | (pl[1] << 16), bl1 = pl[2] | (pl[3] << 16);
    if constexpr (kPackPV) {
      // columns 4..7 of P^T (rows 4..7 of the group, unused) carry the lo parts
      // of heads 0..3: lane (g, c), g >= 4, takes them from lane (g - 4, c)
      const uint32_t xl0 = __shfl_xor_sync(kFull, bl0, 16), xl1 = __shfl_xor_sync(kFull, bl1, 16);
      if (lane >= 16) {
        bh0 = xl0;
        bh1 = xl1;
      }
    }
    // rescale the accumulators when some row's maximum moved
    if (__any_sync(kFull, alpha != 1.f)) {
      const int hc = kPackPV ? (c & 1) : c;           // head pair of this lane's columns
      const float a_even = __shfl_sync(kFull, alpha, 8 * hc);
      const float a_odd = __shfl_sync(kFull, alpha, 8 * hc + 4);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o[mt][0] *= a_even;
        o[mt][1] *= a_odd;
        o[mt][2] *= a_even;
        o[mt][3] *= a_odd;
      }
    }
    // ---- values: vr[blk] = the ldmatrix.trans register of token block blk (8 tokens)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t vr[4];
      ldsm_x4_trans(vb + swz<Tr>(mi * 8 + r8, mt), vr[0], vr[1], vr[2], vr[3]);
      const uint32_t a0 = __byte_perm(vr[0], vr[1], 0x6420);   // column 2g
      const uint32_t a1 = __byte_perm(vr[0], vr[1], 0x7531);   // column 2g + 1
      const uint32_t a2 = __byte_perm(vr[2], vr[3], 0x6420);
      const uint32_t a3 = __byte_perm(vr[2], vr[3], 0x7531);
      mma_e4m3(o[mt], a0, a1, a2, a3, bh0, bh1);
      if constexpr (!kPackPV) mma_e4m3(o[mt], a0, a1, a2, a3, bl0, bl1);
    }
  }

  __device__ __forceinline__ void store(float* macc_w, float* mml_w) {
    float lt = l + __shfl_xor_sync(kFull, l, 1);
    lt += __shfl_xor_sync(kFull, lt, 2);
    const int g = lane >> 2, c = lane & 3;
    if (g < G && c == 0) {
      mml_w[g * 2 + 0] = m;
      mml_w[g * 2 + 1] = lt;
    }
    const int h0 = 2 * c, h1 = 2 * c + 1;
    // V's scale of each column's row (its head of the pair)
    const float vs0 = pshift >= 0 && ((h0 >> pshift) & 1) ? vscale1 : vscale;
    const float vs1 = pshift >= 0 && ((h1 >> pshift) & 1) ? vscale1 : vscale;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      if constexpr (kPackPV) {             // add the lo columns (lane c + 2) to the hi ones
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][e] += __shfl_xor_sync(kFull, o[mt][e], 2);
      }
      const int d0 = 16 * mt + 2 * g, d1 = d0 + 1;     // O^T rows g and g + 8
      if (h0 < G) {
        macc_w[h0 * D + d0] = o[mt][0] * vs0;
        macc_w[h0 * D + d1] = o[mt][2] * vs0;
      }
      if (h1 < G) {
        macc_w[h1 * D + d0] = o[mt][1] * vs1;
        macc_w[h1 * D + d1] = o[mt][3] * vs1;
      }
    }
  }
};

template <bool BF16, int D, int G, bool KV8>
__global__ void __launch_bounds__(DecodeTraits<BF16, D, G, KV8>::THREADS, 1)
    paged_decode_kernel(const __grid_constant__ DecodeKernelParams p) {
  using Tr = DecodeTraits<BF16, D, G, KV8>;
  constexpr int CW = Tr::CW;
  using Consumer = typename std::conditional<
      KV8, Fp8TensorConsumer<Tr>,
      typename std::conditional<Tr::TC, TensorConsumer<Tr>, CoreConsumer<Tr>>::type>::type;
  constexpr int S = Tr::S;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // swizzled tensor-map copies need 1 KiB-aligned stages
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  char* stages = reinterpret_cast<char*>(smem + Tr::OFF_STAGES);
  char* qbuf = reinterpret_cast<char*>(smem + Tr::OFF_QBUF);
  float* macc = reinterpret_cast<float*>(smem + Tr::OFF_MACC);
  float* mml = reinterpret_cast<float*>(smem + Tr::OFF_MML);
  float* ps_all = reinterpret_cast<float*>(smem + Tr::OFF_PS);
  ItemDesc* desc = reinterpret_cast<ItemDesc*>(smem + Tr::OFF_DESC);
  volatile int* stage_bad = reinterpret_cast<volatile int*>(smem + Tr::OFF_SFLAG);
  int* tbl_s = reinterpret_cast<int*>(smem + Tr::OFF_TBL);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Tr::OFF_ABORT);
  volatile uint32_t* issued_by = reinterpret_cast<volatile uint32_t*>(smem + Tr::OFF_ABORT + 8);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tr::OFF_BARS);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* item_full = bars + 2 * S;
  uint64_t* item_empty = item_full + kItemSlots;
  uint64_t* sched_full = item_empty + kItemSlots;
  uint64_t* merge_free = sched_full + kItemSlots;
  uint64_t* merge_full = merge_free + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int k = 0; k < kItemSlots; ++k) {
      mbar_init(&item_full[k], 1);
      // released by every consumer warp (q read), by its producer lane (done
      // issuing) and by the merge warp (descriptor read)
      mbar_init(&item_empty[k], 2 * CW + 1);
      mbar_init(&sched_full[k], 1);
    }
    mbar_init(merge_free, 1);
    mbar_init(merge_full, CW);
    *abort_flag = 0;
    for (int w = 0; w < CW; ++w) issued_by[w] = 0;
    fence_mbar_init();
  }
  // launched as a programmatic dependent of the plan kernel: everything above
  // overlaps its tail; the work list is only read after it has completed
  wait_prior_grids();
  allow_next_grid();
  __syncthreads();
  // no work listed (every sequence empty, or a shared-prefix batch whose own
  // tokens all go to the merge): every warp leaves at once
  if (p.header[1] == 0) return;

  const int Hkv = p.num_kv_heads;
  const int bs = p.block_size;
  // positions per unit: a head-pair stage holds half as many of each head
  const bool paired = KV8 && p.head_pairs != 0;
  const int PU = paired ? Tr::UT / 2 : Tr::UT;

  if (warp == CW + 1) {
    // ----------------------------------------------------------- scheduler
    // Claims work items and resolves them (atomic counter -> work entry ->
    // block-table slice) into the shared item slots, then starts the copy of
    // the item's q rows.  The dependent global round trips never hold up the
    // K/V copies.  It keeps at most kUnitsAhead claimed-but-unissued units,
    // which bounds the work one CTA holds back when the queue runs dry.
    const int total_items = p.header[1] * Hkv;
    uint32_t claimed = 0, q_issued = 0;
    bool ended = false;                          // published the end marker
    for (uint32_t k = 0;; ++k) {
      const int slot = k % kItemSlots;
      for (uint32_t spin = 0; spin < p.wait_limit; ++spin) {
        uint32_t issued = 0;
#pragma unroll
        for (int w = 0; w < CW; ++w) issued += issued_by[w];
        if (*abort_flag || static_cast<int>(claimed - issued) <= kUnitsAhead) break;
        __nanosleep(100);
      }
      int waited = 1;
      if (lane == 0) waited = mbar_wait(&item_empty[slot], ((k / kItemSlots) & 1) ^ 1, p.wait_limit);
      if (!__shfl_sync(kFull, waited, 0)) {
        if (lane == 0) {
          report(p.device_errors, PA_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      if (*abort_flag) break;
      int i = 0;
      if (lane == 0) i = atomicAdd(&p.header[0], 1);
      i = __shfl_sync(kFull, i, 0);
      if (i >= total_items) {
        if (lane == 0) {
          desc[slot].b = -1;                     // the end: producer lanes and consumers stop
          mbar_arrive(&sched_full[slot]);
          mbar_arrive(&item_full[slot]);
        }
        ended = true;
        break;
      }
      const int j = i / Hkv;
      const int h = i - j * Hkv;
      const int4 w = p.work[j];                  // {b, chunk, length, global chunk}
      const int tok0 = w.y;
      const int ntok = min(p.chunk_tokens, w.z - tok0);
      const int n_units = (ntok + PU - 1) / PU;
      const int page0 = tok0 / bs;
      const int npages = (ntok + bs - 1) / bs;
      for (int pg = lane; pg < kItemPages; pg += 32) {
        int phys = -1;
        if (pg < npages) {
          phys = p.block_tables[static_cast<int64_t>(w.x) * p.max_blocks_per_seq + page0 + pg];
          if (phys < 0 || phys >= p.num_blocks) {
            report(p.device_errors, PA_DEVERR_BAD_BLOCK);
            phys = -1;
          }
        }
        tbl_s[slot * kItemPages + pg] = phys;
      }
      if (lane == 0) {
        ItemDesc d;
        d.b = w.x; d.h = h; d.tok0 = w.y; d.len = w.z; d.gchunk = w.w & (kSingleChunk - 1);
        d.n_units = n_units; d.n_tokens = ntok; d.single = (w.w & kSingleChunk) != 0;
        d.rot = i % CW;
        desc[slot] = d;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sched_full[slot]);
        mbar_arrive_expect_tx(&item_full[slot], Tr::Q_BYTES);
        // the G rows: for each new token j, the group's `group` heads (q is
        // [B][q_len][Hq] rows)
        for (int j = 0; j < p.q_len; ++j) {
          const char* qsrc =
              p.q + ((static_cast<int64_t>(w.x) * p.q_len + j) * p.num_q_heads +
                     static_cast<int64_t>(h) * p.group) * Tr::QROW_BYTES;
          bulk_g2s(qbuf + slot * Tr::Q_BYTES + j * p.group * Tr::QROW_BYTES, qsrc,
                   p.group * Tr::QROW_BYTES, &item_full[slot]);
        }
      }
      ++q_issued;
      claimed += static_cast<uint32_t>(n_units);
    }
    // Wait (bounded) for our q copies that may still be in flight: item k's slot
    // was reused for item k + NI only after every consumer had read it, so only
    // the last NI items can be outstanding -- NI - 1 once the end marker has
    // taken the oldest one's slot.
    if (lane == 0) {
      const uint32_t span = ended ? kItemSlots - 1 : kItemSlots;
      for (uint32_t k = q_issued > span ? q_issued - span : 0; k < q_issued; ++k)
        mbar_wait(&item_full[k % kItemSlots], (k / kItemSlots) & 1);
    }
    return;
  }

  if (warp == CW) {
    // ------------------------------------------------------------ producer
    // Lane w < CW feeds consumer warp w: the units u of every item with
    // (u + rot) % CW == w, in order, into w's sub-ring.
    // Each lane runs its own sequence with blocking (bounded) barrier waits;
    // the lanes of the warp diverge freely, so several copies are in issue at
    // once (one issuing thread cannot keep HBM busy) and a consumer that is
    // busy merging only holds back its own sub-ring.
    const int w = lane;
    if (w < CW) {
      uint32_t c = 0;                      // units this lane has issued
      bool ok = true;
      for (uint32_t k = 0; ok; ++k) {
        const int slot = k % kItemSlots;
        if (!mbar_wait(&sched_full[slot], (k / kItemSlots) & 1, p.wait_limit) || *abort_flag) {
          ok = false;
          break;
        }
        const ItemDesc d = desc[slot];
        if (d.b < 0) break;
        for (int u = (w - d.rot + CW) % CW; u < d.n_units; u += CW) {
          const int s = w + CW * static_cast<int>(c % Tr::SPW);
          if (!mbar_wait(&empty[s], ((c / Tr::SPW) & 1) ^ 1, p.wait_limit)) {
            ok = false;
            break;
          }
          const int tok = u * PU;
          char* dst = stages + s * Tr::STAGE_BYTES;
          const int pp = tbl_s[slot * kItemPages + tok / bs];
          if (paired) {
            // one box per pool: the page's 16 rows of head 2h, then of head 2h + 1
            if (pp >= 0) {
              stage_bad[s] = 0;
              mbar_arrive_expect_tx(&full[s], Tr::STAGE_BYTES);
              const int row = (pp * p.pool_heads + 2 * d.h) * bs;
              tma_rows<Tr>(dst, &p.tmap_k, row, &full[s]);
              tma_rows<Tr>(dst + Tr::TILE_BYTES, &p.tmap_v, row, &full[s]);
            } else {
              stage_bad[s] = 1;
              mbar_arrive(&full[s]);
            }
          } else if constexpr (Tr::TC) {
            // one tensor-map box per page the unit touches (a unit longer than
            // a page takes several; the last unit of an item only those it
            // needs) and pool, each taking all 128-byte slabs of its rows
            const int rows_op = bs < Tr::UT ? bs : Tr::UT;
            int n_op = 1;
            bool pages_ok = pp >= 0;
            if (rows_op < Tr::UT) {
              n_op = (min(Tr::UT, d.n_tokens - tok) + rows_op - 1) / rows_op;
              for (int j = 1; j < n_op; ++j)
                pages_ok &= tbl_s[slot * kItemPages + (tok + j * rows_op) / bs] >= 0;
            }
            if (pages_ok) {
              stage_bad[s] = 0;
              mbar_arrive_expect_tx(&full[s], n_op * rows_op * Tr::ROW_BYTES * 2);
              for (int j = 0; j < n_op; ++j) {
                const int t = tok + j * rows_op;
                const int pj = j == 0 ? pp : tbl_s[slot * kItemPages + t / bs];
                const int row = (pj * p.pool_heads + d.h) * bs + t % bs;
                tma_rows<Tr>(dst + j * rows_op * 128, &p.tmap_k, row, &full[s]);
                tma_rows<Tr>(dst + Tr::TILE_BYTES + j * rows_op * 128, &p.tmap_v, row, &full[s]);
              }
            } else {
              stage_bad[s] = 1;
              mbar_arrive(&full[s]);
            }
          } else if (pp >= 0) {
            stage_bad[s] = 0;
            mbar_arrive_expect_tx(&full[s], Tr::STAGE_BYTES);
            const int64_t off =
                ((static_cast<int64_t>(pp) * p.pool_heads + d.h) * bs + (tok % bs)) * Tr::ROW_BYTES;
            bulk_g2s(dst, p.k_cache + off, Tr::TILE_BYTES, &full[s]);
            bulk_g2s(dst + Tr::TILE_BYTES, p.v_cache + off, Tr::TILE_BYTES, &full[s]);
          } else {
            stage_bad[s] = 1;
            mbar_arrive(&full[s]);
          }
          ++c;
          issued_by[w] = c;
        }
        if (!ok) break;
        mbar_arrive(&item_empty[slot]);      // done issuing from this item
      }
      if (!ok) {                             // gave up: tell the others
        report(p.device_errors, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // Wait (bounded) for copies still in flight on warp w's sub-ring: only
      // the last SPW can be (immediate when the consumer took them all).
      const uint32_t first = c > static_cast<uint32_t>(Tr::SPW) ? c - Tr::SPW : 0;
      for (uint32_t cc = first; cc < c; ++cc)
        mbar_wait(&full[w + CW * (cc % Tr::SPW)], (cc / Tr::SPW) & 1);
    }
    return;
  }

  if (warp == CW + 2) {
    // ---------------------------------------------------------------- merger
    // Per item, once every consumer warp has deposited its state: the item's
    // rows out[g] = sum_w 2^(m_w - M) acc_w / sum_w 2^(m_w - M) l_w over the CW
    // warps, written to `out` or as a split-K partial.  A warp of its own, so
    // that no consumer falls behind the others by the merge.
    for (uint32_t k = 0;; ++k) {
      const int slot = k % kItemSlots;
      if (!mbar_wait(&item_full[slot], (k / kItemSlots) & 1, p.wait_limit)) {
        report(p.device_errors, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      const ItemDesc d = desc[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);
      if (d.b < 0 || *abort_flag) break;
      bool ok = false;
      for (uint32_t spin = 0; spin < p.wait_limit && !ok; ++spin) {
        ok = mbar_try_wait(merge_full, k & 1);
        if (*abort_flag) break;
      }
      if (!ok) {
        if (!*abort_flag) {
          report(p.device_errors, PA_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      // out[g] = sum_w 2^(m_w - M) acc_w / sum_w 2^(m_w - M) l_w over the CW warps.
      // The weights of every row first, then all rows' columns together, so
      // that every row's loads are in flight at once.
      float f[G][CW], inv[G], lse[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < CW; ++w) M = fmaxf(M, mml[(w * G + g) * 2]);
        float lam = 0.f;
#pragma unroll
        for (int w = 0; w < CW; ++w) {
          // a row with no visible token in this item (a new token before the
          // item's first position) has M = -inf: it contributes nothing
          f[g][w] = M == -INFINITY ? 0.f : fast_exp2(mml[(w * G + g) * 2] - M);
          lam = fmaf(f[g][w], mml[(w * G + g) * 2 + 1], lam);
        }
        inv[g] = lam > 0.f ? 1.f / lam : 0.f;
        lse[g] = lam > 0.f ? M + __log2f(lam) : -INFINITY;
      }
      const int64_t rows_per_seq = static_cast<int64_t>(p.q_len) * p.num_q_heads;
#pragma unroll
      for (int cp = lane; cp < D / 2; cp += 32) {
        const int dcol = 2 * cp;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float o0 = 0.f, o1 = 0.f;
#pragma unroll
          for (int w = 0; w < CW; ++w) {
            const float2 a = *reinterpret_cast<const float2*>(macc + (w * G + g) * D + dcol);
            o0 = fmaf(f[g][w], a.x, o0);
            o1 = fmaf(f[g][w], a.y, o1);
          }
          o0 *= inv[g];
          o1 *= inv[g];
          // row g = (new token j, head gi of the group): query row j * Hq + h * group + gi
          const int qh = (g >> p.group_log2) * p.num_q_heads + d.h * p.group + (g & (p.group - 1));
          if (d.single) {
            const int64_t o = (static_cast<int64_t>(d.b) * rows_per_seq + qh) * D + dcol;
            if constexpr (BF16) {
              const uint32_t packed = f32_to_bf16_bits(o0) | (f32_to_bf16_bits(o1) << 16);
              *reinterpret_cast<uint32_t*>(static_cast<char*>(p.out) + o * 2) = packed;
            } else {
              *reinterpret_cast<float2*>(static_cast<float*>(p.out) + o) = make_float2(o0, o1);
            }
          } else {
            const int64_t row = static_cast<int64_t>(d.gchunk) * rows_per_seq + qh;
            *reinterpret_cast<float2*>(p.part_out + row * D + dcol) = make_float2(o0, o1);
            if (dcol == 0) p.part_lse[row] = lse[g];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(merge_free);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  Consumer cs;
  cs.init(lane, ps_all + warp * Tr::UT * G);

  uint32_t item_k = 0, consumed = 0;   // items seen; units this warp consumed
  bool aborted = false;
  for (;;) {
    const int slot = item_k % kItemSlots;
    if (!mbar_wait(&item_full[slot], (item_k / kItemSlots) & 1, p.wait_limit)) {
      report(p.device_errors, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
      break;
    }
    const ItemDesc d = desc[slot];
    if (d.b < 0 || *abort_flag) break;
    // fp8 caches: K's head scale folds into the score scale, V's into the output
    const int kvh = paired ? 2 * d.h : d.h;       // (first) kv head of the item
    const float kv_k = KV8 ? p.k_scale[kvh] : 1.f, kv_v = KV8 ? p.v_scale[kvh] : 1.f;
    const float item_scale = p.scale_log2 * kv_k;
    if constexpr (KV8) {
      // a head pair: rows of the second head take its own scales
      if (paired)
        cs.set_pair(p.pair_shift, p.scale_log2 * p.k_scale[kvh + 1], p.v_scale[kvh + 1]);
      else
        cs.set_pair(-1, 0.f, 0.f);
    }
    cs.begin(qbuf + slot * Tr::Q_BYTES, item_scale, kv_v);
    // row j may see positions up to L - q_len + j: relative to the item's first
    // token, the last visible token of this lane's row
    const int qlim0 = d.len - p.q_len - d.tok0 + cs.row_token(p.group_log2);
    __syncwarp();
    if (lane == 0) mbar_arrive(&item_empty[slot]);

    // this warp's units of the item: u = u0, u0 + CW, ... (u + rot == warp mod CW)
    const int u0 = (warp - d.rot + CW) % CW;
    for (int u = u0; u < d.n_units && !aborted; u += CW, ++consumed) {
      const int s = warp + CW * static_cast<int>(consumed % Tr::SPW);
      if (!mbar_wait(&full[s], (consumed / Tr::SPW) & 1, p.wait_limit)) {
        report(p.device_errors, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
        aborted = true;
        break;
      }
      const int nt = min(PU, d.n_tokens - u * PU);     // positions of the unit
      if (!stage_bad[s]) {
        char* kt = stages + s * Tr::STAGE_BYTES;
        char* vt = kt + Tr::TILE_BYTES;
        if constexpr (Tr::TC) {
          // The tensor cores multiply every row of the tile, so value rows past
          // the sequence (stale or never-written slots) must not hold NaN or Inf.
          if (nt < PU) {
            // (a head-pair stage: positions nt.. of both halves)
            const int per_half = PU - nt;
            const int nzero = paired ? 2 * per_half : Tr::UT - nt;
            for (int i = lane; i < nzero * Tr::BOXES * 8; i += 32) {
              const int k = i / (Tr::BOXES * 8);
              const int row = paired ? (k < per_half ? nt + k : PU + nt + (k - per_half)) : nt + k;
              const int rest = i % (Tr::BOXES * 8);
              if (row < Tr::UT)
                *reinterpret_cast<uint4*>(vt + (rest >> 3) * Tr::BOX_BYTES + row * 128 +
                                          (rest & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
          }
        }
        cs.unit(kt, vt, nt, qlim0 - u * PU, item_scale, [&] {
          if constexpr (Tr::TC) {
            // order this warp's generic-proxy writes before the next tensor copy here
            if (nt < PU) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        });
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }

    // ---- hand this warp's state to the merge warp; the warps go on with their
    // next item while it merges (the buffer is free again once it has read it)
    if (item_k > 0 && !mbar_wait(merge_free, (item_k - 1) & 1, p.wait_limit)) {
      report(p.device_errors, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
      aborted = true;
    }
    cs.store(macc + warp * G * D, mml + warp * G * 2);
    __threadfence_block();
    __syncwarp();
    if (lane == 0) mbar_arrive(merge_full);
    ++item_k;
    if (aborted) break;
  }
}

}  // namespace pa
