/*
 * CPU oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline / reference
 * arm may load this file's library.  The product path (the CUDA library in
 * paged_kv_cache_190_gb300/) never links, loads or calls it, and shares no code
 * with it.
 *
 * What it computes is the plain definition, in fp64, with no blocking, fusion
 * or reordering:
 *
 *   "PagedAttention原理" (vLLM long-sequence memory guide, ch. 3), §3.4 closing
 *   paragraph: paging does not change the mathematics of attention, only where
 *   the K/V bytes live.  §3.2: logically contiguous tokens sit in scattered
 *   physical pages, located through a page table.
 *   "PagedAttentionMetal", section "注意力计算优化": look the physical page up in
 *   the block table, load the K/V block, batch variable lengths without padding.
 *
 * So for every sequence b and query head i (kv head h = i / G, G = Hq / Hkv):
 *   1. gather K_b[t] = k_cache[block_tables[b][t / bs]][h][t % bs][:] and V_b[t]
 *      likewise, t = 0 .. L_b - 1, converting every element to double exactly;
 *   2. s_t = scale * sum_d q[b][i][d] * K_b[t][d];
 *      p_t = exp(s_t - max s) / sum_u exp(s_u - max s);
 *   3. out[b][i][d] = sum_t p_t * V_b[t][d].
 *   L_b == 0 gives a zero row.
 *
 * Layouts (row-major, element type f32, bf16, or float8 e4m3 for the caches):
 *   q       [num_seqs][num_q_heads][head_dim]
 *   k_cache [num_blocks][num_kv_heads][block_size][head_dim]   (v_cache alike)
 *   block_tables int32 [num_seqs][max_blocks_per_seq], context_lens int32 [num_seqs]
 *   out     double [num_rows][head_dim]   (rows listed in `rows`, or all
 *           num_seqs * num_q_heads rows in (b, i) order when rows == NULL)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_FP8_E4M3 = 2 };

/* bfloat16 is the upper half of an IEEE binary32: widen by a 16-bit shift. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* float8 e4m3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 fraction
 * bits; no infinities; exponent and fraction all ones is NaN; exponent 0 is
 * subnormal (fraction * 2^-9). */
static double e4m3_bits_to_double(uint8_t bits) {
  const int sign = bits >> 7, e = (bits >> 3) & 15, m = bits & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

static double load_elem(const void* base, size_t index, int dtype) {
  if (dtype == ORACLE_BF16) return bf16_bits_to_double(((const uint16_t*)base)[index]);
  if (dtype == ORACLE_FP8_E4M3) return e4m3_bits_to_double(((const uint8_t*)base)[index]);
  return (double)((const float*)base)[index];
}

/* Widen `n` stored elements to double (exposed so tests can pin the conversion). */
void oracle_widen(double* dst, const void* src, long n, int dtype) {
  for (long j = 0; j < n; ++j) dst[j] = load_elem(src, (size_t)j, dtype);
}

/* One output row: sequence b, query head i.  Returns 0, or -1 when the block
 * table or length is out of range (the oracle refuses rather than guesses). */
static int decode_row(double* out_row, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens, double scale,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      int max_blocks_per_seq, int num_blocks, int q_dtype, int kv_dtype,
                      const double* k_scale, const double* v_scale, int b, int i) {
  const int D = head_dim;
  const int G = num_q_heads / num_kv_heads;
  const int h = i / G;
  const int L = context_lens[b];
  /* stored K/V codes times the kv head's scale (1 when none is given) */
  const double ks = k_scale ? k_scale[h] : 1.0, vs = v_scale ? v_scale[h] : 1.0;
  if (L < 0 || (long)L > (long)max_blocks_per_seq * block_size) return -1;
  for (int d = 0; d < D; ++d) out_row[d] = 0.0;
  if (L == 0) return 0;

  /* Step 1: gather this sequence's keys and values through its block table. */
  double* K = (double*)malloc(sizeof(double) * (size_t)L * D);
  double* V = (double*)malloc(sizeof(double) * (size_t)L * D);
  double* s = (double*)malloc(sizeof(double) * (size_t)L);
  double* p = (double*)malloc(sizeof(double) * (size_t)L);
  if (!K || !V || !s || !p) {
    free(K); free(V); free(s); free(p);
    return -2;
  }
  int rc = 0;
  for (int t = 0; t < L && rc == 0; ++t) {
    const int logical_page = t / block_size;
    const int offset = t % block_size;
    const int32_t phys = block_tables[(size_t)b * max_blocks_per_seq + logical_page];
    if (phys < 0 || phys >= num_blocks) { rc = -1; break; }
    const size_t base = (((size_t)phys * num_kv_heads + h) * block_size + offset) * D;
    for (int d = 0; d < D; ++d) {
      K[(size_t)t * D + d] = load_elem(k_cache, base + d, kv_dtype) * ks;
      V[(size_t)t * D + d] = load_elem(v_cache, base + d, kv_dtype) * vs;
    }
  }

  if (rc == 0) {
    /* Step 2: scaled scores and their softmax. */
    const size_t qbase = ((size_t)b * num_q_heads + i) * D;
    double smax = -INFINITY;
    for (int t = 0; t < L; ++t) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += load_elem(q, qbase + d, q_dtype) * K[(size_t)t * D + d];
      s[t] = scale * dot;
      if (s[t] > smax) smax = s[t];
    }
    double z = 0.0;
    for (int t = 0; t < L; ++t) {
      p[t] = exp(s[t] - smax);
      z += p[t];
    }
    for (int t = 0; t < L; ++t) p[t] = p[t] / z;
    /* Step 3: probability-weighted sum of the values. */
    for (int t = 0; t < L; ++t)
      for (int d = 0; d < D; ++d) out_row[d] += p[t] * V[(size_t)t * D + d];
  }
  free(K); free(V); free(s); free(p);
  return rc;
}

static int decode_rows(double* out, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens, double scale,
                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int max_blocks_per_seq, int num_blocks, int q_dtype,
                       int kv_dtype, const double* k_scale, const double* v_scale,
                       const int32_t* rows, int num_rows, int threads) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0)
    return -3;
  const long n = rows ? (long)num_rows : (long)num_seqs * num_q_heads;
  int status = 0;
#ifdef _OPENMP
  const int nthreads = threads > 0 ? threads : omp_get_num_procs();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (long r = 0; r < n; ++r) {
    const int b = rows ? rows[2 * r] : (int)(r / num_q_heads);
    const int i = rows ? rows[2 * r + 1] : (int)(r % num_q_heads);
    int rc = -1;
    if (b >= 0 && b < num_seqs && i >= 0 && i < num_q_heads)
      rc = decode_row(out + (size_t)r * head_dim, q, k_cache, v_cache, block_tables, context_lens,
                      scale, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                      num_blocks, q_dtype, kv_dtype, k_scale, v_scale, b, i);
    if (rc != 0) {
#ifdef _OPENMP
#pragma omp critical
#endif
      if (status == 0) status = rc;
    }
  }
  return status;
}

/* rows: NULL for every (b, i) row, else num_rows pairs {b, i}.  Returns 0, or
 * the first negative status of any row.  `threads` <= 0 uses every processor.
 * q, k_cache and v_cache share `dtype`. */
int oracle_decode_f64(double* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens, double scale,
                      int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, int max_blocks_per_seq, int num_blocks, int dtype,
                      const int32_t* rows, int num_rows, int threads) {
  return decode_rows(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                     num_blocks, dtype, dtype, NULL, NULL, rows, num_rows, threads);
}

/* The same with float8 e4m3 caches: K = code * k_scale[h], V = code * v_scale[h]
 * for kv head h; q is bf16. */
int oracle_decode_kv8_f64(double* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens, double scale,
                          const double* k_scale, const double* v_scale, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int max_blocks_per_seq, int num_blocks, const int32_t* rows,
                          int num_rows, int threads) {
  return decode_rows(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                     num_blocks, ORACLE_BF16, ORACLE_FP8_E4M3, k_scale, v_scale, rows, num_rows,
                     threads);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_num_procs();
#else
  return 1;
#endif
}
