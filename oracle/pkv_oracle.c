/*
 * Float64 CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or constant table with the CUDA
 * library: every decode, encode and gather below is written out here again
 * from the definitions.
 *
 * What it computes, and where the definition comes from:
 *   - Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V.
 *       "KV Cache에 대해 알아보자 (Feat. Attention)", §1 (the attention formula).
 *     The caller passes the softmax scale (1/sqrt(d_k) in every workload).
 *   - The K/V of a request live in fixed-size physical blocks (16 or 32 tokens);
 *     a per-request block table maps logical block i to a physical block, so
 *     the kernel reads the scattered blocks as one contiguous sequence.
 *       "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 02.
 *     The oracle does exactly that first: it GATHERS the request's K/V into a
 *     contiguous fp64 array, then applies the textbook formula.  No blocking,
 *     no online softmax, no split: a max, an exp, a sum, a divide.
 *   - Decode: one new query token attends over every cached token, the new
 *     token's own K/V included (the new K/V is appended to the cache).
 *       "KV Cache에 대해 알아보자 (Feat. Attention)", §3 (Decode 단계).
 *   - Extend: only the suffix after a cached prefix is computed; suffix row i
 *     of a request with cached prefix length P sees keys 0..P+i (causal,
 *     aligned to the end of the sequence).
 *       "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 03
 *       (2,000-token request with 1,900 cached tokens -> prefill 100).
 *   - fp8_e4m3 cache: "KV Cache 완전 정리 — PagedAttention vs RadixAttention,
 *     SGLang이 빠른 이유", section "FP8 KV 캐시".  The pages name only the
 *     format; the reading used here is one fp32 scale per tensor (separate for
 *     K and V), stored code = e4m3(x / scale) with round-to-nearest-even and
 *     saturation to +-448, and value = code * scale.
 *
 * Layouts (the pages fix none; these are the library's conventions):
 *   cache  [num_blocks][num_kv_heads][block_size][head_dim]
 *   q/out  [tokens][num_q_heads][head_dim]
 *   block_tables [batch][max_blocks_per_seq] int32, seq_lens [batch] int32
 *   slot = physical_block * block_size + offset; slot < 0 means "skip".
 *   GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *
 * Build: plain C99 + OpenMP, compiled with -ffp-contract=off and without
 * -ffast-math so that x86-64 and AArch64 give the same bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };

/* ---- element decoders (exact widening to double) ------------------------ */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double orc_f16_to_double(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, f = h & 0x3FF;
  double v;
  if (e == 0x1F) v = f ? NAN : INFINITY;
  else if (e == 0) v = ldexp((double)f, -24);
  else v = ldexp((double)(f + 1024), e - 25);
  return s ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float x;
  memcpy(&x, &u, 4);
  return (double)x;
}

/* OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
 * infinities, S.1111.111 is NaN, largest finite value 448. */
double orc_e4m3_to_double(uint8_t c) {
  int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 0xF && m == 7) v = NAN;
  else if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp((double)(8 + m), e - 10);
  return s ? -v : v;
}

static double round_half_even(double m) {
  double r = floor(m), frac = m - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  return r;
}

/* Nearest E4M3 code to y (ties to even), finite results saturate to +-448,
 * NaN maps to 0x7F. */
uint8_t orc_e4m3_from_float(float y) {
  if (isnan(y)) return 0x7F;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= 448.0) return sign | 0x7E;
  int e;
  if (a < ldexp(1.0, -6)) {
    e = -6;                      /* subnormal range: spacing 2^-9 */
  } else {
    (void)frexp(a, &e);          /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                      /* now 2^e <= a < 2^(e+1) */
  }
  double quantum = ldexp(1.0, e - 3);
  double r = round_half_even(a / quantum);
  double v = r * quantum;        /* never above 448 because a < 448 */
  if (v == 0.0) return sign;
  if (v < ldexp(1.0, -6)) return sign | (uint8_t)(v / ldexp(1.0, -9));
  int ev;
  double fr = frexp(v, &ev);     /* v = fr * 2^ev, fr in [0.5,1) */
  int biased = (ev - 1) + 7;
  int mant = (int)((fr * 2.0 - 1.0) * 8.0);
  return sign | (uint8_t)(biased << 3) | (uint8_t)mant;
}

/* Correctly rounded fp32 quotient, as the stored-code definition asks. */
float orc_div_f32(float x, float s) {
  volatile float q = x / s;
  return q;
}

static double load_elem(const void* base, int64_t idx, int dtype) {
  if (dtype == ORC_F16) return orc_f16_to_double(((const uint16_t*)base)[idx]);
  if (dtype == ORC_BF16) return orc_bf16_to_double(((const uint16_t*)base)[idx]);
  return orc_e4m3_to_double(((const uint8_t*)base)[idx]);
}

static float load_elem_f32(const void* base, int64_t idx, int dtype) {
  return (float)load_elem(base, idx, dtype);  /* exact: f16/bf16 fit in fp32 */
}

/* ---- gather: request b, kv head g -> contiguous [n][D] fp64 --------------- */
static void gather_kv(const void* cache, int dtype, double scale, int num_blocks,
                      int num_kv_heads, int block_size, int head_dim,
                      const int32_t* table_row, int n, int g, double* dst,
                      int* bad_block) {
  for (int t = 0; t < n; ++t) {
    int logical = t / block_size;
    int offset = t % block_size;
    int32_t phys = table_row[logical];
    if (phys < 0 || phys >= num_blocks) {
      *bad_block = 1;
      for (int d = 0; d < head_dim; ++d) dst[(int64_t)t * head_dim + d] = 0.0;
      continue;
    }
    int64_t base = (((int64_t)phys * num_kv_heads + g) * block_size + offset) * head_dim;
    for (int d = 0; d < head_dim; ++d) {
      double x = load_elem(cache, base + d, dtype);
      if (dtype == ORC_E4M3) x *= scale;
      dst[(int64_t)t * head_dim + d] = x;
    }
  }
}

/* Textbook attention of one query row over n contiguous keys:
 *   s_t = scale * <q, K_t>,  p_t = exp(s_t - max s),  out = sum p_t V_t / sum p_t,
 *   lse = max s + log(sum p_t).  n == 0 gives out = 0 and lse = -inf. */
static void attend_row(const double* qrow, const double* K, const double* V, int n,
                       int head_dim, double sm_scale, double* s_buf, double* out,
                       double* lse) {
  if (n <= 0) {
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int t = 0; t < n; ++t) {
    double acc = 0.0;
    for (int d = 0; d < head_dim; ++d) acc += qrow[d] * K[(int64_t)t * head_dim + d];
    s_buf[t] = sm_scale * acc;
    if (s_buf[t] > m) m = s_buf[t];
  }
  double denom = 0.0;
  for (int t = 0; t < n; ++t) {
    s_buf[t] = exp(s_buf[t] - m);
    denom += s_buf[t];
  }
  for (int d = 0; d < head_dim; ++d) {
    double acc = 0.0;
    for (int t = 0; t < n; ++t) acc += s_buf[t] * V[(int64_t)t * head_dim + d];
    out[d] = acc / denom;
  }
  *lse = m + log(denom);
}

/* Paged decode.  out [batch][num_q_heads][head_dim], lse [batch][num_q_heads]
 * (natural log).  pairs: optional list of (b, h) to evaluate (num_pairs > 0),
 * otherwise every pair.  Returns 0, or 1 if a block id was out of range, or
 * -1 on bad arguments / allocation failure. */
int orc_paged_decode(const void* k_cache, const void* v_cache, int cache_dtype,
                     double k_scale, double v_scale, int num_blocks, int num_kv_heads,
                     int block_size, int head_dim, const void* q, int q_dtype,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* seq_lens, int batch, int num_q_heads, double sm_scale,
                     const int32_t* pairs, int num_pairs, double* out, double* lse,
                     int num_threads) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
      block_size <= 0)
    return -1;
  int group = num_q_heads / num_kv_heads;
  int total = num_pairs > 0 ? num_pairs : batch * num_q_heads;
  int bad = 0, fail = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad, fail)
#endif
  for (int i = 0; i < total; ++i) {
    int b = num_pairs > 0 ? pairs[2 * i] : i / num_q_heads;
    int h = num_pairs > 0 ? pairs[2 * i + 1] : i % num_q_heads;
    int g = h / group;
    int n = seq_lens[b];
    if (n > max_blocks_per_seq * block_size || n < 0) { fail = 1; continue; }
    double* K = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
    double* V = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
    double* s = (double*)malloc(sizeof(double) * ((size_t)n + 1));
    double* qrow = (double*)malloc(sizeof(double) * (size_t)head_dim);
    if (!K || !V || !s || !qrow) { fail = 1; free(K); free(V); free(s); free(qrow); continue; }
    const int32_t* row = block_tables + (int64_t)b * max_blocks_per_seq;
    int bb = 0;
    gather_kv(k_cache, cache_dtype, k_scale, num_blocks, num_kv_heads, block_size,
              head_dim, row, n, g, K, &bb);
    gather_kv(v_cache, cache_dtype, v_scale, num_blocks, num_kv_heads, block_size,
              head_dim, row, n, g, V, &bb);
    bad |= bb;
    int64_t qoff = ((int64_t)b * num_q_heads + h) * head_dim;
    for (int d = 0; d < head_dim; ++d) qrow[d] = load_elem(q, qoff + d, q_dtype);
    int64_t ooff = num_pairs > 0 ? (int64_t)i * head_dim : qoff;
    int64_t loff = num_pairs > 0 ? i : (int64_t)b * num_q_heads + h;
    attend_row(qrow, K, V, n, head_dim, sm_scale, s, out + ooff, lse + loff);
    free(K); free(V); free(s); free(qrow);
  }
  if (fail) return -1;
  return bad ? 1 : 0;
}

/* Paged extend (suffix prefill).  Request b owns query rows
 * q_indptr[b] .. q_indptr[b+1]-1; row i of it sits at absolute position
 * prefix_lens[b] + i and attends to keys 0 .. prefix_lens[b] + i.
 * out [q_indptr[batch]][num_q_heads][head_dim], lse [q_indptr[batch]][num_q_heads].
 * rows: optional list of (global_row, h) pairs to evaluate (num_rows > 0). */
int orc_paged_extend(const void* k_cache, const void* v_cache, int cache_dtype,
                     double k_scale, double v_scale, int num_blocks, int num_kv_heads,
                     int block_size, int head_dim, const void* q, int q_dtype,
                     const int32_t* q_indptr, const int32_t* prefix_lens,
                     const int32_t* block_tables, int max_blocks_per_seq, int batch,
                     int num_q_heads, double sm_scale, const int32_t* rows, int num_rows,
                     double* out, double* lse, int num_threads) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
      block_size <= 0)
    return -1;
  int group = num_q_heads / num_kv_heads;
  int total_rows = q_indptr[batch];
  int total = num_rows > 0 ? num_rows : total_rows * num_q_heads;
  int bad = 0, fail = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad, fail)
#endif
  for (int i = 0; i < total; ++i) {
    int grow = num_rows > 0 ? rows[2 * i] : i / num_q_heads;
    int h = num_rows > 0 ? rows[2 * i + 1] : i % num_q_heads;
    int b = 0;
    while (b + 1 <= batch && q_indptr[b + 1] <= grow) ++b;
    if (b >= batch) { fail = 1; continue; }
    int local = grow - q_indptr[b];
    int n = prefix_lens[b] + local + 1;
    if (n > max_blocks_per_seq * block_size) { fail = 1; continue; }
    int g = h / group;
    double* K = (double*)malloc(sizeof(double) * (size_t)n * head_dim);
    double* V = (double*)malloc(sizeof(double) * (size_t)n * head_dim);
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    double* qrow = (double*)malloc(sizeof(double) * (size_t)head_dim);
    if (!K || !V || !s || !qrow) { fail = 1; free(K); free(V); free(s); free(qrow); continue; }
    const int32_t* row = block_tables + (int64_t)b * max_blocks_per_seq;
    int bb = 0;
    gather_kv(k_cache, cache_dtype, k_scale, num_blocks, num_kv_heads, block_size,
              head_dim, row, n, g, K, &bb);
    gather_kv(v_cache, cache_dtype, v_scale, num_blocks, num_kv_heads, block_size,
              head_dim, row, n, g, V, &bb);
    bad |= bb;
    int64_t qoff = ((int64_t)grow * num_q_heads + h) * head_dim;
    for (int d = 0; d < head_dim; ++d) qrow[d] = load_elem(q, qoff + d, q_dtype);
    int64_t ooff = num_rows > 0 ? (int64_t)i * head_dim : qoff;
    int64_t loff = num_rows > 0 ? i : (int64_t)grow * num_q_heads + h;
    attend_row(qrow, K, V, n, head_dim, sm_scale, s, out + ooff, lse + loff);
    free(K); free(V); free(s); free(qrow);
  }
  if (fail) return -1;
  return bad ? 1 : 0;
}

/* KV append on a byte image of the cache.  new_k/new_v [num_tokens][num_kv_heads]
 * [head_dim] in act dtype (f16/bf16).  Token t goes to slot slot_mapping[t]:
 * block slot / block_size, offset slot % block_size; slot < 0 is skipped.
 * Same cache dtype as act dtype: the 2 bytes are copied.  fp8 cache: the stored
 * code is e4m3(fp32(x) / fp32(scale)).  Returns 1 if a slot pointed outside the
 * pool (that token is skipped), else 0. */
int orc_kv_append(void* k_cache, void* v_cache, int cache_dtype, float k_scale,
                  float v_scale, int num_blocks, int num_kv_heads, int block_size,
                  int head_dim, const void* new_k, const void* new_v, int act_dtype,
                  const int64_t* slot_mapping, int num_tokens) {
  int bad = 0;
  for (int t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t blk = slot / block_size, off = slot % block_size;
    if (blk >= num_blocks) { bad = 1; continue; }
    for (int g = 0; g < num_kv_heads; ++g) {
      int64_t src = ((int64_t)t * num_kv_heads + g) * head_dim;
      int64_t dst = ((blk * num_kv_heads + g) * block_size + off) * head_dim;
      for (int d = 0; d < head_dim; ++d) {
        if (cache_dtype == act_dtype) {
          ((uint16_t*)k_cache)[dst + d] = ((const uint16_t*)new_k)[src + d];
          ((uint16_t*)v_cache)[dst + d] = ((const uint16_t*)new_v)[src + d];
        } else {
          float xk = load_elem_f32(new_k, src + d, act_dtype);
          float xv = load_elem_f32(new_v, src + d, act_dtype);
          ((uint8_t*)k_cache)[dst + d] = orc_e4m3_from_float(orc_div_f32(xk, k_scale));
          ((uint8_t*)v_cache)[dst + d] = orc_e4m3_from_float(orc_div_f32(xv, v_scale));
        }
      }
    }
  }
  return bad;
}

/* Bytes of K+V cache one token occupies across all layers:
 *   2 (K and V) x layers x kv_heads x head_dim x bytes per element.
 *   "KV Cache에 대해 알아보자 (Feat. Attention)", §4 (KV per token). */
uint64_t orc_kv_bytes_per_token(int layers, int kv_heads, int head_dim, int elem_bytes) {
  return 2ull * (uint64_t)layers * (uint64_t)kv_heads * (uint64_t)head_dim *
         (uint64_t)elem_bytes;
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
