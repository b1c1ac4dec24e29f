/*
 * decattn_oracle.c -- plain, slow, fp64 CPU oracle for single-token decode
 * attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * Every function below is the plain definition written out with loops, in
 * double precision, with no blocking, fusion or reordering:
 *
 *   - cache gather: token t of sequence b lives in physical block
 *     block_table[b][t / block_size], slot t % block_size
 *     ("Compressing the KV Cache: DeepSeek's Latent Projections (MLA) vs.
 *     Meta's Grouped Queries (GQA)", "KV-Cache Management Guardrails":
 *     paged KV blocks);
 *   - GQA/MHA/MQA decode: query head i reads KV head i / (h_q / h_kv)
 *     ("MQA, GQA, and MLA", section 8 "Implementation notes", GQA in the
 *     kernel; section 2 "The three answers"), scores q . k scaled,
 *     softmax over the cached tokens (base e, max-subtracted), output the
 *     probability-weighted sum of the values;
 *   - absorbed MLA decode: the query is pre-multiplied by W_uk and scored
 *     against the cached latent, plus a decoupled RoPE part scored against
 *     the cached 64-d RoPE key; the latent itself is the value
 *     ("MQA, GQA, and MLA", section 5 "MLA, mechanically", KEY TRICK;
 *     "Why GQA's KV Cache Savings Don't Fully Reduce TPOT", "What Makes MLA
 *     Different");
 *   - explicit MLA: K and V reconstructed per head from the latent
 *     (k_i = c W_uk^(i), v_i = c W_uv^(i)), then ordinary attention
 *     ("MQA, GQA, and MLA", section 5, "at read time");
 *   - log-sum-exp merge of partial results over disjoint token ranges;
 *   - per-token cache-size formulas ("Why GQA's KV Cache Savings Don't Fully
 *     Reduce TPOT", "KV Cache Size by Attention Variant"; "MQA, GQA, and
 *     MLA", section 5 "CACHE SIZE COMPARISON").
 *
 *   - 8-bit KV cache: e4m3 codes dequantised with one scale per KV head,
 *     then the GQA decode above on the dequantised values ("Why GQA's KV
 *     Cache Savings Don't Fully Reduce TPOT", "When the Serving Engineer
 *     Doesn't Get to Choose the Model Architecture": an fp8 cache halves the
 *     bytes and GQA quantises at KV-head granularity; "07 · MHA/MQA/GQA/MLA
 *     quick learn", the question on changing the KV head count by a flag).
 *
 * Element storage: dtype 0 = IEEE binary16, 1 = bfloat16, 2 = binary64.
 * The two 16-bit formats and the 8-bit e4m3 format are decoded here from
 * their bit-layout definitions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_FP16 0
#define ORACLE_BF16 1
#define ORACLE_F64 2

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_BLOCK (-2)

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/2^10) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 word. */
double oracle_bf16_to_double(uint16_t h) {
  uint32_t w = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* 8-bit float e4m3 (finite-only variant): 1 sign bit, 4 exponent bits
 * (bias 7), 3 fraction bits.  Exponent field 0 holds subnormals
 * frac * 2^-9; exponent field 15 with fraction 7 is NaN (the only
 * non-finite code); every other code is (1 + frac/8) * 2^(e - 7).  Largest
 * finite magnitude 448. */
double oracle_e4m3_to_double(uint8_t c) {
  int sign = (c >> 7) & 1;
  int expo = (c >> 3) & 0xf;
  int frac = c & 0x7;
  double v;
  if (expo == 0xf && frac == 0x7) {
    v = NAN;
  } else if (expo == 0) {
    v = ldexp((double)frac, -9);
  } else {
    v = ldexp((double)(8 + frac), expo - 10); /* (1 + frac/8) * 2^(e-7) */
  }
  return sign ? -v : v;
}

/* Dequantise an e4m3 KV cache laid out [rows][h_kv][d] with one scale per KV
 * head: out[r][j][e] = e4m3(codes[r][j][e]) * scale[j]. */
void oracle_dequant_e4m3(const uint8_t* codes, int64_t rows, int h_kv, int d,
                         const double* scale, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int j = 0; j < h_kv; ++j)
      for (int e = 0; e < d; ++e) {
        const int64_t i = (r * h_kv + j) * d + e;
        out[i] = oracle_e4m3_to_double(codes[i]) * scale[j];
      }
}

/* e4m3 code of the finite e4m3 value nearest to y (largest magnitude 448):
 * ties go to the even code (last fraction bit 0); every magnitude above 448,
 * infinity included, takes 448 (saturation); the sign is kept, zero
 * included; NaN gives the NaN code 0x7F.  Written as a search over the 127
 * non-negative finite codes, so that it is checkable by eye. */
uint8_t oracle_e4m3_from_float(float y) {
  if (isnan(y)) return 0x7F;
  const uint8_t sign = signbit(y) ? 0x80 : 0x00;
  if (isinf(y)) return sign | 0x7E;
  const double a = fabs((double)y);
  int best = 0;
  double best_d = a; /* distance to code 0x00 (value 0) */
  for (int c = 1; c <= 0x7E; ++c) {
    const double d = fabs(oracle_e4m3_to_double((uint8_t)c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)(sign | best);
}

void oracle_e4m3_from_float_array(const float* y, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_from_float(y[i]);
}

/* Quantise 16-bit values laid out [rows][h_kv][d] to e4m3 codes with one
 * scale per KV head: code = e4m3 nearest to (fp32 x) / scale[j], the
 * quotient rounded to fp32 (the cached value is then e4m3(code) * scale[j]). */
void oracle_quant_e4m3(const uint16_t* x, int dtype, int64_t rows, int h_kv, int d,
                       const float* scale, uint8_t* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int j = 0; j < h_kv; ++j)
      for (int e = 0; e < d; ++e) {
        const int64_t i = (r * h_kv + j) * d + e;
        const float xf = (float)(dtype == ORACLE_FP16 ? oracle_half_to_double(x[i])
                                                      : oracle_bf16_to_double(x[i]));
        const float q = xf / scale[j];
        out[i] = oracle_e4m3_from_float(q);
      }
}

void oracle_decode_array(const uint16_t* src, int dtype, int64_t n, double* dst) {
  for (int64_t i = 0; i < n; ++i)
    dst[i] = dtype == ORACLE_FP16 ? oracle_half_to_double(src[i]) : oracle_bf16_to_double(src[i]);
}

static double elem(const void* base, int dtype, int64_t idx) {
  if (dtype == ORACLE_F64) return ((const double*)base)[idx];
  uint16_t h = ((const uint16_t*)base)[idx];
  return dtype == ORACLE_FP16 ? oracle_half_to_double(h) : oracle_bf16_to_double(h);
}

/* Cache gather: physical row (block * block_size + slot) holding token t of
 * sequence b, or -1 when the block id is outside [0, num_blocks). */
int64_t oracle_cache_row(const int32_t* block_table, int max_blocks_per_seq, int block_size,
                         int num_blocks, int b, int t) {
  int32_t blk = block_table[(int64_t)b * max_blocks_per_seq + t / block_size];
  if (blk < 0 || blk >= num_blocks) return -1;
  return (int64_t)blk * block_size + t % block_size;
}

/* Token range [t0, t1) actually attended by sequence b: the requested range
 * clipped to [0, seq_lens[b]). t_end < 0 means "to the end of the sequence". */
static void token_range(const int32_t* seq_lens, int b, int t_begin, int t_end, int* t0, int* t1) {
  int s = seq_lens[b];
  int e = (t_end < 0 || t_end > s) ? s : t_end;
  int a = t_begin < 0 ? 0 : t_begin;
  if (a > e) a = e;
  *t0 = a;
  *t1 = e;
}

/*
 * GQA / MHA / MQA decode (one query token per sequence).
 *
 * q        [batch, h_q, d_head]
 * k_cache  [num_blocks, block_size, h_kv, d_head]
 * v_cache  [num_blocks, block_size, h_kv, d_head]
 * rows     n_rows pairs (b, i); NULL means every (b, i) in order b-major.
 * out      [n_rows, d_head], lse [n_rows] (natural log).
 */
int oracle_gqa_decode(const void* q, const void* k_cache, const void* v_cache, int dtype,
                      const int32_t* block_table, const int32_t* seq_lens, int batch, int h_q,
                      int h_kv, int d_head, int num_blocks, int block_size,
                      int max_blocks_per_seq, double scale, const int32_t* rows, int n_rows,
                      int t_begin, int t_end, double* out, double* lse) {
  if (h_kv <= 0 || h_q % h_kv != 0 || d_head <= 0 || block_size <= 0) return ORACLE_BAD_ARG;
  if (rows == NULL) n_rows = batch * h_q;
  const int group = h_q / h_kv; /* query heads per KV head */
  int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < n_rows; ++r) {
    const int b = rows ? rows[2 * r] : r / h_q;
    const int i = rows ? rows[2 * r + 1] : r % h_q;
    const int j = i / group; /* the KV head this query head reads */
    int t0, t1;
    token_range(seq_lens, b, t_begin, t_end, &t0, &t1);
    double* o = out + (int64_t)r * d_head;
    for (int e = 0; e < d_head; ++e) o[e] = 0.0;
    if (t1 <= t0) {
      lse[r] = -INFINITY;
      continue;
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)(t1 - t0));
    int bad = 0;
    /* scores s_t = scale * q_i . k_{j,t} */
    for (int t = t0; t < t1; ++t) {
      int64_t row = oracle_cache_row(block_table, max_blocks_per_seq, block_size, num_blocks, b, t);
      if (row < 0) { bad = 1; break; }
      double dot = 0.0;
      for (int e = 0; e < d_head; ++e)
        dot += elem(q, dtype, ((int64_t)b * h_q + i) * d_head + e) *
               elem(k_cache, dtype, (row * h_kv + j) * d_head + e);
      s[t - t0] = scale * dot;
    }
    if (bad) {
      free(s);
#pragma omp atomic write
      status = ORACLE_BAD_BLOCK;
      for (int e = 0; e < d_head; ++e) o[e] = NAN;
      lse[r] = NAN;
      continue;
    }
    /* softmax (base e, max-subtracted) and the weighted sum of values */
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) m = s[t - t0] > m ? s[t - t0] : m;
    double den = 0.0;
    for (int t = t0; t < t1; ++t) den += exp(s[t - t0] - m);
    for (int t = t0; t < t1; ++t) {
      double p = exp(s[t - t0] - m) / den;
      int64_t row = oracle_cache_row(block_table, max_blocks_per_seq, block_size, num_blocks, b, t);
      for (int e = 0; e < d_head; ++e)
        o[e] += p * elem(v_cache, dtype, (row * h_kv + j) * d_head + e);
    }
    lse[r] = m + log(den);
    free(s);
  }
  return status;
}

/*
 * Absorbed MLA decode.
 *
 * q_abs    [batch, n_heads, d_c]   query already multiplied by W_uk^(i)
 * q_rope   [batch, n_heads, d_r]   decoupled-RoPE part of the query
 * cache    [num_blocks, block_size, d_c + d_r]: latent c_t in [0, d_c),
 *          the shared RoPE key in [d_c, d_c + d_r)
 * score    s_t = scale * (q_abs . c_t + q_rope . kr_t)
 * output   sum_t p_t c_t  (the latent is the value; W_uv is applied later)
 * rows     n_rows pairs (b, i); NULL means every (b, i) b-major.
 * out      [n_rows, d_c], lse [n_rows].
 */
int oracle_mla_decode(const void* q_abs, const void* q_rope, const void* cache, int dtype,
                      const int32_t* block_table, const int32_t* seq_lens, int batch, int n_heads,
                      int d_c, int d_r, int num_blocks, int block_size, int max_blocks_per_seq,
                      double scale, const int32_t* rows, int n_rows, int t_begin, int t_end,
                      double* out, double* lse) {
  if (n_heads <= 0 || d_c <= 0 || d_r < 0 || block_size <= 0) return ORACLE_BAD_ARG;
  if (rows == NULL) n_rows = batch * n_heads;
  const int width = d_c + d_r; /* elements per cached token */
  int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < n_rows; ++r) {
    const int b = rows ? rows[2 * r] : r / n_heads;
    const int i = rows ? rows[2 * r + 1] : r % n_heads;
    int t0, t1;
    token_range(seq_lens, b, t_begin, t_end, &t0, &t1);
    double* o = out + (int64_t)r * d_c;
    for (int e = 0; e < d_c; ++e) o[e] = 0.0;
    if (t1 <= t0) {
      lse[r] = -INFINITY;
      continue;
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)(t1 - t0));
    int bad = 0;
    for (int t = t0; t < t1; ++t) {
      int64_t row = oracle_cache_row(block_table, max_blocks_per_seq, block_size, num_blocks, b, t);
      if (row < 0) { bad = 1; break; }
      double dot_latent = 0.0, dot_rope = 0.0;
      for (int e = 0; e < d_c; ++e)
        dot_latent += elem(q_abs, dtype, ((int64_t)b * n_heads + i) * d_c + e) *
                      elem(cache, dtype, row * width + e);
      for (int e = 0; e < d_r; ++e)
        dot_rope += elem(q_rope, dtype, ((int64_t)b * n_heads + i) * d_r + e) *
                    elem(cache, dtype, row * width + d_c + e);
      s[t - t0] = scale * (dot_latent + dot_rope);
    }
    if (bad) {
      free(s);
#pragma omp atomic write
      status = ORACLE_BAD_BLOCK;
      for (int e = 0; e < d_c; ++e) o[e] = NAN;
      lse[r] = NAN;
      continue;
    }
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) m = s[t - t0] > m ? s[t - t0] : m;
    double den = 0.0;
    for (int t = t0; t < t1; ++t) den += exp(s[t - t0] - m);
    for (int t = t0; t < t1; ++t) {
      double p = exp(s[t - t0] - m) / den;
      int64_t row = oracle_cache_row(block_table, max_blocks_per_seq, block_size, num_blocks, b, t);
      for (int e = 0; e < d_c; ++e) o[e] += p * elem(cache, dtype, row * width + e);
    }
    lse[r] = m + log(den);
    free(s);
  }
  return status;
}

/*
 * Explicit (non-absorbed) MLA for one sequence, all in fp64: reconstruct
 * k_{i,t} = c_t W_uk^(i) and v_{i,t} = c_t W_uv^(i) for every head, score
 * scale * (q_nope_i . k_{i,t} + q_rope_i . kr_t), softmax, out_i = sum p v.
 *
 * q_nope [h, d_h], q_rope [h, d_r], c [S, d_c], k_rope [S, d_r],
 * w_uk [h, d_c, d_h], w_uv [h, d_c, d_v]; out [h, d_v]; scores [h, S].
 */
int oracle_mla_explicit(const double* q_nope, const double* q_rope, const double* c,
                        const double* k_rope, const double* w_uk, const double* w_uv, int S,
                        int h, int d_c, int d_h, int d_r, int d_v, double scale, double* out,
                        double* scores) {
  if (S <= 0 || h <= 0) return ORACLE_BAD_ARG;
  double* k = (double*)malloc(sizeof(double) * (size_t)d_h);
  double* v = (double*)malloc(sizeof(double) * (size_t)S * d_v);
  for (int i = 0; i < h; ++i) {
    double* s = scores + (int64_t)i * S;
    for (int t = 0; t < S; ++t) {
      /* k_{i,t} = c_t W_uk^(i): row vector times a d_c x d_h matrix */
      for (int e = 0; e < d_h; ++e) {
        double acc = 0.0;
        for (int a = 0; a < d_c; ++a) acc += c[(int64_t)t * d_c + a] * w_uk[((int64_t)i * d_c + a) * d_h + e];
        k[e] = acc;
      }
      for (int e = 0; e < d_v; ++e) {
        double acc = 0.0;
        for (int a = 0; a < d_c; ++a) acc += c[(int64_t)t * d_c + a] * w_uv[((int64_t)i * d_c + a) * d_v + e];
        v[(int64_t)t * d_v + e] = acc;
      }
      double dot = 0.0;
      for (int e = 0; e < d_h; ++e) dot += q_nope[(int64_t)i * d_h + e] * k[e];
      for (int e = 0; e < d_r; ++e) dot += q_rope[(int64_t)i * d_r + e] * k_rope[(int64_t)t * d_r + e];
      s[t] = scale * dot;
    }
    double m = -INFINITY;
    for (int t = 0; t < S; ++t) m = s[t] > m ? s[t] : m;
    double den = 0.0;
    for (int t = 0; t < S; ++t) den += exp(s[t] - m);
    for (int e = 0; e < d_v; ++e) out[(int64_t)i * d_v + e] = 0.0;
    for (int t = 0; t < S; ++t) {
      double p = exp(s[t] - m) / den;
      for (int e = 0; e < d_v; ++e) out[(int64_t)i * d_v + e] += p * v[(int64_t)t * d_v + e];
    }
  }
  free(k);
  free(v);
  return ORACLE_OK;
}

/*
 * Log-sum-exp merge of n_parts partial results over disjoint token ranges.
 * o_parts [n_parts, d] are each normalised softmax outputs over their range,
 * lse_parts [n_parts] their natural-log log-sum-exp (-inf for an empty range).
 * out = sum_j w_j o_j / sum_j w_j with w_j = exp(lse_j - max lse);
 * lse_out = max + log(sum_j w_j).  All parts empty gives out = 0, lse = -inf.
 */
void oracle_lse_merge(int n_parts, int d, const double* o_parts, const double* lse_parts,
                      double* out, double* lse_out) {
  double m = -INFINITY;
  for (int j = 0; j < n_parts; ++j) m = lse_parts[j] > m ? lse_parts[j] : m;
  for (int e = 0; e < d; ++e) out[e] = 0.0;
  if (m == -INFINITY) {
    *lse_out = -INFINITY;
    return;
  }
  double wsum = 0.0;
  for (int j = 0; j < n_parts; ++j) wsum += exp(lse_parts[j] - m);
  for (int j = 0; j < n_parts; ++j) {
    double w = exp(lse_parts[j] - m) / wsum;
    for (int e = 0; e < d; ++e) out[e] += w * o_parts[(int64_t)j * d + e];
  }
  *lse_out = m + log(wsum);
}

/* KV cache bytes per token: n_layers x n_kv x d_head x 2 (K and V) x bytes
 * ("Why GQA's KV Cache Savings Don't Fully Reduce TPOT", "KV Cache Size by
 * Attention Variant"; "MQA, GQA, and MLA", section 1). */
int64_t oracle_kv_bytes_per_token(int n_layers, int n_kv, int d_head, int bytes) {
  return (int64_t)2 * n_layers * n_kv * d_head * bytes;
}

/* MLA cache bytes per token: n_layers x (d_c + d_r) x bytes ("MQA, GQA, and
 * MLA", section 5 "CACHE SIZE COMPARISON": 60 x (512 + 64) x 2). */
int64_t oracle_mla_bytes_per_token(int n_layers, int d_c, int d_r, int bytes) {
  return (int64_t)n_layers * (d_c + d_r) * bytes;
}
