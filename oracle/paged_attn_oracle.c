/*
 * Paged GQA decode / speculative-verify attention: FP64 CPU oracle.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * in __graft_entry__ and the CPU-baseline leg of bench.py may load this
 * library.  It shares no code, header, table or helper with the CUDA path in
 * paged_gqa_decode_split_gb300/csrc, and it is written as the plain definition
 * of the operation, one output row at a time, with no blocking, splitting or
 * online softmax.
 *
 * What it computes (one row = one request b, one verify query qi < q_len, one
 * query head h):
 *
 *   g      = h / (Hq / Hkv)                      query head -> KV head; the six
 *            query heads of a group share one KV head ("DFlash2 concurrent
 *            long-context attention", section "Why the single-request
 *            optimization was missing from concurrent decode": multiple
 *            six-query-head groups, GQA = 6).
 *   L      = ctx_lens[b]; n = L - q_len + qi + 1  keys visible to row qi: the
 *            q_len verify tokens are the last q_len tokens of the context, so
 *            query qi sees keys 0 .. L - q_len + qi (causal verify).
 *   key j  -> page block_table[b][j / page_size], slot j % page_size
 *   k_j    = E4M3(K bytes) * k_scale, v_j = E4M3(V bytes) * v_scale, one FP32
 *            scale per tensor (same section: E4M3 KV, FP16 queries, D = 256 is
 *            the kernel's numerical and shape contract).  An E5M2 cache (a KV
 *            type the same section names beside E4M3) is read the same way
 *            with the E5M2 decoder, and FP16 or BF16 caches (16-bit K/V, no
 *            scales) with the binary16 / bfloat16 decoders.
 *   s_j    = (q . k_j) / sqrt(D)
 *   out    = sum_j exp(s_j - max s) v_j / sum_j exp(s_j - max s)
 *   lse    = max s + log(sum_j exp(s_j - max s))
 *
 * A row with n <= 0 (zero-length request, padded slot, or a context shorter
 * than the verify window) has no keys: out = +0.0 in every element and
 * lse = -inf.  Q is not read for such a row, so a NaN in a padded slot's Q
 * cannot leak ("DFlash2 concurrent long-context attention", same section:
 * padded requests and zero-length rows remain safe).
 *
 * Everything is evaluated in IEEE double precision; the inputs (FP16 Q, E4M3
 * or BF16 K/V, FP32 scales) are widened exactly.  The pages require FP32 or
 * better accumulation for both QK and PV ("SM70 attention and quantized
 * projection coverage across TP sizes", section "Scope"); double is strictly
 * better and serves as the independent FP64 reference the pages check against
 * ("DFlash2 concurrent long-context attention", section "Operator
 * validation": an independent FP64 oracle checks the longest and shortest
 * requests, including multiple KV heads).
 *
 * Element decoders are written from the public format definitions:
 *   E4M3 (OCP 8-bit floating point specification, E4M3 variant): 1 sign bit,
 *     4 exponent bits with bias 7, 3 mantissa bits, no infinities, the two
 *     codes S.1111.111 are NaN; exponent field 0 is subnormal 2^-6 * m/8.
 *   E5M2 (same specification, E5M2 variant): 1 sign bit, 5 exponent bits with
 *     bias 15, 2 mantissa bits; exponent field 31 is infinity (m = 0) or NaN;
 *     exponent field 0 is subnormal 2^-14 * m/4.
 *   binary16 (IEEE 754): 1 sign, 5 exponent bits with bias 15, 10 mantissa.
 *   bfloat16: the upper 16 bits of an IEEE binary32.
 *
 * ORACLE_MUTATION (compile-time, default 0) plants one deliberate mistake; it
 * exists only so that the test suite can show each pin catches a plausible
 * error.  A normal build never defines it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

/* ---- element decoders ---------------------------------------------------- */

double oracle_e4m3_value(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
#if ORACLE_MUTATION == 4
  const int bias = 8;
#else
  const int bias = 7;
#endif
  if (e == 0) {
#if ORACLE_MUTATION == 8
    mag = ldexp(1.0 + m / 8.0, 1 - bias);
#else
    mag = ldexp(m / 8.0, 1 - bias); /* subnormal: 2^(1-bias) * m/8 */
#endif
  } else {
    mag = ldexp(1.0 + m / 8.0, e - bias);
  }
  return sign ? -mag : mag;
}

double oracle_e5m2_value(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 2) & 0x1F;
  int m = code & 0x3;
  double mag;
#if ORACLE_MUTATION == 11
  const int bias = 16;
#else
  const int bias = 15;
#endif
  if (e == 0x1F) {
    if (m != 0) return NAN;
    mag = INFINITY;
  } else if (e == 0) {
#if ORACLE_MUTATION == 12
    mag = ldexp(1.0 + m / 4.0, 1 - bias);
#else
    mag = ldexp(m / 4.0, 1 - bias); /* subnormal: 2^(1-bias) * m/4 */
#endif
  } else {
    mag = ldexp(1.0 + m / 4.0, e - bias);
  }
  return sign ? -mag : mag;
}

double oracle_f16_value(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 10) & 0x1F;
  int m = bits & 0x3FF;
  double mag;
#if ORACLE_MUTATION == 9
  const int bias = 16;
#else
  const int bias = 15;
#endif
  if (e == 0x1F) {
    if (m != 0) return NAN;
    mag = INFINITY;
  } else if (e == 0) {
    mag = ldexp((double)m, 1 - bias - 10);
  } else {
    mag = ldexp(1024.0 + m, e - bias - 10);
  }
  return sign ? -mag : mag;
}

double oracle_bf16_value(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* ---- one output row ------------------------------------------------------- */

enum { KV_BF16 = 0, KV_E4M3 = 1, KV_E5M2 = 2, KV_F16 = 3 };

typedef struct {
  int B, q_len, Hq, Hkv, D, page_size, max_pages_per_req;
  const uint16_t* q;      /* [B][q_len][Hq][D], FP16 or BF16 bits */
  const uint8_t* k_base;  /* byte address of key (page 0, slot 0, head 0, d 0) */
  const uint8_t* v_base;
  int64_t k_page_stride, k_token_stride, k_head_stride; /* bytes */
  int64_t v_page_stride, v_token_stride, v_head_stride;
  const int32_t* block_table; /* [B][max_pages_per_req] */
  const int32_t* ctx_lens;    /* [B] */
  double k_scale, v_scale;    /* 1.0 for BF16 K/V */
  int kv_format;              /* KV_BF16, KV_E4M3, KV_E5M2 or KV_F16 */
  int q_is_bf16;              /* 0: FP16 Q, 1: BF16 Q */
} problem_t;

static double load_q(const problem_t* P, size_t idx) {
  return P->q_is_bf16 ? oracle_bf16_value(P->q[idx]) : oracle_f16_value(P->q[idx]);
}

static double load_kv(const problem_t* P, const uint8_t* row, int d, double scale) {
  if (P->kv_format == KV_E4M3) return oracle_e4m3_value(row[d]) * scale;
  if (P->kv_format == KV_E5M2) return oracle_e5m2_value(row[d]) * scale;
  uint16_t bits;
  memcpy(&bits, row + 2 * (size_t)d, 2);
  return P->kv_format == KV_F16 ? oracle_f16_value(bits) : oracle_bf16_value(bits);
}

static const uint8_t* key_row(const problem_t* P, const uint8_t* base, int64_t ps_, int64_t ts_, int64_t hs_,
                              int b, int j, int g) {
#if ORACLE_MUTATION == 6
  int page = P->block_table[(size_t)b * P->max_pages_per_req + j % P->page_size];
  int slot = j / P->page_size;
#else
  int page = P->block_table[(size_t)b * P->max_pages_per_req + j / P->page_size];
  int slot = j % P->page_size;
#endif
  return base + (int64_t)page * ps_ + (int64_t)slot * ts_ + (int64_t)g * hs_;
}

/* row index r = (b * q_len + qi) * Hq + h ; writes out[0..D) and *lse */
static void attend_row(const problem_t* P, int r, double* out, double* lse, double* s, double* acc) {
  int h = r % P->Hq;
  int qi = (r / P->Hq) % P->q_len;
  int b = r / (P->Hq * P->q_len);
  int D = P->D;
  int group = P->Hq / P->Hkv;
#if ORACLE_MUTATION == 3
  int g = h % P->Hkv;
#else
  int g = h / group;
#endif
  int L = P->ctx_lens[b];
#if ORACLE_MUTATION == 2
  int n = L - P->q_len + qi;
#else
  int n = L - P->q_len + qi + 1;
#endif
  if (n <= 0) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    *lse = -INFINITY;
    return;
  }
  size_t qoff = (size_t)r * D;
#if ORACLE_MUTATION == 1
  double inv_sqrt_d = 1.0;
#else
  double inv_sqrt_d = 1.0 / sqrt((double)D);
#endif
  for (int j = 0; j < n; ++j) {
    const uint8_t* krow = key_row(P, P->k_base, P->k_page_stride, P->k_token_stride, P->k_head_stride, b, j, g);
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += load_q(P, qoff + d) * load_kv(P, krow, d, P->k_scale);
    s[j] = dot * inv_sqrt_d;
  }
  double mx = -INFINITY;
  for (int j = 0; j < n; ++j) mx = s[j] > mx ? s[j] : mx;
  double sum = 0.0;
  for (int j = 0; j < n; ++j) {
#if ORACLE_MUTATION == 7
    s[j] = exp(mx - s[j]);
#else
    s[j] = exp(s[j] - mx);
#endif
    sum += s[j];
  }
  for (int d = 0; d < D; ++d) acc[d] = 0.0;
#if ORACLE_MUTATION == 5
  double vs = 1.0;
#else
  double vs = P->v_scale;
#endif
  for (int j = 0; j < n; ++j) {
    const uint8_t* vrow = key_row(P, P->v_base, P->v_page_stride, P->v_token_stride, P->v_head_stride, b, j, g);
    for (int d = 0; d < D; ++d) acc[d] += s[j] * load_kv(P, vrow, d, vs);
  }
  for (int d = 0; d < D; ++d) out[d] = acc[d] / sum;
#if ORACLE_MUTATION == 10
  *lse = log(sum);
#else
  *lse = mx + log(sum);
#endif
}

static int run(const problem_t* P, const int32_t* rows, int n_rows, double* out, double* lse, int num_threads) {
  int total_rows = P->B * P->q_len * P->Hq;
  int count = rows ? n_rows : total_rows;
  int max_ctx = 0;
  for (int b = 0; b < P->B; ++b) max_ctx = P->ctx_lens[b] > max_ctx ? P->ctx_lens[b] : max_ctx;
  if (rows)
    for (int i = 0; i < n_rows; ++i)
      if (rows[i] < 0 || rows[i] >= total_rows) return -1;
  int failed = 0;
#if ORACLE_MUTATION == 14
  /* planted mistake: one scratch buffer shared by every thread */
  double* shared_s = (double*)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
  double* shared_acc = (double*)malloc(sizeof(double) * (size_t)P->D);
#endif
#ifdef _OPENMP
  if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel num_threads(num_threads)
#endif
  {
    /* each thread owns its score and accumulator scratch */
#if ORACLE_MUTATION == 14
    double* s = shared_s;
    double* acc = shared_acc;
#else
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    double* acc = (double*)malloc(sizeof(double) * (size_t)P->D);
#endif
    if (!s || !acc) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int i = 0; i < count; ++i) {
        int r = rows ? rows[i] : i;
        /* the i-th requested row goes to slot i of out and lse */
#if ORACLE_MUTATION == 13
        attend_row(P, r, out + (size_t)r * P->D, lse + r, s, acc);
#else
        attend_row(P, r, out + (size_t)i * P->D, lse + i, s, acc);
#endif
      }
    }
#if ORACLE_MUTATION != 14
    free(s);
    free(acc);
#endif
  }
#if ORACLE_MUTATION == 14
  free(shared_s);
  free(shared_acc);
#endif
  return failed ? -2 : 0;
}

/*
 * FP16 Q, E4M3 K/V with one FP32 scale per tensor.
 * rows == NULL: every row, out is [B][q_len][Hq][D] and lse [B][q_len][Hq].
 * rows != NULL: only the listed flat rows ((b * q_len + qi) * Hq + h), out is
 * [n_rows][D] and lse [n_rows].  Returns 0, or a negative value on a bad row
 * index or allocation failure.
 */
int oracle_paged_attn_fp8(int B, int q_len, int Hq, int Hkv, int D, int page_size, int max_pages_per_req,
                          const uint16_t* q, const uint8_t* k_base, const uint8_t* v_base,
                          int64_t k_page_stride, int64_t k_token_stride, int64_t k_head_stride,
                          int64_t v_page_stride, int64_t v_token_stride, int64_t v_head_stride,
                          const int32_t* block_table, const int32_t* ctx_lens, float k_scale, float v_scale,
                          const int32_t* rows, int n_rows, double* out, double* lse, int num_threads) {
  problem_t P = {B, q_len, Hq, Hkv, D, page_size, max_pages_per_req, q, k_base, v_base,
                 k_page_stride, k_token_stride, k_head_stride, v_page_stride, v_token_stride, v_head_stride,
                 block_table, ctx_lens, (double)k_scale, (double)v_scale, KV_E4M3, 0};
  return run(&P, rows, n_rows, out, lse, num_threads);
}

/*
 * FP16 Q, E5M2 K/V with one FP32 scale per tensor.  Same arguments, row
 * selection and outputs as oracle_paged_attn_fp8.
 */
int oracle_paged_attn_e5m2(int B, int q_len, int Hq, int Hkv, int D, int page_size, int max_pages_per_req,
                           const uint16_t* q, const uint8_t* k_base, const uint8_t* v_base,
                           int64_t k_page_stride, int64_t k_token_stride, int64_t k_head_stride,
                           int64_t v_page_stride, int64_t v_token_stride, int64_t v_head_stride,
                           const int32_t* block_table, const int32_t* ctx_lens, float k_scale, float v_scale,
                           const int32_t* rows, int n_rows, double* out, double* lse, int num_threads) {
  problem_t P = {B, q_len, Hq, Hkv, D, page_size, max_pages_per_req, q, k_base, v_base,
                 k_page_stride, k_token_stride, k_head_stride, v_page_stride, v_token_stride, v_head_stride,
                 block_table, ctx_lens, (double)k_scale, (double)v_scale, KV_E5M2, 0};
  return run(&P, rows, n_rows, out, lse, num_threads);
}

/*
 * FP16 Q, K, V (no scales).  Strides are in bytes.  Same row selection and
 * outputs as oracle_paged_attn_fp8.
 */
int oracle_paged_attn_f16(int B, int q_len, int Hq, int Hkv, int D, int page_size, int max_pages_per_req,
                          const uint16_t* q, const uint8_t* k_base, const uint8_t* v_base,
                          int64_t k_page_stride, int64_t k_token_stride, int64_t k_head_stride,
                          int64_t v_page_stride, int64_t v_token_stride, int64_t v_head_stride,
                          const int32_t* block_table, const int32_t* ctx_lens,
                          const int32_t* rows, int n_rows, double* out, double* lse, int num_threads) {
  problem_t P = {B, q_len, Hq, Hkv, D, page_size, max_pages_per_req, q, k_base, v_base,
                 k_page_stride, k_token_stride, k_head_stride, v_page_stride, v_token_stride, v_head_stride,
                 block_table, ctx_lens, 1.0, 1.0, KV_F16, 0};
  return run(&P, rows, n_rows, out, lse, num_threads);
}

/*
 * BF16 Q, K, V (no scales).  Strides are in bytes.  Same row selection and
 * outputs as oracle_paged_attn_fp8.
 */
int oracle_paged_attn_bf16(int B, int q_len, int Hq, int Hkv, int D, int page_size, int max_pages_per_req,
                           const uint16_t* q, const uint8_t* k_base, const uint8_t* v_base,
                           int64_t k_page_stride, int64_t k_token_stride, int64_t k_head_stride,
                           int64_t v_page_stride, int64_t v_token_stride, int64_t v_head_stride,
                           const int32_t* block_table, const int32_t* ctx_lens,
                           const int32_t* rows, int n_rows, double* out, double* lse, int num_threads) {
  problem_t P = {B, q_len, Hq, Hkv, D, page_size, max_pages_per_req, q, k_base, v_base,
                 k_page_stride, k_token_stride, k_head_stride, v_page_stride, v_token_stride, v_head_stride,
                 block_table, ctx_lens, 1.0, 1.0, KV_BF16, 1};
  return run(&P, rows, n_rows, out, lse, num_threads);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

int oracle_mutation(void) { return ORACLE_MUTATION; }
