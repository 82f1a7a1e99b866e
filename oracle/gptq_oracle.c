/*
 * gptq_oracle.c -- plain, single-threaded CPU oracle for the GPTQ mixed-precision GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or calls this
 * file; only the test suite, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it follows (page = "增强 vLLM 对 GPTQv2 格式的支持：分析与实现", xxxxyu.github.io):
 *   - section "LLM 的权重量化": the b-bit quantizer
 *         scale = (wmax - wmin) / (2^b - 1),  zero = -round(wmin / scale),
 *         q = clamp(round(w / scale) + zero)
 *     its inverse  w_hat = (q - zero) * scale,  and the symmetric case whose zero is the
 *     fixed value round((2^b - 1) / 2);
 *   - section "从 GPTQv1 到 GPTQv2": GPTQv1 stores clamp(zero - 1) and adds 1 before
 *     dequantizing, GPTQv2 stores zero exactly; v1 -> v2 is lossless;
 *   - section "调整细节：根据格式选择处理方式": zero_offset = use_v2_format ? 0 : 1, and the
 *     reconstruct/dequant kernel that unpacks 16 two-bit codes from one int32 word.
 *
 * Readings taken where the page is silent (each one is listed in the design notes):
 *   - codes are packed LSB-first into a bit stream of consecutive int32 words: code i
 *     occupies stream bits [b*i, b*i + b).  qweight packs along K (column n's stream is
 *     qweight[0][n], qweight[1][n], ...), qzeros packs along N (row g's stream is
 *     qzeros[g][0], qzeros[g][1], ...).  For b = 3 a code may straddle two words;
 *   - words are bit patterns (read as uint32);
 *   - the v1 runtime zero is stored + 1 in plain integer arithmetic (no b-bit wrap);
 *   - round() is round-half-to-even; clamp() is to [0, 2^b - 1]; the zero is clamped to
 *     the same range; the scale is computed in fp32 and stored as fp16, and zero and q
 *     are computed with the stored (fp16) scale; a scale that rounds to 0 becomes 1;
 *   - the symmetric scale is 2 * max|w| / (2^b - 1);
 *   - group = -1 means one group spanning all K rows; with g_idx, row k belongs to group
 *     g_idx[k];
 *   - the dequantized weight is the fp32 product (q - zero) * scale (exact: |q - zero| needs
 *     at most 9 bits, the fp16 scale 11) rounded once, to nearest-even, to the activation
 *     dtype (fp16 or bf16);
 *   - C[m,n] = sum over k ascending of fp32(A[m,k]) * w32[k,n], every product and every
 *     partial sum rounded to fp32 (no fused multiply-add: built with -ffp-contract=off).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_EARG -1
#define OR_ESHAPE -2
#define OR_EOVERFLOW -5
#define OR_ENOMEM -7

#define OR_FMT_V1 1
#define OR_FMT_V2 2
#define OR_F16 0
#define OR_BF16 1

/* ------------------------------------------------------------------------------------ */
/* 16-bit floating point formats, written from their IEEE-754 / bfloat16 definitions.    */
/* ------------------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, f = h & 0x3ff;
  double mag;
  if (e == 0) mag = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
  else if (e == 31) mag = f ? NAN : INFINITY;
  else mag = ldexp((double)(1024 + f), e - 15 - 10);     /* 1.f * 2^(e-15) */
  return sign ? -mag : mag;
}

/* bfloat16: the upper 16 bits of a binary32. */
double oracle_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round x to the nearest value with `p` significant bits whose exponent is at least
 * `emin` (the format's smallest normal exponent), ties to even.  Exact in double for
 * every binary32 input.  Returns the rounded value (may exceed the format's range). */
static double or_round_sig(double x, int p, int emin) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e;
  frexp(fabs(x), &e);          /* |x| = f * 2^e, f in [0.5, 1): unbiased exponent e - 1 */
  int E = e - 1;
  if (E < emin) E = emin;      /* subnormal range: fixed quantum */
  double quantum = ldexp(1.0, E - (p - 1));
  return rint(x / quantum) * quantum;   /* rint: current mode = round-half-even */
}

uint16_t oracle_double_to_half_rne(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return 0x7e00;
  double r = or_round_sig(x, 11, -14);
  double a = fabs(r);
  if (a >= 65536.0 || isinf(a)) return sign | 0x7c00;   /* rounds past 65504: inf */
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);
  int E = e - 1;
  if (E < -14) return sign | (uint16_t)ldexp(a, 24);     /* subnormal: a / 2^-24 */
  uint16_t frac = (uint16_t)(ldexp(a, 10 - E) - 1024.0);
  return sign | (uint16_t)((E + 15) << 10) | frac;
}

uint16_t oracle_double_to_bf16_rne(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return 0x7fc0;
  double r = or_round_sig(x, 8, -126);
  double a = fabs(r);
  if (a >= ldexp(1.0, 128) || isinf(a)) return sign | 0x7f80;
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);
  int E = e - 1;
  if (E < -126) return sign | (uint16_t)ldexp(a, 133);   /* subnormal: a / 2^-133 */
  uint16_t frac = (uint16_t)(ldexp(a, 7 - E) - 128.0);
  return sign | (uint16_t)((E + 127) << 7) | frac;
}

static double or_act_to_double(uint16_t v, int dtype) {
  return dtype == OR_BF16 ? oracle_bf16_to_double(v) : oracle_half_to_double(v);
}

/* ------------------------------------------------------------------------------------ */
/* Bit streams: code i of a stream occupies bits [b*i, b*i+b), LSB first, over words.   */
/* ------------------------------------------------------------------------------------ */

/* Read code i of a stream whose w-th word is words[w * stride]. */
static uint32_t or_stream_get(const int32_t* words, int64_t stride, int bits, int64_t i) {
  uint32_t code = 0;
  for (int t = 0; t < bits; t++) {
    int64_t pos = (int64_t)bits * i + t;
    uint32_t word = (uint32_t)words[(pos / 32) * stride];
    code |= ((word >> (pos % 32)) & 1u) << t;
  }
  return code;
}

/* Write code i (its low `bits` bits) into the stream. */
static void or_stream_put(int32_t* words, int64_t stride, int bits, int64_t i, uint32_t code) {
  for (int t = 0; t < bits; t++) {
    int64_t pos = (int64_t)bits * i + t;
    uint32_t* w = (uint32_t*)&words[(pos / 32) * stride];
    uint32_t m = 1u << (pos % 32);
    if ((code >> t) & 1u) *w |= m; else *w &= ~m;
  }
}

static int or_bits_ok(int bits) { return bits == 2 || bits == 3 || bits == 4 || bits == 8; }

/* Rows of qweight for K codes per column, words of a qzeros row for N codes. */
int64_t oracle_packed_len(int64_t count, int bits) { return count * bits / 32; }

/* Check shapes: K and N must fill whole words, group must divide K. */
static int or_check(int K, int N, int bits, int group, const int32_t* g_idx, int* G) {
  if (!or_bits_ok(bits)) return OR_EARG;
  if (K <= 0 || N <= 0) return OR_ESHAPE;
  if (((int64_t)K * bits) % 32 || ((int64_t)N * bits) % 32) return OR_ESHAPE;
  if (bits == 3 && (K % 32 || N % 32)) return OR_ESHAPE;
  if (group == -1) { *G = 1; return g_idx ? OR_ESHAPE : OR_OK; }
  if (group <= 0 || K % group) return OR_ESHAPE;
  *G = K / group;
  return OR_OK;
}

static int or_group_of(const int32_t* g_idx, int group, int64_t k) {
  if (g_idx) return g_idx[k];
  return group == -1 ? 0 : (int)(k / group);
}

/* Unpack every code of qweight ([K*bits/32, N]) into q[K][N]. */
int oracle_unpack_k(const int32_t* qweight, int K, int N, int bits, uint8_t* q) {
  if (!or_bits_ok(bits)) return OR_EARG;
  for (int64_t k = 0; k < K; k++)
    for (int64_t n = 0; n < N; n++)
      q[k * N + n] = (uint8_t)or_stream_get(qweight + n, N, bits, k);
  return OR_OK;
}

/* Unpack every code of qzeros ([G, N*bits/32]) into z[G][N] (stored values). */
int oracle_unpack_n(const int32_t* qzeros, int G, int N, int bits, int32_t* z) {
  if (!or_bits_ok(bits)) return OR_EARG;
  int64_t words = (int64_t)N * bits / 32;
  for (int64_t g = 0; g < G; g++)
    for (int64_t n = 0; n < N; n++)
      z[g * N + n] = (int32_t)or_stream_get(qzeros + g * words, 1, bits, n);
  return OR_OK;
}

int oracle_pack_k(const uint8_t* q, int K, int N, int bits, int32_t* qweight) {
  if (!or_bits_ok(bits)) return OR_EARG;
  memset(qweight, 0, sizeof(int32_t) * (size_t)((int64_t)K * bits / 32) * (size_t)N);
  for (int64_t k = 0; k < K; k++)
    for (int64_t n = 0; n < N; n++)
      or_stream_put(qweight + n, N, bits, k, q[k * N + n]);
  return OR_OK;
}

int oracle_pack_n(const int32_t* z, int G, int N, int bits, int32_t* qzeros) {
  if (!or_bits_ok(bits)) return OR_EARG;
  int64_t words = (int64_t)N * bits / 32;
  memset(qzeros, 0, sizeof(int32_t) * (size_t)(G * words));
  for (int64_t g = 0; g < G; g++)
    for (int64_t n = 0; n < N; n++)
      or_stream_put(qzeros + g * words, 1, bits, n, (uint32_t)z[g * N + n]);
  return OR_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Dequantization: w = (q - zero) * scale, zero = stored + (v1 ? 1 : 0).                */
/* ------------------------------------------------------------------------------------ */

/* Exact fp32 dequantized weights w32[K][N]. */
int oracle_dequant_f32(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                       const int32_t* g_idx, int K, int N, int bits, int group, int fmt,
                       float* w32) {
  int G, rc = or_check(K, N, bits, group, g_idx, &G);
  if (rc) return rc;
  if (fmt != OR_FMT_V1 && fmt != OR_FMT_V2) return OR_EARG;
  int zero_offset = fmt == OR_FMT_V2 ? 0 : 1;
  int64_t zwords = (int64_t)N * bits / 32;
  for (int64_t k = 0; k < K; k++) {
    int g = or_group_of(g_idx, group, k);
    if (g < 0 || g >= G) return OR_EARG;
    for (int64_t n = 0; n < N; n++) {
      int q = (int)or_stream_get(qweight + n, N, bits, k);
      int z = (int)or_stream_get(qzeros + (int64_t)g * zwords, 1, bits, n) + zero_offset;
      double s = oracle_half_to_double(scales[(int64_t)g * N + n]);
      w32[k * N + n] = (float)((double)(q - z) * s);   /* exact in binary32 */
    }
  }
  return OR_OK;
}

/* Dequantized weights rounded once to fp16 / bf16 (bit patterns). */
int oracle_dequant(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                   const int32_t* g_idx, int K, int N, int bits, int group, int fmt,
                   int out_dtype, uint16_t* W) {
  if (out_dtype != OR_F16 && out_dtype != OR_BF16) return OR_EARG;
  float* w32 = (float*)malloc(sizeof(float) * (size_t)K * (size_t)N);
  if (!w32) return OR_ENOMEM;
  int rc = oracle_dequant_f32(qweight, qzeros, scales, g_idx, K, N, bits, group, fmt, w32);
  if (rc == OR_OK) {
    for (int64_t i = 0; i < (int64_t)K * N; i++)
      W[i] = out_dtype == OR_F16 ? oracle_double_to_half_rne(w32[i])
                                 : oracle_double_to_bf16_rne(w32[i]);
  }
  free(w32);
  return rc;
}

/* ------------------------------------------------------------------------------------ */
/* GEMM: C[m,n] = sum_k A[m,k] * w32[k,n] in fp32, k ascending; also the bound          */
/* B[m,n] = sum_k |A[m,k] * w32[k,n]| (in double) used by the acceptance test.          */
/* `rows` selects which rows m of A to compute (NULL: all M); output row r of C and B   */
/* holds row rows[r].                                                                    */
/* ------------------------------------------------------------------------------------ */
int oracle_gemm_w32(const uint16_t* A, int M, int K, int a_dtype, const float* w32, int N,
                    const int32_t* rows, int nrows, float* C, double* B) {
  if (a_dtype != OR_F16 && a_dtype != OR_BF16) return OR_EARG;
  if (!rows) nrows = M;
  for (int r = 0; r < nrows; r++) {
    int64_t m = rows ? rows[r] : r;
    if (m < 0 || m >= M) return OR_EARG;
    float* c = C + (int64_t)r * N;
    double* b = B ? B + (int64_t)r * N : NULL;
    for (int64_t n = 0; n < N; n++) { c[n] = 0.0f; if (b) b[n] = 0.0; }
    /* k outermost over a row of C: each C[m,n] is still summed in ascending k. */
    for (int64_t k = 0; k < K; k++) {
      float a = (float)or_act_to_double(A[m * K + k], a_dtype);
      const float* w = w32 + k * N;
      for (int64_t n = 0; n < N; n++) {
        float p = a * w[n];
        c[n] = c[n] + p;
        if (b) b[n] += fabs((double)a * (double)w[n]);
      }
    }
  }
  return OR_OK;
}

int oracle_gemm(const uint16_t* A, int M, int K, int a_dtype, const int32_t* qweight,
                const int32_t* qzeros, const uint16_t* scales, const int32_t* g_idx, int N,
                int bits, int group, int fmt, const int32_t* rows, int nrows, float* C,
                double* B) {
  float* w32 = (float*)malloc(sizeof(float) * (size_t)K * (size_t)N);
  if (!w32) return OR_ENOMEM;
  int rc = oracle_dequant_f32(qweight, qzeros, scales, g_idx, K, N, bits, group, fmt, w32);
  if (rc == OR_OK) rc = oracle_gemm_w32(A, M, K, a_dtype, w32, N, rows, nrows, C, B);
  free(w32);
  return rc;
}

/* ------------------------------------------------------------------------------------ */
/* Host v1 -> v2 zero repack: every stored field f becomes f + 1.  A v1 field of 2^b-1   */
/* would need the value 2^b, which v2 cannot store: that is reported, not wrapped.      */
/* ------------------------------------------------------------------------------------ */
int oracle_repack_v1_to_v2(const int32_t* qz_v1, int32_t* qz_v2, int G, int N, int bits) {
  if (!or_bits_ok(bits) || G <= 0 || N <= 0 || ((int64_t)N * bits) % 32) return OR_EARG;
  if (bits == 3 && N % 32) return OR_EARG;
  int64_t words = (int64_t)N * bits / 32;
  uint32_t maxq = (1u << bits) - 1;
  int32_t* out = (int32_t*)calloc((size_t)(G * words), sizeof(int32_t));
  if (!out) return OR_ENOMEM;
  for (int64_t g = 0; g < G; g++)
    for (int64_t n = 0; n < N; n++) {
      uint32_t f = or_stream_get(qz_v1 + g * words, 1, bits, n);
      if (f == maxq) { free(out); return OR_EOVERFLOW; }
      or_stream_put(out + g * words, 1, bits, n, f + 1);
    }
  memcpy(qz_v2, out, sizeof(int32_t) * (size_t)(G * words));
  free(out);
  return OR_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Round-to-nearest quantizer (the page's formula), used to write synthetic checkpoints  */
/* and pinned against hand-worked groups.  Arithmetic in fp32, like the GPU quantizer.  */
/* Outputs: q[K][N] codes, zero[G][N] exact zeros, scale[G][N] fp16 bit patterns.       */
/* ------------------------------------------------------------------------------------ */
int oracle_quantize_rtn(const float* W, int K, int N, int bits, int group,
                        const int32_t* g_idx, int sym, uint8_t* q, int32_t* zero,
                        uint16_t* scale) {
  int G, rc = or_check(K, N, bits, group, g_idx, &G);
  if (rc) return rc;
  const float maxq = (float)((1 << bits) - 1);
  float* wmin = (float*)malloc(sizeof(float) * (size_t)G * (size_t)N);
  float* wmax = (float*)malloc(sizeof(float) * (size_t)G * (size_t)N);
  float* s = (float*)malloc(sizeof(float) * (size_t)G * (size_t)N);
  if (!wmin || !wmax || !s) { free(wmin); free(wmax); free(s); return OR_ENOMEM; }
  for (int64_t i = 0; i < (int64_t)G * N; i++) { wmin[i] = INFINITY; wmax[i] = -INFINITY; }
  for (int64_t k = 0; k < K; k++) {
    int g = or_group_of(g_idx, group, k);
    if (g < 0 || g >= G) { rc = OR_EARG; goto done; }
    for (int64_t n = 0; n < N; n++) {
      float w = W[k * N + n];
      if (w < wmin[(int64_t)g * N + n]) wmin[(int64_t)g * N + n] = w;
      if (w > wmax[(int64_t)g * N + n]) wmax[(int64_t)g * N + n] = w;
    }
  }
  for (int64_t i = 0; i < (int64_t)G * N; i++) {
    if (wmin[i] > wmax[i]) { rc = OR_EARG; goto done; }      /* a group with no rows */
    float s32, z;
    if (sym) {
      float amax = fabsf(wmin[i]) > fabsf(wmax[i]) ? fabsf(wmin[i]) : fabsf(wmax[i]);
      s32 = (2.0f * amax) / maxq;
    } else {
      s32 = (wmax[i] - wmin[i]) / maxq;
    }
    uint16_t h = oracle_double_to_half_rne(s32);
    if ((h & 0x7fff) == 0) h = 0x3c00;                          /* degenerate group: 1.0 */
    if ((h & 0x7c00) == 0x7c00) { rc = OR_EOVERFLOW; goto done; }
    scale[i] = h;
    s[i] = (float)oracle_half_to_double(h);
    if (sym) {
      z = rintf(maxq / 2.0f);
    } else {
      z = -rintf(wmin[i] / s[i]);
      if (z < 0.0f) z = 0.0f;
      if (z > maxq) z = maxq;
    }
    zero[i] = (int32_t)z;
  }
  for (int64_t k = 0; k < K; k++) {
    int g = or_group_of(g_idx, group, k);
    for (int64_t n = 0; n < N; n++) {
      int64_t i = (int64_t)g * N + n;
      float v = rintf(W[k * N + n] / s[i]) + (float)zero[i];
      if (v < 0.0f) v = 0.0f;
      if (v > maxq) v = maxq;
      q[k * N + n] = (uint8_t)v;
    }
  }
done:
  free(wmin); free(wmax); free(s);
  return rc;
}

/* Stored zero of each checkpoint format: v2 keeps zero, v1 keeps clamp(zero - 1). */
int oracle_store_zeros(const int32_t* zero, int64_t count, int bits, int fmt, int32_t* stored) {
  if (!or_bits_ok(bits) || (fmt != OR_FMT_V1 && fmt != OR_FMT_V2)) return OR_EARG;
  int32_t maxq = (1 << bits) - 1;
  for (int64_t i = 0; i < count; i++) {
    int32_t v = fmt == OR_FMT_V1 ? zero[i] - 1 : zero[i];
    if (v < 0) v = 0;
    if (v > maxq) v = maxq;
    stored[i] = v;
  }
  return OR_OK;
}

/* Array forms of the 16-bit conversions (for the rounding pins). */
void oracle_half_to_double_array(const uint16_t* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_half_to_double(h[i]);
}
void oracle_bf16_to_double_array(const uint16_t* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_bf16_to_double(h[i]);
}
void oracle_float_to_half_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_double_to_half_rne(x[i]);
}
void oracle_float_to_bf16_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_double_to_bf16_rne(x[i]);
}
