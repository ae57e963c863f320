/*
 * Oracle for the FP8-quantized MoE expert FFN.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow and obviously correct
 * CPU statement of what the expert-FFN path computes.  Only the tests, the
 * package smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code with the CUDA path and includes none of its headers.
 *
 * Sources.  Three MaxText pull-request pages define the path:
 *   [Q-EP]   "Quantize activations before EP all gather" (PR #4812): quantize
 *            the activations before the all-gather and the activation sort;
 *            gather the scale rows only when the scale is per token (review
 *            thread on ragged_sort); gmm_v2 takes rhs_scale and group_offset
 *            and the lhs scale multiplies the output (review thread on the
 *            unit test); an fp8 or missing output dtype means bf16 output
 *            (review thread on ops.py).
 *   [Q-GMM]  "Support quantization for tokamax gmm v2" (PR #4451): gmm and
 *            tgmm with quantization; fp8_dynamic = absmax scales for weights,
 *            activations and gradients; fp8_static_wa = fixed weight and
 *            activation scales with absmax gradients (review reply, tables 1
 *            and 2 list output, grad_wi_0, grad_wi_1 and grad_wo).
 *   [Q-FUSE] "Keep qwix out of tpu-inference's fused MoE kernel and
 *            pre-quantize weights" (PR #5136): float8_e4m3fn weights with
 *            [E, blocks, 1, N] scales; the matmul accumulator must be 32-bit
 *            (the Mosaic error quoted in the description).
 *
 *   [MX]     The MXFP8 variant is not a method of the pages: it is the
 *            Blackwell block-scaled form of the same path, defined by the OCP
 *            "Microscaling Formats (MX) Specification" v1.0 (MXFP8: blocks of
 *            32 e4m3 elements along the contracted dimension sharing one
 *            power-of-two E8M0 scale).  Its functions are marked [MX].
 *   [W8]     The int8-weight variant follows [Q-FUSE]'s other weight type
 *            ("float8_e4m3fn (or int8)" with the same [E, blocks, 1, N]
 *            scales): symmetric absmax codes in [-127, 127], activations and
 *            h still e4m3.  Its functions are marked [W8].
 *
 * Arithmetic.  fp8 codes and bf16 values are decoded exactly to double and
 * every contraction accumulates in double.  Products of two e4m3 values carry
 * at most 8 significant bits and lie in [2^-18, 2^17.6], so every raw code
 * dot product used here (K or group rows up to 2^16) is exact in double; the
 * only roundings are the scale products and the final bf16 or fp32 store.
 * Where floating point decides a quantised code (the scale amax/448, the
 * quotient x/s, and the SwiGLU value that is requantised), the oracle takes
 * that decision in IEEE fp32, the precision the pages fix for scales and the
 * precision the kernels compute in.  Build with -ffp-contract=off and without
 * fast-math so that every fp32 operation below rounds once, as written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_PER_ROW 0
#define OR_PER_ROW_BLOCK128 1
#define OR_PER_TENSOR 2
#define OR_PER_GROUP_COL 3
#define OR_MX32 4 /* [MX]: uint8 E8M0 codes, one per 32 values along K */

#define E4M3_MAX 448.0

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* bfloat16: the upper half of an IEEE binary32. */
double or_bf16_to_f64(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static uint16_t f32_bits_hi(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* Round a double to the nearest bfloat16, ties to even, in one step (no
 * intermediate fp32 rounding).  bf16 has 8 significant bits, exponent range
 * of binary32, subnormal quantum 2^-133; results at or above 2^128 are inf. */
uint16_t or_f64_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  frexp(a, &e); /* a = m 2^e, m in [0.5, 1) */
  int q = e - 8;
  if (q < -133) q = -133;
  double r = nearbyint(ldexp(a, -q)); /* default rounding mode: ties to even */
  double res = ldexp(r, q);
  if (res >= 0x1p128) return sign | 0x7F80;
  return sign | f32_bits_hi((float)res); /* exact: res has <= 8 significant bits */
}

/* OCP 8-bit floating point, E4M3 ("float8_e4m3fn"): exponent bias 7, three
 * mantissa bits, no infinities, 0x7F/0xFF are NaN, largest finite 448,
 * smallest subnormal 2^-9. */
double or_e4m3_to_f64(uint8_t c) {
  int s = c >> 7, E = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (E == 15 && m == 7) return NAN;
  if (E == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, E - 7);
  return s ? -v : v;
}

/* Nearest e4m3 value, ties to even mantissa, magnitudes beyond 448 saturate
 * to 448 (satfinite), the sign of zero is kept.  NaN input is outside the
 * contract and maps to 0x7F. */
uint8_t or_f32_to_e4m3(float vf) {
  double v = (double)vf;
  if (isnan(v)) return 0x7F;
  uint8_t s = signbit(v) ? 0x80 : 0;
  double a = fabs(v);
  if (a == 0.0) return s;
  double res;
  if (isinf(a)) {
    res = E4M3_MAX;
  } else {
    int e;
    frexp(a, &e);
    int q = e - 4; /* quantum of a normal with 4 significant bits */
    if (q < -9) q = -9;
    res = ldexp(nearbyint(ldexp(a, -q)), q);
    if (res > E4M3_MAX) res = E4M3_MAX;
  }
  if (res == 0.0) return s;
  if (res < 0x1p-6) return s | (uint8_t)(res * 512.0); /* subnormal: m 2^-9 */
  int e;
  double m = frexp(res, &e); /* res = m 2^e, m in [0.5, 1) */
  int E = e - 1 + 7;
  int mant = (int)((m * 2.0 - 1.0) * 8.0);
  return s | (uint8_t)(E << 3) | (uint8_t)mant;
}

/* ------------------------------------------------------------------------ */
/* fp32 exponential used by SwiGLU.                                         */
/*                                                                          */
/* Cody-Waite argument reduction (W. J. Cody and W. Waite, Software Manual  */
/* for the Elementary Functions, 1980): x = n ln2 + r with n = rint(x/ln2)  */
/* and ln2 split into a 16-bit head and a tail, then the degree-7 Taylor    */
/* polynomial of e^r evaluated by Horner's rule with fused multiply-adds,   */
/* then scaling by 2^n in two exact power-of-two steps.  Every operation is */
/* a single IEEE fp32 rounding, so the result is a fixed function of x.     */
/* ------------------------------------------------------------------------ */

static float pow2_f32(int i) { /* 2^i for i in [-126, 127] */
  uint32_t u = (uint32_t)(i + 127) << 23;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

float or_exp_f32(float x) {
  if (x != x) return x;
  if (x > 88.72283935546875f) return INFINITY;
  if (x < -103.972076416015625f) return 0.0f;
  const float log2e = 1.44269502162933349609375f;
  const float ln2_head = 0.693145751953125f;      /* 16 significant bits */
  const float ln2_tail = 1.428606765330187045e-6f; /* ln2 - ln2_head */
  float t = x * log2e;
  float n = rintf(t);
  float r = fmaf(-n, ln2_head, x);
  r = fmaf(-n, ln2_tail, r);
  float p = 1.0f / 5040.0f;
  p = fmaf(p, r, 1.0f / 720.0f);
  p = fmaf(p, r, 1.0f / 120.0f);
  p = fmaf(p, r, 1.0f / 24.0f);
  p = fmaf(p, r, 1.0f / 6.0f);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  int ni = (int)n;
  int n1 = ni / 2, n2 = ni - n1;
  p = p * pow2_f32(n1);
  p = p * pow2_f32(n2);
  return p;
}

/* silu(z) = z / (1 + e^-z) in fp32 ([Q-GMM] names the wi_0 / wi_1 / wo
 * projections; SwiGLU applies silu to the wi_0 branch). */
float or_silu_f32(float z) {
  float e = or_exp_f32(-z);
  float d = 1.0f + e;
  return z / d;
}

/* ------------------------------------------------------------------------ */
/* Activation and weight quantisation ([Q-EP] description; [Q-GMM] review   */
/* reply: absmax scales; [Q-FUSE]: float8_e4m3fn with fp32 scales).         */
/*   s = fp32(amax / 448), s = 1 when amax = 0;  q = e4m3(fp32(x / s)).     */
/* ------------------------------------------------------------------------ */

static float absmax_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  return amax / 448.0f;
}

static void quantize_span_f32(const float* x, int64_t n, float s, uint8_t* q) {
  for (int64_t i = 0; i < n; ++i) q[i] = or_f32_to_e4m3(x[i] / s);
}

static float amax_f32(const float* x, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > m) m = a;
  }
  return m;
}

/* Quantise fp32 rows (values already rounded as the caller wants them).
 * mode OR_PER_ROW: scale[rows]; OR_PER_ROW_BLOCK128: scale[rows, ceil(cols/128)];
 * OR_PER_TENSOR: the fixed scale static_scale is used and scale is not written. */
static void quantize_rows_f32(const float* x, int64_t rows, int64_t cols, int mode, float static_scale,
                              uint8_t* q, float* scale) {
  int64_t nb = (cols + 127) / 128;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const float* xr = x + r * cols;
    uint8_t* qr = q + r * cols;
    if (mode == OR_PER_ROW) {
      float s = absmax_scale(amax_f32(xr, cols));
      scale[r] = s;
      quantize_span_f32(xr, cols, s, qr);
    } else if (mode == OR_PER_ROW_BLOCK128) {
      for (int64_t b = 0; b < nb; ++b) {
        int64_t c0 = b * 128, n = cols - c0 < 128 ? cols - c0 : 128;
        float s = absmax_scale(amax_f32(xr + c0, n));
        scale[r * nb + b] = s;
        quantize_span_f32(xr + c0, n, s, qr + c0);
      }
    } else {
      quantize_span_f32(xr, cols, static_scale, qr);
    }
  }
}

/* bf16 rows -> e4m3 codes and fp32 scales. */
void or_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, int mode, float static_scale,
                      uint8_t* q, float* scale) {
  float* xf = (float*)malloc(sizeof(float) * (size_t)(rows * cols));
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < rows * cols; ++i) xf[i] = (float)or_bf16_to_f64(x[i]);
  quantize_rows_f32(xf, rows, cols, mode, static_scale, q, scale);
  free(xf);
}

/* Expert weights in the device layout w[E, N, K] (K contracted).  Each
 * (e, n) row of length K is quantised as above.  Scale layouts:
 *   per channel  (OR_PER_ROW):          scale[E, N]
 *   blockwise    (OR_PER_ROW_BLOCK128): scale[E, K/128, N], the pages'
 *                                       [E, blocks, 1, N] without the 1
 *   per tensor   (OR_PER_TENSOR):       static_scale, scale not written. */
void or_quantize_weights(const uint16_t* w, int64_t E, int64_t N, int64_t K, int mode, float static_scale,
                         uint8_t* q, float* scale) {
  int64_t nb = (K + 127) / 128;
  float* tmp = NULL;
  if (mode == OR_PER_ROW_BLOCK128) tmp = (float*)malloc(sizeof(float) * (size_t)(E * N * nb));
  or_quantize_rows(w, E * N, K, mode, static_scale, q, mode == OR_PER_ROW_BLOCK128 ? tmp : scale);
  if (mode == OR_PER_ROW_BLOCK128) {
    for (int64_t e = 0; e < E; ++e)
      for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b) scale[(e * nb + b) * N + n] = tmp[(e * N + n) * nb + b];
    free(tmp);
  }
}

/* ------------------------------------------------------------------------ */
/* [W8] int8 weight quantisation ([Q-FUSE]: weights pre-quantised to int8   */
/* with [E, blocks, 1, N] scales).  Symmetric absmax, the largest magnitude */
/* mapping to 127:                                                          */
/*   s = fp32(amax / 127), s = 1 when amax = 0;                             */
/*   q = rint(fp32(x / s)) (nearest integer, ties to even), limited to      */
/*       [-127, 127].                                                       */
/* ------------------------------------------------------------------------ */

static float int8_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  return amax / 127.0f;
}

static int8_t f32_to_int8(float v) {
  float r = rintf(v); /* the default rounding mode: nearest, ties to even */
  if (r > 127.0f) r = 127.0f;
  if (r < -127.0f) r = -127.0f;
  return (int8_t)r;
}

static void quantize_span_i8(const float* x, int64_t n, float s, int8_t* q) {
  for (int64_t i = 0; i < n; ++i) q[i] = f32_to_int8(x[i] / s);
}

/* [W8] Expert weights w[E, N, K] -> int8 codes and fp32 scales, in the scale
 * layouts of or_quantize_weights: per channel [E, N], blockwise
 * [E, K/128, N], per tensor (static_scale; scale not written). */
void or_quantize_weights_int8(const uint16_t* w, int64_t E, int64_t N, int64_t K, int mode, float static_scale,
                              int8_t* q, float* scale) {
  const int64_t nb = (K + 127) / 128;
#pragma omp parallel for schedule(static)
  for (int64_t row = 0; row < E * N; ++row) {
    const int64_t e = row / N, n = row % N;
    float* x = (float*)malloc(sizeof(float) * (size_t)K);
    for (int64_t kk = 0; kk < K; ++kk) x[kk] = (float)or_bf16_to_f64(w[row * K + kk]);
    int8_t* qr = q + row * K;
    if (mode == OR_PER_ROW) {
      const float s = int8_scale(amax_f32(x, K));
      scale[row] = s;
      quantize_span_i8(x, K, s, qr);
    } else if (mode == OR_PER_ROW_BLOCK128) {
      for (int64_t b = 0; b < nb; ++b) {
        const int64_t c0 = b * 128, len = K - c0 < 128 ? K - c0 : 128;
        const float s = int8_scale(amax_f32(x + c0, len));
        scale[(e * nb + b) * N + n] = s;
        quantize_span_i8(x + c0, len, s, qr + c0);
      }
    } else {
      quantize_span_i8(x, K, static_scale, qr);
    }
    free(x);
  }
}

/* ------------------------------------------------------------------------ */
/* [MX] MXFP8 quantisation (OCP MX v1.0, MXFP8 with E4M3 elements).  Each   */
/* block of 32 consecutive values of a row shares the scale 2^X with        */
/*   X = floor(log2(amax)) - 8,                                             */
/* 8 being the exponent of the largest power of two that e4m3 holds (256),  */
/* clamped to the E8M0 range [-127, 127]; the block's E8M0 code is X + 127. */
/* The elements are e4m3(v / 2^X), nearest with ties to even and saturating */
/* at 448 (v / 2^X < 512, so only the top binade can saturate).  A block of */
/* zeros takes X = -127 (code 0), the smallest scale.                       */
/* ------------------------------------------------------------------------ */

static int mx_shared_exp(float amax) {
  if (amax == 0.0f) return -127;
  int e;
  frexp((double)amax, &e); /* amax = f 2^e with f in [0.5, 1): floor(log2 amax) = e - 1 */
  int X = e - 1 - 8;
  if (X < -127) X = -127;
  if (X > 127) X = 127;
  return X;
}

/* fp32 rows [rows, cols] (cols a multiple of 32) -> codes and E8M0 codes [rows, cols/32]. */
static void quantize_rows_mx_f32(const float* x, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sf) {
  int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      const float* xb = x + r * cols + b * 32;
      int X = mx_shared_exp(amax_f32(xb, 32));
      sf[r * nb + b] = (uint8_t)(X + 127);
      /* v / 2^X is exact in double; as fp32 it is exact too unless it falls
       * below 2^-126, far under e4m3's smallest half-step (2^-10) */
      for (int i = 0; i < 32; ++i) q[r * cols + b * 32 + i] = or_f32_to_e4m3((float)ldexp((double)xb[i], -X));
    }
}

/* [MX] bf16 rows -> MXFP8 codes [rows, cols] and E8M0 codes [rows, cols/32].
 * Expert weights w[E, N, K] are the rows e*N + n, so their scales come out
 * as [E, N, K/32]. */
void or_quantize_rows_mx(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sf) {
  float* xf = (float*)malloc(sizeof(float) * (size_t)(rows * cols));
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < rows * cols; ++i) xf[i] = (float)or_bf16_to_f64(x[i]);
  quantize_rows_mx_f32(xf, rows, cols, q, sf);
  free(xf);
}

/* ------------------------------------------------------------------------ */
/* Ragged sort by routed expert ([Q-EP]: ragged_sort / ragged_gather).      */
/* Flat pair i = t*k + j goes to expert ids[i].  Stable counting sort: by   */
/* expert ascending, then by i ascending.  sorted_src[r] = i, pos[i] = r.   */
/* Returns 0, or -1 when an id lies outside [0, E).                         */
/* ------------------------------------------------------------------------ */
int or_ragged_sort(const int32_t* ids, int64_t T, int k, int E, int32_t* sorted_src, int32_t* pos,
                   int32_t* group_sizes, int32_t* group_offsets) {
  int64_t R = T * k;
  for (int e = 0; e < E; ++e) group_sizes[e] = 0;
  for (int64_t i = 0; i < R; ++i) {
    if (ids[i] < 0 || ids[i] >= E) return -1;
    group_sizes[ids[i]]++;
  }
  group_offsets[0] = 0;
  for (int e = 0; e < E; ++e) group_offsets[e + 1] = group_offsets[e] + group_sizes[e];
  int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  for (int e = 0; e < E; ++e) next[e] = group_offsets[e];
  for (int64_t i = 0; i < R; ++i) {
    int32_t r = next[ids[i]]++;
    sorted_src[r] = (int32_t)i;
    pos[i] = r;
  }
  free(next);
  return 0;
}

/* Gather the quantised rows and, for per-token scales only, the scale rows
 * ([Q-EP] review: gather the scale only when its leading dimension is the
 * token dimension; a per-tensor scale passes through unchanged).
 * xs_q[r] = x_q[sorted_src[r] / k]. */
void or_gather_rows(const uint8_t* x_q, const float* x_scale, int mode, int64_t D, const int32_t* sorted_src,
                    int64_t R, int k, uint8_t* xs_q, float* xs_scale) {
  int64_t nb = (D + 127) / 128;
  for (int64_t r = 0; r < R; ++r) {
    int64_t t = sorted_src[r] / k;
    memcpy(xs_q + r * D, x_q + t * D, (size_t)D);
    if (mode == OR_PER_ROW) xs_scale[r] = x_scale[t];
    if (mode == OR_PER_ROW_BLOCK128)
      for (int64_t b = 0; b < nb; ++b) xs_scale[r * nb + b] = x_scale[t * nb + b];
  }
}

/* ------------------------------------------------------------------------ */
/* Grouped matmul ([Q-EP] review on gmm_v2: gmm(lhs, rhs, group_sizes,      */
/* rhs_scale, group_offset) with the lhs scale multiplying the output; bf16 */
/* output for an fp8 operand type; [Q-FUSE]: 32-bit accumulation).          */
/*   out[m, n] = sum_k deq(lhs)[m, k] * deq(rhs)[g(m), n, k]                */
/* where g(m) is the group holding row m and deq multiplies each code by    */
/* the scale that covers it.  Groups outside [g0, g0 + E_local) give zero   */
/* rows.                                                                    */
/* ------------------------------------------------------------------------ */

/* [MX] the power of two an E8M0 code stands for: 2^(c - 127) (c = 255, NaN,
 * is never produced by the quantiser). */
static double e8m0_to_f64(uint8_t c) { return ldexp(1.0, (int)c - 127); }

/* Scale of lhs element (m, k): fp32 scales per row, per (row, 128-column
 * block) or per tensor; [MX] E8M0 codes per (row, 32-column block). */
static double lhs_scale_at(const void* s, int mode, int64_t m, int64_t kk, int64_t K) {
  const float* f = (const float*)s;
  if (mode == OR_PER_ROW) return f[m];
  if (mode == OR_PER_ROW_BLOCK128) return f[m * ((K + 127) / 128) + kk / 128];
  if (mode == OR_MX32) return e8m0_to_f64(((const uint8_t*)s)[m * (K / 32) + kk / 32]);
  return f[0];
}

/* Scale of rhs element (e, n, k) of w[E_local, N, K]: per channel [E, N],
 * blockwise [E, K/128, N], per tensor; [MX] E8M0 codes [E, N, K/32]. */
static double rhs_scale_at(const void* s, int mode, int64_t e, int64_t n, int64_t kk, int64_t N, int64_t K) {
  const float* f = (const float*)s;
  if (mode == OR_PER_ROW) return f[e * N + n];
  if (mode == OR_PER_ROW_BLOCK128) return f[(e * ((K + 127) / 128) + kk / 128) * N + n];
  if (mode == OR_MX32) return e8m0_to_f64(((const uint8_t*)s)[(e * N + n) * (K / 32) + kk / 32]);
  return f[0];
}

static int group_of_row(const int64_t* starts, int E, int64_t m) {
  int lo = 0, hi = E; /* starts[E] = total rows; find g with starts[g] <= m < starts[g+1] */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (starts[mid] <= m) lo = mid; else hi = mid;
  }
  return lo;
}

/* rows: optional list of nrows output rows to compute (NULL = all M rows).
 * out_bf16 / out_f64 (either may be NULL) are [nrows, N]. */
/* rhs_int8: [W8] the rhs codes are int8 integers instead of e4m3 codes. */
static void gmm_core(const uint8_t* lhs, const void* lhs_scale, int lhs_mode, const uint8_t* rhs, int rhs_int8,
                     const void* rhs_scale, int rhs_mode, const int32_t* group_sizes, int E, int g0, int E_local,
                     int64_t M, int64_t K, int64_t N, const int64_t* rows, int64_t nrows, uint16_t* out_bf16,
                     double* out_f64) {
  int64_t* starts = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E + 1));
  starts[0] = 0;
  for (int e = 0; e < E; ++e) starts[e + 1] = starts[e] + group_sizes[e];
  if (!rows) nrows = M;
  /* dequantised lhs rows, one per output row */
  double* a = (double*)malloc(sizeof(double) * (size_t)(nrows * K));
  int* grp = (int*)malloc(sizeof(int) * (size_t)nrows);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t m = rows ? rows[i] : i;
    int g = (m < starts[E]) ? group_of_row(starts, E, m) : -1;
    grp[i] = (g >= g0 && g < g0 + E_local) ? g : -1;
    for (int64_t kk = 0; kk < K; ++kk)
      a[i * K + kk] = or_e4m3_to_f64(lhs[m * K + kk]) * lhs_scale_at(lhs_scale, lhs_mode, m, kk, K);
  }
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 4)
    for (int64_t n = 0; n < N; ++n) {
      int cur = -2;
      for (int64_t i = 0; i < nrows; ++i) {
        double acc = 0.0;
        int g = grp[i];
        if (g >= 0) {
          if (g != cur) {
            int64_t el = g - g0;
            const uint8_t* wr = rhs + (el * N + n) * K;
            for (int64_t kk = 0; kk < K; ++kk)
              w[kk] = (rhs_int8 ? (double)(int8_t)wr[kk] : or_e4m3_to_f64(wr[kk])) *
                      rhs_scale_at(rhs_scale, rhs_mode, el, n, kk, N, K);
            cur = g;
          }
          const double* ar = a + i * K;
          for (int64_t kk = 0; kk < K; ++kk) acc += ar[kk] * w[kk];
        }
        if (out_f64) out_f64[i * N + n] = acc;
        if (out_bf16) out_bf16[i * N + n] = or_f64_to_bf16(acc);
      }
    }
    free(w);
  }
  free(a);
  free(grp);
  free(starts);
}

void or_gmm(const uint8_t* lhs, const float* lhs_scale, int lhs_mode, const uint8_t* rhs, const float* rhs_scale,
            int rhs_mode, const int32_t* group_sizes, int E, int g0, int E_local, int64_t M, int64_t K, int64_t N,
            const int64_t* rows, int64_t nrows, uint16_t* out_bf16, double* out_f64) {
  gmm_core(lhs, lhs_scale, lhs_mode, rhs, 0, rhs_scale, rhs_mode, group_sizes, E, g0, E_local, M, K, N, rows,
           nrows, out_bf16, out_f64);
}

/* [W8] The grouped matmul with int8 weights: deq(rhs)[e, n, k] = q[e, n, k] *
 * s, the code taken as the integer it holds and s covering it (per channel,
 * blockwise [E, K/128, N] or per tensor); lhs as in or_gmm. */
void or_gmm_w8(const uint8_t* lhs, const float* lhs_scale, int lhs_mode, const int8_t* rhs, const float* rhs_scale,
               int rhs_mode, const int32_t* group_sizes, int E, int g0, int E_local, int64_t M, int64_t K, int64_t N,
               const int64_t* rows, int64_t nrows, uint16_t* out_bf16, double* out_f64) {
  gmm_core(lhs, lhs_scale, lhs_mode, (const uint8_t*)rhs, 1, rhs_scale, rhs_mode, group_sizes, E, g0, E_local, M, K,
           N, rows, nrows, out_bf16, out_f64);
}

/* [MX] The same grouped matmul on MXFP8 operands: lhs_sf [M, K/32] and
 * rhs_sf [E_local, N, K/32] hold the E8M0 codes of each 32-element block
 * along K, so deq(x)[.., k] = e4m3(x[.., k]) * 2^(sf[.., k/32] - 127).  K is a
 * multiple of 32. */
void or_gmm_mx(const uint8_t* lhs, const uint8_t* lhs_sf, const uint8_t* rhs, const uint8_t* rhs_sf,
               const int32_t* group_sizes, int E, int g0, int E_local, int64_t M, int64_t K, int64_t N,
               const int64_t* rows, int64_t nrows, uint16_t* out_bf16, double* out_f64) {
  gmm_core(lhs, lhs_sf, OR_MX32, rhs, 0, rhs_sf, OR_MX32, group_sizes, E, g0, E_local, M, K, N, rows, nrows,
           out_bf16, out_f64);
}

/* The same contraction on double operands (no quantisation), used to pin
 * the adjoint and finite-difference identities of the backward pass.
 * rhs is [E_local, N, K]. */
void or_gmm_f64(const double* lhs, const double* rhs, const int32_t* group_sizes, int E, int g0, int E_local,
                int64_t M, int64_t K, int64_t N, double* out) {
  int64_t start = 0;
  for (int e = 0; e < g0; ++e) start += group_sizes[e];
  memset(out, 0, sizeof(double) * (size_t)(M * N));
  for (int el = 0; el < E_local; ++el) {
    int64_t sz = group_sizes[g0 + el];
#pragma omp parallel for schedule(static)
    for (int64_t m = start; m < start + sz; ++m)
      for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t kk = 0; kk < K; ++kk) acc += lhs[m * K + kk] * rhs[(el * N + n) * K + kk];
        out[m * N + n] = acc;
      }
    start += sz;
  }
}

/* ------------------------------------------------------------------------ */
/* SwiGLU and requantisation.  a = [a0 | a1] is the bf16 output of the      */
/* wi_0 / wi_1 gmm ([R, 2F]); h = bf16(silu(a0) * a1) in fp32, then h is    */
/* quantised exactly as the activations are.                                */
/* ------------------------------------------------------------------------ */
static float* swiglu_rows(const uint16_t* a, int64_t R, int64_t F, uint16_t* h_bf16) {
  float* h = (float*)malloc(sizeof(float) * (size_t)(R * F));
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r)
    for (int64_t f = 0; f < F; ++f) {
      float a0 = (float)or_bf16_to_f64(a[r * 2 * F + f]);
      float a1 = (float)or_bf16_to_f64(a[r * 2 * F + F + f]);
      float v = or_silu_f32(a0) * a1;
      uint16_t hb = or_f64_to_bf16((double)v);
      if (h_bf16) h_bf16[r * F + f] = hb;
      h[r * F + f] = (float)or_bf16_to_f64(hb);
    }
  return h;
}

void or_swiglu_quant(const uint16_t* a, int64_t R, int64_t F, int mode, float static_scale, uint8_t* h_q,
                     float* h_scale, uint16_t* h_bf16) {
  float* h = swiglu_rows(a, R, F, h_bf16);
  quantize_rows_f32(h, R, F, mode, static_scale, h_q, h_scale);
  free(h);
}

/* [MX] The same h, requantised to MXFP8 along F (the wo gmm's contracted
 * dimension): codes [R, F], E8M0 codes [R, F/32]. */
void or_swiglu_quant_mx(const uint16_t* a, int64_t R, int64_t F, uint8_t* h_q, uint8_t* h_sf, uint16_t* h_bf16) {
  float* h = swiglu_rows(a, R, F, h_bf16);
  quantize_rows_mx_f32(h, R, F, h_q, h_sf);
  free(h);
}

/* ------------------------------------------------------------------------ */
/* Ragged gather-reduce (combine) ([Q-EP]: ragged_gather_reduce): undo the  */
/* sort and sum the k expert rows of each token weighted by its router      */
/* probabilities.  y[t] = bf16(sum_j w[t, j] o[pos[t k + j]]); w = NULL     */
/* means all weights are 1.  toks: optional list of ntoks tokens.           */
/* ------------------------------------------------------------------------ */
void or_combine(const uint16_t* o, const int32_t* pos, const float* w, int64_t T, int k, int64_t D,
                const int64_t* toks, int64_t ntoks, uint16_t* y_bf16, double* y_f64) {
  if (!toks) ntoks = T;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < ntoks; ++i) {
    int64_t t = toks ? toks[i] : i;
    for (int64_t d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) {
        double wj = w ? (double)w[t * k + j] : 1.0;
        acc += wj * or_bf16_to_f64(o[(int64_t)pos[t * k + j] * D + d]);
      }
      if (y_f64) y_f64[i * D + d] = acc;
      if (y_bf16) y_bf16[i * D + d] = or_f64_to_bf16(acc);
    }
  }
}

/* Double-operand combine for the adjoint identities. */
void or_combine_f64(const double* o, const int32_t* pos, const float* w, int64_t T, int k, int64_t D, double* y) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += (w ? (double)w[t * k + j] : 1.0) * o[(int64_t)pos[t * k + j] * D + d];
      y[t * D + d] = acc;
    }
}

/* ------------------------------------------------------------------------ */
/* Backward pass ([Q-GMM]: gmm for the input gradient, tgmm for grad_wi_0,  */
/* grad_wi_1 and grad_wo; gradients quantised by absmax).                   */
/* ------------------------------------------------------------------------ */

/* Adjoint of the combine: dO[r] = bf16(fp32(w[i] * G[i / k])), i = sorted_src[r]. */
void or_gather_scale(const uint16_t* G, const float* w, const int32_t* sorted_src, int64_t R, int k, int64_t D,
                     uint16_t* dO) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    int64_t i = sorted_src[r];
    float wi = w ? w[i] : 1.0f;
    for (int64_t d = 0; d < D; ++d) {
      float g = (float)or_bf16_to_f64(G[(i / k) * D + d]);
      float v = wi * g;
      dO[r * D + d] = or_f64_to_bf16((double)v);
    }
  }
}

void or_gather_scale_f64(const double* G, const float* w, const int32_t* sorted_src, int64_t R, int k, int64_t D,
                         double* dO) {
  for (int64_t r = 0; r < R; ++r) {
    int64_t i = sorted_src[r];
    for (int64_t d = 0; d < D; ++d) dO[r * D + d] = (w ? (double)w[i] : 1.0) * G[(i / k) * D + d];
  }
}

/* SwiGLU backward in fp32, rounded to bf16:
 *   sigma = 1 / (1 + e^-a0), silu = a0 / (1 + e^-a0),
 *   silu' = sigma (1 + a0 (1 - sigma)),
 *   dA0 = (dH a1) silu',  dA1 = dH silu.        dA = [dA0 | dA1]  [R, 2F]. */
void or_swiglu_bwd(const uint16_t* dH, const uint16_t* a, int64_t R, int64_t F, uint16_t* dA) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r)
    for (int64_t f = 0; f < F; ++f) {
      float z = (float)or_bf16_to_f64(a[r * 2 * F + f]);
      float a1 = (float)or_bf16_to_f64(a[r * 2 * F + F + f]);
      float dh = (float)or_bf16_to_f64(dH[r * F + f]);
      float e = or_exp_f32(-z);
      float d = 1.0f + e;
      float sig = 1.0f / d;
      float silu = z / d;
      float t1 = 1.0f - sig;
      float t2 = z * t1;
      float t3 = 1.0f + t2;
      float ds = sig * t3;
      float p = dh * a1;
      float da0 = p * ds;
      float da1 = dh * silu;
      dA[r * 2 * F + f] = or_f64_to_bf16((double)da0);
      dA[r * 2 * F + F + f] = or_f64_to_bf16((double)da1);
    }
}

/* The same formulas in double, unrounded (for the finite-difference pin). */
void or_swiglu_f64(const double* a, int64_t R, int64_t F, double* h) {
  for (int64_t r = 0; r < R; ++r)
    for (int64_t f = 0; f < F; ++f) {
      double z = a[r * 2 * F + f], a1 = a[r * 2 * F + F + f];
      h[r * F + f] = z / (1.0 + exp(-z)) * a1;
    }
}

void or_swiglu_bwd_f64(const double* dH, const double* a, int64_t R, int64_t F, double* dA) {
  for (int64_t r = 0; r < R; ++r)
    for (int64_t f = 0; f < F; ++f) {
      double z = a[r * 2 * F + f], a1 = a[r * 2 * F + F + f], dh = dH[r * F + f];
      double sig = 1.0 / (1.0 + exp(-z));
      dA[r * 2 * F + f] = dh * a1 * sig * (1.0 + z * (1.0 - sig));
      dA[r * 2 * F + F + f] = dh * z * sig;
    }
}

/* Gradient requantisation for the weight-gradient contraction: one absmax
 * scale per (expert, column) over that expert's rows, so that both scales
 * factor out of the sum over rows.  q[M, N] (rows outside the local groups
 * are left untouched), scale[E_local, N]; an expert with no rows, or an
 * all-zero column, gets scale 1. */
void or_quantize_group_cols(const uint16_t* g, const int32_t* group_sizes, int E, int g0, int E_local, int64_t M,
                            int64_t N, uint8_t* q, float* scale) {
  (void)M;
  int64_t start = 0;
  for (int e = 0; e < g0; ++e) start += group_sizes[e];
  for (int el = 0; el < E_local; ++el) {
    int64_t sz = group_sizes[g0 + el];
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
      float amax = 0.0f;
      for (int64_t m = start; m < start + sz; ++m) {
        float v = fabsf((float)or_bf16_to_f64(g[m * N + n]));
        if (v > amax) amax = v;
      }
      float s = absmax_scale(amax);
      scale[(int64_t)el * N + n] = s;
      for (int64_t m = start; m < start + sz; ++m)
        q[m * N + n] = or_f32_to_e4m3((float)or_bf16_to_f64(g[m * N + n]) / s);
    }
    start += sz;
  }
}

/* Transposed grouped matmul (tgmm):
 *   out[e, k, n] = sum_{m in group e} deq(lhs)[m, k] * deq(rhs)[m, n]
 * lhs scale: OR_PER_TENSOR ([1]) or OR_PER_GROUP_COL ([E_local, K]);
 * rhs scale: OR_PER_TENSOR or OR_PER_GROUP_COL ([E_local, N]).  Both factor
 * out of the sum over rows.  out is fp32 [E_local, K, N] (optional) and/or
 * double.  samples: optional list of nsamp flat output indices
 * (e * K + k) * N + n; then out/out_f64 hold nsamp values. */
static double grp_scale(const float* s, int mode, int64_t el, int64_t c, int64_t C) {
  return mode == OR_PER_GROUP_COL ? (double)s[el * C + c] : (double)s[0];
}

void or_tgmm(const uint8_t* lhs, const float* lhs_scale, int lhs_mode, const uint8_t* rhs, const float* rhs_scale,
             int rhs_mode, const int32_t* group_sizes, int E, int g0, int E_local, int64_t M, int64_t K, int64_t N,
             const int64_t* samples, int64_t nsamp, float* out, double* out_f64) {
  (void)M;
  int64_t* starts = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E_local + 1));
  int64_t s0 = 0;
  for (int e = 0; e < g0; ++e) s0 += group_sizes[e];
  starts[0] = s0;
  for (int el = 0; el < E_local; ++el) starts[el + 1] = starts[el] + group_sizes[g0 + el];
  int64_t total = samples ? nsamp : (int64_t)E_local * K * N;
#pragma omp parallel for schedule(dynamic, 256)
  for (int64_t i = 0; i < total; ++i) {
    int64_t flat = samples ? samples[i] : i;
    int64_t el = flat / (K * N), kk = (flat / N) % K, n = flat % N;
    double acc = 0.0;
    for (int64_t m = starts[el]; m < starts[el + 1]; ++m)
      acc += or_e4m3_to_f64(lhs[m * K + kk]) * or_e4m3_to_f64(rhs[m * N + n]);
    acc *= grp_scale(lhs_scale, lhs_mode, el, kk, K) * grp_scale(rhs_scale, rhs_mode, el, n, N);
    if (out) out[i] = (float)acc;
    if (out_f64) out_f64[i] = acc;
  }
  free(starts);
}

/* Double-operand tgmm for the adjoint identities: out[E_local, K, N]. */
void or_tgmm_f64(const double* lhs, const double* rhs, const int32_t* group_sizes, int E, int g0, int E_local,
                 int64_t M, int64_t K, int64_t N, double* out) {
  (void)M;
  int64_t start = 0;
  for (int e = 0; e < g0; ++e) start += group_sizes[e];
  for (int el = 0; el < E_local; ++el) {
    int64_t sz = group_sizes[g0 + el];
    for (int64_t kk = 0; kk < K; ++kk)
      for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t m = start; m < start + sz; ++m) acc += lhs[m * K + kk] * rhs[m * N + n];
        out[((int64_t)el * K + kk) * N + n] = acc;
      }
    start += sz;
  }
}

/* ------------------------------------------------------------------------ */
/* Router ("Support quantization for tokamax gmm v2", table 1: the gate      */
/* kernel's gradient grad_gate-kernel and the state gradient state_grad are  */
/* measured beside the expert weights' gradients).  The gate is a dense      */
/* bf16 layer W_gate [E, D]; routing takes a softmax over all E logits and   */
/* the k most probable experts, weighted by their probabilities, not         */
/* renormalised, ties to the lower expert index.                             */
/* ------------------------------------------------------------------------ */

/* logits[t, e] = sum_d x[t, d] W_gate[e, d] in double (products of two bf16
 * values are exact). */
void or_router_logits(const uint16_t* x, const uint16_t* wg, int64_t T, int64_t D, int64_t E, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t d = 0; d < D; ++d) acc += or_bf16_to_f64(x[t * D + d]) * or_bf16_to_f64(wg[e * D + d]);
      out[t * E + e] = acc;
    }
}

/* Softmax probabilities of one row of fp32 logits, in fp32 (the precision in
 * which the kernels take the top-k decision): m = max l, e_i = exp(l_i - m)
 * with the fp32 exponential above, Z = e_0 + e_1 + ... summed in ascending i,
 * p_i = e_i / Z correctly rounded. */
static void softmax_row_f32(const float* l, int64_t E, float* p) {
  float m = -INFINITY;
  for (int64_t i = 0; i < E; ++i) m = l[i] > m ? l[i] : m;
  float z = 0.0f;
  for (int64_t i = 0; i < E; ++i) {
    p[i] = or_exp_f32(l[i] - m);
    z = z + p[i];
  }
  for (int64_t i = 0; i < E; ++i) p[i] = p[i] / z;
}

/* Top-k routing from fp32 logits [T, E]: ids [T, k] in descending order of
 * probability (ties to the lower expert index), weights w [T, k] = the
 * selected probabilities; p [T, E] (optional) receives every probability. */
void or_router_topk(const float* logits, int64_t T, int64_t E, int k, int32_t* ids, float* w, float* p_out) {
#pragma omp parallel
  {
    float* p = (float*)malloc(sizeof(float) * (size_t)E);
    char* taken = (char*)malloc((size_t)E);
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      softmax_row_f32(logits + t * E, E, p);
      memset(taken, 0, (size_t)E);
      for (int j = 0; j < k; ++j) {
        int64_t best = -1;
        for (int64_t i = 0; i < E; ++i)
          if (!taken[i] && (best < 0 || p[i] > p[best])) best = i; /* strict >: the lower index wins a tie */
        taken[best] = 1;
        ids[t * k + j] = (int32_t)best;
        w[t * k + j] = p[best];
      }
      if (p_out) memcpy(p_out + t * E, p, sizeof(float) * (size_t)E);
    }
    free(p);
    free(taken);
  }
}

/* Gradient of the loss with respect to the routing weights: the combine
 * y[t] = sum_j w[t, j] o[pos[t k + j]] gives dL/dw[t, j] = <G[t], o[pos]>, in
 * double. */
void or_router_dw(const uint16_t* G, const uint16_t* o, const int32_t* pos, int64_t T, int k, int64_t D,
                  double* dw) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      const int64_t r = pos[t * k + j];
      double acc = 0.0;
      for (int64_t d = 0; d < D; ++d) acc += or_bf16_to_f64(G[t * D + d]) * or_bf16_to_f64(o[r * D + d]);
      dw[t * k + j] = acc;
    }
}

/* Softmax backward through the selected probabilities, in fp32, rounded to
 * bf16 (gradients are bf16 between steps):
 *   w_j = p[id_j],  s = sum_j w_j dw_j (ascending j),
 *   dlogits[t, i] = bf16( p_i (g_i - s) ),  g_i = dw_j if i = id_j, else 0. */
void or_router_dlogits(const float* logits, const int32_t* ids, const float* dw, int64_t T, int64_t E, int k,
                       uint16_t* dlogits) {
#pragma omp parallel
  {
    float* p = (float*)malloc(sizeof(float) * (size_t)E);
    float* g = (float*)malloc(sizeof(float) * (size_t)E);
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      softmax_row_f32(logits + t * E, E, p);
      float s = 0.0f;
      for (int64_t i = 0; i < E; ++i) g[i] = 0.0f;
      for (int j = 0; j < k; ++j) {
        const int32_t e = ids[t * k + j];
        const float wj = p[e];
        const float pr = wj * dw[t * k + j];
        s = s + pr;
        g[e] = dw[t * k + j];
      }
      for (int64_t i = 0; i < E; ++i) {
        const float diff = g[i] - s;
        const float v = p[i] * diff;
        dlogits[t * E + i] = or_f64_to_bf16((double)v); /* an fp32 value rounds to bf16 in one step */
      }
    }
    free(p);
    free(g);
  }
}

/* Gradients of the gate from bf16 dlogits [T, E], in double:
 *   grad_gate[e, d] = sum_t dlogits[t, e] x[t, d]     (W_gate's layout [E, D])
 *   state_grad[t, d] = sum_e dlogits[t, e] W_gate[e, d]. */
void or_router_grads(const uint16_t* x, const uint16_t* wg, const uint16_t* dl, int64_t T, int64_t D, int64_t E,
                     double* grad_gate, double* state_grad) {
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < E; ++e)
    for (int64_t d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int64_t t = 0; t < T; ++t) acc += or_bf16_to_f64(dl[t * E + e]) * or_bf16_to_f64(x[t * D + d]);
      grad_gate[e * D + d] = acc;
    }
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int64_t e = 0; e < E; ++e) acc += or_bf16_to_f64(dl[t * E + e]) * or_bf16_to_f64(wg[e * D + d]);
      state_grad[t * D + d] = acc;
    }
}
