// Shared device helpers for the sm_103a kernels of libmoefp8.
//
// Inline PTX wrappers for mbarriers, TMA (cp.async.bulk.tensor), tcgen05
// (tensor-memory allocation, MMA, commit, loads), number-format conversion
// (bf16 and e4m3 packing via cvt), the fp32 exponential used by SwiGLU, and
// the per-translation-unit device error word.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moefp8.h"

#define MOE_HOST_CHECK(cond, status) \
  do {                               \
    if (!(cond)) return (status);    \
  } while (0)

#define MOE_CUDA_TRY(expr)                         \
  do {                                             \
    cudaError_t e_ = (expr);                       \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA;    \
  } while (0)

namespace moe {

constexpr float kE4M3Max = 448.0f;

#ifndef MOE_IDLE_WAIT_HINT_NS
#define MOE_IDLE_WAIT_HINT_NS 1000
#endif

// ------------------------------------------------------------------------
// Device error word.  Each translation unit owns one (no relocatable device
// code); moe_get_device_error reads and clears all of them.
// ------------------------------------------------------------------------
__device__ __forceinline__ void raise_error(unsigned int* word, unsigned int bits) { atomicOr(word, bits); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// ------------------------------------------------------------------------
// Number formats
// ------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Two fp32 -> bf16x2, round to nearest even; `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Round an fp32 value to the nearest bf16 and return it as fp32 (exact).
__device__ __forceinline__ float round_bf16(float v) { return bf16lo(pack_bf16x2(v, 0.0f)); }

// Packed fp32 pair arithmetic (two lanes of work per instruction).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Two fp32 -> e4m3x2 (float8_e4m3fn), round to nearest even, saturating to
// +-448; `lo` lands in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight values -> eight e4m3 codes (little-endian order) in a uint2.
__device__ __forceinline__ uint2 pack_e4m3x8(const float* v) {
  uint2 r;
  r.x = pack_e4m3x2(v[0], v[1]) | (pack_e4m3x2(v[2], v[3]) << 16);
  r.y = pack_e4m3x2(v[4], v[5]) | (pack_e4m3x2(v[6], v[7]) << 16);
  return r;
}

// Absmax scale in fp32: amax / 448, or 1 for an all-zero span.
__device__ __forceinline__ float absmax_scale(float amax) { return amax > 0.0f ? __fdiv_rn(amax, kE4M3Max) : 1.0f; }

// int8 weights: symmetric absmax scale amax / 127 (1 for an all-zero span),
// and eight quotients -> the nearest integers (ties to even) limited to
// [-127, 127], as int8 bytes in little-endian order.
__device__ __forceinline__ float int8_scale(float amax) { return amax > 0.0f ? __fdiv_rn(amax, 127.0f) : 1.0f; }
__device__ __forceinline__ uint2 pack_i8x8(const float* v) {
  uint32_t b[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = static_cast<uint32_t>(min(127, max(-127, __float2int_rn(v[j])))) & 0xFFu;
  return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

// MXFP8 (OCP MX v1.0) shared exponent of a 32-value block: floor(log2(amax))
// - 8, clamped to [-127, 127], -127 for amax = 0.  Read off the fp32 exponent
// field: a normal amax = 1.f * 2^(field - 127); every subnormal (and zero)
// amax is below 2^-119 and clamps to -127.
__device__ __forceinline__ int mx_shared_exp(float amax) {
  const int field = static_cast<int>(__float_as_uint(amax) >> 23);  // amax >= 0
  const int x = field - 127 - 8;
  return field == 0 ? -127 : (x < -127 ? -127 : (x > 127 ? 127 : x));
}
// 2^-X as an fp32 value, for the X of a finite bf16 or fp32 amax (X <= 119,
// so 127 - X lies in [8, 254]): multiplying by it is exact, so the element
// code is e4m3(v / 2^X) as the format defines it.
__device__ __forceinline__ float mx_inv_scale(int x) { return __uint_as_float(static_cast<uint32_t>(127 - x) << 23); }

// ------------------------------------------------------------------------
// fp32 exponential for SwiGLU, written from Cody and Waite's method (Software
// Manual for the Elementary Functions, 1980): x = n ln2 + r, n = rint(x
// log2 e), ln2 split into a 16-bit head and its tail; e^r by its degree-7
// Taylor polynomial in Horner form with fused multiply-adds; the result
// scaled by 2^n in two exact power-of-two steps.  Each step is one IEEE fp32
// rounding (no contraction, no flush to zero), so the value is a fixed
// function of x.
// ------------------------------------------------------------------------
__device__ __forceinline__ float pow2i(int i) { return __int_as_float((i + 127) << 23); }

__device__ __forceinline__ float exp_poly(float x, float& n) {
  n = rintf(__fmul_rn(x, 1.44269502162933349609375f));
  float r = __fmaf_rn(-n, 0.693145751953125f, x);
  r = __fmaf_rn(-n, 1.428606765330187045e-6f, r);
  float p = 1.0f / 5040.0f;
  p = __fmaf_rn(p, r, 1.0f / 720.0f);
  p = __fmaf_rn(p, r, 1.0f / 120.0f);
  p = __fmaf_rn(p, r, 1.0f / 24.0f);
  p = __fmaf_rn(p, r, 1.0f / 6.0f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  return p;
}

__device__ __forceinline__ float exp_f32(float x) {
  float n;
  if (fabsf(x) <= 87.0f) {
    // n lies in [-126, 126], so 2^n is a normal float and the single product
    // rounds once -- the same value as the two-step scaling below, whose
    // first step is exact.
    const float p = exp_poly(x, n);
    return __fmul_rn(p, pow2i(static_cast<int>(n)));
  }
  if (x != x) return x;
  if (x > 88.72283935546875f) return __int_as_float(0x7f800000);
  if (x < -103.972076416015625f) return 0.0f;
  float p = exp_poly(x, n);
  const int ni = static_cast<int>(n);
  const int n1 = ni / 2, n2 = ni - n1;
  p = __fmul_rn(p, pow2i(n1));
  p = __fmul_rn(p, pow2i(n2));
  return p;
}

__device__ __forceinline__ float silu_f32(float z) { return __fdiv_rn(z, __fadd_rn(1.0f, exp_f32(-z))); }

// ---- branch-free forms of the same arithmetic ----------------------------
// The per-element code below has no data-dependent branch in its common
// range, so that a thread's elements form one basic block the compiler can
// interleave.  Each helper flags the rare inputs it does not cover and the
// caller recomputes those with the exact per-element path, so the values are
// bit-identical to exp_f32 / __fdiv_rn / quant_quotient.

__device__ __forceinline__ float rcp_approx(float b) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(b));
  return y;
}

// exp_f32 for |x| <= 87 (no range checks; same value).
__device__ __forceinline__ float exp_fast(float x) {
  float n;
  const float p = exp_poly(x, n);
  return __fmul_rn(p, pow2i(static_cast<int>(n)));
}

// fp32(a / b), correctly rounded, for b in [1, 2^30] and a = 0 or
// 2^-60 <= |a| <= 2^20.  A reciprocal estimate y and one correction step
// (Markstein's method, q1 = q0 + (a - b q0) y) give a candidate q1; q1 is the
// correctly rounded quotient iff |a/b - q1| < ulp(q1)/2, i.e. iff
// |a - b q1| * 2^(24 - E(q1)) < b.  The residual is computed with one fused
// multiply-add and the scaling by a power of two is exact, so the test is
// rounding-monotone and never accepts a wrong q1 (a quotient of two fp32
// values is never exactly halfway between two floats).  `ok` is cleared when
// the test fails.
__device__ __forceinline__ float div_checked(float a, float b, bool& ok) {
  const float y = rcp_approx(b);
  const float q0 = __fmul_rn(a, y);
  const float r0 = __fmaf_rn(-b, q0, a);
  const float q1 = __fmaf_rn(r0, y, q0);
  const float r1 = __fmaf_rn(-b, q1, a);
  const uint32_t eb = (__float_as_uint(q1) >> 23) & 0xFFu;
  const float sc = __uint_as_float((278u - eb) << 23);  // 2^(24 - E(q1))
  ok = ok && (a == 0.0f || __fmul_rn(fabsf(r1), sc) < b);
  return a == 0.0f ? a : q1;  // keeps the sign of a zero numerator
}

// Range in which the SwiGLU fast path applies: |z| <= 20 keeps e^-z in
// [2^-29, 2^29] and the quotients normal.
__device__ __forceinline__ bool swiglu_fast_range(float z) {
  const float a = fabsf(z);
  return a <= 20.0f && (a >= 0x1p-60f || a == 0.0f);
}

// h[j] = bf16(silu(a0[j]) * a1[j]) for N elements (N even), on pairs of
// elements with packed fp32 arithmetic.  The fast path takes the steps of
// exp_fast, div_checked and round_bf16 lane by lane, so its values are those
// of the exact per-element path that takes over when a check fails.  rint(t)
// is (t + 1.5 * 2^23) - 1.5 * 2^23 (exact round-to-nearest-even for
// |t| < 2^22), whose bit pattern also gives 2^n; negations are exact sign
// flips folded into products.  hb receives the h pairs as packed bf16 (the
// storage format).
template <int N>
__device__ __forceinline__ void swiglu_h_x2(const float* a0, const float* a1, float* h, uint32_t* hb) {
  bool fast = true;
#pragma unroll
  for (int j = 0; j < N; ++j) fast = fast && swiglu_fast_range(a0[j]);
  if (fast) {
    bool ok = true;
    const uint64_t kMagic = f2_pack(12582912.0f, 12582912.0f);
    const uint64_t kNegOne = f2_pack(-1.0f, -1.0f);
#pragma unroll
    for (int j = 0; j < N; j += 2) {
      const uint64_t z = f2_pack(a0[j], a0[j + 1]);
      const uint64_t x = f2_mul(z, kNegOne);  // -z
      const uint64_t t = f2_mul(x, f2_pack(1.44269502162933349609375f, 1.44269502162933349609375f));
      const uint64_t m = f2_add(t, kMagic);
      const uint64_t n = f2_sub(m, kMagic);  // rint(t)
      uint64_t r = f2_fma(n, f2_pack(-0.693145751953125f, -0.693145751953125f), x);
      r = f2_fma(n, f2_pack(-1.428606765330187045e-6f, -1.428606765330187045e-6f), r);
      uint64_t p = f2_pack(1.0f / 5040.0f, 1.0f / 5040.0f);
      p = f2_fma(p, r, f2_pack(1.0f / 720.0f, 1.0f / 720.0f));
      p = f2_fma(p, r, f2_pack(1.0f / 120.0f, 1.0f / 120.0f));
      p = f2_fma(p, r, f2_pack(1.0f / 24.0f, 1.0f / 24.0f));
      p = f2_fma(p, r, f2_pack(1.0f / 6.0f, 1.0f / 6.0f));
      p = f2_fma(p, r, f2_pack(0.5f, 0.5f));
      p = f2_fma(p, r, f2_pack(1.0f, 1.0f));
      p = f2_fma(p, r, f2_pack(1.0f, 1.0f));
      float m0, m1;
      f2_unpack(m, m0, m1);
      // bits(m) = 0x4B400000 + n, so (bits(m) << 23) + (127 << 23) = (n + 127) << 23 = 2^n
      const float s0 = __uint_as_float((__float_as_uint(m0) << 23) + (127u << 23));
      const float s1 = __uint_as_float((__float_as_uint(m1) << 23) + (127u << 23));
      const uint64_t d = f2_add(f2_mul(p, f2_pack(s0, s1)), f2_pack(1.0f, 1.0f));  // 1 + e^-z
      // silu = z / d (div_checked, lane by lane)
      float d0, d1;
      f2_unpack(d, d0, d1);
      const uint64_t y = f2_pack(rcp_approx(d0), rcp_approx(d1));
      const uint64_t q0 = f2_mul(z, y);
      const uint64_t nd = f2_mul(d, kNegOne);
      const uint64_t r0 = f2_fma(nd, q0, z);
      const uint64_t q1 = f2_fma(r0, y, q0);
      const uint64_t r1 = f2_fma(nd, q1, z);
      float q10, q11, r10, r11;
      f2_unpack(q1, q10, q11);
      f2_unpack(r1, r10, r11);
      const float sc0 = __uint_as_float((278u - ((__float_as_uint(q10) >> 23) & 0xFFu)) << 23);
      const float sc1 = __uint_as_float((278u - ((__float_as_uint(q11) >> 23) & 0xFFu)) << 23);
      ok = ok && (a0[j] == 0.0f || __fmul_rn(fabsf(r10), sc0) < d0);
      ok = ok && (a0[j + 1] == 0.0f || __fmul_rn(fabsf(r11), sc1) < d1);
      const float si0 = a0[j] == 0.0f ? a0[j] : q10, si1 = a0[j + 1] == 0.0f ? a0[j + 1] : q11;
      float h0, h1;
      f2_unpack(f2_mul(f2_pack(si0, si1), f2_pack(a1[j], a1[j + 1])), h0, h1);
      const uint32_t pk = pack_bf16x2(h0, h1);
      hb[j / 2] = pk;
      h[j] = bf16lo(pk);
      h[j + 1] = bf16hi(pk);
    }
    if (ok) return;
  }
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    h[j] = round_bf16(__fmul_rn(silu_f32(a0[j]), a1[j]));
    h[j + 1] = round_bf16(__fmul_rn(silu_f32(a0[j + 1]), a1[j + 1]));
    hb[j / 2] = pack_bf16x2(h[j], h[j + 1]);
  }
}

// Fast e4m3 quotient.  y = x * inv_s with inv_s = 1/s rounded to nearest lies
// within 2 ulp of x / s (two roundings of relative size 2^-24).  Rounding to
// e4m3 keeps 3 mantissa bits, so y and fp32(x / s) can only round to
// different e4m3 values when a midpoint between two neighbouring e4m3 values
// lies within those ulp.  For |y| >= 2^-6 (normal e4m3) the midpoints are the
// fp32 values whose low 20 mantissa bits are 0x80000.  Below 2^-6 the e4m3
// grid is uniform with step 2^-9, the same step as the normal binade
// [2^-6, 2^-5); adding 2^-6 maps that grid and its midpoints onto the
// binade's, and the addition rounds by at most 2^-30, far inside the +-8 ulp
// (8 * 2^-29) window tested.  So one test on the low mantissa bits of
// |y| (+ 2^-6 when small) finds every value that may round differently; those
// rare values take the exact division, everywhere else
// e4m3(y) == e4m3(fp32(x / s)).  Above 448 every value saturates to 448 either
// way.
__device__ __forceinline__ bool quant_needs_division(float y) {
  const float a = fabsf(y);
  const float v = a < 0x1p-6f ? __fadd_rn(a, 0x1p-6f) : a;
  return ((__float_as_uint(v) & 0xFFFFFu) - 0x80000u + 8u) <= 16u;
}

// out[j] = fp32(x[j] / s) as far as e4m3 rounding can tell, for N elements.
template <int N>
__device__ __forceinline__ void quant_n(const float* x, float s, float inv, float* out) {
  bool slow = false;
  const uint64_t inv2 = f2_pack(inv, inv);
#pragma unroll
  for (int j = 0; j < N; j += 2) {  // the products in pairs (packed fp32, one rounding each)
    f2_unpack(f2_mul(f2_pack(x[j], x[j + 1]), inv2), out[j], out[j + 1]);
    slow = slow || quant_needs_division(out[j]) || quant_needs_division(out[j + 1]);
  }
  if (slow) {
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (quant_needs_division(out[j])) out[j] = __fdiv_rn(x[j], s);
  }
}

// The quotient that e4m3 quantisation rounds, fp32(x / s), for one element.
__device__ __forceinline__ float quant_quotient(float x, float s, float inv_s) {
  const float y = __fmul_rn(x, inv_s);
  return quant_needs_division(y) ? __fdiv_rn(x, s) : y;
}

// ------------------------------------------------------------------------
// Shared-memory addresses, mbarriers, timers
// ------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the thread may sleep up to `hint_ns`
// waiting for the phase instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Time limit of every bounded mbarrier wait.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// Bounded wait for warps whose waiting should not take issue slots from the
// warps they share an SM sub-partition with: the same contract as
// mbar_wait_bounded, with each poll allowed to sleep up to
// MOE_IDLE_WAIT_HINT_NS.
__device__ __forceinline__ bool mbar_wait_bounded_idle(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                                       uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_hint(bar, parity, MOE_IDLE_WAIT_HINT_NS)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Bounded wait: true once the phase with `parity` has completed; false if
// `abort_flag` becomes non-zero or `limit_ns` of wall time pass first.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// The same wait taken by all 32 lanes of a warp, with one outcome for the
// whole warp: a lane that saw the phase complete while another lane of the
// warp ran out of time follows the timeout, so that the warp never splits
// ahead of a warp-wide synchronisation.
__device__ __forceinline__ bool mbar_wait_bounded_warp(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                                       uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort_flag, limit_ns));
}

// ------------------------------------------------------------------------
// TMA
// ------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled as
// transaction bytes on `bar`.  x is the innermost coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// CTA-pair form: the completion is signalled on `bar`, a shared::cluster
// address that may lie in the peer CTA of the pair (the pair's MMA issuer
// waits there for both CTAs' operands).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Contiguous copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global to this CTA's shared memory; completion is signalled
// as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// 4-byte asynchronous copy global -> shared through L1 (cp.async); with
// src_bytes 0 nothing is read and the destination is zero-filled.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed cp.async groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 3-D tiled store of one box from this CTA's shared memory; completion is
// tracked by bulk async-groups (commit, then wait).
__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed groups may still be reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed group has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make this thread's shared-memory writes visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------------
// Thread-block clusters (CTA pairs)
// ------------------------------------------------------------------------
// shared::cluster address of the variable at shared::cta address `addr` in
// CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
// Arrive (release, cluster scope) on an mbarrier of any CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Relaxed form, for a release that orders nothing but completed tensor-memory
// loads (tcgen05.wait::ld has returned, so the registers already hold the
// data): measured about 900 clocks cheaper per arrive than the release form.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// All threads of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, tensor memory)
// ------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// CTA-pair forms: one warp of each CTA of the pair allocates together; the
// columns are allocated at the same address in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Barrier among `count` threads (a multiple of 32) on hardware barrier `id`
// (1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Per-warpgroup register budget (every warp of the warpgroup executes the
// same instruction).  An increase draws on registers released by decreases in
// the same CTA, within what the CTA was launched with.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4, one CTA.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 with bf16 A and B (K = 16 per
// instruction: 32 bytes, the same byte step as kind::f8f6f4), one CTA.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// MXFP8 block-scaled MMA: D[tmem] (+)= (A * 2^(sfa - 127)) (B * 2^(sfb - 127))^T,
// kind::mxf8f6f4 with one E8M0 scale per 32 elements of K (scale_vec::1X),
// one CTA, K = 32 per instruction.  The scales are read from tensor memory:
// A's for row m at (lane m, column sfa + m / 32) and B's for column n at
// (lane 32 q + n % 32, column sfb + n / 32) in every lane quarter q; each
// 32-bit cell holds four E8M0 bytes, of which the instruction descriptor's
// a_sf_id / b_sf_id selects one (the K block of this instruction within the
// cell's four).
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Shared memory -> tensor memory: 32 rows of 16 bytes (an unswizzled K-major
// matrix, see smem_desc_plain) to 32 lanes x 4 columns, replicated into all
// four lane quarters.  Asynchronous; ordered with the tcgen05.mma that this
// thread issues after it.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 with f16 A and B, one CTA:
// the A operand (M = 128 rows, K = 16) is read from tensor memory, row m in
// lane m and elements 2c, 2c + 1 of K in column c (low, high half).
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far has
// completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// D (+)= A * B^T over a CTA pair (issued by the even CTA): M = 256 rows, 128
// from each CTA's shared memory at the same offset; the B tile's N rows are
// split the same way; each CTA's tensor memory receives its own 128 rows.
__device__ __forceinline__ void mma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier at offset `bar` of every CTA in `mask` once the
// pair MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp receives the
// 32 columns of TMEM lane (lane base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// 32 lanes x 16 consecutive fp32 columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// The same 16 columns delivered as 8 packed fp32 pairs (columns 2i, 2i+1 in
// pair i), so that packed f32x2 arithmetic takes them without register moves.
__device__ __forceinline__ void tmem_ld_32x32b_x16_pairs(uint32_t taddr, uint64_t (&r)[8]) {
  asm volatile(
      "{\n\t.reg .b32 t<16>;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, "
      "t15}, [%8];\n\t"
      "mov.b64 %0, {t0, t1};\n\tmov.b64 %1, {t2, t3};\n\tmov.b64 %2, {t4, t5};\n\tmov.b64 %3, {t6, t7};\n\t"
      "mov.b64 %4, {t8, t9};\n\tmov.b64 %5, {t10, t11};\n\tmov.b64 %6, {t12, t13};\n\tmov.b64 %7, {t14, t15};\n\t}"
      : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]), "=l"(r[7])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns from registers: thread i of the
// warp writes the 32 columns of TMEM lane (lane base + i).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// The tensor-memory stores this thread issued have completed.
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle (rows of 128 bytes, 8-row / 1024-byte swizzle atoms, tile
// base 1024-byte aligned): start address >> 4 in bits [0,14), leading byte
// offset (unused for this layout, 16 B) in [16,30), stride byte offset 1024 B
// (between 8-row atoms) in [32,46), descriptor version 1 at bit 46, base
// offset 0, layout type 2 (128-byte swizzle) in bits [61,64).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor for kind::f8f6f4: fp32 accumulator (bits [4,6) = 1),
// A and B e4m3 (format 0), both K-major, N >> 3 in bits [17,23), M >> 4 in
// bits [24,29).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// Shared-memory descriptor of an unswizzled K-major matrix whose 16-byte rows
// lie back to back: 8-row core matrices 128 bytes apart (leading and stride
// byte offsets both 128), version 1, layout type 0.  Used for the 32 x 16-byte
// scale-factor atoms that tcgen05.cp copies.
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
         (static_cast<uint64_t>(128 >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
}

// Instruction descriptor for kind::mxf8f6f4 block scaling: b_sf_id in bits
// [4,6), A and B e4m3 (format 0), both K-major, N >> 3 in [17,23), E8M0
// scale type (bit 23), M >> 4 in [24,29), a_sf_id in [29,31).
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int m, int n, int a_sf_id, int b_sf_id) {
  return (static_cast<uint32_t>(b_sf_id) << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(m >> 4) << 24) | (static_cast<uint32_t>(a_sf_id) << 29);
}

// Instruction descriptor for kind::f16 with f16 A and B (format 0), fp32
// accumulator, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Instruction descriptor for kind::f16 with bf16 A and B (format 1 in bits
// [7,10) and [10,13)), fp32 accumulator, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}


}  // namespace moe
