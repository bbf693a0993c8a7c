// common.cuh -- device helpers shared by the sm_103a kernels of this library.
//
// Number formats (e4m3, e2m1, UE8M0, bf16), the exp/SiLU specification that
// makes the activation quantisation reproducible bit for bit, warp helpers and
// the device error word. Everything here is written for sm_103a; every float
// operation whose rounding matters uses an explicit _rn intrinsic so that the
// compiler cannot contract it into an fma.
//
// Sources cited by tag and section:
//  [LR] "Blackwell FP4 MoE：把 live-row 边界贯穿整个 FFN"
//  [DG] "Blackwell 上的 DeepGEMM FusedMoE（sglang）"
//  [SD] "Phase 20: Sparse MoE Decode — 只算被路由到的专家"
//  [KM] "kimi3_pro6000_sglang_sm120_flashinfer_mxfp4" experiment log
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

// ----------------------------------------------------------------- errors
// Device-side anomalies set bits in a context-owned word; nothing traps.
__device__ __forceinline__ void raise_error(uint32_t* err, uint32_t bit) {
  if (err) atomicOr(err, bit);
}

// ------------------------------------------------------------------ bf16
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// fp32 -> bf16 bits, round to nearest even, NaN kept quiet.
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return (u >> 16) | 0x40u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return u >> 16;
}
// Two fp32 -> packed bf16x2 (lo in bits 0-15), hardware round-to-nearest-even
// (one cvt.rn.bf16x2.f32); equal to f32_to_bf16_bits on every non-NaN input.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------------- e4m3
// Two fp32 values -> two e4m3 codes with the hardware's round-to-nearest-even
// and saturation to the largest finite value (+-448); `lo` lands in bits 0-7.
__device__ __forceinline__ uint32_t e4m3x2_satfinite(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// e4m3 pair (bits 0-7 and 8-15) -> two fp32 values (exact, through f16).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(two_codes & 0xFFFFu)));
  float2 out;
  asm("{.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;}"
      : "=f"(out.x), "=f"(out.y) : "r"(h2));
  return out;
}

// ------------------------------------------------------------------ UE8M0
// Smallest power of two not below s (s >= 0, finite), as a biased exponent
// byte: the fp32 exponent field, plus one when the mantissa is non-zero,
// except at exponent 0xFE and for subnormals not above 2^-127
// ([DG] 附录 A, rounding-up cast).
__device__ __forceinline__ uint32_t ue8m0_ceil(float s) {
  uint32_t bits = __float_as_uint(s);
  uint32_t e = (bits >> 23) & 0xFFu;
  uint32_t m = bits & 0x7FFFFFu;
  uint32_t ru = (m > 0u && e != 0xFEu) && !(e == 0u && m <= 0x400000u);
  return (e + ru) & 0xFFu;
}

// 2^k for k in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float pow2_f32(int k) {
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}

// Scale byte for a group with absolute maximum `amax` (NaN never reaches it:
// the callers reduce with fmaxf, which drops NaN). A non-finite amax keeps the
// scale finite at 0xFE ([KM] NaN/Inf decision: E8M0 must never be 0xFF).
__device__ __forceinline__ uint32_t group_scale_byte(float amax) {
  if (isinf(amax)) return 0xFEu;
  return ue8m0_ceil(__fdiv_rn(amax, 448.0f));
}

// ----------------------------------------------------- exp specification
// The pages leave exp unspecified; this library fixes one definition so that
// SiLU and the routing weights are reproducible bit for bit:
//   n = rint(x * fl(log2 e)); r = fma(-n, L_hi, x); r = fma(-n, L_lo, r)
//   with L_hi = fl(ln 2) with its 12 low significand bits cleared (exact
//   products n * L_hi for |n| < 4096) and L_lo = fl(ln 2 - L_hi);
//   p = Taylor series of e^r to degree 7 by Horner, coefficients fl(1/k!),
//   one fma per step (Cody & Waite reduction, textbook series);
//   e^x = (p * 2^(n/2)) * 2^(n - n/2), n/2 truncated toward zero;
//   x >= 128 -> +inf, x <= -150 -> +0, NaN -> NaN.
// Constants as fp32 bit patterns:
//   fl(log2 e) 0x3fb8aa3b, L_hi 0x3f317000, L_lo 0x3805fdf4,
//   1/3! 0x3e2aaaab, 1/4! 0x3d2aaaab, 1/5! 0x3c088889, 1/6! 0x3ab60b61,
//   1/7! 0x39500d01.
__device__ __forceinline__ float spec_exp(float x) {
  if (isnan(x)) return x;
  if (x >= 128.0f) return __uint_as_float(0x7F800000u);
  if (x <= -150.0f) return 0.0f;
  const float t = __fmul_rn(x, __uint_as_float(0x3fb8aa3bu));
  const float fn = rintf(t);
  const int n = (int)fn;
  float r = __fmaf_rn(-fn, __uint_as_float(0x3f317000u), x);
  r = __fmaf_rn(-fn, __uint_as_float(0x3805fdf4u), r);
  float p = __uint_as_float(0x39500d01u);
  p = __fmaf_rn(p, r, __uint_as_float(0x3ab60b61u));
  p = __fmaf_rn(p, r, __uint_as_float(0x3c088889u));
  p = __fmaf_rn(p, r, __uint_as_float(0x3d2aaaabu));
  p = __fmaf_rn(p, r, __uint_as_float(0x3e2aaaabu));
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int n1 = n / 2;
  const int n2 = n - n1;
  return __fmul_rn(__fmul_rn(p, pow2_f32(n1)), pow2_f32(n2));
}

// silu(g) = g / (1 + exp(-g)), one add and one IEEE division.
__device__ __forceinline__ float spec_silu(float g) {
  return __fdiv_rn(g, __fadd_rn(1.0f, spec_exp(-g)));
}
__device__ __forceinline__ float spec_sigmoid(float x) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, spec_exp(-x)));
}

// gpt-oss GLU of the decode path ([SD] §3): g = min(g, L), u = clamp(u, -L, L)
// when L > 0; act = (g * sigmoid(alpha g)) * (u + beta).
__device__ __forceinline__ float glu_value(float g, float u, float alpha, float beta, float limit) {
  if (limit > 0.0f) {
    g = fminf(g, limit);
    u = fminf(fmaxf(u, -limit), limit);
  }
  const float s = spec_sigmoid(__fmul_rn(alpha, g));
  return __fmul_rn(__fmul_rn(g, s), __fadd_rn(u, beta));
}

// tanh specification (the pages use tanh in SiTU without defining it; the
// oracle implements the same definition independently):
//   |y| < 2^-12  -> y
//   |y| < 1/4    -> fma(y*y^2, P(y^2), y), P the Taylor series of
//                   (tanh y - y)/y^3 through the y^8 term, coefficients the
//                   fp32 roundings of -1/3, 2/15, -17/315, 62/2835,
//                   -1382/155925, Horner with one fma per step
//   |y| >= 9     -> sign(y)
//   otherwise    -> sign(y) (1 - e) / (1 + e), e = spec_exp(-2|y|)
constexpr float kTanhP0 = (float)(-1.0 / 3.0);
constexpr float kTanhP1 = (float)(2.0 / 15.0);
constexpr float kTanhP2 = (float)(-17.0 / 315.0);
constexpr float kTanhP3 = (float)(62.0 / 2835.0);
constexpr float kTanhP4 = (float)(-1382.0 / 155925.0);

__device__ __forceinline__ float spec_tanh(float y) {
  if (isnan(y)) return y;
  const float a = fabsf(y);
  if (a < 0x1p-12f) return y;
  if (a < 0.25f) {
    const float z = __fmul_rn(y, y);
    float p = kTanhP4;
    p = __fmaf_rn(p, z, kTanhP3);
    p = __fmaf_rn(p, z, kTanhP2);
    p = __fmaf_rn(p, z, kTanhP1);
    p = __fmaf_rn(p, z, kTanhP0);
    return __fmaf_rn(__fmul_rn(y, z), p, y);
  }
  if (a >= 9.0f) return copysignf(1.0f, y);
  const float e = spec_exp(__fmul_rn(-2.0f, a));
  return copysignf(__fdiv_rn(__fsub_rn(1.0f, e), __fadd_rn(1.0f, e)), y);
}

// SiTU halves: gate' = (beta_s * tanh(g / beta_s)) * sigmoid(g) and
// up' = beta_l * tanh(u / beta_l), one IEEE operation each, in this order.
__device__ __forceinline__ float spec_situ_gate(float g, float beta_s) {
  return __fmul_rn(__fmul_rn(beta_s, spec_tanh(__fdiv_rn(g, beta_s))), spec_sigmoid(g));
}
__device__ __forceinline__ float spec_situ_up(float u, float beta_l) {
  return __fmul_rn(beta_l, spec_tanh(__fdiv_rn(u, beta_l)));
}

// ------------------------------------------------ packed pairs (f32x2)
// Blackwell executes fp32 add / mul / fma on register pairs; each half is the
// ordinary IEEE round-to-nearest operation, so results are bitwise those of
// the scalar forms.
__device__ __forceinline__ uint64_t pk(float2 a) {
  return ((uint64_t)__float_as_uint(a.y) << 32) | __float_as_uint(a.x);
}
__device__ __forceinline__ float2 upk(uint64_t r) {
  return make_float2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)), "l"(pk(c)));
  return upk(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)));
  return upk(d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)));
  return upk(d);
}
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// SiLU of a bf16 gate value through the per-context table (65,536 entries,
// entry i = spec_silu(bf16 with bits i)); with the clamp, gate values above
// the limit (or NaN) take spec_silu(limit) instead, as min(g, L) does.
template <bool kClamp>
__device__ __forceinline__ float silu_of_bf16(const float* __restrict__ tbl, uint32_t gbits, float g, float limit,
                                              float silu_limit) {
  if (kClamp && !(g <= limit) && !isnan(limit)) return silu_limit;
  return __ldg(tbl + (gbits & 0xFFFFu));
}

// ------------------------------------------------------------------- e2m1
// e2m1 nibble -> fp32: 1 sign, 2 exponent (bias 1), 1 mantissa bit.
__device__ __forceinline__ float e2m1_to_f32(uint32_t nib) {
  const uint32_t e = (nib >> 1) & 3u, m = nib & 1u;
  float mag = (e == 0u) ? (m ? 0.5f : 0.0f)
                        : __uint_as_float(((e - 1u + 127u) << 23) | (m << 22));
  return (nib & 8u) ? -mag : mag;
}

// Two e2m1 values in one byte (low nibble first) -> two fp32 values (exact).
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte) {
  uint32_t h2;
  asm("{.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;}" : "=r"(h2) : "h"((uint16_t)byte));
  float2 out;
  asm("{.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;}"
      : "=f"(out.x), "=f"(out.y) : "r"(h2));
  return out;
}

// ------------------------------------------------------------------ warps
__device__ __forceinline__ float warp_max_xor(float v, int width_log2) {
  for (int o = 1 << (width_log2 - 1); o > 0; o >>= 1)
    v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__host__ __device__ __forceinline__ int64_t align_up64(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

}  // namespace moe
