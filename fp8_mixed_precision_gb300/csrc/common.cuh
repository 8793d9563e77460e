// Shared device helpers for the FP8 linear library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <float.h>

#include "../../include/fp8lin.h"
#include "internal.h"

namespace fp8lin {

constexpr float kE4M3Max = 448.0f;
constexpr float kE5M2Max = 57344.0f;

// count_launch / LaunchScope are declared in internal.h.

// ---------------------------------------------------------------------------
// Scale rule: scale = fp32(fmax / amax) with IEEE round-to-nearest-even
// division; amax == 0 -> 1; overflow -> FLT_MAX; scale_inv = fp32(1 / scale).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void scale_from_amax(float amax, float fmax, float &s, float &s_inv) {
  if (amax == 0.0f) {
    s = 1.0f;
    s_inv = 1.0f;
    return;
  }
  s = __fdiv_rn(fmax, amax);
  if (isinf(s)) s = FLT_MAX;
  s_inv = __fdiv_rn(1.0f, s);
}

// |x| max that ignores NaN (fmaxf returns the non-NaN operand).
__device__ __forceinline__ float amax_acc(float acc, float v) { return fmaxf(acc, fabsf(v)); }

// Two fp32 -> two FP8 bytes, saturating round-to-nearest-even; lo lands in
// the low byte.  NaN maps to 0x7F in both formats.
template <int FMT>
__device__ __forceinline__ uint32_t cvt2(float lo, float hi) {
  uint16_t r;
  if (FMT == FP8_FORMAT_E4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  uint32_t v = r;
  if (isnan(lo)) v = (v & 0xFF00u) | 0x7Fu;
  if (isnan(hi)) v = (v & 0x00FFu) | 0x7F00u;
  return v;
}

// Four fp32 -> four FP8 bytes packed little-endian into a 32-bit word.
template <int FMT>
__device__ __forceinline__ uint32_t cvt4(float a, float b, float c, float d) {
  return cvt2<FMT>(a, b) | (cvt2<FMT>(c, d) << 16);
}

// As cvt2 without the NaN fix-up: only for values known not to be NaN.
template <int FMT>
__device__ __forceinline__ uint32_t cvt2_finite(float lo, float hi) {
  uint16_t r;
  if (FMT == FP8_FORMAT_E4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
template <int FMT>
__device__ __forceinline__ uint32_t cvt4_finite(float a, float b, float c, float d) {
  return cvt2_finite<FMT>(a, b) | (cvt2_finite<FMT>(c, d) << 16);
}

// True if any bf16 of the packed pairs is inf or NaN (exponent all ones).
__device__ __forceinline__ bool any_nonfinite_bf16(uint4 a, uint4 b) {
  const uint32_t e = 0x7F807F80u;
  uint32_t m = __vcmpeq2(a.x & e, e) | __vcmpeq2(a.y & e, e) | __vcmpeq2(a.z & e, e) |
               __vcmpeq2(a.w & e, e) | __vcmpeq2(b.x & e, e) | __vcmpeq2(b.y & e, e) |
               __vcmpeq2(b.z & e, e) | __vcmpeq2(b.w & e, e);
  return m != 0;
}

// Exact-erf GELU and its derivative in fp32 (shared by the standalone GELU
// kernels and the fused GELU + quantize path, so both round identically).
// Phi(h) via erfc keeps full relative precision for large negative h.
__device__ __forceinline__ float gelu_f(float h) {
  return 0.5f * h * erfcf(-h * 0.70710678118654752f);
}
__device__ __forceinline__ float gelu_grad_f(float h) {
  const float cdf = 0.5f * erfcf(-h * 0.70710678118654752f);
  const float pdf = expf(-0.5f * h * h) * 0.39894228040143268f;
  return fmaf(h, pdf, cdf);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace fp8lin
