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

// Programmatic dependent launch.  Every kernel of this library calls one of
// these before its first global-memory access (after its barrier setup,
// descriptor prefetch and TMEM allocation): the thread waits until the kernel
// before it on the stream has completed with its memory visible (at once when
// the launch did not allow overlap).  Results are those of serial launches.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// ... and then lets the next kernel's CTAs start their own setup on whatever
// SM resources are free.  The GEMM does not release early: the small kernels
// that follow it (amax pass, split-K reduce, gradient accumulation) fit beside
// a running GEMM CTA, and with an early release the step ran slower (fp8
// linear step at N = 131072 on four shapes: 3.84 ms with the GEMM releasing
// at exit, 3.93 ms with it releasing at once).
__device__ __forceinline__ void pdl_wait_then_release() {
  pdl_wait();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// Exact-erf GELU and its derivative in fp32, two elements at a time (shared
// by the standalone GELU kernels and the fused GELU + quantize path, so both
// round identically).
//   GELU(h) = h Phi(h),  GELU'(h) = Phi(h) + h phi(h),
//   Phi(h) = erfc(-h / sqrt 2) / 2,  phi(h) = exp(-h^2 / 2) / sqrt(2 pi).
// With z = |h| / sqrt 2: erfc(z) = exp(-z^2) erfcx(z), and erfcx(z) is
// approximated as t Q(t), t = 1 / (1 + z/2), Q the degree-7 polynomial that
// gelu_fit.py fits (relative error 3e-6 for all z >= 0).  Phi(h) is then
// erfc(z)/2 for h < 0 and 1 - erfc(z)/2 for h >= 0, with full relative
// precision in the negative tail, and exp(-z^2) serves phi as well.  The
// exponential is taken as 2^64 exp(-z^2) (normal down to the smallest
// results bf16 can hold) and the product is scaled by 2^-64 last, so tiny
// results round once, subnormals included.  The arithmetic runs on packed
// fp32 pairs (f32x2: one instruction, two IEEE operations); the reciprocal
// and the base-2 exponential, the hardware's approximate instructions, are
// per element.
// Every finite bf16 input lands within 1 bf16 ulp of the exact value (tested
// over all of them).
namespace gelu2 {
__device__ __forceinline__ uint64_t pk(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk(uint64_t r, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t dup(float a) { return pk(a, a); }
// For z = |h| / sqrt 2, both elements: tq = t Q(t) / 2 ~ erfcx(z) / 2 and e64 = 2^64 exp(-z^2).
// The 1/sqrt 2 is folded into the constants (d = 1 + |h| / (2 sqrt 2), exponent 64 - h^2 log2(e) / 2)
// and the 1/2 into Q's coefficients, both exact or within a rounding of the unfolded forms.
__device__ __forceinline__ void parts(float h0, float h1, uint64_t &tq, uint64_t &e64) {
  const uint64_t a = pk(fabsf(h0), fabsf(h1));
  float d0, d1;
  upk(fma2(a, dup(0.35355339059327376f), dup(1.0f)), d0, d1);
  float t0, t1;  // the hardware's approximate reciprocal (within 1 ulp of 1/d)
  asm("rcp.approx.f32 %0, %1;" : "=f"(t0) : "f"(d0));
  asm("rcp.approx.f32 %0, %1;" : "=f"(t1) : "f"(d1));
  const uint64_t t = pk(t0, t1);
  uint64_t q = fma2(dup(0.025493290275335312f), t, dup(-0.05529460310935974f));
  q = fma2(q, t, dup(-0.020236637443304062f));
  q = fma2(q, t, dup(0.062468305230140686f));
  q = fma2(q, t, dup(0.08111003786325455f));
  q = fma2(q, t, dup(0.12441571056842804f));
  q = fma2(q, t, dup(0.14099758863449097f));
  q = fma2(q, t, dup(0.14104776084423065f));
  tq = mul2(t, q);
  float a0, a1;
  upk(fma2(mul2(a, a), dup(-0.72134752044448170f), dup(64.0f)), a0, a1);
  float x0, x1;  // the hardware's approximate base-2 exponential (relative error ~2^-22)
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(x0) : "f"(a0));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(x1) : "f"(a1));
  e64 = pk(x0, x1);
}
}  // namespace gelu2

// GELU of two values.
__device__ __forceinline__ void gelu_f2(float h0, float h1, float &g0, float &g1) {
  using namespace gelu2;
  uint64_t tq, e64;
  parts(h0, h1, tq, e64);
  // h erfc(z) / 2
  const uint64_t hq = mul2(mul2(mul2(pk(h0, h1), tq), e64), dup(5.42101086242752217e-20f));
  float q0, q1;
  upk(hq, q0, q1);
  g0 = h0 >= 0.0f ? __fsub_rn(h0, q0) : q0;
  g1 = h1 >= 0.0f ? __fsub_rn(h1, q1) : q1;
}
// GELU'(h) of two values.
__device__ __forceinline__ void gelu_grad_f2(float h0, float h1, float &g0, float &g1) {
  using namespace gelu2;
  uint64_t tq, e64;
  parts(h0, h1, tq, e64);
  // h >= 0: 1 - erfc(z)/2 + h phi(h);  h < 0: erfc(z)/2 + h phi(h)
  const uint64_t s = pk(h0 >= 0.0f ? -1.0f : 1.0f, h1 >= 0.0f ? -1.0f : 1.0f);
  const uint64_t v = mul2(mul2(fma2(s, tq, mul2(pk(h0, h1), dup(0.39894228040143268f))), e64),
                          dup(5.42101086242752217e-20f));
  float v0, v1;
  upk(v, v0, v1);
  g0 = __fadd_rn(h0 >= 0.0f ? 1.0f : 0.0f, v0);
  g1 = __fadd_rn(h1 >= 0.0f ? 1.0f : 0.0f, v1);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace fp8lin
