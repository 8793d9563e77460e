// MLP glue around the FP8 linears: exact-erf GELU forward/backward (fp32
// arithmetic, bf16 in/out) and fp32 gradient accumulation over microbatches.
// Elementwise and HBM-bound: 16-byte vector loads/stores, grid-stride over a
// grid sized in multiples of the SM count.
#include "common.cuh"
#include "internal.h"

namespace fp8lin {

namespace {

constexpr int kThreads = 256;

// gelu_f2 / gelu_grad_f2 / pack_bf16x2 live in common.cuh (shared with the
// fused GELU + quantize path).

__global__ void gelu_fwd_kernel(const uint4 *__restrict__ H, uint4 *__restrict__ A, int64_t n8) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 h = H[i];
    const uint32_t w[4] = {h.x, h.y, h.z, h.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float g0, g1;
      gelu_f2(bf16lo(w[k]), bf16hi(w[k]), g0, g1);
      o[k] = pack_bf16x2(g0, g1);
    }
    A[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void gelu_bwd_kernel(const uint4 *__restrict__ dA, const uint4 *__restrict__ H,
                                uint4 *__restrict__ dH, int64_t n8) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 h = H[i], d = dA[i];
    const uint32_t hw[4] = {h.x, h.y, h.z, h.w}, dw[4] = {d.x, d.y, d.z, d.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float g0, g1;
      gelu_grad_f2(bf16lo(hw[k]), bf16hi(hw[k]), g0, g1);
      o[k] = pack_bf16x2(__fmul_rn(bf16lo(dw[k]), g0), __fmul_rn(bf16hi(dw[k]), g1));
    }
    dH[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void grad_accumulate_kernel(float4 *__restrict__ acc, const uint2 *__restrict__ dW,
                                       int64_t n4) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 a = acc[i];
    const uint2 d = dW[i];
    a.x = __fadd_rn(a.x, bf16lo(d.x));
    a.y = __fadd_rn(a.y, bf16hi(d.x));
    a.z = __fadd_rn(a.z, bf16lo(d.y));
    a.w = __fadd_rn(a.w, bf16hi(d.y));
    acc[i] = a;
  }
}

unsigned grid_for(int64_t items) {
  const int64_t want = (items + kThreads - 1) / kThreads;
  return (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms() * 8));
}

}  // namespace

cudaError_t launch_gelu_fwd(const void *H, void *A, int64_t n, cudaStream_t st) {
  const int64_t n8 = n / 8;
  LaunchScope ls("gelu_fwd", st, 4.0 * n, 0.0, n);
  gelu_fwd_kernel<<<grid_for(n8), kThreads, 0, st>>>(static_cast<const uint4 *>(H),
                                                      static_cast<uint4 *>(A), n8);
  return cudaGetLastError();
}

cudaError_t launch_gelu_bwd(const void *dA, const void *H, void *dH, int64_t n, cudaStream_t st) {
  const int64_t n8 = n / 8;
  LaunchScope ls("gelu_bwd", st, 6.0 * n, 0.0, n);
  gelu_bwd_kernel<<<grid_for(n8), kThreads, 0, st>>>(static_cast<const uint4 *>(dA),
                                                      static_cast<const uint4 *>(H),
                                                      static_cast<uint4 *>(dH), n8);
  return cudaGetLastError();
}

cudaError_t launch_grad_accumulate(float *acc, const void *dW, int64_t n, cudaStream_t st) {
  const int64_t n4 = n / 4;
  LaunchScope ls("grad_accumulate", st, 10.0 * n, (double)n, n);
  grad_accumulate_kernel<<<grid_for(n4), kThreads, 0, st>>>(
      reinterpret_cast<float4 *>(acc), static_cast<const uint2 *>(dW), n4);
  return cudaGetLastError();
}

}  // namespace fp8lin
