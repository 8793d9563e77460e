// MLP glue around the FP8 linears: exact-erf GELU forward/backward (fp32
// arithmetic, bf16 in/out) and fp32 gradient accumulation over microbatches.
// Elementwise: 16-byte vector loads/stores, grid-stride over a grid sized in
// multiples of the SM count (the GELU kernels: exactly the resident blocks).
#include "common.cuh"
#include "internal.h"

namespace fp8lin {

namespace {

constexpr int kThreads = 256;

// gelu_f2 / gelu_grad_f2 / pack_bf16x2 live in common.cuh (shared with the
// fused GELU + quantize path).

__device__ __forceinline__ uint4 gelu8(uint4 h) {
  const uint32_t w[4] = {h.x, h.y, h.z, h.w};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float g0, g1;
    gelu_f2(bf16lo(w[k]), bf16hi(w[k]), g0, g1);
    o[k] = pack_bf16x2(g0, g1);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 gelu_bwd8(uint4 d, uint4 h) {
  const uint32_t hw[4] = {h.x, h.y, h.z, h.w}, dw[4] = {d.x, d.y, d.z, d.w};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float g0, g1;
    gelu_grad_f2(bf16lo(hw[k]), bf16hi(hw[k]), g0, g1);
    o[k] = pack_bf16x2(__fmul_rn(bf16lo(dw[k]), g0), __fmul_rn(bf16hi(dw[k]), g1));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Grid-stride over 8-element vectors on a grid of exactly the resident
// blocks, at full occupancy (32 registers: 8 blocks of 256 threads per SM).
// Measured on 131072 x 2048 with an earlier form of the GELU arithmetic:
// forward 0.255 ms, backward 0.293 ms; two vectors per iteration at 40-52
// registers ran 0.267 / 0.314-0.339 ms.
__global__ void __launch_bounds__(kThreads, 8) gelu_fwd_kernel(const uint4 *__restrict__ H,
                                                               uint4 *__restrict__ A, int64_t n8) {
  pdl_wait_then_release();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride)
    A[i] = gelu8(H[i]);
}

__global__ void __launch_bounds__(kThreads, 8) gelu_bwd_kernel(const uint4 *__restrict__ dA,
                                                               const uint4 *__restrict__ H,
                                                               uint4 *__restrict__ dH, int64_t n8) {
  pdl_wait_then_release();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride)
    dH[i] = gelu_bwd8(dA[i], H[i]);
}

__global__ void grad_accumulate_kernel(float4 *__restrict__ acc, const uint2 *__restrict__ dW,
                                       int64_t n4) {
  pdl_wait_then_release();
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

// Grid of the glue kernels: every block resident at once (blocks per SM from
// the occupancy calculator, per kernel and device), so that no block starts
// after the others have finished their grid-stride share.
template <typename Kernel>
unsigned grid_resident(Kernel kernel, int64_t items, int *per_dev) {
  const int bps = blocks_per_sm(kernel, kThreads, per_dev);
  const int64_t want = (items + kThreads - 1) / kThreads;
  return (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms() * bps));
}
int g_gelu_fwd_bps[64], g_gelu_bwd_bps[64], g_acc_bps[64];

}  // namespace

cudaError_t launch_gelu_fwd(const void *H, void *A, int64_t n, cudaStream_t st) {
  const int64_t n8 = n / 8;
  LaunchScope ls("gelu_fwd", st, 4.0 * n, 0.0, n);
  const unsigned grid = grid_resident(gelu_fwd_kernel, n8, g_gelu_fwd_bps);
  return launch_kernel(gelu_fwd_kernel, dim3(grid), dim3(kThreads), 0, st,
                       static_cast<const uint4 *>(H), static_cast<uint4 *>(A), n8);
}

cudaError_t launch_gelu_bwd(const void *dA, const void *H, void *dH, int64_t n, cudaStream_t st) {
  const int64_t n8 = n / 8;
  LaunchScope ls("gelu_bwd", st, 6.0 * n, 0.0, n);
  const unsigned grid = grid_resident(gelu_bwd_kernel, n8, g_gelu_bwd_bps);
  return launch_kernel(gelu_bwd_kernel, dim3(grid), dim3(kThreads), 0, st,
                       static_cast<const uint4 *>(dA), static_cast<const uint4 *>(H),
                       static_cast<uint4 *>(dH), n8);
}

cudaError_t launch_grad_accumulate(float *acc, const void *dW, int64_t n, cudaStream_t st) {
  const int64_t n4 = n / 4;
  LaunchScope ls("grad_accumulate", st, 10.0 * n, (double)n, n);
  const unsigned grid = grid_resident(grad_accumulate_kernel, n4, g_acc_bps);
  return launch_kernel(grad_accumulate_kernel, dim3(grid), dim3(kThreads), 0, st,
                       reinterpret_cast<float4 *>(acc), static_cast<const uint2 *>(dW), n4);
}

}  // namespace fp8lin
