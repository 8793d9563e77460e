// Internal launcher interface between the C-ABI layer (api.cpp) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>  // CUtensorMap (type only)
#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>
#include <algorithm>

namespace fp8lin {

// Host-side launch counter (defined in api.cpp).
void count_launch();

// Brackets one kernel launch with CUDA events on its stream while kernel
// timing is enabled (fp8_profile_begin/end); also counts the launch.
// bytes/flops: the launch's algorithmic HBM traffic and floating-point work;
// m, n, k: its problem shape (GEMM M, N, K; quantizer rows, columns; glue
// element count), which keeps launches of one kernel on different shapes
// apart in the timing records.
class LaunchScope {
 public:
  LaunchScope(const char *name, cudaStream_t st, double bytes, double flops, int64_t m = 0,
              int64_t n = 0, int64_t k = 0);
  ~LaunchScope();

 private:
  int rec_ = -1;
  cudaStream_t st_;
};

// Tensorwise quantization keeps one fp32 partial amax per CTA of its first
// pass in the caller's workspace; at most this many.
constexpr int kMaxPartials = 1024;

int num_sms();

// Kernel launches allow programmatic dependent launch (the kernel may be
// scheduled while the previous kernel on the stream drains; each kernel waits
// for it in pdl_wait or pdl_wait_then_release before touching global memory,
// see common.cuh) unless the
// environment sets FP8LIN_PDL=0 when the library first launches.
bool pdl_enabled();

// Blocks of `kernel` (threads per block, no dynamic shared memory) that fit on
// one SM of the current device, cached per device in per_dev[64].  Grids of
// grid-stride kernels are sized to this many blocks per SM: under overlapped
// launch the blocks are placed on SMs in the order the previous kernel frees
// them, and a smaller grid would crowd onto the first SMs freed.
template <typename Kernel>
int blocks_per_sm(Kernel kernel, int threads, int *per_dev) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 1;
  if (per_dev[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1)
      n = 1;
    per_dev[dev] = n;
  }
  return per_dev[dev];
}

// overlap = false: a plain launch (the kernel starts once the previous one on
// the stream has completed).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_as(bool overlap, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                             size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap && pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, Args... args) {
  return launch_kernel_as(true, kernel, grid, block, smem, st, args...);
}
int tensorwise_partials_count(int64_t rows, int64_t cols);

// mode: 0 tensorwise, 1 1x128 blocks, 2 128x128 tiles; fmt: fp8_format.
// Tensorwise with amax_done: the first pass already wrote `partials`
// (launch_amax_partials on the same tensor); only the cast runs.
cudaError_t launch_quantize(const void *x, int64_t rows, int64_t cols, int mode, int fmt,
                            uint8_t *out_row, uint8_t *out_col, float *row_scale,
                            float *row_scale_inv, float *col_scale, float *col_scale_inv,
                            float *partials, cudaStream_t st, bool amax_done = false);
// Tensorwise first pass alone: tensorwise_partials_count(rows, cols) partial maxima.
cudaError_t launch_amax_partials(const void *x, int64_t rows, int64_t cols, float *partials,
                                 cudaStream_t st);

// Delayed scaling: cast with the scale of the history's maximum, then write
// this tensor's amax to hist[step % hist_len] (partials: >= 2 x SMs floats).
cudaError_t launch_quantize_delayed(const void *x, int64_t rows, int64_t cols, int fmt,
                                    uint8_t *out_row, uint8_t *out_col, float *scale,
                                    float *scale_inv, float *hist, int hist_len, int64_t step,
                                    float *partials, cudaStream_t st);

// Fused GELU (bwd = 0: A = GELU(H), E4M3) or GELU backward (bwd = 1:
// dH = H * GELU'(H2) with H = dA, E5M2) with the 1x128 quantizer.
cudaError_t launch_gelu_quantize(const void *H, const void *H2, int64_t rows, int64_t cols,
                                 int bwd, uint8_t *out_row, uint8_t *out_col, float *row_scale,
                                 float *row_scale_inv, float *col_scale, float *col_scale_inv,
                                 cudaStream_t st);

// TMA descriptor of a bf16 [rows, cols] row-major tensor (row stride cols,
// 16-byte aligned base) for box_rows x box_cols boxes, no swizzle, zeros read
// outside the tensor.
bool make_bf16_tile_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows,
                        int box_cols);
// Reads and clears the quantizer kernels' device status word (0 = ok).
cudaError_t quant_read_status(unsigned *status);

// FP8 GEMM (tcgen05).  scaling: fp8_scaling.  ws may be null when
// gemm_workspace_bytes() is 0.
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int scaling);
cudaError_t launch_gemm(const uint8_t *A, int a_fmt, const float *a_sinv, const uint8_t *B,
                        int b_fmt, const float *b_sinv, int64_t M, int64_t N, int64_t K,
                        int scaling, void *C, void *ws, cudaStream_t st);
// Launches the bounded-wait probe (a wait nobody satisfies; limit_ns <= 1 s).
cudaError_t launch_wait_timeout_probe(uint64_t limit_ns, cudaStream_t st);
// Reads and clears the GEMM kernels' device status word (0 = ok).
cudaError_t gemm_read_status(unsigned *status, cudaStream_t st);

cudaError_t launch_gelu_fwd(const void *H, void *A, int64_t n, cudaStream_t st);
cudaError_t launch_gelu_bwd(const void *dA, const void *H, void *dH, int64_t n, cudaStream_t st);
cudaError_t launch_grad_accumulate(float *acc, const void *dW, int64_t n, cudaStream_t st);

}  // namespace fp8lin
