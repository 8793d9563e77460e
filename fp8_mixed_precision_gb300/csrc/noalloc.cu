// Allocation-free variant of the tensorwise quantizer.
//
// Tensorwise quantization needs scratch memory between its two passes: one
// fp32 partial amax per CTA of the first pass, read back by the cast pass.
// fp8_quantize takes that scratch from a caller-supplied workspace.  Some
// callers cannot allocate one: code running inside a custom device allocator
// or memory-pool hook (allocating again would re-enter the allocator),
// latency-critical paths that must not pay for cudaMalloc/cudaFree (which can
// synchronise the whole device), and plugins whose host framework owns all
// device memory and hands them only their inputs and outputs.  For them,
// fp8_quantize_tensorwise_noalloc keeps the scratch in a fixed device array
// that is part of this library: every GPU that loads the library holds it
// (kNoAllocPartials floats, 4 KiB) until the process exits.
#include "common.cuh"
#include "internal.h"

namespace fp8lin {
namespace {

constexpr int kNoAllocPartials = kMaxPartials;  // 1024 fp32 partial maxima

// Shared by every call of fp8_quantize_tensorwise_noalloc on a device.  The
// first pass overwrites exactly the slots the second pass reads, so nothing
// has to be cleared between calls; calls whose work overlaps on the GPU
// (different streams without ordering) race on it.
static __device__ __align__(256) float g_noalloc_partials[kNoAllocPartials];

// Device address of the array in the current device's context.  Host code
// must not use the symbol itself (that is a host-side stand-in).  The address
// is looked up on every call, with the caller's device current: a context
// that was torn down and created again (cudaDeviceReset, a released primary
// context) loads the module anew and may place the array elsewhere, so a
// remembered address could be stale.  The first call on a device also loads
// the module there.
cudaError_t partials_for_current_device(float **out) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_partials);
  if (e != cudaSuccess) return e;
  *out = static_cast<float *>(p);
  return cudaSuccess;
}

}  // namespace
}  // namespace fp8lin

using namespace fp8lin;

extern "C" fp8_status fp8_quantize_tensorwise_noalloc(const void *x, int64_t rows, int64_t cols,
                                                      fp8_role role, uint8_t *rowwise_out,
                                                      uint8_t *colwise_out, float *scale,
                                                      float *scale_inv, fp8_stream_t stream) {
  if (role < FP8_ROLE_ACT || role > FP8_ROLE_GRAD) return FP8_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0) return FP8_ERR_INVALID_ARG;
  if (rows % 16 || cols % 16) return FP8_ERR_SHAPE;
  if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31)) return FP8_ERR_SHAPE;
  if (!rowwise_out && !colwise_out) return FP8_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (!x || !scale || !scale_inv) return FP8_ERR_INVALID_ARG;
  auto mis = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
  if (mis(x) || (rowwise_out && mis(rowwise_out)) || (colwise_out && mis(colwise_out)))
    return FP8_ERR_ALIGN;
  // The first pass uses one partial per CTA; refuse a launch that would need
  // more slots than the fixed array holds.
  if (tensorwise_partials_count(rows, cols) > kNoAllocPartials) return FP8_ERR_WORKSPACE;
  float *partials = nullptr;
  if (partials_for_current_device(&partials) != cudaSuccess) return FP8_ERR_CUDA;
  const int fmt = role == FP8_ROLE_GRAD ? FP8_FORMAT_E5M2 : FP8_FORMAT_E4M3;
  const cudaError_t e =
      launch_quantize(x, rows, cols, /*mode tensorwise*/ 0, fmt, rowwise_out, colwise_out, scale,
                      scale_inv, nullptr, nullptr, partials, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}
