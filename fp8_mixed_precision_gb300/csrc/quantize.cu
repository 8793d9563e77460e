// Fused FP8 quantizers: amax -> fp32 scale -> saturating RNE cast, writing the
// row-major and the transposed FP8 layout in one pass over a 128x128 tile.
//
// "Native FP8 MLP reconstruction", implementation paragraph: current
// tensorwise amax, E4M3 for inputs and weights, E5M2 for incoming gradients,
// one fused cast emitting the ordinary and the transposed layout.  Block
// recipe (Float8BlockScaling reading, TransformerEngine issue #2852 opening
// post: blockwise, no amax history): 1x128 blocks for activations and
// gradients, 128x128 tiles for weights.
//
// Work decomposition (all modes): one CTA of 256 threads owns a 128x128 tile.
//   phase 1  thread t holds 16 consecutive columns (cg = t & 7) of 4 rows
//            (rr = t >> 3, rows rr + 32 i): two 16-byte loads per row, the
//            bf16 kept packed in registers.  Scales are formed, the rowwise
//            bytes are stored with one 16-byte store per row (8 lanes = one
//            128-byte row segment), and the bytes meant for the transposed
//            layout go to a swizzled 16 KB shared-memory tile.
//   phase 2  thread t reads a 16-row x 4-column byte block (16 conflict-free
//            32-bit shared loads), transposes it in registers with byte
//            permutes and writes 4 transposed rows of 16 bytes (8 lanes = one
//            128-byte segment of a transposed row).
// Ragged tails: the last tile may have fewer rows/columns (multiples of 16);
// absent elements are zeros for the amax and are never stored.
#include "common.cuh"
#include "internal.h"

namespace fp8lin {

enum QMode { Q_TENSOR = 0, Q_BLOCK1x128 = 1, Q_BLOCK128 = 2 };

constexpr int kQThreads = 256;
constexpr int kAmaxThreads = 512;

// Word w (4 bytes = 4 columns) of tile row r lives at word index
// r*32 + (w ^ swz(r)); swz keeps 4-word groups contiguous and makes the
// phase-2 column reads hit 32 distinct banks.
__device__ __forceinline__ int swz(int r) { return ((r >> 4) & 7) << 2; }

// ---------------------------------------------------------------------------
// Tensorwise pass 1: per-CTA max |x| over a grid-stride sweep (NaN ignored).
// bf16 magnitudes order like unsigned integers, so the sweep works on the
// packed bit patterns with SIMD 16-bit max.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kAmaxThreads) amax_partials_kernel(const uint4 *__restrict__ x,
                                                                     int64_t n16,
                                                                     float *__restrict__ partials) {
  uint32_t m = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  auto fold = [&](uint4 v) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t a = w[k] & 0x7FFF7FFFu;
      a &= ~__vcmpgtu2(a, 0x7F807F80u);  // NaN halves -> 0
      m = __vmaxu2(m, a);
    }
  };
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 v0 = __ldcs(x + i), v1 = __ldcs(x + i + stride), v2 = __ldcs(x + i + 2 * stride),
          v3 = __ldcs(x + i + 3 * stride);
    fold(v0); fold(v1); fold(v2); fold(v3);
  }
  for (; i < n16; i += stride) fold(__ldcs(x + i));
  uint32_t bits = max(m & 0xFFFFu, m >> 16) << 16;  // as fp32 bit pattern
#pragma unroll
  for (int o = 16; o; o >>= 1) bits = max(bits, __shfl_xor_sync(0xffffffffu, bits, o));
  __shared__ uint32_t red[kAmaxThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = bits;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
    for (int k = 0; k < kAmaxThreads / 32; ++k) b = max(b, red[k]);
    partials[blockIdx.x] = __uint_as_float(b);
  }
}

// ---------------------------------------------------------------------------
// Fused cast, one 128x128 tile per loop iteration (persistent grid).
// ---------------------------------------------------------------------------
struct QParams {
  const uint16_t *x;
  int64_t R, C;
  uint8_t *out_row;  // [R, C] or null
  uint8_t *out_col;  // [C, R] or null
  float *row_scale, *row_scale_inv;
  float *col_scale, *col_scale_inv;
  const float *partials;  // tensorwise: per-CTA amax of pass 1
  int n_partials;
};

// A product x * scale can only be NaN when x is inf or NaN (scale is finite
// and non-negative; inf * 0 needs an infinite x), so a row slot whose 16
// inputs are all finite converts without the NaN fix-up.
template <int FMT>
__device__ __forceinline__ uint4 cast16(const float (&v)[16], bool special) {
  uint4 q;
  if (!special) {
    q.x = cvt4_finite<FMT>(v[0], v[1], v[2], v[3]);
    q.y = cvt4_finite<FMT>(v[4], v[5], v[6], v[7]);
    q.z = cvt4_finite<FMT>(v[8], v[9], v[10], v[11]);
    q.w = cvt4_finite<FMT>(v[12], v[13], v[14], v[15]);
  } else {
    q.x = cvt4<FMT>(v[0], v[1], v[2], v[3]);
    q.y = cvt4<FMT>(v[4], v[5], v[6], v[7]);
    q.z = cvt4<FMT>(v[8], v[9], v[10], v[11]);
    q.w = cvt4<FMT>(v[12], v[13], v[14], v[15]);
  }
  return q;
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(kQThreads, MODE == 0 ? 4 : 2) quant_tile_kernel(QParams p) {
  __shared__ __align__(16) uint32_t tile[128 * 32];   // FP8 bytes for the transposed layout
  __shared__ float colred[8][128];                     // 1x128: per-warp column maxima
  __shared__ __align__(16) float colsc[128];           // 1x128: column scales
  __shared__ float red8[8];
  __shared__ float tscale[2];

  const float fmax = (FMT == FP8_FORMAT_E4M3) ? kE4M3Max : kE5M2Max;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int cg = t & 7, rr = t >> 3;
  const int64_t tiles_r = (p.R + 127) / 128, tiles_c = (p.C + 127) / 128;
  const int64_t ntiles = tiles_r * tiles_c;

  float ts = 1.0f, tsi = 1.0f;
  if (MODE == Q_TENSOR) {
    float a = 0.0f;
    for (int k = t; k < p.n_partials; k += kQThreads) a = fmaxf(a, p.partials[k]);
#pragma unroll
    for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) red8[warp] = a;
    __syncthreads();
    if (t == 0) {
      float m = 0.0f;
      for (int k = 0; k < 8; ++k) m = fmaxf(m, red8[k]);
      float s, si;
      scale_from_amax(m, fmax, s, si);
      tscale[0] = s;
      tscale[1] = si;
      if (blockIdx.x == 0) {
        if (p.row_scale) { p.row_scale[0] = s; p.row_scale_inv[0] = si; }
        if (p.col_scale) { p.col_scale[0] = s; p.col_scale_inv[0] = si; }
      }
    }
    __syncthreads();
    ts = tscale[0];
    tsi = tscale[1];
  }
  (void)tsi;

  for (int64_t tile_id = blockIdx.x; tile_id < ntiles; tile_id += gridDim.x) {
    const int64_t tr = tile_id / tiles_c, tc = tile_id % tiles_c;
    const int64_t r0 = tr * 128, c0 = tc * 128;
    const int rows_here = (int)(p.R - r0 < 128 ? p.R - r0 : 128);
    const int cols_here = (int)(p.C - c0 < 128 ? p.C - c0 : 128);
    const bool col_ok = 16 * cg < cols_here;

    // ---- load 4 rows x 16 columns, packed bf16
    uint4 raw[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = rr + 32 * i;
      if (col_ok && r < rows_here) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (r0 + r) * p.C + c0 + 16 * cg);
        raw[i][0] = __ldcs(src);
        raw[i][1] = __ldcs(src + 1);
      } else {
        raw[i][0] = make_uint4(0, 0, 0, 0);
        raw[i][1] = make_uint4(0, 0, 0, 0);
      }
    }
    auto val = [&](int i, int j) -> float {  // element j (0..15) of row slot i
      const uint4 &q = raw[i][j >> 3];
      const uint32_t w = ((j & 7) < 2) ? q.x : ((j & 7) < 4) ? q.y : ((j & 7) < 6) ? q.z : q.w;
      return (j & 1) ? bf16hi(w) : bf16lo(w);
    };

    // ---- scales
    float rs[4], rsi[4];
    if (MODE == Q_TENSOR) {
#pragma unroll
      for (int i = 0; i < 4; ++i) { rs[i] = ts; rsi[i] = tsi; }
    } else if (MODE == Q_BLOCK128) {
      float a = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 16; ++j) a = amax_acc(a, val(i, j));
#pragma unroll
      for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      if (lane == 0) red8[warp] = a;
      __syncthreads();
      float m = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) m = fmaxf(m, red8[k]);
      float s, si;
      scale_from_amax(m, fmax, s, si);
#pragma unroll
      for (int i = 0; i < 4; ++i) { rs[i] = s; rsi[i] = si; }
      if (t == 0) {
        if (p.row_scale) {
          p.row_scale[tr * tiles_c + tc] = s;
          p.row_scale_inv[tr * tiles_c + tc] = si;
        }
        if (p.col_scale) {
          p.col_scale[tc * tiles_r + tr] = s;
          p.col_scale_inv[tc * tiles_r + tr] = si;
        }
      }
    } else {  // Q_BLOCK1x128
      // row blocks: the 128 columns of a row are spread over the 8 lanes of one cg group
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j) a = amax_acc(a, val(i, j));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        scale_from_amax(a, fmax, rs[i], rsi[i]);
        const int r = rr + 32 * i;
        if (cg == 0 && r < rows_here && p.out_row) {
          p.row_scale[(r0 + r) * tiles_c + tc] = rs[i];
          p.row_scale_inv[(r0 + r) * tiles_c + tc] = rsi[i];
        }
      }
      if (p.out_col) {
        // column blocks: 4 rows per thread, 4 row groups per warp (lane bits 3,4), 8 warps
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float a = 0.0f;
#pragma unroll
          for (int i = 0; i < 4; ++i) a = amax_acc(a, val(i, j));
          a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
          a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
          if (lane < 8) colred[warp][16 * cg + j] = a;
        }
        __syncthreads();
        if (t < 128) {
          float m = 0.0f;
#pragma unroll
          for (int k = 0; k < 8; ++k) m = fmaxf(m, colred[k][t]);
          float s, si;
          scale_from_amax(m, fmax, s, si);
          colsc[t] = s;
          if (t < cols_here) {
            p.col_scale[(c0 + t) * tiles_r + tr] = s;
            p.col_scale_inv[(c0 + t) * tiles_r + tr] = si;
          }
        }
        __syncthreads();
      }
    }

    // ---- cast: rowwise bytes (and, for one-scale tiles, the transposed source)
    float cs[16];
    if (MODE == Q_BLOCK1x128 && p.out_col) {
      const float4 *c4 = reinterpret_cast<const float4 *>(colsc + 16 * cg);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 f = c4[k];
        cs[4 * k] = f.x; cs[4 * k + 1] = f.y; cs[4 * k + 2] = f.z; cs[4 * k + 3] = f.w;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = rr + 32 * i;
      const bool special = any_nonfinite_bf16(raw[i][0], raw[i][1]);
      const bool need_row = p.out_row || (MODE != Q_BLOCK1x128 && p.out_col);
      if (need_row) {
        const float s = rs[i];
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(val(i, j), s);
        const uint4 q = cast16<FMT>(v, special);
        if (p.out_row && col_ok && r < rows_here)
          *reinterpret_cast<uint4 *>(p.out_row + (r0 + r) * p.C + c0 + 16 * cg) = q;
        if (MODE != Q_BLOCK1x128 && p.out_col)
          *reinterpret_cast<uint4 *>(&tile[r * 32 + ((4 * cg) ^ swz(r))]) = q;
      }
      if (MODE == Q_BLOCK1x128 && p.out_col) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(val(i, j), cs[j]);
        *reinterpret_cast<uint4 *>(&tile[r * 32 + ((4 * cg) ^ swz(r))]) = cast16<FMT>(v, special);
      }
    }

    // ---- transposed layout
    if (p.out_col) {
      __syncthreads();
      const int seg = t & 7, w = t >> 3;  // rows seg*16..+15, columns 4w..4w+3
      if (4 * w < cols_here && 16 * seg < rows_here) {
        uint32_t a[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = seg * 16 + i;
          a[i] = tile[r * 32 + (w ^ swz(r))];
        }
        uint32_t o[4][4];  // o[jj][g]: transposed row 4w+jj, word g (rows 4g..4g+3 of the segment)
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint32_t t0 = __byte_perm(a[4 * g + 0], a[4 * g + 1], 0x5140);
          const uint32_t t1 = __byte_perm(a[4 * g + 0], a[4 * g + 1], 0x7362);
          const uint32_t t2 = __byte_perm(a[4 * g + 2], a[4 * g + 3], 0x5140);
          const uint32_t t3 = __byte_perm(a[4 * g + 2], a[4 * g + 3], 0x7362);
          o[0][g] = __byte_perm(t0, t2, 0x5410);
          o[1][g] = __byte_perm(t0, t2, 0x7632);
          o[2][g] = __byte_perm(t1, t3, 0x5410);
          o[3][g] = __byte_perm(t1, t3, 0x7632);
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          *reinterpret_cast<uint4 *>(p.out_col + (c0 + 4 * w + jj) * p.R + r0 + 16 * seg) =
              make_uint4(o[jj][0], o[jj][1], o[jj][2], o[jj][3]);
      }
    }
    __syncthreads();  // tile / colred / colsc reused by the next iteration
  }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

int tensorwise_partials_count(int64_t rows, int64_t cols) {
  const int64_t n16 = rows * cols / 8;
  const int64_t want = (n16 + (int64_t)kAmaxThreads * 4 - 1) / ((int64_t)kAmaxThreads * 4);
  const int64_t cap = std::min<int64_t>(2 * (int64_t)num_sms(), kMaxPartials);
  return (int)std::max<int64_t>(1, std::min<int64_t>(want, cap));
}

template <int MODE, int FMT>
static cudaError_t launch_tile(const QParams &p, cudaStream_t st) {
  static const char *names[3] = {"quant_cast_tensorwise", "quant_block_1x128", "quant_block_128x128"};
  const int64_t tr = (p.R + 127) / 128, tc = (p.C + 127) / 128;
  const int64_t ntiles = tr * tc;
  const int64_t grid = std::min<int64_t>(ntiles, (int64_t)num_sms() * 8);
  // algorithmic bytes: bf16 read + one byte per written layout + scale arrays
  double bytes = 2.0 * p.R * p.C + (p.out_row ? 1.0 * p.R * p.C : 0.0) +
                 (p.out_col ? 1.0 * p.R * p.C : 0.0);
  if (MODE == Q_BLOCK1x128)
    bytes += (p.out_row ? 8.0 * p.R * tc : 0.0) + (p.out_col ? 8.0 * p.C * tr : 0.0);
  else if (MODE == Q_BLOCK128)
    bytes += 16.0 * ntiles;
  else
    bytes += 16.0;
  LaunchScope ls(names[MODE], st, bytes, 0.0);
  quant_tile_kernel<MODE, FMT><<<(unsigned)grid, kQThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const void *x, int64_t rows, int64_t cols, int mode, int fmt,
                            uint8_t *out_row, uint8_t *out_col, float *row_scale,
                            float *row_scale_inv, float *col_scale, float *col_scale_inv,
                            float *partials, cudaStream_t st) {
  QParams p;
  p.x = static_cast<const uint16_t *>(x);
  p.R = rows;
  p.C = cols;
  p.out_row = out_row;
  p.out_col = out_col;
  p.row_scale = row_scale;
  p.row_scale_inv = row_scale_inv;
  p.col_scale = col_scale;
  p.col_scale_inv = col_scale_inv;
  p.partials = partials;
  p.n_partials = 0;
  if (mode == Q_TENSOR) {
    const int g = tensorwise_partials_count(rows, cols);
    {
      LaunchScope ls("quant_amax_tensorwise", st, 2.0 * rows * cols, 0.0);
      amax_partials_kernel<<<g, kAmaxThreads, 0, st>>>(static_cast<const uint4 *>(x),
                                                       rows * cols / 8, partials);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.n_partials = g;
    return fmt == FP8_FORMAT_E4M3 ? launch_tile<Q_TENSOR, FP8_FORMAT_E4M3>(p, st)
                                  : launch_tile<Q_TENSOR, FP8_FORMAT_E5M2>(p, st);
  }
  if (mode == Q_BLOCK1x128)
    return fmt == FP8_FORMAT_E4M3 ? launch_tile<Q_BLOCK1x128, FP8_FORMAT_E4M3>(p, st)
                                  : launch_tile<Q_BLOCK1x128, FP8_FORMAT_E5M2>(p, st);
  return fmt == FP8_FORMAT_E4M3 ? launch_tile<Q_BLOCK128, FP8_FORMAT_E4M3>(p, st)
                                : launch_tile<Q_BLOCK128, FP8_FORMAT_E5M2>(p, st);
}

}  // namespace fp8lin
