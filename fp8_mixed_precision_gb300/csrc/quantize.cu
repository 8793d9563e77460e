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
// Work decomposition (all modes): persistent CTAs of 256 threads, one 128x128
// bf16 tile per loop iteration, staged in shared memory by one TMA tensor
// load per tile into two buffers (completion on an mbarrier per buffer), so
// the next tile's load overlaps the current tile's work.
// Thread t owns 8 consecutive columns (cg = t & 15) of 8 rows (rr = t >> 4,
// rows rr + 16 i): 16 lanes cover one 256-byte row, so every shared read is
// conflict-free and every rowwise store is a contiguous 128-byte segment.
//   maxima    one pass over the registers (128x128: the tile maximum with
//             the NaN-ignoring packed bf16 max; 1x128: row maxima over the 16
//             lanes of a row and column maxima over the CTA, as unsigned
//             16-bit maxima of the magnitude bits, which also flag inf/NaN;
//             a tile holding one redoes them with the bf16 max), then one
//             IEEE division per thread forms the 128 row scales and the 128
//             column scales (tensorwise: the scale comes from the first
//             pass's partial maxima)
//   cast      packed fp32 multiplies, saturating RNE conversion; the rowwise
//             bytes are stored, the bytes of the transposed layout go to a
//             swizzled 16 KB tile
//   transpose thread t reads a 16-row x 4-column byte block (conflict-free
//             32-bit shared loads), transposes it with byte permutes and writes
//             4 transposed rows of 16 bytes (8 lanes = one 128-byte segment)
// Fused producers (1x128 only): PRE = 1 applies GELU, PRE = 2 forms
// dA * GELU'(H), to the thread's register tile right after its shared read,
// rounding to bf16 there, so the quantizer sees exactly the bf16 tensor the
// unfused GELU kernels would write.  PRE = 2 loads dA and H into the two
// buffers together and refills both with the next tile as soon as every
// thread holds its elements (after the maxima).
// Ragged tails: the last tile may have fewer rows/columns (multiples of 16);
// absent elements are zero-filled by the TMA load (zeros never raise an amax)
// and never stored.  Every wait on a tile is bounded: on expiry the kernel
// records FP8_ERR_TIMEOUT in its status word and carries on (no trap).
#include <cstdlib>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8lin {

enum QMode { Q_TENSOR = 0, Q_BLOCK1x128 = 1, Q_BLOCK128 = 2 };

constexpr int kQThreads = 256;
constexpr int kAmaxThreads = 512;

// Word w (4 bytes = 4 columns) of tile row r lives at word index
// r*32 + (w ^ swz(r)); swz keeps 4-word groups contiguous and makes the
// transpose reads hit 32 distinct banks.
__device__ __forceinline__ int swz(int r) { return ((r >> 4) & 7) << 2; }

// ---------------------------------------------------------------------------
// Tensorwise pass 1: per-CTA max |x| over a grid-stride sweep, first to last
// (NaN ignored).
// bf16 magnitudes order like unsigned integers, so the sweep works on the
// packed bit patterns with SIMD 16-bit max.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kAmaxThreads) amax_partials_kernel(const uint4 *__restrict__ x,
                                                                     int64_t n16,
                                                                     float *__restrict__ partials) {
  pdl_wait_then_release();
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
// Fused cast, one 128x128 tile per loop iteration (persistent grid).  Tiles
// are visited last to first: the amax pass sweeps the tensor first to last,
// so the cast starts on the rows still in L2, and it finishes on the first
// rows, which the GEMM that consumes its output reads first.
// ---------------------------------------------------------------------------
struct QParams {
  const uint16_t *x;
  const uint16_t *x2;  // fused GELU backward: H (x holds dA)
  int64_t R, C;
  uint8_t *out_row;  // [R, C] or null
  uint8_t *out_col;  // [C, R] or null
  float *row_scale, *row_scale_inv;
  float *col_scale, *col_scale_inv;
  const float *partials;  // tensorwise: per-CTA amax of pass 1
  int n_partials;
  const float *hist;      // delayed: amax history ring (scale source) or null
  int hist_len;
  float *cur_partials;    // delayed: per-CTA amax of this tensor, written by the cast pass
};

struct __align__(128) QSmem {
  uint16_t in[2][128 * 128];  // bf16 tiles, 256 bytes per row (TMA destinations)
  uint32_t tile[128 * 32];    // FP8 bytes for the transposed layout (swizzled words)
  float colred[8][128];       // 1x128: per-warp column maxima
  float colsc[128];           // 1x128: column scales
  float rowmx[128];           // 1x128: row maxima
  float rowsc[128];           // 1x128: row scales
  float red[8];
  float tscale[2];
  uint64_t full[2];           // TMA completion, one per tile buffer
};
constexpr size_t kQSmemBytes = sizeof(QSmem);

__device__ unsigned g_quant_status;
constexpr uint64_t kQWaitLimitNs = 2000000000ull;  // 2 s

// Bounded wait for phase `parity` of a tile buffer's barrier.  On expiry the
// status word records FP8_ERR_TIMEOUT and the caller proceeds (its results
// are then invalid and the status reports it; nothing hangs or traps).
__device__ __forceinline__ void wait_tile(uint64_t *bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return;
    if ((it & 63) == 0 && ptx::globaltimer() - t0 > kQWaitLimitNs) {
      atomicCAS(&g_quant_status, 0u, (unsigned)FP8_ERR_TIMEOUT);
      return;
    }
  }
}

// Eight fp32 values -> eight FP8 bytes (two little-endian words).  A product
// x * scale can only be NaN when x is inf or NaN (scale is finite and
// non-negative), so `special` (some input non-finite) selects the NaN fix-up.
template <int FMT>
__device__ __forceinline__ uint2 cast8(const float (&v)[8], bool special) {
  uint2 q;
  if (!special) {
    q.x = cvt4_finite<FMT>(v[0], v[1], v[2], v[3]);
    q.y = cvt4_finite<FMT>(v[4], v[5], v[6], v[7]);
  } else {
    q.x = cvt4<FMT>(v[0], v[1], v[2], v[3]);
    q.y = cvt4<FMT>(v[4], v[5], v[6], v[7]);
  }
  return q;
}

// True if any of the 64 bf16 values is inf or NaN: a NaN-propagating packed
// max of the magnitudes reaches the all-ones exponent exactly then.
__device__ __forceinline__ bool any_nonfinite64(const uint4 (&w)[8]) {
  __nv_bfloat162 m = __float2bfloat162_rn(0.0f);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t q[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      m = __hmax2_nan(m, __habs2(*reinterpret_cast<const __nv_bfloat162 *>(&q[j])));
  }
  const uint32_t b = *reinterpret_cast<uint32_t *>(&m);
  return (b & 0x7F80u) == 0x7F80u || (b & 0x7F800000u) == 0x7F800000u;
}

// max(acc, |w|) on packed bf16 pairs; NaN lanes of w are ignored (max.bf16x2
// returns the non-NaN operand).
__device__ __forceinline__ uint32_t absmax2(uint32_t acc, uint32_t w) {
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&acc);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&w);
  __nv_bfloat162 r = __hmax2(a, __habs2(b));
  return *reinterpret_cast<uint32_t *>(&r);
}
// Larger of the two non-negative bf16 halves, as an fp32 value.
__device__ __forceinline__ float bf16pair_max(uint32_t w) {
  return __uint_as_float(max(w & 0xFFFFu, w >> 16) << 16);
}

// Packed fp32 pair multiply (two IEEE round-to-nearest products).
__device__ __forceinline__ void mul2(float a0, float a1, float s0, float s1, float &r0, float &r1) {
  uint64_t a, s, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(s) : "f"(s0), "f"(s1));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(s));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r0), "=f"(r1) : "l"(r));
}

__device__ __forceinline__ void unpack8(uint4 w, float (&v)[8]) {
  v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
  v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
}

// PRE selects a producer fused in front of the quantizer, applied by each
// thread to its own register tile of the staged input and rounded to bf16
// exactly as the standalone kernels round (so fused and unfused results are
// bitwise equal):
//   0  none
//   1  A = bf16(GELU(x))                 (activation of the next linear)
//   2  dH = bf16(x * GELU'(x2)), x = dA  (gradient entering the linear below)
template <int MODE, int FMT, int PRE = 0>
__global__ void __launch_bounds__(kQThreads, 2)
    quant_tile_kernel(const __grid_constant__ CUtensorMap tmx,
                      const __grid_constant__ CUtensorMap tmx2, QParams p) {
  static_assert(PRE == 0 || MODE == Q_BLOCK1x128, "fused producers use 1x128 blocks");
  extern __shared__ __align__(1024) uint8_t q_smem_raw[];
  QSmem &S = *reinterpret_cast<QSmem *>(q_smem_raw);

  const float fmax = (FMT == FP8_FORMAT_E4M3) ? kE4M3Max : kE5M2Max;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int cg = t & 15, rr = t >> 4;
  const int64_t tiles_r = (p.R + 127) / 128, tiles_c = (p.C + 127) / 128;
  const int64_t ntiles = tiles_r * tiles_c;

  if (t == 0) {
    ptx::mbar_init(&S.full[0], 1);
    ptx::mbar_init(&S.full[1], 1);
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tmx);
    if (PRE == 2) ptx::tma_prefetch_desc(&tmx2);
  }
  __syncthreads();
  pdl_wait_then_release();
  // Thread 0 loads tile `id` into buffer b with one TMA tensor load (two for
  // the fused GELU backward: dA into buffer 0, H into buffer 1, both on
  // barrier 0); parts of the box outside the tensor arrive as zeros.
  auto prefetch = [&](int64_t id, int b) {
    if (t != 0 || id >= ntiles) return;
    const int64_t tr = (ntiles - 1 - id) / tiles_c, tc = (ntiles - 1 - id) % tiles_c;
    ptx::fence_proxy_async_smem();  // earlier generic writes to the buffer come first
    if (PRE == 2) {
      ptx::mbar_arrive_expect_tx(&S.full[0], 2u * 128 * 128 * 2);
      ptx::tma_load_2d(S.in[0], &tmx, &S.full[0], (int)(tc * 128), (int)(tr * 128));
      ptx::tma_load_2d(S.in[1], &tmx2, &S.full[0], (int)(tc * 128), (int)(tr * 128));
    } else {
      ptx::mbar_arrive_expect_tx(&S.full[b], 128u * 128 * 2);
      ptx::tma_load_2d(S.in[b], &tmx, &S.full[b], (int)(tc * 128), (int)(tr * 128));
    }
  };

  // the first tiles do not depend on the scale: request them now
  int64_t id = blockIdx.x;
  prefetch(id, 0);
  if (PRE != 2) prefetch(id + gridDim.x, 1);

  float ts = 1.0f, tsi = 1.0f;
  if (MODE == Q_TENSOR) {
    float a = 0.0f;
    if (p.hist) {  // delayed scaling: the history's maximum, before this tensor
      for (int k = t; k < p.hist_len; k += kQThreads) a = fmaxf(a, p.hist[k]);
    } else {
      for (int k = t; k < p.n_partials; k += kQThreads) a = fmaxf(a, p.partials[k]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) S.red[warp] = a;
    __syncthreads();
    if (t == 0) {
      float m = 0.0f;
      for (int k = 0; k < 8; ++k) m = fmaxf(m, S.red[k]);
      float s, si;
      scale_from_amax(m, fmax, s, si);
      S.tscale[0] = s;
      S.tscale[1] = si;
      if (blockIdx.x == 0) {
        if (p.row_scale) { p.row_scale[0] = s; p.row_scale_inv[0] = si; }
        if (p.col_scale) { p.col_scale[0] = s; p.col_scale_inv[0] = si; }
      }
    }
    __syncthreads();
    ts = S.tscale[0];
    tsi = S.tscale[1];
  }
  (void)tsi;

  const bool want_row = p.out_row != nullptr;
  const bool want_col = p.out_col != nullptr;
  uint32_t cur_max = 0;  // delayed: running |max| of this CTA's tiles (bf16 pair)
  for (int k = 0; id < ntiles; ++k, id += gridDim.x) {
    const int b = PRE == 2 ? 0 : (k & 1);
    uint16_t *in = S.in[b];
    const int64_t tr = (ntiles - 1 - id) / tiles_c, tc = (ntiles - 1 - id) % tiles_c;
    const int64_t r0 = tr * 128, c0 = tc * 128;
    const int rows_here = (int)(p.R - r0 < 128 ? p.R - r0 : 128);
    const int cols_here = (int)(p.C - c0 < 128 ? p.C - c0 : 128);
    const bool col_ok = 8 * cg < cols_here;
    // this tile is in shared memory (fused GELU backward: dA and H, loaded
    // once the previous tile was in registers)
    if (PRE == 2)
      wait_tile(&S.full[0], k & 1);
    else
      wait_tile(&S.full[b], (k >> 1) & 1);
    // every thread has finished the previous tile's transpose reads of S.tile
    // before this tile's cast writes it
    __syncthreads();
    // this thread's 8 rows x 8 columns of the tile, read from shared memory
    // once and kept in registers for the maxima and the cast
    uint4 xw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) xw[i] = *reinterpret_cast<const uint4 *>(&in[(rr + 16 * i) * 128 + 8 * cg]);
    if (PRE != 0) {  // fused producer on the thread's own elements, rounded to bf16
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t wi[4] = {xw[i].x, xw[i].y, xw[i].z, xw[i].w};
        uint32_t o4[4];
        if (PRE == 1) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float g0, g1;
            gelu_f2(bf16lo(wi[j]), bf16hi(wi[j]), g0, g1);
            o4[j] = pack_bf16x2(g0, g1);
          }
        } else {
          const uint4 hw = *reinterpret_cast<const uint4 *>(&S.in[1][(rr + 16 * i) * 128 + 8 * cg]);
          const uint32_t hi4[4] = {hw.x, hw.y, hw.z, hw.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float g0, g1;
            gelu_grad_f2(bf16lo(hi4[j]), bf16hi(hi4[j]), g0, g1);
            o4[j] = pack_bf16x2(__fmul_rn(bf16lo(wi[j]), g0), __fmul_rn(bf16hi(wi[j]), g1));
          }
        }
        xw[i] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
    }
    // any inf or NaN among these 64 values selects the cast's NaN fix-up
    // (1x128: found by the maxima pass)
    bool special = MODE == Q_BLOCK1x128 ? false : any_nonfinite64(xw);

    // ---- maxima: one pass over the tile
    float s_tile = ts;
    if (MODE == Q_BLOCK1x128) {
      uint32_t cm[4];  // column maxima of this thread's 8 columns (bf16 pairs)
      // rows rr+16i and rr+16(i+1): each row's maximum over this thread's 8
      // columns, the two packed as one bf16 pair, reduced over the 16 lanes
      // of the row group with 4 shuffles for both rows at once; then the two
      // row groups of the warp combine their column maxima, stored per warp.
      // EXACT: bf16 max that ignores NaN; otherwise unsigned 16-bit max of the
      // magnitude bits (finite bf16 magnitudes order like unsigned integers).
      auto maxima = [&](auto exact) {
        constexpr bool kExact = decltype(exact)::value;
        auto mx = [](uint32_t acc, uint32_t w) {
          return kExact ? absmax2(acc, w) : __vmaxu2(acc, w & 0x7FFF7FFFu);
        };
#pragma unroll
        for (int j = 0; j < 4; ++j) cm[j] = 0;
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          uint32_t rm[2];  // per row: two partial maxima (the halves of the pair)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 w = xw[i + h];
            cm[0] = mx(cm[0], w.x); cm[1] = mx(cm[1], w.y);
            cm[2] = mx(cm[2], w.z); cm[3] = mx(cm[3], w.w);
            if (kExact)  // max with 0 drops NaN lanes
              rm[h] = mx(mx(mx(mx(0u, w.x), w.y), w.z), w.w);
            else
              rm[h] = __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                               __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
          }
          // lo: row i, hi: row i+1 (the max of each row's two halves)
          uint32_t pr = mx(__byte_perm(rm[0], rm[1], 0x5410), __byte_perm(rm[0], rm[1], 0x7632));
#pragma unroll
          for (int o = 1; o < 16; o <<= 1) pr = mx(pr, __shfl_xor_sync(0xffffffffu, pr, o));
          if (cg == 0) {
            S.rowmx[rr + 16 * i] = __uint_as_float(pr << 16);
            S.rowmx[rr + 16 * (i + 1)] = __uint_as_float(pr & 0xFFFF0000u);
          }
        }
        // a magnitude >= 0x7F80 (inf or NaN) among this thread's 64 values
        if (!kExact)
          special = __vcmpgeu2(__vmaxu2(__vmaxu2(cm[0], cm[1]), __vmaxu2(cm[2], cm[3])),
                               0x7F807F80u) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) cm[j] = mx(cm[j], __shfl_xor_sync(0xffffffffu, cm[j], 16));
        if (lane < 16 && want_col) {
          float4 *dst = reinterpret_cast<float4 *>(&S.colred[warp][8 * cg]);
          dst[0] = make_float4(__uint_as_float(cm[0] << 16), __uint_as_float(cm[0] & 0xFFFF0000u),
                               __uint_as_float(cm[1] << 16), __uint_as_float(cm[1] & 0xFFFF0000u));
          dst[1] = make_float4(__uint_as_float(cm[2] << 16), __uint_as_float(cm[2] & 0xFFFF0000u),
                               __uint_as_float(cm[3] << 16), __uint_as_float(cm[3] & 0xFFFF0000u));
        }
      };
      maxima(std::false_type{});
      // NaN must not win a maximum: a tile holding inf or NaN anywhere redoes
      // the maxima with the NaN-ignoring bf16 max (each thread rewrites the
      // same shared entries it wrote above)
      if (__syncthreads_or(special)) {
        maxima(std::true_type{});
        __syncthreads();
      }
      // fused GELU backward: every thread holds its elements in registers,
      // so both buffers may take the next tile now (the single-input modes
      // keep a second buffer in flight and refill this one after the cast,
      // measured 1-3% faster than refilling it here)
      if (PRE == 2) prefetch(id + (int64_t)gridDim.x, 0);
      // one division per thread: row scale of row t, column scale of column t
      if (t < 128) {
        float s, si;
        scale_from_amax(S.rowmx[t], fmax, s, si);
        S.rowsc[t] = s;
        if (want_row && t < rows_here) {
          p.row_scale[(r0 + t) * tiles_c + tc] = s;
          p.row_scale_inv[(r0 + t) * tiles_c + tc] = si;
        }
      } else if (want_col) {
        const int c = t - 128;
        float m = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) m = fmaxf(m, S.colred[w][c]);
        float s, si;
        scale_from_amax(m, fmax, s, si);
        S.colsc[c] = s;
        if (c < cols_here) {
          p.col_scale[(c0 + c) * tiles_r + tr] = s;
          p.col_scale_inv[(c0 + c) * tiles_r + tr] = si;
        }
      }
      __syncthreads();
    } else if (MODE == Q_BLOCK128) {
      uint32_t tm = 0;  // running tile maximum (bf16 pair)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 w = xw[i];
        tm = absmax2(absmax2(absmax2(absmax2(tm, w.x), w.y), w.z), w.w);
      }
      float a = bf16pair_max(tm);
#pragma unroll
      for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      if (lane == 0) S.red[warp] = a;
      __syncthreads();
      float m = 0.0f;
#pragma unroll
      for (int w = 0; w < 8; ++w) m = fmaxf(m, S.red[w]);
      float si;
      scale_from_amax(m, fmax, s_tile, si);
      if (t == 0) {
        if (p.row_scale) {
          p.row_scale[tr * tiles_c + tc] = s_tile;
          p.row_scale_inv[tr * tiles_c + tc] = si;
        }
        if (p.col_scale) {
          p.col_scale[tc * tiles_r + tr] = s_tile;
          p.col_scale_inv[tc * tiles_r + tr] = si;
        }
      }
    }

    // ---- cast: rowwise bytes and the source of the transposed layout
    float cs[8];
    if (MODE == Q_BLOCK1x128 && want_col) {
      const float4 *c4 = reinterpret_cast<const float4 *>(&S.colsc[8 * cg]);
      const float4 f0 = c4[0], f1 = c4[1];
      cs[0] = f0.x; cs[1] = f0.y; cs[2] = f0.z; cs[3] = f0.w;
      cs[4] = f1.x; cs[5] = f1.y; cs[6] = f1.z; cs[7] = f1.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = rr + 16 * i;
      const uint4 w = xw[i];
      float v[8];
      unpack8(w, v);
      if (MODE == Q_TENSOR && p.cur_partials)
        cur_max = absmax2(absmax2(absmax2(absmax2(cur_max, w.x), w.y), w.z), w.w);
      const float s = MODE == Q_BLOCK1x128 ? S.rowsc[r] : s_tile;
      if (want_row || (MODE != Q_BLOCK1x128 && want_col)) {
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; j += 2) mul2(v[j], v[j + 1], s, s, y[j], y[j + 1]);
        const uint2 q = cast8<FMT>(y, special);
        if (want_row && col_ok && r < rows_here)
          *reinterpret_cast<uint2 *>(p.out_row + (r0 + r) * p.C + c0 + 8 * cg) = q;
        if (MODE != Q_BLOCK1x128 && want_col)
          *reinterpret_cast<uint2 *>(&S.tile[r * 32 + ((2 * cg) ^ swz(r))]) = q;
      }
      if (MODE == Q_BLOCK1x128 && want_col) {
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; j += 2) mul2(v[j], v[j + 1], cs[j], cs[j + 1], y[j], y[j + 1]);
        *reinterpret_cast<uint2 *>(&S.tile[r * 32 + ((2 * cg) ^ swz(r))]) = cast8<FMT>(y, special);
      }
    }
    __syncthreads();  // tile complete; the bf16 buffer is free again
    if (PRE != 2) prefetch(id + 2 * (int64_t)gridDim.x, b);

    // ---- transposed layout
    if (want_col) {
      const int seg = t & 7, w = t >> 3;  // rows seg*16..+15, columns 4w..4w+3
      if (4 * w < cols_here && 16 * seg < rows_here) {
        uint32_t a[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = seg * 16 + i;
          a[i] = S.tile[r * 32 + (w ^ swz(r))];
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
  }
  if (MODE == Q_TENSOR && p.cur_partials) {
    float a = bf16pair_max(cur_max);
#pragma unroll
    for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    __syncthreads();
    if (lane == 0) S.red[warp] = a;
    __syncthreads();
    if (t == 0) {
      float m = 0.0f;
      for (int w = 0; w < 8; ++w) m = fmaxf(m, S.red[w]);
      p.cur_partials[blockIdx.x] = m;
    }
  }
}

// Delayed scaling, after the cast pass: this tensor's amax (the maximum of
// the per-CTA partials) enters the history ring at position step mod len.
__global__ void delayed_history_update_kernel(const float *__restrict__ partials, int n,
                                              float *__restrict__ hist, int hist_len,
                                              int64_t step) {
  pdl_wait_then_release();
  __shared__ float red[8];
  float a = 0.0f;
  for (int k = threadIdx.x; k < n; k += blockDim.x) a = fmaxf(a, partials[k]);
#pragma unroll
  for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
    hist[step % hist_len] = m;
  }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
bool pdl_enabled() {
  static const bool on = [] {
    const char *e = getenv("FP8LIN_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

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

static int g_amax_bps[64];

int tensorwise_partials_count(int64_t rows, int64_t cols) {
  const int64_t n16 = rows * cols / 8;
  const int64_t want = (n16 + (int64_t)kAmaxThreads * 4 - 1) / ((int64_t)kAmaxThreads * 4);
  // every SM filled: as many blocks as fit on one, times the SMs
  const int64_t cap = std::min<int64_t>(
      (int64_t)blocks_per_sm(amax_partials_kernel, kAmaxThreads, g_amax_bps) * num_sms(), kMaxPartials);
  return (int)std::max<int64_t>(1, std::min<int64_t>(want, cap));
}

template <int MODE, int FMT, int PRE = 0>
static cudaError_t launch_tile(const QParams &p, cudaStream_t st) {
  CUtensorMap tmx, tmx2;
  if (!make_bf16_tile_map(&tmx, p.x, p.R, p.C, 128, 128)) return cudaErrorInvalidValue;
  if (PRE == 2) {
    if (!make_bf16_tile_map(&tmx2, p.x2, p.R, p.C, 128, 128)) return cudaErrorInvalidValue;
  } else {
    tmx2 = tmx;
  }
  static const char *names[3] = {"quant_cast_tensorwise", "quant_block_1x128", "quant_block_128x128"};
  static const char *pre_names[3] = {"", "gelu_quant_block_1x128", "gelu_bwd_quant_block_1x128"};
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(quant_tile_kernel<MODE, FMT, PRE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kQSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t tr = (p.R + 127) / 128, tc = (p.C + 127) / 128;
  const int64_t ntiles = tr * tc;
  const int64_t grid = std::min<int64_t>(ntiles, (int64_t)num_sms() * 2);
  // algorithmic bytes: bf16 read + one byte per written layout + scale arrays
  double bytes = 2.0 * p.R * p.C + (p.out_row ? 1.0 * p.R * p.C : 0.0) +
                 (p.out_col ? 1.0 * p.R * p.C : 0.0);
  if (MODE == Q_BLOCK1x128)
    bytes += (p.out_row ? 8.0 * p.R * tc : 0.0) + (p.out_col ? 8.0 * p.C * tr : 0.0);
  else if (MODE == Q_BLOCK128)
    bytes += 16.0 * ntiles;
  else
    bytes += 16.0;
  if (PRE == 2) bytes += 2.0 * p.R * p.C;  // the second input (H)
  LaunchScope ls(PRE ? pre_names[PRE] : names[MODE], st, bytes, 0.0, p.R, p.C);
  return launch_kernel(quant_tile_kernel<MODE, FMT, PRE>, dim3((unsigned)grid), dim3(kQThreads),
                       kQSmemBytes, st, tmx, tmx2, p);
}

cudaError_t quant_read_status(unsigned *status) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_quant_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_quant_status, &zero, sizeof(unsigned));
}

cudaError_t launch_amax_partials(const void *x, int64_t rows, int64_t cols, float *partials,
                                 cudaStream_t st) {
  const int g = tensorwise_partials_count(rows, cols);
  LaunchScope ls("quant_amax_tensorwise", st, 2.0 * rows * cols, 0.0, rows, cols);
  // a plain launch: overlapped with the kernel before it, the step measured
  // 0.5% slower (3.84 against 3.82 ms, fp8 linear step at N = 131072)
  return launch_kernel_as(false, amax_partials_kernel, dim3(g), dim3(kAmaxThreads), 0, st,
                          static_cast<const uint4 *>(x), (int64_t)(rows * cols / 8), partials);
}

cudaError_t launch_quantize(const void *x, int64_t rows, int64_t cols, int mode, int fmt,
                            uint8_t *out_row, uint8_t *out_col, float *row_scale,
                            float *row_scale_inv, float *col_scale, float *col_scale_inv,
                            float *partials, cudaStream_t st, bool amax_done) {
  QParams p;
  p.x = static_cast<const uint16_t *>(x);
  p.x2 = nullptr;
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
  p.hist = nullptr;
  p.hist_len = 0;
  p.cur_partials = nullptr;
  if (mode == Q_TENSOR) {
    if (!amax_done) {
      cudaError_t e = launch_amax_partials(x, rows, cols, partials, st);
      if (e != cudaSuccess) return e;
    }
    p.n_partials = tensorwise_partials_count(rows, cols);
    return fmt == FP8_FORMAT_E4M3 ? launch_tile<Q_TENSOR, FP8_FORMAT_E4M3>(p, st)
                                  : launch_tile<Q_TENSOR, FP8_FORMAT_E5M2>(p, st);
  }
  if (mode == Q_BLOCK1x128)
    return fmt == FP8_FORMAT_E4M3 ? launch_tile<Q_BLOCK1x128, FP8_FORMAT_E4M3>(p, st)
                                  : launch_tile<Q_BLOCK1x128, FP8_FORMAT_E5M2>(p, st);
  return fmt == FP8_FORMAT_E4M3 ? launch_tile<Q_BLOCK128, FP8_FORMAT_E4M3>(p, st)
                                : launch_tile<Q_BLOCK128, FP8_FORMAT_E5M2>(p, st);
}

cudaError_t launch_quantize_delayed(const void *x, int64_t rows, int64_t cols, int fmt,
                                    uint8_t *out_row, uint8_t *out_col, float *scale,
                                    float *scale_inv, float *hist, int hist_len, int64_t step,
                                    float *partials, cudaStream_t st) {
  QParams p;
  p.x = static_cast<const uint16_t *>(x);
  p.x2 = nullptr;
  p.R = rows;
  p.C = cols;
  p.out_row = out_row;
  p.out_col = out_col;
  p.row_scale = scale;
  p.row_scale_inv = scale_inv;
  p.col_scale = nullptr;
  p.col_scale_inv = nullptr;
  p.partials = nullptr;
  p.n_partials = 0;
  p.hist = hist;
  p.hist_len = hist_len;
  p.cur_partials = partials;
  const int64_t ntiles = ((rows + 127) / 128) * ((cols + 127) / 128);
  const int grid = (int)std::min<int64_t>(ntiles, (int64_t)num_sms() * 2);
  cudaError_t e = fmt == FP8_FORMAT_E4M3 ? launch_tile<Q_TENSOR, FP8_FORMAT_E4M3>(p, st)
                                         : launch_tile<Q_TENSOR, FP8_FORMAT_E5M2>(p, st);
  if (e != cudaSuccess) return e;
  LaunchScope ls("quant_delayed_history", st, 4.0 * grid + 4.0, 0.0);
  return launch_kernel(delayed_history_update_kernel, dim3(1), dim3(256), 0, st,
                       (const float *)partials, (int)grid, hist, hist_len, (int64_t)step);
}

cudaError_t launch_gelu_quantize(const void *H, const void *H2, int64_t rows, int64_t cols,
                                 int bwd, uint8_t *out_row, uint8_t *out_col, float *row_scale,
                                 float *row_scale_inv, float *col_scale, float *col_scale_inv,
                                 cudaStream_t st) {
  QParams p;
  p.x = static_cast<const uint16_t *>(H);
  p.x2 = static_cast<const uint16_t *>(H2);
  p.R = rows;
  p.C = cols;
  p.out_row = out_row;
  p.out_col = out_col;
  p.row_scale = row_scale;
  p.row_scale_inv = row_scale_inv;
  p.col_scale = col_scale;
  p.col_scale_inv = col_scale_inv;
  p.partials = nullptr;
  p.n_partials = 0;
  p.hist = nullptr;
  p.hist_len = 0;
  p.cur_partials = nullptr;
  return bwd ? launch_tile<Q_BLOCK1x128, FP8_FORMAT_E5M2, 2>(p, st)
             : launch_tile<Q_BLOCK1x128, FP8_FORMAT_E4M3, 1>(p, st);
}

}  // namespace fp8lin
