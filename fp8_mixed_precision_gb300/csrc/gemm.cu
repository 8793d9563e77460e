// FP8 GEMM on the sm_103a 5th-generation tensor cores.
//
//   C[M, N] = sum_k (A[m, k] * sa) * (B[n, k] * sb),   A, B K-major FP8, C bf16
//
// Used for the fprop, dgrad and wgrad GEMMs of the FP8 linear layer
// ("Native FP8 MLP reconstruction", implementation paragraph: FP8 operands,
// BF16 GEMM outputs, use_fast_accum=False).  fp32 accumulation throughout:
//   FP8_SCALING_TENSOR        one accumulator over the whole K range in TMEM,
//                             scaled by sa*sb in the epilogue;
//   FP8_SCALING_1x128_*       every 128-deep K block is accumulated into a
//                             fresh TMEM partial; the epilogue warps multiply
//                             it by that block's scales and add it to an fp32
//                             register accumulator (software promotion).
//
// Structure: persistent CTAs (one per SM), warp-specialised, tile BM x BN
// (128 x 256 when N allows; 128 x 192 for 1x128 x 1x128 scaling of outputs
// at least 320 wide; 128 x 128 for narrow outputs).
//   warp 0      TMA producer: A (128 rows) and B (BN rows) tiles of 128 bytes
//               along K, 128B swizzle, into a shared-memory ring guarded by
//               full/empty mbarriers
//   warp 1      TMEM allocator (all 512 columns) + single-thread tcgen05.mma
//               issuer (kind::f8f6f4, M = 128, N = BN, K = 32 per instruction)
//   warps 2-9   epilogue: tcgen05.ld from TMEM, scale, round to bf16, stage
//               32x64 slabs in 128B-swizzled shared memory, TMA bulk stores.
//               Warp w reads TMEM lanes 32*(w%4)..+31 and column half (w-2)/4.
//   1x128 x 1x128, 128 x 128 tiles: warps 2-17 are the epilogue, warp w
//               taking column quarter (w-2)/4 of lanes 32*(w%4)..+31, read
//               with the 16x256b shape (4 rows x 8 columns per thread) and
//               staged as unswizzled 32x32 slabs.
//   1x128 x 1x128, 128 x 192 tiles: warpgroup 0 = producer, MMA issuer and
//               two scale-loader warps; warps 4-15 the epilogue (64 columns
//               each, 16x256b reads), results stored from registers once per
//               tile; a register split between the warpgroups (setmaxnreg).
// TMEM holds 512/BN accumulator buffers used round-robin, so the epilogue of
// one tile (tensor scaling) or one K block (block scaling) overlaps the
// following MMAs.  Deep-K tensor-scaled GEMMs use 256-row tiles (two M
// halves sharing each B stage), and for the deepest units run them as CTA
// pairs (cluster of 2, cta_group::2 MMAs, each SM holding half of every B
// tile).  Split-K (small M*N, deep K): each split writes an fp32 partial to
// the workspace; a second kernel sums the splits in a fixed order.  The
// tile shape and split count come from a cost model of the GPU's measured
// per-SM and whole-GPU operand rates.  Every wait is bounded: on expiry the
// kernel records FP8_ERR_TIMEOUT, drains what it has in flight, frees its
// TMEM and returns.
#include <cstddef>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8lin {

namespace {

constexpr int BM = 128, BK = 128;
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemBudget = 227 * 1024;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint64_t kDrainLimitNs = 100000000ull;  // 0.1 s
constexpr int kSplitTargetCtas = 152;  // wave size the plan assumes (one CTA per SM)
constexpr int kMaxStages = 8;

struct SmemCtl {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t acc_full[4], acc_empty[4];
  uint64_t mma_done;
  // 128 x 256 1x128 x 1x128 tiles: the scale ring's slots (filled by the
  // producer warp's cp.async, drained by the epilogue warps)
  uint64_t sfull[4], sempty[4];
  uint32_t tmem_base;
  int abort;
  // 1x128 x 1x128 only: per epilogue warp, the column and row scales of the
  // current group of 4 K blocks as [K block][column] and [K block][row], and
  // the cp.async staging slots of the next group's column and row scales
  float bscale[4096];
  float4 sstage[1024];
};
constexpr int kCtlFull = (int)((sizeof(SmemCtl) + 127) / 128 * 128);
// barriers and flags only (the column-scale area serves 1x128 x 1x128 alone)
constexpr int kCtlSmall = (int)((offsetof(SmemCtl, bscale) + 127) / 128 * 128);

// 1x128 x 1x128 scaling with 128 x 192 tiles ("wide"): the row and column
// scales of a group of 4 K blocks sit in a CTA-wide ring of kScaleSlots
// slots, each [4 K blocks][128 row scales + 192 column scales] fp32.
constexpr int kWideBN = 192;
constexpr int kScaleGroup = 4;
constexpr int kScaleSlots = 3;
constexpr int kScaleRowStride = BM + kWideBN;  // floats per K block in a slot
constexpr int kScaleSlotFloats = kScaleGroup * kScaleRowStride;
// ring slots, then the scale loaders' staging area (384 entries x 16 bytes)
constexpr int kScaleRingBytes = kScaleSlots * kScaleSlotFloats * 4 + kScaleRowStride * 16;

// Per-CTA configuration.
//   MH  M halves per tile: MH = 2 gives 256 x BN tiles made of two M = 128
//       MMAs sharing each B stage (for BN = 256, 1.5x fewer operand bytes per
//       flop enter the SM); the two accumulators fill TMEM, so a tile's
//       epilogue does not overlap the next tile's MMAs (deep-K tensor-scaled
//       GEMMs only).
//   PR  CTA pair (cluster of 2, cta_group::2 MMAs): each CTA stages its own
//       A rows and half of the B tile.
// Epilogue warps: 8 (two per TMEM lane quarter, each taking half of the
// tile's columns), or for the 1x128 x 1x128 promotion 16 (128-wide tiles:
// four per lane quarter, 32 columns each) or 12 (192-wide tiles: three per
// lane quarter, 64 columns each), whose per-K-block TMEM drain is
// latency-bound and needs more warps per scheduler to overlap it.
// Shared memory: operand ring, bf16 output staging (none for split-K, which
// writes fp32 partials from registers) and the control block (the column
// scale area only for 1x128 x 1x128).  Output slabs are 32 rows x 64 columns
// (128 bytes per row, 128-byte swizzle) for 64-column warps and 32 x 32
// (64 bytes per row, unswizzled) for 32-column warps.
template <int SCALING, bool SPLIT, int BN, int MH = 1, bool PR = false>
struct Cfg {
  // 1x128 x 1x128 with 192-wide tiles: scale ring, 12 epilogue warps of 64
  // columns, bf16 results stored from registers once per tile
  static constexpr bool kWide = SCALING == FP8_SCALING_1x128_1x128 && BN == kWideBN;
  static constexpr int kEpi =
      kWide ? 12 : (SCALING == FP8_SCALING_1x128_1x128 ? 16 : 8);  // epilogue warps
  // Control warps before the epilogue: producer, MMA issuer and, for wide
  // tiles, the two scale-loader warps completing warpgroup 0.  Wide tiles run
  // as 4 whole warpgroups launched at kLaunchRegs registers per thread;
  // warpgroup 0 then gives registers back (setmaxnreg.dec to kCtlRegs) and
  // the three epilogue warpgroups take them (setmaxnreg.inc to kEpiRegs),
  // which holds their 64 fp32 accumulators, half a partial and its scales.
  static constexpr int kCtlWarps = kWide ? 4 : 2;
  static constexpr int kThreads = 32 * (kCtlWarps + kEpi);
  static constexpr int kLaunchRegs = 128, kCtlRegs = 32, kEpiRegs = 152;
  static constexpr int kCols = BN * 4 / kEpi;  // tile columns per epilogue warp
  static constexpr int kStageA = MH * BM * BK;  // bytes
  static constexpr int kStageB = (PR ? BN / 2 : BN) * BK;  // a pair CTA holds half of B
  static constexpr int kStageBytes = kStageA + kStageB;
  static constexpr int kAccBufs = (int)kTmemCols / BN;
  static constexpr int kCtlBytes =
      SCALING == FP8_SCALING_1x128_1x128 && !kWide ? kCtlFull : kCtlSmall;
  static constexpr int kScaleBytes = kWide ? kScaleRingBytes : 0;
  static constexpr int kOutSlabBytes = kCols == 32 ? 32 * 64 : 32 * 128;
  // Tensor scaling keeps one slab buffer per warp, which leaves room for a
  // fourth 48 KB operand stage of 128 x 256 tiles: their K = 512 GEMMs are
  // limited by operand bytes in flight (measured 4-5% faster with 4 stages
  // than with 3 and two slab buffers); the 1x128 x 128x128 epilogue
  // overlaps more with two (one buffer: 6% slower at K = 512).
  static constexpr int kOutSlabs =
      SPLIT || kWide ? 0 : (MH == 2 || kCols == 32 || SCALING == FP8_SCALING_TENSOR ? 1 : 2);
  static constexpr int kOutBytes = kEpi * kOutSlabs * kOutSlabBytes;
  static constexpr int kRing = kSmemBudget - 1024 - kOutBytes - kCtlBytes - kScaleBytes;
  static constexpr int kStages = kRing / kStageBytes < kMaxStages ? kRing / kStageBytes : kMaxStages;
  static constexpr size_t kSmemBytes =
      1024 + (size_t)kStages * kStageBytes + (size_t)kOutBytes + kCtlBytes + kScaleBytes;
  static_assert(kStages >= 2, "shared memory too small for the operand ring");
  static_assert(MH == 1 || (MH == 2 && kAccBufs == 2), "two M halves fill TMEM exactly");
  static_assert(kCols == 32 || kCols % 64 == 0, "epilogue column split");
  static_assert(SCALING != FP8_SCALING_1x128_1x128 || kWide ||
                    (kCols == 32 && kEpi * 256 <= 4096 && kEpi * 64 <= 1024),
                "scale staging areas");
  static_assert(!kWide || (kCols == 64 && MH == 1 && !PR && kAccBufs == 2), "wide 1x128 tiles");
  // the register split never asks for more than the launch provides
  static_assert(!kWide || (kThreads == 512 && 128 * kCtlRegs + 32 * kEpi * kEpiRegs <=
                                                  kThreads * kLaunchRegs),
                "register split");
};

__device__ unsigned g_gemm_status;

struct GemmArgs {
  int64_t M, N, K;
  int tiles_m, tiles_n, kbs, splits, kb_per_split;
  int64_t units;
  const float *a_sinv;
  const float *b_sinv;
  int64_t lds_a, lds_b;  // row strides (floats) of the block scale arrays
  void *out;             // bf16 C [M, N], or fp32 partials [splits, M, N]
  uint32_t idesc;
  int vec4;              // scale rows are 16-byte aligned in groups of 4 K blocks
  int group_m;           // > 0: units run in groups of group_m M tiles (N tiles within a group)
};


// Bounded wait on phase `parity` of `bar`; false on abort or timeout.
// CLUSTER: the barrier's arrivals may come from the other CTA of a pair.
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort) {
  auto probe = [&]() {
    return CLUSTER ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (probe()) return true;
    if ((it & 63) == 0) {
      if (*abort) return false;
      if (ptx::globaltimer() - t0 > kWaitLimitNs) {
        atomicCAS(&g_gemm_status, 0u, (unsigned)FP8_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag (used only to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer() - t0 > kDrainLimitNs) {
      atomicCAS(&g_gemm_status, 0u, (unsigned)FP8_ERR_TIMEOUT);
      return;
    }
}

// Unit u = (M tile, N tile, K split); for a CTA pair (PR) the M index is a
// pair of 128-row tiles and CTA `rank` takes tile 2 * pair + rank (which may
// lie past the last M tile).
// Tiles run N-tile fastest, or (group_m > 0) in groups of group_m M units
// (tiles, or tile pairs for CTA pairs), M unit fastest within a group: the
// CTAs running at one time then share few A and B tiles, which L2 serves to
// all of them.
template <bool PR>
__device__ __forceinline__ void decode_unit(const GemmArgs &g, int64_t u64, uint32_t rank, int &tm,
                                            int &tn, int &kb0, int &kb1) {
  // 32-bit arithmetic: the host refuses launches of 2^31 units or more (an
  // output of over 2^45 elements), so every quotient here fits
  const uint32_t u = (uint32_t)u64, splits = (uint32_t)g.splits;
  const uint32_t split = u % splits;
  const uint32_t t = u / splits;
  const uint32_t tiles_n = (uint32_t)g.tiles_n;
  if (g.group_m > 0) {
    // M units: tiles, or pairs of tiles for a CTA pair
    const uint32_t m_units = PR ? ((uint32_t)g.tiles_m + 1) / 2 : (uint32_t)g.tiles_m;
    const uint32_t gmax = (uint32_t)g.group_m;
    const uint32_t per_group = gmax * tiles_n;
    const uint32_t m0 = t / per_group * gmax;
    const uint32_t rem = t - (m0 / gmax) * per_group;
    const uint32_t gm = min(gmax, m_units - m0);  // last group may be short
    const uint32_t mu = m0 + rem % gm;
    tm = PR ? (int)mu * 2 + (int)rank : (int)mu;
    tn = (int)(rem / gm);
  } else {
    tm = PR ? (int)(t / tiles_n) * 2 + (int)rank : (int)(t / tiles_n);
    tn = (int)(t % tiles_n);
  }
  kb0 = (int)split * g.kb_per_split;
  kb1 = min(g.kbs, kb0 + g.kb_per_split);
}

// fp32 split-K partial: 32 consecutive outputs of row m from column col0.
__device__ __forceinline__ void store32_f32(const GemmArgs &g, int split, int64_t m, int64_t col0,
                                            const float (&v)[32], float scale) {
  if (m >= g.M) return;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int64_t n = col0 + 8 * p;
    if (n >= g.N) continue;
    float *dst = static_cast<float *>(g.out) + ((int64_t)split * g.M + m) * g.N + n;
    reinterpret_cast<float4 *>(dst)[0] =
        make_float4(__fmul_rn(v[8 * p], scale), __fmul_rn(v[8 * p + 1], scale),
                    __fmul_rn(v[8 * p + 2], scale), __fmul_rn(v[8 * p + 3], scale));
    reinterpret_cast<float4 *>(dst)[1] =
        make_float4(__fmul_rn(v[8 * p + 4], scale), __fmul_rn(v[8 * p + 5], scale),
                    __fmul_rn(v[8 * p + 6], scale), __fmul_rn(v[8 * p + 7], scale));
  }
}

// Row `row` of a 32x64 bf16 output slab (128 bytes, 128-byte swizzle: the
// 16-byte chunk j of row r sits at chunk j ^ (r & 7), which is also the
// layout the TMA store expects); writes chunks chunk0..chunk0+3 from v*scale.
__device__ __forceinline__ void stage32(uint8_t *slab, int row, int chunk0, const float (&v)[32],
                                        float scale) {
  uint8_t *rp = slab + row * 128;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(v[8 * p + 2 * j], scale),
                                               __fmul_rn(v[8 * p + 2 * j + 1], scale));
      w[j] = *reinterpret_cast<uint32_t *>(&b);
    }
    const int chunk = (chunk0 + p) ^ (row & 7);
    *reinterpret_cast<uint4 *>(rp + chunk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Packed fp32 pair arithmetic (two IEEE operations per instruction).
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

template <int SCALING, bool SPLIT, int BN, int MH, bool PR>
__global__ void __launch_bounds__(Cfg<SCALING, SPLIT, BN, MH, PR>::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const GemmArgs g) {
  using C = Cfg<SCALING, SPLIT, BN, MH, PR>;
  static_assert(MH == 1 || SCALING == FP8_SCALING_TENSOR, "M halves: tensor scaling only");
  static_assert(!PR || (SCALING == FP8_SCALING_TENSOR && BN == 256),
                "CTA pairs: tensor scaling, 256-wide tiles");
  // PR: a cluster of two CTAs computes a (2 * MH * 128) x BN tile with
  // cta_group::2 MMAs issued by rank 0 (the leader), one M = 256 MMA per M
  // half taking 128 rows from each CTA.  Each CTA loads its MH x 128 rows of A
  // and its BN/2 rows of B into its own shared memory; all loads complete on
  // the leader's full barrier; the leader's commits release the stages and
  // hand the accumulators to both CTAs; both CTAs' epilogues drain their own
  // TMEM rows and report to the leader's acc_empty barrier.
  const uint32_t rank = PR ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int64_t u0 = PR ? blockIdx.x / 2 : blockIdx.x;
  const int64_t ustep = PR ? gridDim.x / 2 : gridDim.x;
  constexpr uint16_t kBoth = 0x3;
  constexpr int kStages = C::kStages;
  constexpr int NB = C::kAccBufs;
  constexpr int kHalf = C::kCols;         // columns per epilogue warp
  constexpr int kSlabs = kHalf / 64;      // 64-column slabs per epilogue warp per tile
  // 1x128 x 128x128 scaling: the partial is consumed in kCw-column TMEM
  // loads (16 for 256-wide tiles, which keep 128 fp32 accumulators per
  // thread in registers)
  constexpr int kCw = BN == 256 ? 16 : 32;
  constexpr int kChunks = kHalf / kCw;
  constexpr int kPre = BN == 256 ? 2 : 4; // K blocks of scales held ahead in registers

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, by pointer arithmetic on the shared array (so the
  // compiler keeps every derived pointer in the shared window)
  uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *out_stage = smem + (size_t)kStages * C::kStageBytes;
  SmemCtl *ctl = reinterpret_cast<SmemCtl *>(out_stage + C::kOutBytes);
  // wide 1x128 x 1x128 tiles: ring of scale slots after the control block
  float *scale_ring = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ctl) + C::kCtlBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&ctl->full[s], 1);
      ptx::mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < NB; ++b) {
      ptx::mbar_init(&ctl->acc_full[b], 1);
      ptx::mbar_init(&ctl->acc_empty[b], PR ? 2 * C::kEpi : C::kEpi);
    }
    ptx::mbar_init(&ctl->mma_done, 1);
    if (C::kWide)
      for (int sl = 0; sl < kScaleSlots; ++sl) {
        ptx::mbar_init(&ctl->sfull[sl], 64);  // every lane of the two scale-loader warps
        ptx::mbar_init(&ctl->sempty[sl], C::kEpi);
      }
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    if (!SPLIT && !C::kWide) ptx::tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    if (PR) {
      ptx::tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&ctl->tmem_base, kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (PR) ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  ptx::tc_fence_after();
  pdl_wait();  // dependents launch as this grid exits
  const uint32_t tmem = ctl->tmem_base;
  volatile int *abort = &ctl->abort;

  if (warp < C::kCtlWarps) {
  // wide tiles: registers move from the control warpgroup to the epilogue
  if constexpr (C::kWide) ptx::setmaxnreg_dec<C::kCtlRegs>();
  if (C::kWide && (warp == 2 || warp == 3)) {
    // ------------------------------------------------------------ scale loaders (wide 1x128 x 1x128)
    // For every group of 4 K blocks of a unit, the two warps copy the group's
    // 128 row scales and 256 column scales (4 K blocks each: 16 bytes per row
    // or column) into a staging area with cp.async (one 16-byte copy per row
    // when the scale rows allow it), wait for their own copies, and store the
    // values transposed, [K block][row or column], into the next ring slot;
    // each lane then arrives on the slot's full barrier.  Rows or columns
    // past the tensor and K blocks past the unit read as zeros.  A slot is
    // reused once all epilogue warps released it.
    const int part = warp - 2;                  // entries part*192 .. +191 of the 384
    constexpr int kPer = kScaleRowStride / 2 / 32;
    float4 *stg = reinterpret_cast<float4 *>(scale_ring + kScaleSlots * kScaleSlotFloats) +
                  part * (kScaleRowStride / 2);
    uint32_t ngrp = 0;
    bool ok = true;
    for (int64_t u = u0; ok && u < g.units; u += ustep) {
      int tm, tn, kb0, kb1;
      decode_unit<PR>(g, u, rank, tm, tn, kb0, kb1);
      const int m0 = tm * BM, n0 = tn * BN;
      for (int g0 = kb0; g0 < kb1; g0 += kScaleGroup) {
        const uint32_t slot = ngrp % kScaleSlots;
        if (!wait_bar(&ctl->sempty[slot], ((ngrp / kScaleSlots) & 1) ^ 1, abort)) { ok = false; break; }
        const bool whole = g.vec4 && g0 + kScaleGroup <= kb1;
#pragma unroll 1
        for (int e = 0; e < kPer; ++e) {
          const int idx = part * (kScaleRowStride / 2) + e * 32 + lane;
          const bool is_row = idx < BM;
          const int rix = is_row ? m0 + idx : n0 + (idx - BM);
          const bool rok = rix < (is_row ? g.M : g.N);
          const float *src = (is_row ? g.a_sinv + (int64_t)(rok ? rix : 0) * g.lds_a
                                     : g.b_sinv + (int64_t)(rok ? rix : 0) * g.lds_b) + g0;
          if (whole) {
            ptx::cp_async16_zfill(stg + e * 32 + lane, src, rok ? 16u : 0u);
          } else {
            float *d = reinterpret_cast<float *>(stg + e * 32 + lane);
#pragma unroll
            for (int kk = 0; kk < kScaleGroup; ++kk) {
              const bool v = rok && g0 + kk < kb1;
              ptx::cp_async4(d + kk, v ? src + kk : g.a_sinv, v ? 4u : 0u);
            }
          }
        }
        ptx::cp_async_commit();
        ptx::cp_async_wait_all();  // this lane's copies have landed (it reads only its own)
        float *dst = scale_ring + slot * kScaleSlotFloats;
#pragma unroll 1
        for (int e = 0; e < kPer; ++e) {
          const int idx = part * (kScaleRowStride / 2) + e * 32 + lane;
          const float4 v = stg[e * 32 + lane];
          dst[0 * kScaleRowStride + idx] = v.x;
          dst[1 * kScaleRowStride + idx] = v.y;
          dst[2 * kScaleRowStride + idx] = v.z;
          dst[3 * kScaleRowStride + idx] = v.w;
        }
        ptx::mbar_arrive(&ctl->sfull[slot]);
        ++ngrp;
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int last_phase[kStages];
      for (int s = 0; s < kStages; ++s) last_phase[s] = -1;
      bool ok = true;
      for (int64_t u = u0; ok && u < g.units; u += ustep) {
        int tm, tn, kb0, kb1;
        decode_unit<PR>(g, u, rank, tm, tn, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar<PR>(&ctl->empty[stage], phase ^ 1, abort)) { ok = false; break; }
          uint8_t *sa = smem + (size_t)stage * C::kStageBytes;
          if (PR) {  // both halves' bytes complete on the leader's full barrier
            const uint32_t fb = ptx::mapa_shared(ptx::smem_u32(&ctl->full[stage]), 0);
            if (leader) ptx::mbar_arrive_expect_tx(&ctl->full[stage], 2u * C::kStageBytes);
            for (int mh = 0; mh < MH; ++mh)  // rows past M (or wholly outside) read as zeros
              ptx::tma_load_2d_pair(sa + mh * BM * BK, &tmA, fb, kb * BK, (tm * MH + mh) * BM);
            ptx::tma_load_2d_pair(sa + C::kStageA, &tmB, fb, kb * BK,
                                  tn * BN + (int)rank * (BN / 2));
            last_phase[stage] = (int)phase;
            if (++stage == kStages) { stage = 0; phase ^= 1; }
            continue;
          }
          // an M half that starts past the last row is not loaded (its
          // accumulator is never stored)
          const int64_t row0 = (int64_t)tm * MH * BM;
          const int halves = (MH == 2 && row0 + BM >= g.M) ? 1 : MH;
          ptx::mbar_arrive_expect_tx(&ctl->full[stage],
                                     (uint32_t)(C::kStageBytes - (MH - halves) * BM * BK));
          for (int mh = 0; mh < halves; ++mh)
            ptx::tma_load_2d(sa + mh * BM * BK, &tmA, &ctl->full[stage], kb * BK,
                             (int)(row0 + mh * BM));
          ptx::tma_load_2d(sa + C::kStageA, &tmB, &ctl->full[stage], kb * BK, tn * BN);
          last_phase[stage] = (int)phase;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok && leader)  // let every issued copy land before the CTA can exit
        for (int s = 0; s < kStages; ++s)
          if (last_phase[s] >= 0) drain_wait(&ctl->full[s], (uint32_t)last_phase[s]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t nacc = 0;  // accumulator-buffer uses so far
      bool ok = true;
      for (int64_t u = u0; ok && u < g.units; u += ustep) {
        int tm, tn, kb0, kb1;
        decode_unit<PR>(g, u, rank, tm, tn, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          // tensor scaling: one accumulator per tile; block scaling: one per K block
          const bool first = SCALING != FP8_SCALING_TENSOR || kb == kb0;
          const bool last = SCALING != FP8_SCALING_TENSOR || kb == kb1 - 1;
          if (first) {  // the accumulator buffer(s) of this tile have been drained
            for (int mh = 0; ok && mh < MH; ++mh) {
              const uint32_t n = nacc + mh;
              if (!wait_bar<PR>(&ctl->acc_empty[n % NB], ((n / NB) & 1) ^ 1, abort)) ok = false;
            }
            if (!ok) break;
            ptx::tc_fence_after();
          }
          if (!wait_bar<PR>(&ctl->full[stage], phase, abort)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(smem + (size_t)stage * C::kStageBytes);
          const uint64_t bdesc = ptx::smem_desc_sw128(a_addr + C::kStageA);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
#pragma unroll
            for (int mh = 0; mh < MH; ++mh) {
              const uint32_t d = tmem + ((nacc + mh) % NB) * BN;
              const uint64_t adesc = ptx::smem_desc_sw128(a_addr + mh * BM * BK);
              if (PR)
                ptx::mma_f8f6f4_pair(d, adesc + 2 * k, bdesc + 2 * k, g.idesc,
                                     (!first || k > 0) ? 1u : 0u);
              else
                ptx::mma_f8f6f4(d, adesc + 2 * k, bdesc + 2 * k, g.idesc,
                                (!first || k > 0) ? 1u : 0u);
            }
          if (PR)
            ptx::mma_commit_pair(&ctl->empty[stage], kBoth);
          else
            ptx::mma_commit(&ctl->empty[stage]);
          if (last) {
            for (int mh = 0; mh < MH; ++mh) {
              if (PR)
                ptx::mma_commit_pair(&ctl->acc_full[(nacc + mh) % NB], kBoth);
              else
                ptx::mma_commit(&ctl->acc_full[(nacc + mh) % NB]);
            }
            nacc += MH;
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      // all issued MMAs complete before TMEM is freed / the CTA exits
      if (PR)
        ptx::mma_commit_pair(&ctl->mma_done, 0x1);
      else
        ptx::mma_commit(&ctl->mma_done);
      drain_wait(&ctl->mma_done, 0);
    }
  }
  } else {
    // ------------------------------------------------------------ epilogue
    if constexpr (C::kWide) ptx::setmaxnreg_inc<C::kEpiRegs>();
    const int ew = warp - C::kCtlWarps;  // epilogue warp index
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int h = ew >> 2;           // column group of the tile (kHalf columns)
    const int r = q * 32 + lane;     // tile row owned by this thread
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * kHalf);
    uint32_t nacc = 0;
    uint32_t ngrp = 0;  // scale-ring slots consumed (wide 1x128 x 1x128 tiles)
    uint32_t nout = 0;  // bf16 slabs this warp has handed to TMA stores
    uint8_t *slabs = out_stage + (size_t)ew * C::kOutSlabs * C::kOutSlabBytes;
    float s_tensor = 0.0f;
    if (SCALING == FP8_SCALING_TENSOR) s_tensor = __fmul_rn(g.a_sinv[0], g.b_sinv[0]);
    // TMEM buffer ab drained by this warp: tell the MMA issuer (the leader's
    // barrier, for a CTA pair)
    auto release_acc = [&](uint32_t ab) {
      if (PR)
        ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&ctl->acc_empty[ab]), 0));
      else
        ptx::mbar_arrive(&ctl->acc_empty[ab]);
    };

    // Hands one 32x64 slab (columns col0.. of rows slab_y..) to a TMA store
    // (bf16) or writes it as an fp32 split-K partial.
    auto emit = [&](const float (&v0)[32], const float (&v1)[32], float scale, int64_t col0,
                    int64_t slab_y, int split) {
      if constexpr (SPLIT) {
        store32_f32(g, split, slab_y + lane, col0, v0, scale);
        store32_f32(g, split, slab_y + lane, col0 + 32, v1, scale);
      } else if constexpr (C::kOutSlabs > 0) {
        if (slab_y >= g.M || col0 >= g.N) return;  // slab entirely outside C
        uint8_t *slab = slabs + (nout % C::kOutSlabs) * C::kOutSlabBytes;
        // the store kOutSlabs slabs ago has finished reading this buffer
        if (lane == 0) ptx::bulk_wait_read<C::kOutSlabs - 1>();
        __syncwarp();
        stage32(slab, lane, 0, v0, scale);
        stage32(slab, lane, 4, v1, scale);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(&tmC, slab, (int)col0, (int)slab_y);
          ptx::bulk_commit();
        }
        ++nout;
      }
    };

    for (int64_t u = u0; u < g.units; u += ustep) {
      int tm, tn, kb0, kb1;
      decode_unit<PR>(g, u, rank, tm, tn, kb0, kb1);
      const int split = (int)(u % g.splits);
      const int64_t m = (int64_t)tm * MH * BM + r;
      const int64_t colbase = (int64_t)tn * BN + h * kHalf;
      const int64_t slab_y0 = (int64_t)tm * MH * BM + q * 32;
      if (SCALING == FP8_SCALING_TENSOR) {
        bool ok = true;
        for (int mh = 0; mh < MH; ++mh) {  // one accumulator buffer per M half
          const int64_t slab_y = slab_y0 + (int64_t)mh * BM;
          const uint32_t ab = nacc % NB, aph = (nacc / NB) & 1;
          if (!wait_bar<PR>(&ctl->acc_full[ab], aph, abort)) { ok = false; break; }
          ptx::tc_fence_after();
#pragma unroll
          for (int s = 0; s < kSlabs; ++s) {
            uint32_t raw0[32], raw1[32];
            ptx::tmem_ld32(tl + ab * BN + 64 * s, raw0);
            ptx::tmem_ld32(tl + ab * BN + 64 * s + 32, raw1);
            ptx::tmem_ld_wait();
            if (s == kSlabs - 1) {  // accumulator fully in registers: free the TMEM buffer
              ptx::tc_fence_before();
              __syncwarp();
              if (lane == 0) release_acc(ab);
            }
            float v0[32], v1[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              v0[j] = __uint_as_float(raw0[j]);
              v1[j] = __uint_as_float(raw1[j]);
            }
            emit(v0, v1, s_tensor, colbase + 64 * s, slab_y, split);
          }
          ++nacc;
        }
        if (!ok) break;
      } else if constexpr (C::kWide) {
        // Every element's scale is (row scale) x (column scale) of its K
        // block, both read from the scale ring.  The partial is read with the
        // 16x256b TMEM shape, 64 columns per load: thread (rr, cc) =
        // (lane / 4, lane % 4) holds rows rr + 8i (i = 0..3) of the warp's
        // 32-row quarter and columns 8k + 2cc, +1 (k = 0..7) of its 64, so per
        // K block it needs 4 row scales and 16 column scales (8-byte shared
        // loads, 4 distinct per warp) instead of all 64 columns' scales.
        // acc[8i + k] is the column pair k of row i.
        const int rr = lane >> 2, cc = lane & 3;
        uint64_t acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0;
        bool ok = true;
        for (int g0 = kb0; ok && g0 < kb1; g0 += kScaleGroup) {
          const uint32_t slot = ngrp % kScaleSlots;
          if (!wait_bar(&ctl->sfull[slot], (ngrp / kScaleSlots) & 1, abort)) { ok = false; break; }
          const float *srow = scale_ring + slot * kScaleSlotFloats + q * 32 + rr;
          const float *scol = scale_ring + slot * kScaleSlotFloats + BM + h * 64 + 2 * cc;
#pragma unroll 1
          for (int kk = 0; kk < kScaleGroup; ++kk) {
            if (g0 + kk >= kb1) break;
            const uint32_t ab = nacc % NB, aph = (nacc / NB) & 1;
            if (!wait_bar<PR>(&ctl->acc_full[ab], aph, abort)) { ok = false; break; }
            ptx::tc_fence_after();
            uint64_t sb[8];  // column-scale pairs of this thread's 8 column pairs
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float2 b2 = *reinterpret_cast<const float2 *>(scol + kk * kScaleRowStride + 8 * k);
              sb[k] = pk(b2.x, b2.y);
            }
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {  // TMEM lanes q*32 + 16 hb .. +15: rows rr + 8i, i = 2hb, 2hb+1
              uint32_t raw[32];
              ptx::tmem_ld16x256b_x8(tl + ((uint32_t)(16 * hb) << 16) + ab * BN, raw);
              const float sa0 = srow[kk * kScaleRowStride + 16 * hb];
              const float sa1 = srow[kk * kScaleRowStride + 16 * hb + 8];
              ptx::tmem_ld_wait();
              if (hb == 1) {  // the partial is in registers: free the TMEM buffer
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(ab);
              }
#pragma unroll
              for (int ii = 0; ii < 2; ++ii) {
                const uint64_t sa2 = ii ? pk(sa1, sa1) : pk(sa0, sa0);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  uint64_t &a = acc[8 * (2 * hb + ii) + k];
                  a = fma2(pk(__uint_as_float(raw[4 * k + 2 * ii]), __uint_as_float(raw[4 * k + 2 * ii + 1])),
                           mul2(sa2, sb[k]), a);
                }
              }
            }
            ++nacc;
          }
          __syncwarp();  // every lane's reads of the slot are done
          if (lane == 0) ptx::mbar_arrive(&ctl->sempty[slot]);
          ++ngrp;
        }
        if (!ok) break;
        // results straight from registers (once per tile): rows
        // slab_y0 + rr + 8i, columns colbase + 8k + 2cc and +1 (N is a multiple
        // of 16, so n < N covers n + 1)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int64_t mm = slab_y0 + rr + 8 * i;
          if (mm >= g.M) continue;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int64_t n = colbase + 8 * k + 2 * cc;
            if (n >= g.N) continue;
            float x, y;
            upk(acc[8 * i + k], x, y);
            if constexpr (SPLIT) {
              *reinterpret_cast<float2 *>(static_cast<float *>(g.out) +
                                          ((int64_t)split * g.M + mm) * g.N + n) = make_float2(x, y);
            } else {
              *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(g.out) + mm * g.N + n) =
                  __floats2bfloat162_rn(x, y);
            }
          }
        }
      } else {
        const int64_t slab_y = slab_y0;
        uint64_t acc[kHalf / 2];  // kHalf fp32 accumulators as packed pairs
#pragma unroll
        for (int j = 0; j < kHalf / 2; ++j) acc[j] = 0;
        const int64_t mrow = m < g.M ? m : g.M - 1;  // clamp for the scale read only
        const float *arow = g.a_sinv + mrow * g.lds_a;
        const float *bt = g.b_sinv + (colbase / 128) * g.lds_b;  // 128x128: this warp's column block
        // Scales of K blocks kb .. kb+kPre-1 in a register ring (slot 0 = current):
        // the loads are issued kPre blocks before their use, hiding their latency.
        bool ok = true;
        if constexpr (SCALING == FP8_SCALING_1x128_1x128) {
          // Every element's scale is (row scale) x (column scale) of its K
          // block.  The partial is read with the 16x256b TMEM shape: thread
          // (rr, cc) = (lane / 4, lane % 4) holds rows rr + 8i (i = 0..3) of
          // the warp's 32-row quarter and columns 8j + 2cc, +1 (j = 0..3) of
          // its 32 columns, so it needs 8 column scales and 4 row scales per
          // K block instead of 32 column scales (32x32b shape) - fewer bytes
          // through the shared-memory / TMEM load path into registers, which
          // bounds this promotion.  acc[4i + j] holds the pair (row i, pair j).
          static_assert(kHalf == 32, "16x256b promotion: 32 columns per warp");
          const int rr = lane >> 2, cc = lane & 3;
          const int64_t n_st = colbase + lane;  // column whose scales this lane stages
          const bool nok = n_st < g.N;
          const float *brow = g.b_sinv + (nok ? n_st : g.N - 1) * g.lds_b;
          // per warp: current group as [K block][32 columns] and [K block][32 rows]
          float *bsw = ctl->bscale + ew * 256;
          float *asw = bsw + 128;
          // cp.async staging, one group ahead: [lane] column scales, then [lane] row scales
          float4 *stg = ctl->sstage + ew * 64;
          // Scales move in groups of 4 K blocks; each lane copies the 4 scales
          // of its staging column and of row q*32 + lane with cp.async
          // (nothing held in registers while in flight).
          auto fetch4 = [&](float4 *dst, const float *row, int k) {
            if (g.vec4 && k + 3 < kb1) {
              ptx::cp_async16(dst, row + k);
            } else {
              float *d = reinterpret_cast<float *>(dst);
#pragma unroll
              for (int i = 0; i < 4; ++i)  // past kb1: zero fill from a valid address
                ptx::cp_async4(d + i, row + (k + i < kb1 ? k + i : kb0), k + i < kb1 ? 4u : 0u);
            }
          };
          auto fetch = [&](int k) {
            fetch4(stg + lane, brow, k);
            fetch4(stg + 32 + lane, arow, k);
            ptx::cp_async_commit();
          };
          fetch(kb0);
          for (int g0 = kb0; ok && g0 < kb1; g0 += 4) {
            ptx::cp_async_wait_all();
            const float4 bv = stg[lane], av = stg[32 + lane];  // this lane's own slots
            if (g0 + 4 < kb1) fetch(g0 + 4);
            __syncwarp();  // the previous group's reads of bsw / asw are done
            bsw[0 * 32 + lane] = nok ? bv.x : 0.0f;
            bsw[1 * 32 + lane] = nok ? bv.y : 0.0f;
            bsw[2 * 32 + lane] = nok ? bv.z : 0.0f;
            bsw[3 * 32 + lane] = nok ? bv.w : 0.0f;
            asw[0 * 32 + lane] = av.x;
            asw[1 * 32 + lane] = av.y;
            asw[2 * 32 + lane] = av.z;
            asw[3 * 32 + lane] = av.w;
            __syncwarp();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              if (g0 + kk >= kb1) break;
              const uint32_t ab = nacc % NB, aph = (nacc / NB) & 1;
              if (!wait_bar<PR>(&ctl->acc_full[ab], aph, abort)) { ok = false; break; }
              ptx::tc_fence_after();
              uint64_t sb[4];  // column-scale pairs of this thread's 4 column pairs
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float2 b2 = *reinterpret_cast<const float2 *>(bsw + kk * 32 + 8 * j + 2 * cc);
                sb[j] = pk(b2.x, b2.y);
              }
#pragma unroll
              for (int hb = 0; hb < 2; ++hb) {  // TMEM lanes q*32 + 16 hb .. +15
                uint32_t raw[16];
                ptx::tmem_ld16x256b_x4(tl + ((uint32_t)(16 * hb) << 16) + ab * BN, raw);
                ptx::tmem_ld_wait();
                if (hb == 1) {  // the partial is in registers: free the TMEM buffer
                  ptx::tc_fence_before();
                  __syncwarp();
                  if (lane == 0) release_acc(ab);
                }
#pragma unroll
                for (int ii = 0; ii < 2; ++ii) {
                  const int i = 2 * hb + ii;  // row rr + 8i
                  const float sa = asw[kk * 32 + rr + 8 * i];
                  const uint64_t sa2 = pk(sa, sa);
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    const uint64_t sc = mul2(sa2, sb[j]);
                    acc[4 * i + j] = fma2(pk(__uint_as_float(raw[4 * j + 2 * ii]),
                                             __uint_as_float(raw[4 * j + 2 * ii + 1])),
                                          sc, acc[4 * i + j]);
                  }
                }
              }
              ++nacc;
            }
          }
          ptx::cp_async_wait_all();  // no scale copy in flight past the tile (abort path)
        } else {
        float ra[kPre], rb[kPre];  // row scale, B tile scale
        auto load_scales = [&](int k, float &a, float &b) {
          a = k < kb1 ? arow[k] : 0.0f;
          b = k < kb1 ? bt[k] : 0.0f;
        };
#pragma unroll
        for (int i = 0; i < kPre; ++i) load_scales(kb0 + i, ra[i], rb[i]);
        for (int kb = kb0; kb < kb1; ++kb) {
          const uint32_t ab = nacc % NB, aph = (nacc / NB) & 1;
          const float sa_cur = ra[0], sbt_cur = rb[0];
#pragma unroll
          for (int i = 0; i + 1 < kPre; ++i) {
            ra[i] = ra[i + 1];
            rb[i] = rb[i + 1];
          }
          load_scales(kb + kPre, ra[kPre - 1], rb[kPre - 1]);
          if (!wait_bar<PR>(&ctl->acc_full[ab], aph, abort)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint64_t st2 = pk(__fmul_rn(sa_cur, sbt_cur), __fmul_rn(sa_cur, sbt_cur));
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            uint32_t raw[kCw];
            if constexpr (kCw == 16) ptx::tmem_ld16(tl + ab * BN + kCw * c, raw);
            else ptx::tmem_ld32(tl + ab * BN + kCw * c, raw);
            ptx::tmem_ld_wait();
            if (c == kChunks - 1) {  // the partial is in registers: free the TMEM buffer
              ptx::tc_fence_before();
              __syncwarp();
              if (lane == 0) release_acc(ab);
            }
#pragma unroll
            for (int j = 0; j < kCw / 2; ++j) {
              const int p = (kCw / 2) * c + j;  // accumulator pair index
              acc[p] = fma2(pk(__uint_as_float(raw[2 * j]), __uint_as_float(raw[2 * j + 1])), st2,
                            acc[p]);
            }
          }
          ++nacc;
        }
        }
        if (!ok) break;
        if constexpr (SCALING == FP8_SCALING_1x128_1x128) {
          // rows slab_y + rr + 8i, columns colbase + 8j + 2cc and +1
          const int rr = lane >> 2, cc = lane & 3;
          if constexpr (SPLIT) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int64_t mm = slab_y + rr + 8 * i;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int64_t n = colbase + 8 * j + 2 * cc;  // N is even: n < N covers n + 1
                if (mm >= g.M || n >= g.N) continue;
                float2 v;
                upk(acc[4 * i + j], v.x, v.y);
                *reinterpret_cast<float2 *>(static_cast<float *>(g.out) +
                                            ((int64_t)split * g.M + mm) * g.N + n) = v;
              }
            }
          } else if (slab_y < g.M && colbase < g.N) {
            // one 32 x 32 bf16 slab (64-byte rows, unswizzled), staged once per tile
            uint8_t *slab = slabs + (nout % C::kOutSlabs) * C::kOutSlabBytes;
            if (lane == 0) ptx::bulk_wait_read<C::kOutSlabs - 1>();
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                float x, y;
                upk(acc[4 * i + j], x, y);
                __nv_bfloat162 b = __floats2bfloat162_rn(x, y);
                *reinterpret_cast<__nv_bfloat162 *>(slab + (rr + 8 * i) * 64 + 16 * j + 4 * cc) = b;
              }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_2d(&tmC, slab, (int)colbase, (int)slab_y);
              ptx::bulk_commit();
            }
            ++nout;
          }
        } else {
#pragma unroll
          for (int s = 0; s < kSlabs; ++s) {
            float v0[32], v1[32];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              upk(acc[32 * s + j], v0[2 * j], v0[2 * j + 1]);
              upk(acc[32 * s + 16 + j], v1[2 * j], v1[2 * j + 1]);
            }
            emit(v0, v1, 1.0f, colbase + 64 * s, slab_y, split);
          }
        }
      }
    }
    if (!SPLIT && lane == 0) ptx::bulk_wait<0>();  // stores complete before the CTA exits
  }

  ptx::tc_fence_before();
  __syncthreads();
  // neither CTA of a pair frees its TMEM or exits while the other may still
  // signal its barriers or the leader's MMAs may still write its TMEM
  if (PR) ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (PR)
      ptx::tmem_dealloc_pair(tmem, kTmemCols);
    else
      ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Failure-detection test hook: one warp initialises an mbarrier that nothing
// will ever arrive at and waits on it with the same bounded wait the GEMM
// uses, but with a caller-chosen limit; on expiry it records FP8_ERR_TIMEOUT
// in the status word and returns.  No trap, no fault, the context stays usable.
__global__ void wait_timeout_probe_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(&bar, 0)) {
      if (ptx::globaltimer() - t0 > limit_ns) {
        atomicCAS(&g_gemm_status, 0u, (unsigned)FP8_ERR_TIMEOUT);
        break;
      }
    }
  }
}

// Fixed-order sum of the split-K partials, rounded once to bf16.
__global__ void splitk_reduce_kernel(const float *__restrict__ ws, int splits, int64_t mn,
                                     __nv_bfloat16 *__restrict__ C) {
  pdl_wait_then_release();
  const int64_t n4 = mn / 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 a = reinterpret_cast<const float4 *>(ws)[i];
    for (int s = 1; s < splits; ++s) {
      const float4 b = reinterpret_cast<const float4 *>(ws + (int64_t)s * mn)[i];
      a.x = __fadd_rn(a.x, b.x);
      a.y = __fadd_rn(a.y, b.y);
      a.z = __fadd_rn(a.z, b.z);
      a.w = __fadd_rn(a.w, b.w);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t *>(&lo);
    w.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(C)[i] = w;
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 [rows, cols] row-major output, boxes of 32 rows x 64 columns (128 bytes),
// 128-byte swizzle, or (narrow) 32 rows x 32 columns unswizzled; out-of-range
// parts of a box are not written.
bool make_out_map(CUtensorMap *m, void *base, int64_t rows, int64_t cols, bool narrow) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {narrow ? 32u : 64u, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            narrow ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, cols] u8 row-major operand, boxes of box_rows rows x 128 bytes,
// 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
  int bn, mh, pr, tiles_m, tiles_n, kbs, splits, kb_per_split;
  double est_s;  // estimated kernel time, seconds (plan selection only)
};

// Rates used to compare plans (flop/s).  A CTA alone on the GPU runs a
// 128 x 256 tile at about kSmRate; with every SM busy the operand traffic
// through L2 caps the whole GPU at about kGpuRate.  A 256 x 256 tile (two M
// halves) moves 1.5x fewer operand bytes per flop, so both rates are higher.
struct TileRates {
  double sm, gpu;
};
constexpr TileRates kRatesBn128{14e12, 2.0e15}, kRatesBn192{12e12, 1.9e15},
    kRatesBn256{20e12, 2.6e15}, kRatesBn256Mh2{23.5e12, 3.1e15};
constexpr double kPlanHbmBps = 6e12;   // fp32 split partials, written and read once
constexpr double kPlanEpiBps = 60e9;   // per-SM epilogue drain rate (not overlapped, MH = 2)
constexpr double kPlanReduceLaunchS = 4e-6;

// One candidate: tile shape (bn, mh) and the split count that minimises
//   max(waves x time per unit, all units' work at the GPU-wide rate)
//   + split-partial traffic,
// a unit's time being its K blocks at the per-SM rate plus, for MH = 2, its
// unoverlapped epilogue.  Splits start on 4-block groups.
Plan plan_for(int64_t M, int64_t N, int64_t K, int bn, int mh) {
  Plan p;
  p.bn = bn;
  p.mh = mh;
  p.pr = 0;
  p.tiles_m = (int)((M + BM * mh - 1) / (BM * mh));
  p.tiles_n = (int)((N + bn - 1) / bn);
  p.kbs = (int)((K + BK - 1) / BK);
  const int64_t tiles = (int64_t)p.tiles_m * p.tiles_n;
  const TileRates r = bn == 128 ? kRatesBn128
                      : bn == kWideBN ? kRatesBn192
                                      : (mh == 2 ? kRatesBn256Mh2 : kRatesBn256);
  const double kb_flops = 2.0 * BM * mh * bn * BK;
  const double all_s = (double)tiles * p.kbs * kb_flops / r.gpu;
  p.splits = 1;
  p.kb_per_split = p.kbs;
  p.est_s = 1e30;
  const int max_s = std::min(32, std::max(1, p.kbs / 4));
  for (int s = 1; s <= max_s; ++s) {
    int kbp = (p.kbs + s - 1) / s;
    if (s > 1) kbp = (kbp + 3) / 4 * 4;
    const int splits = (p.kbs + kbp - 1) / kbp;
    if (splits != s) continue;  // same as a smaller split count
    const int64_t waves = (tiles * splits + kSplitTargetCtas - 1) / kSplitTargetCtas;
    double unit_s = kbp * kb_flops / r.sm;
    if (mh == 2) unit_s += (double)BM * mh * bn * (splits > 1 ? 4 : 2) / kPlanEpiBps;
    double est = std::max((double)waves * unit_s, all_s);
    if (splits > 1) est += 8.0 * splits * M * N / kPlanHbmBps + kPlanReduceLaunchS;
    if (est < p.est_s * 0.98) {  // a larger split must win clearly
      p.est_s = est;
      p.splits = splits;
      p.kb_per_split = kbp;
    }
  }
  return p;
}

// Kernel configuration as a function of (M, N, K, scaling) only.
Plan make_plan(int64_t M, int64_t N, int64_t K, int scaling) {
  // 256-wide tiles halve the A re-reads and the per-SM operand traffic per
  // flop; under 1x128 x 1x128 scaling the tiles are 192 wide (the widest
  // whose fp32 promotion fits the epilogue's registers), for outputs at least
  // 320 wide (narrower ones would waste most of a second tile)
  const int bn = scaling == FP8_SCALING_1x128_1x128 ? (N >= 320 ? kWideBN : 128)
                                                    : (N >= 256 ? 256 : 128);
  Plan p = plan_for(M, N, K, bn, 1);
  if (scaling == FP8_SCALING_TENSOR && bn == 256 && M > BM) {
    const Plan p2 = plan_for(M, N, K, bn, 2);
    if (p2.est_s < p.est_s) p = p2;
  }
  // Deep-K 256-row tiles run as CTA pairs (512 x 256 per pair): each SM then
  // stores and reads half of every B tile.  Measured on GB300: 1-4% faster
  // when a unit spans >= 64 K blocks, slower for shorter units (the pair's
  // epilogues must both drain before the next tile starts) and for 128-row
  // tiles.
  if (scaling == FP8_SCALING_TENSOR && p.bn == 256 && p.mh == 2 && p.tiles_m >= 2 &&
      p.kb_per_split >= 64)
    p.pr = 1;
  return p;
}

template <int SCALING, bool SPLIT, int BN, int MH = 1, bool PR = false>
cudaError_t launch_variant(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                           const GemmArgs &g, cudaStream_t st) {
  using C = Cfg<SCALING, SPLIT, BN, MH, PR>;
  constexpr int kCl = PR ? 2 : 1;  // CTAs per cluster
  auto kernel = fp8_gemm_kernel<SCALING, SPLIT, BN, MH, PR>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = PR ? 1 : 0;  // the occupancy query below sees the cluster shape only
  // per device: the shared-memory opt-in, and how many CTAs can be resident
  // at once (whole clusters for pairs), which sizes the persistent grid
  static int resident[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (resident[dev] == 0) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (C::kWide) {  // the setmaxnreg split needs the launch allocation it was sized for
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kernel);
      if (e != cudaSuccess) return e;
      if (fa.numRegs < C::kLaunchRegs) return cudaErrorInvalidConfiguration;
    }
    int n = num_sms();
    if (PR) {
      int clusters = 0;
      cfg.gridDim = dim3((unsigned)(num_sms() / kCl * kCl));
      e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
      if (e != cudaSuccess) return e;
      if (clusters < 1) return cudaErrorInvalidConfiguration;
      n = std::min(n / kCl, clusters) * kCl;
    }
    resident[dev] = n;
  }
  static const char *names[3] = {"gemm_fp8_tensor", "gemm_fp8_block_1x128_128x128",
                                 "gemm_fp8_block_1x128_1x128"};
  const int64_t grid = std::min<int64_t>(g.units * kCl, resident[dev]);
  // algorithmic bytes: FP8 operands once, bf16 output once, block scales
  double bytes = (double)g.M * g.K + (double)g.N * g.K + 2.0 * g.M * g.N;
  if (SCALING == FP8_SCALING_1x128_128x128) bytes += 4.0 * g.kbs * (g.M + (g.N + 127) / 128);
  if (SCALING == FP8_SCALING_1x128_1x128) bytes += 4.0 * g.kbs * (g.M + g.N);
  LaunchScope ls(names[SCALING], st, bytes, 2.0 * g.M * g.N * g.K, g.M, g.N, g.K);
  cfg.gridDim = dim3((unsigned)grid);
  if (pdl_enabled()) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  }
  return cudaLaunchKernelEx(&cfg, kernel, ta, tb, tc, g);
}

template <int SCALING>
cudaError_t launch_scaling(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                           const GemmArgs &g, bool split, int bn, int mh, int pr,
                           cudaStream_t st) {
  if constexpr (SCALING == FP8_SCALING_TENSOR) {
    if (bn == 256 && mh == 2 && pr)
      return split ? launch_variant<SCALING, true, 256, 2, true>(ta, tb, tc, g, st)
                   : launch_variant<SCALING, false, 256, 2, true>(ta, tb, tc, g, st);
    if (bn == 256 && mh == 2)
      return split ? launch_variant<SCALING, true, 256, 2>(ta, tb, tc, g, st)
                   : launch_variant<SCALING, false, 256, 2>(ta, tb, tc, g, st);
  }
  if constexpr (SCALING == FP8_SCALING_1x128_1x128) {
    if (bn == kWideBN)
      return split ? launch_variant<SCALING, true, kWideBN>(ta, tb, tc, g, st)
                   : launch_variant<SCALING, false, kWideBN>(ta, tb, tc, g, st);
  } else if (bn == 256) {
    return split ? launch_variant<SCALING, true, 256>(ta, tb, tc, g, st)
                 : launch_variant<SCALING, false, 256>(ta, tb, tc, g, st);
  }
  return split ? launch_variant<SCALING, true, 128>(ta, tb, tc, g, st)
               : launch_variant<SCALING, false, 128>(ta, tb, tc, g, st);
}

}  // namespace

bool make_bf16_tile_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows,
                        int box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int scaling) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  const Plan p = make_plan(M, N, K, scaling);
  return p.splits > 1 ? (size_t)p.splits * (size_t)M * (size_t)N * sizeof(float) : 0;
}

cudaError_t launch_gemm(const uint8_t *A, int a_fmt, const float *a_sinv, const uint8_t *B,
                        int b_fmt, const float *b_sinv, int64_t M, int64_t N, int64_t K,
                        int scaling, void *Cout, void *ws, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (K == 0) return cudaMemsetAsync(Cout, 0, (size_t)M * N * 2, st);
  const Plan p = make_plan(M, N, K, scaling);
  CUtensorMap ta, tb, tc;
  // a CTA pair loads the B tile as two halves of bn / 2 rows
  if (!make_map(&ta, A, M, K, BM) || !make_map(&tb, B, N, K, p.pr ? p.bn / 2 : p.bn))
    return cudaErrorInvalidValue;
  if (p.splits == 1 && !(scaling == FP8_SCALING_1x128_1x128 && p.bn == kWideBN)) {
    // the 128-wide 1x128 x 1x128 kernel's epilogue warps own 32 columns each
    if (!make_out_map(&tc, Cout, M, N, scaling == FP8_SCALING_1x128_1x128))
      return cudaErrorInvalidValue;
  } else {
    tc = ta;  // unused: split-K partials and wide 1x128 x 1x128 results are stored from registers
  }
  GemmArgs g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.tiles_m = p.tiles_m;
  g.tiles_n = p.tiles_n;
  g.kbs = p.kbs;
  g.splits = p.splits;
  g.kb_per_split = p.kb_per_split;
  g.units = (int64_t)(p.pr ? (p.tiles_m + 1) / 2 : p.tiles_m) * p.tiles_n * p.splits;
  if (g.units >= (int64_t(1) << 31)) return cudaErrorInvalidValue;  // units are decoded in 32 bits
  g.a_sinv = a_sinv;
  g.b_sinv = b_sinv;
  g.lds_a = p.kbs;
  g.lds_b = p.kbs;
  g.out = p.splits > 1 ? ws : Cout;
  g.idesc = ptx::idesc_f8f6f4((uint32_t)a_fmt, (uint32_t)b_fmt, p.pr ? 2 * BM : BM, (uint32_t)p.bn);
  g.vec4 = (p.kbs % 4 == 0) && (reinterpret_cast<uintptr_t>(a_sinv) % 16 == 0) &&
           (reinterpret_cast<uintptr_t>(b_sinv) % 16 == 0);
  // Wide 1x128 x 1x128 tiles stream both operands per 128-deep K block for
  // the whole K range: grouping 16 M tiles keeps the concurrently running
  // tiles' A and B blocks shared through L2.  Other GEMMs keep the N-tile
  // fastest order (measured faster for the K = 512 shapes, whose output
  // rows are then written across all N tiles at once).
  // Deep-K 1x128 x 128x128 GEMMs (fprop/dgrad, K >= 2048) gain the same way
  // (16384 x 14336 x 4096: 0.82 -> 0.78 ms).
  g.group_m = ((scaling == FP8_SCALING_1x128_1x128 && p.bn == kWideBN) ||
               (scaling == FP8_SCALING_1x128_128x128 && p.kbs >= 16))
                  ? std::min(16, p.tiles_m)
                  : 0;
  const bool split = p.splits > 1;
  cudaError_t e;
  switch (scaling) {
    case FP8_SCALING_TENSOR:
      e = launch_scaling<FP8_SCALING_TENSOR>(ta, tb, tc, g, split, p.bn, p.mh, p.pr, st);
      break;
    case FP8_SCALING_1x128_128x128:
      e = launch_scaling<FP8_SCALING_1x128_128x128>(ta, tb, tc, g, split, p.bn, p.mh, p.pr, st);
      break;
    default:
      e = launch_scaling<FP8_SCALING_1x128_1x128>(ta, tb, tc, g, split, p.bn, p.mh, p.pr, st);
      break;
  }
  if (e != cudaSuccess || !split) return e;
  const int64_t mn = M * N;
  static int reduce_bps[64];
  const int64_t blocks = std::min<int64_t>(
      (mn / 4 + 255) / 256, (int64_t)num_sms() * blocks_per_sm(splitk_reduce_kernel, 256, reduce_bps));
  LaunchScope ls("gemm_splitk_reduce", st, 4.0 * p.splits * mn + 2.0 * mn, (double)p.splits * mn, M, N,
                 p.splits);
  return launch_kernel(splitk_reduce_kernel, dim3((unsigned)std::max<int64_t>(blocks, 1)), dim3(256),
                       0, st, static_cast<const float *>(ws), p.splits, mn,
                       static_cast<__nv_bfloat16 *>(Cout));
}

cudaError_t launch_wait_timeout_probe(uint64_t limit_ns, cudaStream_t st) {
  LaunchScope ls("wait_timeout_probe", st, 0.0, 0.0);
  wait_timeout_probe_kernel<<<1, 32, 0, st>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t gemm_read_status(unsigned *status, cudaStream_t st) {
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(status, g_gemm_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(unsigned));
}

}  // namespace fp8lin
