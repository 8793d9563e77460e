// C-ABI layer of the FP8 linear library: argument validation, workspace
// carving, the weight cache (is_first_microbatch semantics) and the
// orchestration of quantize + GEMM calls for the linear layer's forward and
// backward.  Host code only; every arithmetic step runs in the kernels.
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <map>
#include <tuple>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/fp8lin.h"
#include "internal.h"

namespace fp8lin {
static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// ---- per-kernel event timing (fp8_profile_begin / fp8_profile_end)
namespace {
struct ProfRec {
  const char *name;
  cudaEvent_t start, stop;
  double bytes, flops;
  int64_t m, n, k;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

LaunchScope::LaunchScope(const char *name, cudaStream_t st, double bytes, double flops, int64_t m,
                         int64_t n, int64_t k)
    : st_(st) {
  count_launch();
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) return;
  ProfRec r{name, take_event(), take_event(), bytes, flops, m, n, k};
  if (!r.start || !r.stop) return;
  cudaEventRecord(r.start, st);
  g_prof.push_back(r);
  rec_ = (int)g_prof.size() - 1;
}

LaunchScope::~LaunchScope() {
  if (rec_ < 0) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (rec_ < (int)g_prof.size()) cudaEventRecord(g_prof[rec_].stop, st_);
}
}  // namespace fp8lin

using namespace fp8lin;

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline cudaStream_t cs(fp8_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

fp8_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA; }

int format_of(fp8_role role) { return role == FP8_ROLE_GRAD ? FP8_FORMAT_E5M2 : FP8_FORMAT_E4M3; }

// 0 tensorwise, 1 1x128, 2 128x128
int qmode_of(fp8_recipe recipe, fp8_role role) {
  if (recipe != FP8_RECIPE_BLOCK) return 0;
  return role == FP8_ROLE_WEIGHT ? 2 : 1;
}

bool valid_recipe(int r) { return r == FP8_RECIPE_TENSORWISE || r == FP8_RECIPE_BLOCK; }
// Recipes a linear layer / weight cache accepts (delayed scaling needs per-tensor state).
bool valid_linear_recipe(int r) { return valid_recipe(r) || r == FP8_RECIPE_DELAYED; }
// Activations and gradients of a delayed-scaling linear use current tensorwise scaling.
fp8_recipe act_recipe(fp8_recipe r) { return r == FP8_RECIPE_DELAYED ? FP8_RECIPE_TENSORWISE : r; }
bool valid_role(int r) { return r >= FP8_ROLE_ACT && r <= FP8_ROLE_GRAD; }

fp8_status check_dims(int64_t a, int64_t b) {
  if (a < 0 || b < 0) return FP8_ERR_INVALID_ARG;
  if (a % 16 || b % 16) return FP8_ERR_SHAPE;
  if (a > (int64_t(1) << 31) || b > (int64_t(1) << 31)) return FP8_ERR_SHAPE;
  return FP8_OK;
}

// number of floats in one scale array of a layout
int64_t scale_elems(fp8_recipe recipe, fp8_role role, int64_t rows, int64_t cols, int colwise) {
  int64_t sr = 0, sc = 0;
  fp8_scale_shape(recipe, role, rows, cols, colwise, &sr, &sc);
  return sr * sc;
}

// Carves consecutive 256-byte-aligned regions out of a base pointer.
struct Carver {
  uint8_t *base;
  size_t off = 0;
  explicit Carver(void *b) : base(static_cast<uint8_t *>(b)) {}
  template <class T>
  T *take(size_t bytes) {
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off += align_up(bytes);
    return p;
  }
};

}  // namespace

extern "C" {

const char *fp8_status_string(fp8_status s) {
  switch (s) {
    case FP8_OK: return "ok";
    case FP8_ERR_INVALID_ARG: return "invalid argument";
    case FP8_ERR_SHAPE: return "unsupported shape (dimensions must be multiples of 16)";
    case FP8_ERR_ALIGN: return "pointer not 16-byte aligned";
    case FP8_ERR_STALE: return "weight-cache entry stale or version changed mid-cycle";
    case FP8_ERR_TIMEOUT: return "device-side wait timed out";
    case FP8_ERR_CUDA: return "CUDA error";
    case FP8_ERR_UNSUPPORTED: return "unsupported";
    case FP8_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

uint64_t fp8_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

fp8_status fp8_scale_shape(fp8_recipe recipe, fp8_role role, int64_t rows, int64_t cols,
                           int colwise, int64_t *srows, int64_t *scols) {
  if (!srows || !scols || !valid_linear_recipe(recipe) || !valid_role(role))
    return FP8_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0) return FP8_ERR_INVALID_ARG;
  const int mode = qmode_of(recipe, role);
  if (mode == 0) {
    *srows = 1;
    *scols = 1;
  } else if (mode == 1) {
    *srows = colwise ? cols : rows;
    *scols = colwise ? cdiv(rows, 128) : cdiv(cols, 128);
  } else {
    *srows = colwise ? cdiv(cols, 128) : cdiv(rows, 128);
    *scols = colwise ? cdiv(rows, 128) : cdiv(cols, 128);
  }
  return FP8_OK;
}

fp8_status fp8_quantize_workspace_size(fp8_recipe recipe, int64_t rows, int64_t cols,
                                       size_t *bytes) {
  if (!bytes || !valid_linear_recipe(recipe) || rows < 0 || cols < 0) return FP8_ERR_INVALID_ARG;
  *bytes = recipe != FP8_RECIPE_BLOCK ? (size_t)kMaxPartials * sizeof(float) : 0;
  return FP8_OK;
}

fp8_status fp8_quantize(const void *x, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_role role,
                        uint8_t *rowwise_out, uint8_t *colwise_out, float *row_scale,
                        float *row_scale_inv, float *col_scale, float *col_scale_inv,
                        void *workspace, size_t workspace_bytes, fp8_stream_t stream) {
  if (!valid_recipe(recipe) || !valid_role(role)) return FP8_ERR_INVALID_ARG;
  fp8_status st = check_dims(rows, cols);
  if (st != FP8_OK) return st;
  if (!rowwise_out && !colwise_out) return FP8_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (!x) return FP8_ERR_INVALID_ARG;
  const int mode = qmode_of(recipe, role);
  if ((rowwise_out || mode == 0) && (!row_scale || !row_scale_inv)) return FP8_ERR_INVALID_ARG;
  if (colwise_out && mode != 0 && (!col_scale || !col_scale_inv)) return FP8_ERR_INVALID_ARG;
  if (mode != 0 && !rowwise_out) row_scale = row_scale_inv = nullptr;
  if (mode == 0 && (!col_scale || !col_scale_inv)) col_scale = col_scale_inv = nullptr;
  if (!aligned16(x) || (rowwise_out && !aligned16(rowwise_out)) ||
      (colwise_out && !aligned16(colwise_out)))
    return FP8_ERR_ALIGN;
  size_t need = 0;
  fp8_quantize_workspace_size(recipe, rows, cols, &need);
  if (workspace_bytes < need || (need && !workspace)) return FP8_ERR_WORKSPACE;
  return from_cuda(launch_quantize(x, rows, cols, mode, format_of(role), rowwise_out, colwise_out,
                                   row_scale, row_scale_inv, col_scale, col_scale_inv,
                                   static_cast<float *>(workspace), cs(stream)));
}

fp8_status fp8_quantize_delayed(const void *x, int64_t rows, int64_t cols, fp8_role role,
                                uint8_t *rowwise_out, uint8_t *colwise_out, float *scale,
                                float *scale_inv, float *amax_history, int32_t history_len,
                                int64_t step, void *workspace, size_t workspace_bytes,
                                fp8_stream_t stream) {
  if (!valid_role(role) || history_len <= 0 || history_len > 1 << 20 || step < 0)
    return FP8_ERR_INVALID_ARG;
  fp8_status st = check_dims(rows, cols);
  if (st != FP8_OK) return st;
  if (!rowwise_out && !colwise_out) return FP8_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (!x || !scale || !scale_inv || !amax_history) return FP8_ERR_INVALID_ARG;
  if (!aligned16(x) || (rowwise_out && !aligned16(rowwise_out)) ||
      (colwise_out && !aligned16(colwise_out)))
    return FP8_ERR_ALIGN;
  if (workspace_bytes < (size_t)kMaxPartials * sizeof(float) || !workspace)
    return FP8_ERR_WORKSPACE;
  return from_cuda(launch_quantize_delayed(x, rows, cols, format_of(role), rowwise_out,
                                           colwise_out, scale, scale_inv, amax_history,
                                           history_len, step, static_cast<float *>(workspace),
                                           cs(stream)));
}

fp8_status fp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K, fp8_scaling scaling,
                                   size_t *bytes) {
  if (!bytes || M < 0 || N < 0 || K < 0 || scaling < 0 || scaling > 2) return FP8_ERR_INVALID_ARG;
  *bytes = gemm_workspace_bytes(M, N, K, scaling);
  return FP8_OK;
}

fp8_status fp8_gemm(const uint8_t *A, fp8_format a_fmt, const float *a_scale_inv, const uint8_t *B,
                    fp8_format b_fmt, const float *b_scale_inv, int64_t M, int64_t N, int64_t K,
                    fp8_scaling scaling, void *C, void *workspace, size_t workspace_bytes,
                    fp8_stream_t stream) {
  if (scaling < 0 || scaling > 2 || (a_fmt != 0 && a_fmt != 1) || (b_fmt != 0 && b_fmt != 1))
    return FP8_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return FP8_ERR_INVALID_ARG;
  if (M % 16 || N % 16 || K % 16) return FP8_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8_OK;
  if (!C || (K > 0 && (!A || !B || !a_scale_inv || !b_scale_inv))) return FP8_ERR_INVALID_ARG;
  if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B)))) return FP8_ERR_ALIGN;
  const size_t need = gemm_workspace_bytes(M, N, K, scaling);
  if (workspace_bytes < need || (need && !workspace)) return FP8_ERR_WORKSPACE;
  if (need && !aligned16(workspace)) return FP8_ERR_ALIGN;
  return from_cuda(launch_gemm(A, a_fmt, a_scale_inv, B, b_fmt, b_scale_inv, M, N, K, scaling, C,
                               workspace, cs(stream)));
}

// ---------------------------------------------------------------- weight cache
struct fp8_weight_cache {
  struct Entry {
    const void *w;
    int64_t O, K;
    fp8_recipe recipe;
    uint8_t *w_row, *w_col;
    float *row_scale, *row_scale_inv, *col_scale, *col_scale_inv;
    void *ws;
    size_t ws_bytes;
    uint64_t cycle;    // cycle in which the FP8 copy was last made (0 = never)
    uint64_t version;  // caller's weight version at that time
    float *hist;       // delayed scaling: amax history ring (caller-owned), else null
    int32_t hist_len;
    int64_t steps;     // delayed scaling: quantizations so far (ring position)
  };
  std::vector<Entry> entries;
  uint64_t cycle = 1;
};

fp8_status fp8_weight_cache_create(fp8_weight_cache **out) {
  if (!out) return FP8_ERR_INVALID_ARG;
  *out = new (std::nothrow) fp8_weight_cache();
  return *out ? FP8_OK : FP8_ERR_INVALID_ARG;
}

void fp8_weight_cache_destroy(fp8_weight_cache *cache) { delete cache; }

fp8_status fp8_weight_cache_register(fp8_weight_cache *cache, const void *w, int64_t O, int64_t K,
                                     fp8_recipe recipe, uint8_t *w_row, uint8_t *w_col,
                                     float *row_scale, float *row_scale_inv, float *col_scale,
                                     float *col_scale_inv, void *workspace, size_t workspace_bytes,
                                     fp8_weight_handle *out) {
  if (!cache || !out || !valid_recipe(recipe)) return FP8_ERR_INVALID_ARG;
  fp8_status st = check_dims(O, K);
  if (st != FP8_OK) return st;
  if (O == 0 || K == 0) return FP8_ERR_SHAPE;
  if (!w || !w_row || !w_col || !row_scale || !row_scale_inv || !col_scale || !col_scale_inv)
    return FP8_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(w_row) || !aligned16(w_col)) return FP8_ERR_ALIGN;
  size_t need = 0;
  fp8_quantize_workspace_size(recipe, O, K, &need);
  if (workspace_bytes < need || (need && !workspace)) return FP8_ERR_WORKSPACE;
  fp8_weight_cache::Entry e{w,         O,          K,         recipe,        w_row,
                            w_col,     row_scale,  row_scale_inv, col_scale, col_scale_inv,
                            workspace, workspace_bytes, 0,     0,             nullptr,
                            0,         0};
  cache->entries.push_back(e);
  *out = (fp8_weight_handle)(cache->entries.size() - 1);
  return FP8_OK;
}

fp8_status fp8_weight_cache_register_delayed(fp8_weight_cache *cache, const void *w, int64_t O,
                                             int64_t K, uint8_t *w_row, uint8_t *w_col,
                                             float *scale, float *scale_inv, float *amax_history,
                                             int32_t history_len, void *workspace,
                                             size_t workspace_bytes, fp8_weight_handle *out) {
  if (!amax_history || history_len <= 0 || history_len > 1 << 20) return FP8_ERR_INVALID_ARG;
  fp8_status st = fp8_weight_cache_register(cache, w, O, K, FP8_RECIPE_TENSORWISE, w_row, w_col,
                                            scale, scale_inv, scale, scale_inv, workspace,
                                            workspace_bytes, out);
  if (st != FP8_OK) return st;
  auto &e = cache->entries[*out];
  e.recipe = FP8_RECIPE_DELAYED;
  e.hist = amax_history;
  e.hist_len = history_len;
  return FP8_OK;
}

fp8_status fp8_weight_cache_begin_cycle(fp8_weight_cache *cache) {
  if (!cache) return FP8_ERR_INVALID_ARG;
  ++cache->cycle;
  return FP8_OK;
}

fp8_status fp8_weight_cache_get(fp8_weight_cache *cache, fp8_weight_handle h, uint64_t w_version,
                                int use_cache, fp8_stream_t stream, int *requantized) {
  if (requantized) *requantized = 0;
  if (!cache || h < 0 || (size_t)h >= cache->entries.size()) return FP8_ERR_INVALID_ARG;
  auto &e = cache->entries[h];
  if (use_cache && e.cycle == cache->cycle) {
    if (e.version != w_version) return FP8_ERR_STALE;
    return FP8_OK;  // is_first_microbatch=False: reuse the FP8 copy
  }
  fp8_status st;
  if (e.recipe == FP8_RECIPE_DELAYED) {
    st = fp8_quantize_delayed(e.w, e.O, e.K, FP8_ROLE_WEIGHT, e.w_row, e.w_col, e.row_scale,
                              e.row_scale_inv, e.hist, e.hist_len, e.steps, e.ws, e.ws_bytes,
                              stream);
    if (st == FP8_OK) ++e.steps;
  } else {
    st = fp8_quantize(e.w, e.O, e.K, e.recipe, FP8_ROLE_WEIGHT, e.w_row, e.w_col, e.row_scale,
                      e.row_scale_inv, e.col_scale, e.col_scale_inv, e.ws, e.ws_bytes, stream);
  }
  if (st != FP8_OK) return st;
  e.cycle = cache->cycle;
  e.version = w_version;
  if (requantized) *requantized = 1;
  return FP8_OK;
}

// ---------------------------------------------------------------- linear layer
namespace {

struct CtxLayout {
  size_t xq_col, scale, scale_inv, total;
};
CtxLayout ctx_layout(fp8_recipe recipe, int64_t N, int64_t K) {
  recipe = act_recipe(recipe);
  CtxLayout L;
  const int64_t ns = scale_elems(recipe, FP8_ROLE_ACT, N, K, 1);
  L.xq_col = 0;
  L.scale = align_up((size_t)N * K);
  L.scale_inv = L.scale + align_up((size_t)ns * 4);
  L.total = L.scale_inv + align_up((size_t)ns * 4);
  return L;
}

fp8_scaling fwd_scaling(fp8_recipe r) {
  return r == FP8_RECIPE_BLOCK ? FP8_SCALING_1x128_128x128 : FP8_SCALING_TENSOR;
}
fp8_scaling wgrad_scaling(fp8_recipe r) {
  return r == FP8_RECIPE_BLOCK ? FP8_SCALING_1x128_1x128 : FP8_SCALING_TENSOR;
}

size_t fwd_ws(fp8_recipe r, int64_t N, int64_t K, int64_t O) {
  r = act_recipe(r);
  const int64_t ns = scale_elems(r, FP8_ROLE_ACT, N, K, 0);
  size_t qws = 0;
  fp8_quantize_workspace_size(r, N, K, &qws);
  return align_up((size_t)N * K) + 2 * align_up((size_t)ns * 4) + align_up(qws) +
         align_up(gemm_workspace_bytes(N, O, K, fwd_scaling(r)));
}
size_t bwd_ws(fp8_recipe r, int64_t N, int64_t K, int64_t O) {
  r = act_recipe(r);
  const int64_t nr = scale_elems(r, FP8_ROLE_GRAD, N, O, 0);
  const int64_t nc = scale_elems(r, FP8_ROLE_GRAD, N, O, 1);
  size_t qws = 0;
  fp8_quantize_workspace_size(r, N, O, &qws);
  const size_t g = std::max(gemm_workspace_bytes(N, K, O, fwd_scaling(r)),
                            gemm_workspace_bytes(O, K, N, wgrad_scaling(r)));
  return 2 * align_up((size_t)N * O) + 2 * align_up((size_t)nr * 4) + 2 * align_up((size_t)nc * 4) +
         align_up(qws) + align_up(g);
}

}  // namespace

fp8_status fp8_linear_ctx_size(fp8_recipe recipe, int64_t N, int64_t K, size_t *bytes) {
  if (!bytes || !valid_linear_recipe(recipe) || N < 0 || K < 0) return FP8_ERR_INVALID_ARG;
  *bytes = ctx_layout(recipe, N, K).total;
  return FP8_OK;
}

fp8_status fp8_linear_workspace_size(fp8_recipe recipe, int64_t N, int64_t K, int64_t O,
                                     size_t *bytes) {
  if (!bytes || !valid_linear_recipe(recipe) || N < 0 || K < 0 || O < 0)
    return FP8_ERR_INVALID_ARG;
  *bytes = std::max(fwd_ws(recipe, N, K, O), bwd_ws(recipe, N, K, O));
  return FP8_OK;
}

}  // extern "C"

namespace {
// x_partials: the tensorwise first pass over X already ran (fp8_amax_partials)
fp8_status linear_fwd_impl(const void *X, int64_t N, int64_t K, fp8_weight_cache *cache,
                           fp8_weight_handle h, fp8_recipe recipe, void *Y, void *ctx, void *ws,
                           size_t ws_bytes, fp8_stream_t stream, const float *x_partials) {
  if (!cache || h < 0 || (size_t)h >= cache->entries.size() || !valid_linear_recipe(recipe))
    return FP8_ERR_INVALID_ARG;
  const auto &e = cache->entries[h];
  if (e.recipe != recipe || e.K != K) return FP8_ERR_INVALID_ARG;
  const fp8_recipe ar = act_recipe(recipe);
  fp8_status st = check_dims(N, K);
  if (st != FP8_OK) return st;
  if (e.cycle != cache->cycle) return FP8_ERR_STALE;
  if (N == 0) return FP8_OK;
  if (!X || !Y || !ctx || !ws) return FP8_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Y) || !aligned16(ctx) || !aligned16(ws)) return FP8_ERR_ALIGN;
  const int64_t O = e.O;
  if (ws_bytes < fwd_ws(recipe, N, K, O)) return FP8_ERR_WORKSPACE;
  const CtxLayout L = ctx_layout(recipe, N, K);
  uint8_t *c = static_cast<uint8_t *>(ctx);
  const int64_t ns = scale_elems(ar, FP8_ROLE_ACT, N, K, 0);
  size_t qws = 0;
  fp8_quantize_workspace_size(ar, N, K, &qws);
  Carver w(ws);
  uint8_t *xq_row = w.take<uint8_t>((size_t)N * K);
  float *rs = w.take<float>((size_t)ns * 4);
  float *rsi = w.take<float>((size_t)ns * 4);
  float *part = w.take<float>(qws);
  void *gws = w.take<void>(gemm_workspace_bytes(N, O, K, fwd_scaling(recipe)));
  if (x_partials) {
    if (ar != FP8_RECIPE_TENSORWISE) return FP8_ERR_UNSUPPORTED;
    st = from_cuda(launch_quantize(X, N, K, 0, FP8_FORMAT_E4M3, xq_row, c + L.xq_col, rs, rsi,
                                   reinterpret_cast<float *>(c + L.scale),
                                   reinterpret_cast<float *>(c + L.scale_inv),
                                   const_cast<float *>(x_partials), cs(stream), true));
  } else {
    st = fp8_quantize(X, N, K, ar, FP8_ROLE_ACT, xq_row, c + L.xq_col, rs, rsi,
                      reinterpret_cast<float *>(c + L.scale),
                      reinterpret_cast<float *>(c + L.scale_inv), part, qws, stream);
  }
  if (st != FP8_OK) return st;
  return fp8_gemm(xq_row, FP8_FORMAT_E4M3, rsi, e.w_row, FP8_FORMAT_E4M3, e.row_scale_inv, N, O, K,
                  fwd_scaling(recipe), Y, gws, gemm_workspace_bytes(N, O, K, fwd_scaling(recipe)),
                  stream);
}

// dy_partials: the tensorwise first pass over dY already ran (fp8_amax_partials)
fp8_status linear_bwd_impl(const void *dY, int64_t N, int64_t O, const void *ctx,
                           fp8_weight_cache *cache, fp8_weight_handle h, fp8_recipe recipe,
                           void *dX, void *dW, void *ws, size_t ws_bytes, fp8_stream_t stream,
                           const float *dy_partials) {
  if (!cache || h < 0 || (size_t)h >= cache->entries.size() || !valid_linear_recipe(recipe))
    return FP8_ERR_INVALID_ARG;
  const auto &e = cache->entries[h];
  if (e.recipe != recipe || e.O != O) return FP8_ERR_INVALID_ARG;
  const fp8_recipe ar = act_recipe(recipe);
  fp8_status st = check_dims(N, O);
  if (st != FP8_OK) return st;
  if (e.cycle != cache->cycle) return FP8_ERR_STALE;
  const int64_t K = e.K;
  if (N == 0) return FP8_OK;  // dW of an empty batch is not written
  if (!dY || !ctx || !dW || !ws) return FP8_ERR_INVALID_ARG;
  if (!aligned16(dY) || !aligned16(ctx) || !aligned16(dW) || !aligned16(ws) ||
      (dX && !aligned16(dX)))
    return FP8_ERR_ALIGN;
  if (ws_bytes < bwd_ws(recipe, N, K, O)) return FP8_ERR_WORKSPACE;
  const CtxLayout L = ctx_layout(recipe, N, K);
  const uint8_t *c = static_cast<const uint8_t *>(ctx);
  const int64_t nr = scale_elems(ar, FP8_ROLE_GRAD, N, O, 0);
  const int64_t nc = scale_elems(ar, FP8_ROLE_GRAD, N, O, 1);
  size_t qws = 0;
  fp8_quantize_workspace_size(ar, N, O, &qws);
  const size_t gbytes = std::max(gemm_workspace_bytes(N, K, O, fwd_scaling(recipe)),
                                 gemm_workspace_bytes(O, K, N, wgrad_scaling(recipe)));
  Carver w(ws);
  uint8_t *g_row = w.take<uint8_t>((size_t)N * O);
  uint8_t *g_col = w.take<uint8_t>((size_t)N * O);
  float *grs = w.take<float>((size_t)nr * 4);
  float *grsi = w.take<float>((size_t)nr * 4);
  float *gcs = w.take<float>((size_t)nc * 4);
  float *gcsi = w.take<float>((size_t)nc * 4);
  float *part = w.take<float>(qws);
  void *gws = w.take<void>(gbytes);
  if (dy_partials) {
    if (ar != FP8_RECIPE_TENSORWISE) return FP8_ERR_UNSUPPORTED;
    st = from_cuda(launch_quantize(dY, N, O, 0, FP8_FORMAT_E5M2, g_row, g_col, grs, grsi, gcs,
                                   gcsi, const_cast<float *>(dy_partials), cs(stream), true));
  } else {
    st = fp8_quantize(dY, N, O, ar, FP8_ROLE_GRAD, g_row, g_col, grs, grsi, gcs, gcsi, part, qws,
                      stream);
  }
  if (st != FP8_OK) return st;
  if (dX) {
    st = fp8_gemm(g_row, FP8_FORMAT_E5M2, grsi, e.w_col, FP8_FORMAT_E4M3, e.col_scale_inv, N, K, O,
                  fwd_scaling(recipe), dX, gws, gbytes, stream);
    if (st != FP8_OK) return st;
  }
  return fp8_gemm(g_col, FP8_FORMAT_E5M2, gcsi, c + L.xq_col, FP8_FORMAT_E4M3,
                  reinterpret_cast<const float *>(c + L.scale_inv), O, K, N, wgrad_scaling(recipe),
                  dW, gws, gbytes, stream);
}
}  // namespace

extern "C" {

fp8_status fp8_linear_fwd(const void *X, int64_t N, int64_t K, fp8_weight_cache *cache,
                          fp8_weight_handle h, fp8_recipe recipe, void *Y, void *ctx, void *ws,
                          size_t ws_bytes, fp8_stream_t stream) {
  return linear_fwd_impl(X, N, K, cache, h, recipe, Y, ctx, ws, ws_bytes, stream, nullptr);
}

fp8_status fp8_linear_bwd(const void *dY, int64_t N, int64_t O, const void *ctx,
                          fp8_weight_cache *cache, fp8_weight_handle h, fp8_recipe recipe, void *dX,
                          void *dW, void *ws, size_t ws_bytes, fp8_stream_t stream) {
  return linear_bwd_impl(dY, N, O, ctx, cache, h, recipe, dX, dW, ws, ws_bytes, stream, nullptr);
}

fp8_status fp8_amax_partials(const void *x, int64_t rows, int64_t cols, void *partials,
                             size_t partials_bytes, fp8_stream_t stream) {
  fp8_status st = check_dims(rows, cols);
  if (st != FP8_OK) return st;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (!x || !partials) return FP8_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(partials)) return FP8_ERR_ALIGN;
  size_t need = 0;
  fp8_quantize_workspace_size(FP8_RECIPE_TENSORWISE, rows, cols, &need);
  if (partials_bytes < need) return FP8_ERR_WORKSPACE;
  return from_cuda(launch_amax_partials(x, rows, cols, static_cast<float *>(partials), cs(stream)));
}

fp8_status fp8_linear_fwd_after_amax(const void *X, const void *x_partials, int64_t N, int64_t K,
                                     fp8_weight_cache *cache, fp8_weight_handle h,
                                     fp8_recipe recipe, void *Y, void *ctx, void *ws,
                                     size_t ws_bytes, fp8_stream_t stream) {
  if (!x_partials && N > 0) return FP8_ERR_INVALID_ARG;
  if (x_partials && !aligned16(x_partials)) return FP8_ERR_ALIGN;
  return linear_fwd_impl(X, N, K, cache, h, recipe, Y, ctx, ws, ws_bytes, stream,
                         static_cast<const float *>(x_partials));
}

fp8_status fp8_linear_bwd_after_amax(const void *dY, const void *dy_partials, int64_t N, int64_t O,
                                     const void *ctx, fp8_weight_cache *cache, fp8_weight_handle h,
                                     fp8_recipe recipe, void *dX, void *dW, void *ws,
                                     size_t ws_bytes, fp8_stream_t stream) {
  if (!dy_partials && N > 0) return FP8_ERR_INVALID_ARG;
  if (dy_partials && !aligned16(dy_partials)) return FP8_ERR_ALIGN;
  return linear_bwd_impl(dY, N, O, ctx, cache, h, recipe, dX, dW, ws, ws_bytes, stream,
                         static_cast<const float *>(dy_partials));
}

// ---------------------------------------------------------------- fused producers
namespace {
fp8_status check_block_outputs(const void *x, int64_t rows, int64_t cols, fp8_recipe recipe,
                               uint8_t *row, uint8_t *col, float *rs, float *rsi, float *cs,
                               float *csi) {
  if (recipe != FP8_RECIPE_BLOCK) return FP8_ERR_UNSUPPORTED;
  fp8_status st = check_dims(rows, cols);
  if (st != FP8_OK) return st;
  if (!row && !col) return FP8_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (!x || (row && (!rs || !rsi)) || (col && (!cs || !csi))) return FP8_ERR_INVALID_ARG;
  if (!aligned16(x) || (row && !aligned16(row)) || (col && !aligned16(col))) return FP8_ERR_ALIGN;
  return FP8_OK;
}
}  // namespace

fp8_status fp8_gelu_quantize(const void *H, int64_t rows, int64_t cols, fp8_recipe recipe,
                             uint8_t *rowwise_out, uint8_t *colwise_out, float *row_scale,
                             float *row_scale_inv, float *col_scale, float *col_scale_inv,
                             fp8_stream_t stream) {
  fp8_status st = check_block_outputs(H, rows, cols, recipe, rowwise_out, colwise_out, row_scale,
                                      row_scale_inv, col_scale, col_scale_inv);
  if (st != FP8_OK || rows == 0 || cols == 0) return st;
  return from_cuda(launch_gelu_quantize(H, nullptr, rows, cols, 0, rowwise_out, colwise_out,
                                        row_scale, row_scale_inv, col_scale, col_scale_inv,
                                        cs(stream)));
}

fp8_status fp8_gelu_bwd_quantize(const void *dA, const void *H, int64_t rows, int64_t cols,
                                 fp8_recipe recipe, uint8_t *rowwise_out, uint8_t *colwise_out,
                                 float *row_scale, float *row_scale_inv, float *col_scale,
                                 float *col_scale_inv, fp8_stream_t stream) {
  fp8_status st = check_block_outputs(dA, rows, cols, recipe, rowwise_out, colwise_out, row_scale,
                                      row_scale_inv, col_scale, col_scale_inv);
  if (st != FP8_OK || rows == 0 || cols == 0) return st;
  if (!H) return FP8_ERR_INVALID_ARG;
  if (!aligned16(H)) return FP8_ERR_ALIGN;
  return from_cuda(launch_gelu_quantize(dA, H, rows, cols, 1, rowwise_out, colwise_out,
                                        row_scale, row_scale_inv, col_scale, col_scale_inv,
                                        cs(stream)));
}

fp8_status fp8_linear_ctx_layout(fp8_recipe recipe, int64_t N, int64_t K, void *ctx,
                                 uint8_t **xq_col, float **col_scale, float **col_scale_inv) {
  if (!valid_linear_recipe(recipe) || N < 0 || K < 0 || !ctx || !xq_col || !col_scale ||
      !col_scale_inv)
    return FP8_ERR_INVALID_ARG;
  const CtxLayout L = ctx_layout(recipe, N, K);
  uint8_t *c = static_cast<uint8_t *>(ctx);
  *xq_col = c + L.xq_col;
  *col_scale = reinterpret_cast<float *>(c + L.scale);
  *col_scale_inv = reinterpret_cast<float *>(c + L.scale_inv);
  return FP8_OK;
}

fp8_status fp8_linear_fwd_quantized(const uint8_t *xq_row, const float *xq_row_scale_inv,
                                    int64_t N, int64_t K, fp8_weight_cache *cache,
                                    fp8_weight_handle h, fp8_recipe recipe, void *Y, void *ws,
                                    size_t ws_bytes, fp8_stream_t stream) {
  if (!cache || h < 0 || (size_t)h >= cache->entries.size() || !valid_linear_recipe(recipe))
    return FP8_ERR_INVALID_ARG;
  const auto &e = cache->entries[h];
  if (e.recipe != recipe || e.K != K) return FP8_ERR_INVALID_ARG;
  fp8_status st = check_dims(N, K);
  if (st != FP8_OK) return st;
  if (e.cycle != cache->cycle) return FP8_ERR_STALE;
  if (N == 0) return FP8_OK;
  if (!xq_row || !xq_row_scale_inv || !Y || !ws) return FP8_ERR_INVALID_ARG;
  const size_t g = gemm_workspace_bytes(N, e.O, K, fwd_scaling(recipe));
  if (ws_bytes < g) return FP8_ERR_WORKSPACE;
  return fp8_gemm(xq_row, FP8_FORMAT_E4M3, xq_row_scale_inv, e.w_row, FP8_FORMAT_E4M3,
                  e.row_scale_inv, N, e.O, K, fwd_scaling(recipe), Y, ws, ws_bytes, stream);
}

fp8_status fp8_linear_bwd_quantized(const uint8_t *gq_row, const float *gq_row_scale_inv,
                                    const uint8_t *gq_col, const float *gq_col_scale_inv,
                                    int64_t N, int64_t O, const void *ctx, fp8_weight_cache *cache,
                                    fp8_weight_handle h, fp8_recipe recipe, void *dX, void *dW,
                                    void *ws, size_t ws_bytes, fp8_stream_t stream) {
  if (!cache || h < 0 || (size_t)h >= cache->entries.size() || !valid_linear_recipe(recipe))
    return FP8_ERR_INVALID_ARG;
  const auto &e = cache->entries[h];
  if (e.recipe != recipe || e.O != O) return FP8_ERR_INVALID_ARG;
  fp8_status st = check_dims(N, O);
  if (st != FP8_OK) return st;
  if (e.cycle != cache->cycle) return FP8_ERR_STALE;
  const int64_t K = e.K;
  if (N == 0) return FP8_OK;
  if (!gq_col || !gq_col_scale_inv || !ctx || !dW || !ws || (dX && (!gq_row || !gq_row_scale_inv)))
    return FP8_ERR_INVALID_ARG;
  const size_t gbytes = std::max(gemm_workspace_bytes(N, K, O, fwd_scaling(recipe)),
                                 gemm_workspace_bytes(O, K, N, wgrad_scaling(recipe)));
  if (ws_bytes < gbytes) return FP8_ERR_WORKSPACE;
  const CtxLayout L = ctx_layout(recipe, N, K);
  const uint8_t *c = static_cast<const uint8_t *>(ctx);
  if (dX) {
    st = fp8_gemm(gq_row, FP8_FORMAT_E5M2, gq_row_scale_inv, e.w_col, FP8_FORMAT_E4M3,
                  e.col_scale_inv, N, K, O, fwd_scaling(recipe), dX, ws, ws_bytes, stream);
    if (st != FP8_OK) return st;
  }
  return fp8_gemm(gq_col, FP8_FORMAT_E5M2, gq_col_scale_inv, c + L.xq_col, FP8_FORMAT_E4M3,
                  reinterpret_cast<const float *>(c + L.scale_inv), O, K, N,
                  wgrad_scaling(recipe), dW, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- glue + status
fp8_status fp8_gelu_fwd(const void *H, void *A, int64_t n, fp8_stream_t stream) {
  if (n < 0) return FP8_ERR_INVALID_ARG;
  if (n % 8) return FP8_ERR_SHAPE;
  if (n == 0) return FP8_OK;
  if (!H || !A) return FP8_ERR_INVALID_ARG;
  if (!aligned16(H) || !aligned16(A)) return FP8_ERR_ALIGN;
  return from_cuda(launch_gelu_fwd(H, A, n, cs(stream)));
}

fp8_status fp8_gelu_bwd(const void *dA, const void *H, void *dH, int64_t n, fp8_stream_t stream) {
  if (n < 0) return FP8_ERR_INVALID_ARG;
  if (n % 8) return FP8_ERR_SHAPE;
  if (n == 0) return FP8_OK;
  if (!dA || !H || !dH) return FP8_ERR_INVALID_ARG;
  if (!aligned16(dA) || !aligned16(H) || !aligned16(dH)) return FP8_ERR_ALIGN;
  return from_cuda(launch_gelu_bwd(dA, H, dH, n, cs(stream)));
}

fp8_status fp8_grad_accumulate(float *acc, const void *dW, int64_t n, fp8_stream_t stream) {
  if (n < 0) return FP8_ERR_INVALID_ARG;
  if (n % 8) return FP8_ERR_SHAPE;
  if (n == 0) return FP8_OK;
  if (!acc || !dW) return FP8_ERR_INVALID_ARG;
  if (!aligned16(acc) || !aligned16(dW)) return FP8_ERR_ALIGN;
  return from_cuda(launch_grad_accumulate(acc, dW, n, cs(stream)));
}

fp8_status fp8_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto &r : g_prof) {
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  g_prof.clear();
  g_prof_on = true;
  return FP8_OK;
}

fp8_status fp8_profile_end(fp8_kernel_stat *out, int cap, int *n) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = false;
  std::map<std::tuple<std::string, int64_t, int64_t, int64_t>, fp8_kernel_stat> agg;
  fp8_status st = FP8_OK;
  for (auto &r : g_prof) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
      st = FP8_ERR_CUDA;
      continue;
    }
    fp8_kernel_stat &k = agg[std::make_tuple(std::string(r.name), r.m, r.n, r.k)];
    if (k.launches == 0) {
      std::memset(&k, 0, sizeof(k));
      std::strncpy(k.name, r.name, sizeof(k.name) - 1);
      k.m = r.m;
      k.n = r.n;
      k.k = r.k;
    }
    k.launches += 1;
    k.total_ms += ms;
    k.bytes += r.bytes;
    k.flops += r.flops;
  }
  for (auto &r : g_prof) {
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  g_prof.clear();
  if (n) *n = (int)agg.size();
  int i = 0;
  for (auto &kv : agg) {
    if (out && i < cap) out[i] = kv.second;
    ++i;
  }
  return st;
}

// ---------------------------------------------------------------- host-buffer steps
struct fp8_host_pipeline {
  int device = 0;
  cudaStream_t copy_in = nullptr, compute = nullptr, copy_out = nullptr;
  // Per slot, the forward and the backward halves of a step are tracked
  // apart, so that dY streams in while the forward runs and Y streams out
  // while the backward runs.
  struct Slot {
    cudaEvent_t in_fwd = nullptr;    // X and W are on the device
    cudaEvent_t in_bwd = nullptr;    // dY is on the device
    cudaEvent_t fwd_done = nullptr;  // the forward's kernels (the last readers of X, W) finished
    cudaEvent_t bwd_done = nullptr;  // the backward's kernels (the last readers of dY) finished
    cudaEvent_t out_fwd = nullptr;   // Y is on the host
    cudaEvent_t out_bwd = nullptr;   // dX and dW are on the host
  };
  std::vector<Slot> slots;
  cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
};

void fp8_host_pipeline_destroy(fp8_host_pipeline *p) {
  if (!p) return;
  for (auto &s : p->slots)
    for (cudaEvent_t e : {s.in_fwd, s.in_bwd, s.fwd_done, s.bwd_done, s.out_fwd, s.out_bwd})
      if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : {p->fork_ev, p->join_ev})
    if (e) cudaEventDestroy(e);
  for (cudaStream_t s : {p->copy_in, p->compute, p->copy_out})
    if (s) cudaStreamDestroy(s);
  delete p;
}

fp8_status fp8_host_pipeline_create(int slots, fp8_host_pipeline **out) {
  if (!out || slots <= 0 || slots > 4096) return FP8_ERR_INVALID_ARG;
  *out = nullptr;
  auto *p = new (std::nothrow) fp8_host_pipeline();
  if (!p) return FP8_ERR_INVALID_ARG;
  bool ok = cudaGetDevice(&p->device) == cudaSuccess;
  for (cudaStream_t *s : {&p->copy_in, &p->compute, &p->copy_out})
    ok = ok && cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) == cudaSuccess;
  p->slots.resize((size_t)slots);
  for (auto &s : p->slots)
    for (cudaEvent_t *e : {&s.in_fwd, &s.in_bwd, &s.fwd_done, &s.bwd_done, &s.out_fwd, &s.out_bwd})
      ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
  for (cudaEvent_t *e : {&p->fork_ev, &p->join_ev})
    ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    fp8_host_pipeline_destroy(p);
    return FP8_ERR_CUDA;
  }
  *out = p;
  return FP8_OK;
}

fp8_status fp8_linear_step_host(fp8_host_pipeline *p, int slot, int64_t N,
                                const fp8_linear_host_io *host, const fp8_linear_device_io *dev,
                                fp8_weight_cache *cache, fp8_weight_handle h, fp8_recipe recipe,
                                uint64_t w_version) {
  // every check the enqueued calls would make, before anything is enqueued
  if (!p || slot < 0 || (size_t)slot >= p->slots.size() || !host || !dev || !cache || h < 0 ||
      (size_t)h >= cache->entries.size() || !valid_linear_recipe(recipe))
    return FP8_ERR_INVALID_ARG;
  const auto &e = cache->entries[h];
  if (e.recipe != recipe) return FP8_ERR_INVALID_ARG;
  const int64_t K = e.K, O = e.O;
  fp8_status st = check_dims(N, K);
  if (st != FP8_OK) return st;
  if (N == 0) return FP8_OK;
  if (!host->X || !host->W || !host->dY || !host->Y || !host->dW || !dev->X || !dev->dY ||
      !dev->Y || !dev->dW || !dev->ctx || !dev->ws)
    return FP8_ERR_INVALID_ARG;
  if (!aligned16(dev->X) || !aligned16(dev->dY) || !aligned16(dev->Y) || !aligned16(dev->dW) ||
      !aligned16(dev->ctx) || !aligned16(dev->ws) || (dev->dX && !aligned16(dev->dX)))
    return FP8_ERR_ALIGN;
  size_t need = 0;
  fp8_linear_workspace_size(recipe, N, K, O, &need);
  if (dev->ws_bytes < need) return FP8_ERR_WORKSPACE;
  if (e.cycle == cache->cycle && e.version != w_version) return FP8_ERR_STALE;
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != p->device) return FP8_ERR_INVALID_ARG;

  auto &s = p->slots[(size_t)slot];
  const size_t xb = (size_t)N * K * 2, wb = (size_t)O * K * 2, gb = (size_t)N * O * 2;
  // copy-in: X and W once this slot's previous forward has read them, dY once
  // its previous backward has
  bool ok = cudaStreamWaitEvent(p->copy_in, s.fwd_done, 0) == cudaSuccess &&
            cudaMemcpyAsync(dev->X, host->X, xb, cudaMemcpyHostToDevice, p->copy_in) ==
                cudaSuccess &&
            cudaMemcpyAsync(const_cast<void *>(e.w), host->W, wb, cudaMemcpyHostToDevice,
                            p->copy_in) == cudaSuccess &&
            cudaEventRecord(s.in_fwd, p->copy_in) == cudaSuccess &&
            cudaStreamWaitEvent(p->copy_in, s.bwd_done, 0) == cudaSuccess &&
            cudaMemcpyAsync(dev->dY, host->dY, gb, cudaMemcpyHostToDevice, p->copy_in) ==
                cudaSuccess &&
            cudaEventRecord(s.in_bwd, p->copy_in) == cudaSuccess &&
            // forward: its inputs are in, and the previous Y has left the device
            cudaStreamWaitEvent(p->compute, s.in_fwd, 0) == cudaSuccess &&
            cudaStreamWaitEvent(p->compute, s.out_fwd, 0) == cudaSuccess;
  if (!ok) return FP8_ERR_CUDA;
  fp8_stream_t cst = reinterpret_cast<fp8_stream_t>(p->compute);
  st = fp8_weight_cache_get(cache, h, w_version, 1, cst, nullptr);
  if (st == FP8_OK)
    st = fp8_linear_fwd(dev->X, N, K, cache, h, recipe, dev->Y, dev->ctx, dev->ws, dev->ws_bytes,
                        cst);
  if (st != FP8_OK) return st;
  // backward: dY is in, and the previous dX and dW have left the device
  ok = cudaEventRecord(s.fwd_done, p->compute) == cudaSuccess &&
       cudaStreamWaitEvent(p->compute, s.in_bwd, 0) == cudaSuccess &&
       cudaStreamWaitEvent(p->compute, s.out_bwd, 0) == cudaSuccess;
  if (!ok) return FP8_ERR_CUDA;
  st = fp8_linear_bwd(dev->dY, N, O, dev->ctx, cache, h, recipe, dev->dX, dev->dW, dev->ws,
                      dev->ws_bytes, cst);
  if (st != FP8_OK) return st;
  // copy-out: Y as soon as the forward is done, dX and dW after the backward
  ok = cudaEventRecord(s.bwd_done, p->compute) == cudaSuccess &&
       cudaStreamWaitEvent(p->copy_out, s.fwd_done, 0) == cudaSuccess &&
       cudaMemcpyAsync(host->Y, dev->Y, gb, cudaMemcpyDeviceToHost, p->copy_out) == cudaSuccess &&
       cudaEventRecord(s.out_fwd, p->copy_out) == cudaSuccess &&
       cudaStreamWaitEvent(p->copy_out, s.bwd_done, 0) == cudaSuccess &&
       (!host->dX || !dev->dX ||
        cudaMemcpyAsync(host->dX, dev->dX, xb, cudaMemcpyDeviceToHost, p->copy_out) ==
            cudaSuccess) &&
       cudaMemcpyAsync(host->dW, dev->dW, wb, cudaMemcpyDeviceToHost, p->copy_out) ==
           cudaSuccess &&
       cudaEventRecord(s.out_bwd, p->copy_out) == cudaSuccess;
  return ok ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status fp8_host_pipeline_fork(fp8_host_pipeline *p, fp8_stream_t s) {
  if (!p) return FP8_ERR_INVALID_ARG;
  bool ok = cudaEventRecord(p->fork_ev, cs(s)) == cudaSuccess;
  for (cudaStream_t t : {p->copy_in, p->compute, p->copy_out})
    ok = ok && cudaStreamWaitEvent(t, p->fork_ev, 0) == cudaSuccess;
  return ok ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status fp8_host_pipeline_join(fp8_host_pipeline *p, fp8_stream_t s) {
  if (!p) return FP8_ERR_INVALID_ARG;
  bool ok = true;
  for (cudaStream_t t : {p->copy_in, p->compute, p->copy_out})
    ok = ok && cudaEventRecord(p->join_ev, t) == cudaSuccess &&
         cudaStreamWaitEvent(cs(s), p->join_ev, 0) == cudaSuccess;
  return ok ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status fp8_host_pipeline_sync(fp8_host_pipeline *p) {
  if (!p) return FP8_ERR_INVALID_ARG;
  bool ok = true;
  for (cudaStream_t t : {p->copy_in, p->compute, p->copy_out})
    ok = ok && cudaStreamSynchronize(t) == cudaSuccess;
  return ok ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status fp8_debug_wait_timeout(uint64_t limit_ns, fp8_stream_t stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return FP8_ERR_INVALID_ARG;
  return from_cuda(launch_wait_timeout_probe(limit_ns, cs(stream)));
}

fp8_status fp8_get_device_status(fp8_stream_t stream) {
  unsigned s = 0, q = 0;
  if (gemm_read_status(&s, cs(stream)) != cudaSuccess) return FP8_ERR_CUDA;
  if (quant_read_status(&q) != cudaSuccess) return FP8_ERR_CUDA;
  return (fp8_status)(s ? s : q);
}

}  // extern "C"
