// api.cu -- the C ABI of libexl3 (declared in include/exl3.h): argument
// validation, workspace layout and kernel dispatch.  No entry point
// allocates device memory or synchronises the caller's stream (except the
// test helper exl3_check_device_error).
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "exl3_common.cuh"

// ---- kernels (other translation units)
cudaError_t exl3_launch_decode_tile(const uint16_t *trellis, int n, int K, int tk0, int tk_cnt, int tn0,
                                    int tn_cnt, uint16_t *w_out, int64_t ld, cudaStream_t s);
cudaError_t exl3_launch_reconstruct_t(const uint16_t *trellis, int k, int n, int K, uint16_t *wt,
                                      cudaStream_t s);
cudaError_t exl3_launch_input_rht(const uint16_t *x, int M, int k, const uint16_t *suh, void *out,
                                  bool f32out, cudaStream_t s, float *xsum = nullptr);
cudaError_t exl3_launch_gemv_m1(const uint16_t *x, const uint16_t *trellis, const uint16_t *suh,
                                const uint16_t *svh, int k, int n, int K, void *y, bool f32out,
                                float *partials, int *counters, int *err, int grid, cudaStream_t s,
                                bool prefetch = false);
cudaError_t exl3_launch_gemv_m1_bias(const uint16_t *x, const uint16_t *trellis, const uint16_t *suh,
                                     const uint16_t *svh, const uint16_t *bias, int k, int n, int K, void *y,
                                     bool f32out, float *partials, int *counters, int *err, int grid,
                                     cudaStream_t s, bool prefetch);
void exl3_gemv_plan(int k, int n, int K, int *grid, size_t *partial_floats);
bool exl3_gemv_fits(int k, int n, int K);
cudaError_t exl3_launch_copy_in(const void *src, void *dst, size_t bytes, cudaStream_t s, bool chained);
int exl3_launch_gemm_tc(const uint16_t *xh, const uint16_t *wt, int M, int n, int k, const uint16_t *svh,
                        void *y, bool f32out, const float *row_scale, float pre, int *err, cudaStream_t s,
                        bool q8 = false, int32_t *acc_out = nullptr, const uint16_t *bias = nullptr);
cudaError_t exl3_launch_quant_act(const uint16_t *x, int M, int k, const uint16_t *suh, uint16_t *qh,
                                  int8_t *q8, float *row_scale, cudaStream_t s);
cudaError_t exl3_launch_reconstruct_q8_t(const uint16_t *trellis, int k, int n, int K, uint16_t *wq,
                                         cudaStream_t s);
int exl3_fused_tc_splits(int k, int n);
int exl3_launch_fused_tc(const uint16_t *xh, const float *xsum, const uint16_t *trellis, const uint16_t *svh, int M,
                         int k, int n, int K, void *y, bool f32out, float *partials, int *counters, int *err,
                         int splits, cudaStream_t s, int npad_fixed, const uint16_t *bias = nullptr);

cudaError_t exl3_launch_moe_remap(const int32_t *ids, int U, int E, int *counts, int *offsets, int *perm, int *pos,
                                  int *mtiles, int *n_mtiles, int max_mtiles, int cap, int *chunk_tab, int *err,
                                  cudaStream_t s);
int exl3_moe_remap_chunk(int E);
cudaError_t exl3_launch_moe_gather(const uint16_t *x, int U, int hidden, int topk, const int *perm, const int *offsets,
                                   int E, const int32_t *ids, const uint16_t *suh13, uint16_t *xg, uint16_t *xu,
                                   cudaStream_t s);
cudaError_t exl3_launch_moe_combine(const float *d, const int *pos, int T, int topk, int hidden, void *y,
                                    bool f32out, cudaStream_t s);
bool exl3_moe_gemv_plan(int U, int nslots, int k, int n, int K, int *grid, size_t *partial_floats, int *blocks,
                        int *xops = nullptr);
bool exl3_gemv_shards_plan(int S, int k, int n, int K, int *grid, size_t *partial_floats, int *blocks);
bool exl3_gemv_shards_var_plan(int S, int k, const int *n, int K, int *grid, size_t *partial_floats, int *blocks);
cudaError_t exl3_launch_gemv_shards_var(const uint16_t *x, int S, int k, const int *n, int K, const uint16_t *trellis,
                                        const uint16_t *suh, const uint16_t *svh, void *y, bool f32out,
                                        float *partials, int *counters, int *err, cudaStream_t s, bool prefetch);
cudaError_t exl3_launch_gemv_shards(const uint16_t *x, int S, int k, int n, int K, const uint16_t *trellis,
                                    const uint16_t *suh, const uint16_t *svh, void *y, bool f32out,
                                    float *partials, int *counters, int *err, cudaStream_t s, bool prefetch);
cudaError_t exl3_launch_moe_gemv(const uint16_t *x, const float *act_in, int *pos_out, const int32_t *ids,
                                 const float *weights, int U, int topk, int E, int nslots, int k, int n, int K,
                                 const uint16_t *trellis, const uint16_t *suh, const uint16_t *svh, float *y,
                                 float *partials, int *counters, int *err, cudaStream_t s);
bool exl3_moe_gemv_widths_plan(int U, int nslots, int k, int n, int runs, const int *K, int *grid,
                               size_t *partial_floats, int *counters_needed, int *xops = nullptr);
cudaError_t exl3_launch_moe_gemv_widths(const uint16_t *x, const float *act_in, int *pos_out, const int32_t *ids,
                                        const float *weights, int U, int topk, int E, int nslots, int k, int n,
                                        int runs, const int *K, const int *e_lo, const int *cnt, const size_t *words,
                                        const uint16_t *trellis, const uint16_t *suh, const uint16_t *svh, float *y,
                                        float *partials, int *counters, int *err, cudaStream_t s, bool prefetch);
int exl3_launch_moe_fused_gateup(const uint16_t *xg, const uint16_t *xu, int U, int hidden, int inter, int K, int E,
                                 const uint16_t *w13_trellis, const int *mtiles, const int *n_mtiles, int max_mtiles,
                                 int cap, const uint16_t *svh13, const uint16_t *suh2, uint16_t *hout, int splits,
                                 float *partials, int *counters, int *err, cudaStream_t s, int e_lo = 0,
                                 int e_cnt = -1);
bool exl3_moe_fused_cap_fits(int cap, int K);
int exl3_launch_moe_fused_down(const uint16_t *hin, int U, int hidden, int inter, int K, int E,
                               const uint16_t *w2_trellis, const int *mtiles, const int *n_mtiles, int max_mtiles,
                               int cap, const uint16_t *svh2, const float *weights, const int *perm, float *dout,
                               int *err, cudaStream_t s, int e_lo = 0, int e_cnt = -1);

// ---------------------------------------------------------------- errors --

static thread_local std::string g_last_error;
static std::atomic<int> g_weight_prefetch{0};
static std::atomic<int> g_row_invariant{0};

int exl3_fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int exl3_cuda_check(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return EXL3_OK;
  return exl3_fail(EXL3_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int exl3_sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;
  }
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && (v = cache[dev].load(std::memory_order_relaxed)) > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
    cudaGetLastError();
    return 152;
  }
  if (cached) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

PFN_cuTensorMapEncodeTiled_v12000 exl3_tmap_encode_fn() {
  // a function-local static is initialised once, even with concurrent callers
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

cudaError_t exl3_ensure_smem(const void *kfn, size_t bytes, std::atomic<size_t> *per_dev) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && per_dev[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess || !cached) return e;
  size_t cur = per_dev[dev].load(std::memory_order_relaxed);
  while (cur < bytes && !per_dev[dev].compare_exchange_weak(cur, bytes, std::memory_order_release)) {
  }
  return cudaSuccess;
}

#define EXL3_TRY(expr)            \
  do {                            \
    int _rc = (expr);             \
    if (_rc != EXL3_OK) return _rc; \
  } while (0)

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kCtrlBytes = 256;   // device error word and reserved control words
// Arrival counters live at one fixed place of every workspace, right after
// the control block, so calls of any shape find them zero (each call resets
// the counters it used).  Capacity bounds n / 128 of one call.
constexpr size_t kMaxCounters = 8192;
constexpr size_t kCounterOff = kCtrlBytes;
constexpr size_t kDataOff = kCounterOff + kMaxCounters * sizeof(int);
constexpr int kFusedMaxM = 128;      // 2 <= M <= this: fused decode + tcgen05; above: reconstruct + tcgen05
constexpr int kRowInvChunk = 32;     // row-invariant mode: MMA width and rows per fused launch
constexpr int kMaxGemvK = 49152;     // the M = 1 GEMV keeps x' for all of k in shared memory

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


int check_ptr(const void *p, const char *name, bool required = true) {
  if (!p) return required ? exl3_fail(EXL3_ERR_ARG, "%s is NULL", name) : EXL3_OK;
  if (!aligned16(p)) return exl3_fail(EXL3_ERR_ARG, "%s is not 16-byte aligned", name);
  return EXL3_OK;
}

int check_bits_codebook(int K, int codebook) {
  if (codebook == EXL3_CB_MCG || codebook == EXL3_CB_3INST)
    return exl3_fail(EXL3_ERR_CODEBOOK,
                     "codebook %d is not implemented (only mul1 = %d); refusing rather than guessing",
                     codebook, EXL3_CB_MUL1);
  if (codebook != EXL3_CB_MUL1) return exl3_fail(EXL3_ERR_CODEBOOK, "unknown codebook id %d", codebook);
  if (K < 1 || K > 8) return exl3_fail(EXL3_ERR_BITS, "K = %d outside 1..8", K);
  return EXL3_OK;
}

int check_linear_shape(int M, int k, int n) {
  if (M < 1) return exl3_fail(EXL3_ERR_SHAPE, "M = %d < 1", M);
  if (k <= 0 || n <= 0 || k % 128 || n % 128)
    return exl3_fail(EXL3_ERR_SHAPE, "k = %d and n = %d must be positive multiples of 128", k, n);
  if ((int64_t)M * k > INT32_MAX || (int64_t)M * n > INT32_MAX || (int64_t)k * n > ((int64_t)1 << 40) ||
      (size_t)(n / 128) > kMaxCounters || (M == 1 && k > kMaxGemvK))
    return exl3_fail(EXL3_ERR_SHAPE, "shape too large (n <= %zu, and k <= %d at M = 1)", 128 * kMaxCounters,
                     kMaxGemvK);
  return EXL3_OK;
}

// ---- exl3_linear workspace layout
struct LinearWs {
  size_t ctrl = 0, counters = 0, partials = 0, xh = 0, xsum = 0, wt = 0, total = 0;
  int grid = 1, splits = 1;
};

// row_invariant: every M takes the 128-token-wide fused kernel, 128 rows at
// a time (x' and its sums for all M rows, partials for one chunk).
LinearWs linear_ws(int M, int k, int n, int K, bool row_invariant) {
  LinearWs w;
  size_t off = kDataOff;
  w.counters = kCounterOff;
  if (row_invariant) {
    const int Mc = M < kRowInvChunk ? M : kRowInvChunk;
    w.xh = off;
    off = align_up(off + sizeof(uint16_t) * (size_t)M * k);
    w.xsum = off;
    off = align_up(off + sizeof(float) * (size_t)M * ((k + 255) / 256));
    w.splits = exl3_fused_tc_splits(k, n);
    w.partials = off;
    off = align_up(off + (w.splits > 1 ? sizeof(float) * (size_t)w.splits * Mc * n : 0));
  } else if (M == 1 && exl3_gemv_fits(k, n, K)) {
    size_t floats = 0;
    exl3_gemv_plan(k, n, K, &w.grid, &floats);
    w.partials = off;
    off = align_up(off + sizeof(float) * floats);
  } else if (M <= kFusedMaxM) {
    w.xh = off;
    off = align_up(off + sizeof(uint16_t) * (size_t)M * k);
    w.xsum = off;   // per-token sums of x' over 256-element units
    off = align_up(off + sizeof(float) * (size_t)M * ((k + 255) / 256));
    w.splits = exl3_fused_tc_splits(k, n);
    w.partials = off;
    off = align_up(off + (w.splits > 1 ? sizeof(float) * (size_t)w.splits * M * n : 0));
  } else {
    w.xh = off;
    off = align_up(off + sizeof(uint16_t) * (size_t)M * k);
    w.wt = off;
    off = align_up(off + sizeof(uint16_t) * (size_t)k * n);
  }
  w.total = off;
  return w;
}

// ---- exl3_linear_int8 workspace layout
struct LinearInt8Ws {
  size_t qh = 0, wq = 0, rs = 0, total = 0;
};

LinearInt8Ws linear_int8_ws(int M, int k, int n) {
  LinearInt8Ws w;
  size_t off = kDataOff;
  w.qh = off;
  off = align_up(off + sizeof(uint16_t) * (size_t)M * k);
  w.wq = off;
  off = align_up(off + sizeof(uint16_t) * (size_t)k * n);
  w.rs = off;
  off = align_up(off + sizeof(float) * (size_t)M);
  w.total = off;
  return w;
}

// ---- exl3_moe_grouped workspace layout
struct MoeWs {
  size_t counts, offsets, pos, perm, mtiles, n_mtiles, chunk, xg, xu, h, d, partials, total;
  int max_mtiles, grid_mtiles, splits;
  int cap;            // rows per expert tile: 32, 128, 160 or 256 (chosen in moe_ws)
  bool gemv;          // few routed rows: grouped M = 1 GEMVs instead of the tile kernels
  size_t y13;         // gemv: gate/up outputs [U][2][inter] fp32 (d, pos, partials as above)
};

// The few-token path (one grouped CUDA-core GEMV launch per projection, no
// sort) runs instead of the tensor-core tiles for up to 32 routed rows, and
// for up to 1.25 routed rows per expert (at most 512 rows, and as long as
// no CTA's share spans more ops than the GEMV keeps x' for): it decodes
// every routed row's expert weights separately, at about twice the rate per
// weight of the tile kernels' decoders, which pays while few rows share an
// expert (E = 256, top-8: T = 16 0.090 against 0.124 ms, T = 40 0.196
// against about 0.205 ms; at T = 48 the tiles are faster).
constexpr int kMoeGemvMaxU = 32;
constexpr int kMoeGemvMaxUPerExpert = 512;


// Few routed rows (grouped M = 1 GEMVs): gate and up outputs [U][2][inter]
// fp32, d [U][hidden] fp32, pos [U] and the GEMVs' split-k partials.
MoeWs moe_gemv_layout(size_t U, int hidden, int inter, size_t partial_floats) {
  MoeWs w{};
  w.gemv = true;
  size_t off = kDataOff;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes); return o; };
  w.y13 = take(sizeof(float) * U * 2 * inter);
  w.d = take(sizeof(float) * U * hidden);
  w.pos = take(sizeof(int) * U);
  w.partials = take(sizeof(float) * partial_floats);
  w.total = off;
  return w;
}

// allow_gemv = false keeps every token count on the tile kernels (the
// mixed-width call, which plans its few-token path itself).
MoeWs moe_ws(int T, int topk, int E, int hidden, int inter, int K13, int K2, bool allow_gemv = true) {
  MoeWs w{};
  const size_t U = (size_t)T * topk;
  if (allow_gemv) {
    int g1 = 0, g2 = 0, b1 = 0, b2 = 0;
    size_t p1 = 0, p2 = 0;
    const bool few =
        U <= (size_t)kMoeGemvMaxU || (4 * U <= (size_t)5 * E && U <= (size_t)kMoeGemvMaxUPerExpert);
    if (few && exl3_moe_gemv_plan((int)U, 2, hidden, inter, K13, &g1, &p1, &b1) &&
        exl3_moe_gemv_plan((int)U, 1, inter, hidden, K2, &g2, &p2, &b2) && (size_t)b1 <= kMaxCounters &&
        (size_t)b2 <= kMaxCounters) {
      return moe_gemv_layout(U, hidden, inter, p1 > p2 ? p1 : p2);
    }
  }
  // Tiles of 32 rows (the grouped kernels then run MMAs 16 or 32 rows wide,
  // with four issuers) when the call routes at most 16 rows per expert on
  // average; when it routes at least 96, tiles that keep an expert's rows
  // together (its weights are then decoded once): 160 rows up to 136 rows
  // per expert on average (room for three x' stages), 256 above; 128 rows
  // otherwise.  The larger tiles need widths that fit their rings.
  w.cap = U <= (size_t)16 * E ? 32 : 128;
  const int kmax = K13 > K2 ? K13 : K2;
  if (U >= (size_t)96 * E) {
    const int big = U < (size_t)136 * E ? 160 : 256;
    if (exl3_moe_fused_cap_fits(big, kmax)) w.cap = big;
    else if (big == 160 && exl3_moe_fused_cap_fits(256, kmax)) w.cap = 256;
  }
  w.max_mtiles = (int)(U / w.cap + E + 1);
  size_t off = kDataOff;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes); return o; };
  w.counts = take(sizeof(int) * E);
  w.offsets = take(sizeof(int) * (E + 1));
  w.pos = take(sizeof(int) * U);
  w.perm = take(sizeof(int) * U);
  w.mtiles = take(sizeof(int) * 4 * (size_t)w.max_mtiles);
  w.n_mtiles = take(sizeof(int));
  const size_t ch = (size_t)exl3_moe_remap_chunk(E);
  w.chunk = take(sizeof(int) * ((U + ch - 1) / ch) * (size_t)E);
  w.xg = take(sizeof(uint16_t) * U * hidden);
  w.xu = take(sizeof(uint16_t) * U * hidden);
  w.h = take(sizeof(uint16_t) * U * inter);
  w.d = take(sizeof(float) * U * hidden);
  // Every tile holds at least one unit, so the grouped kernels need
  // at most min(U, max_mtiles) tiles per output column block.  When those
  // tiles cannot fill half the SMs (few tokens), the gate+up projection is
  // split over k into an even number of k steps (at least 4) per CTA.
  w.grid_mtiles = (int)(U < (size_t)w.max_mtiles ? U : (size_t)w.max_mtiles);
  const long tiles1 = (long)w.grid_mtiles * (inter / 128);
  const int kb = hidden / 64, sms = exl3_sm_count();
  w.splits = 1;
  for (int sp = 2; sp <= 8 && w.cap <= 128; ++sp)
    if (kb % sp == 0 && (kb / sp) % 2 == 0 && kb / sp >= 4 && tiles1 * sp <= sms) w.splits = sp;
  if (w.splits > 1) w.partials = take(sizeof(float) * (size_t)tiles1 * w.splits * 2 * w.cap * 128);
  w.total = off;
  return w;
}

int check_moe(int T, int hidden, int topk, int E, const exl3_expert_proj *w13, const exl3_expert_proj *w2) {
  if (!w13 || !w2) return exl3_fail(EXL3_ERR_ARG, "w13 / w2 descriptor is NULL");
  if (T < 1 || topk < 1 || E < 1 || E > 1024 || (int64_t)T * topk > (1 << 24))
    return exl3_fail(EXL3_ERR_SHAPE, "T = %d, topk = %d, E = %d out of range (E <= 1024)", T, topk, E);
  EXL3_TRY(check_ptr(w13->trellis, "w13.trellis"));
  EXL3_TRY(check_ptr(w13->suh, "w13.suh"));
  EXL3_TRY(check_ptr(w13->svh, "w13.svh"));
  EXL3_TRY(check_ptr(w2->trellis, "w2.trellis"));
  EXL3_TRY(check_ptr(w2->suh, "w2.suh"));
  EXL3_TRY(check_ptr(w2->svh, "w2.svh"));
  EXL3_TRY(check_bits_codebook(w13->K, w13->codebook));
  EXL3_TRY(check_bits_codebook(w2->K, w2->codebook));
  if (w13->nslots != 2 || w2->nslots != 1)
    return exl3_fail(EXL3_ERR_SHAPE, "w13 must have nslots = 2 (gate, up) and w2 nslots = 1");
  const int inter = w13->n;
  if (w13->k != hidden || w2->k != inter || w2->n != hidden)
    return exl3_fail(EXL3_ERR_SHAPE, "projection shapes do not chain: w13 %d->%d, w2 %d->%d, hidden %d",
                     w13->k, w13->n, w2->k, w2->n, hidden);
  if (hidden <= 0 || inter <= 0 || hidden % 256 || inter % 128)
    return exl3_fail(EXL3_ERR_SHAPE, "hidden = %d must be a multiple of 256 and inter = %d of 128", hidden, inter);
  return EXL3_OK;
}

// Runs of equal width in expert order: [e_lo, e_lo + cnt) of width K, whose
// trellis starts `words` uint16 words into the arena.
struct WidthRun {
  int e_lo, cnt, K;
  size_t words;
};

int check_mixed_proj(const exl3_expert_proj_mixed *p, const char *name, int E, int nslots, int k, int n) {
  if (!p) return exl3_fail(EXL3_ERR_ARG, "%s descriptor is NULL", name);
  EXL3_TRY(check_ptr(p->trellis, "trellis"));
  EXL3_TRY(check_ptr(p->suh, "suh"));
  EXL3_TRY(check_ptr(p->svh, "svh"));
  if (!p->K) return exl3_fail(EXL3_ERR_ARG, "%s.K (host array of %d widths) is NULL", name, E);
  EXL3_TRY(check_bits_codebook(1, p->codebook));
  for (int e = 0; e < E; ++e)
    if (p->K[e] < 1 || p->K[e] > 8)
      return exl3_fail(EXL3_ERR_BITS, "%s.K[%d] = %d outside 1..8", name, e, p->K[e]);
  if (p->nslots != nslots || p->k != k || p->n != n)
    return exl3_fail(EXL3_ERR_SHAPE, "%s is %d slots of %d -> %d, expected %d slots of %d -> %d", name, p->nslots,
                     p->k, p->n, nslots, k, n);
  return EXL3_OK;
}

std::vector<WidthRun> width_runs(const exl3_expert_proj_mixed *p, int E) {
  std::vector<WidthRun> runs;
  const size_t per_bit = (size_t)p->nslots * (p->k / 16) * (p->n / 16) * 16;   // words per expert per bit of width
  size_t off = 0;
  for (int e = 0; e < E; ++e) {
    if (runs.empty() || runs.back().K != p->K[e]) runs.push_back(WidthRun{e, 0, p->K[e], off});
    ++runs.back().cnt;
    off += per_bit * (size_t)p->K[e];
  }
  return runs;
}

// Few routed rows of experts with mixed widths: one grouped-GEMV launch per
// projection over all its runs of equal width (at most 8 of them).  False
// when the path does not apply; *partial_floats: the larger launch's
// split-k partials.
bool mixed_gemv_plan(size_t U, int E, int hidden, int inter, const exl3_expert_proj_mixed *w13,
                     const exl3_expert_proj_mixed *w2, size_t *partial_floats) {
  // as for one width, but up to one routed row per expert (measured at the
  // MoE shape with two widths: T = 32 0.219 against 0.233 ms through the
  // tiles, T = 40 0.261 against 0.246 ms)
  if (!(U <= (size_t)kMoeGemvMaxU || (U <= (size_t)E && U <= (size_t)kMoeGemvMaxUPerExpert))) return false;
  size_t pmax = 0;
  for (int proj = 0; proj < 2; ++proj) {
    const std::vector<WidthRun> runs = width_runs(proj == 0 ? w13 : w2, E);
    if (runs.size() > 8) return false;
    int K[8];
    for (size_t r = 0; r < runs.size(); ++r) K[r] = runs[r].K;
    int grid = 0, counters = 0;
    size_t pf = 0;
    if (!exl3_moe_gemv_widths_plan((int)U, proj == 0 ? 2 : 1, proj == 0 ? hidden : inter,
                                   proj == 0 ? inter : hidden, (int)runs.size(), K, &grid, &pf, &counters) ||
        (size_t)counters > kMaxCounters)
      return false;
    pmax = pf > pmax ? pf : pmax;
  }
  *partial_floats = pmax;
  return true;
}

int check_workspace(const void *ws, size_t have, size_t need) {
  if (need == 0) return EXL3_OK;
  if (!ws) return exl3_fail(EXL3_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
    return exl3_fail(EXL3_ERR_WORKSPACE, "workspace must be %zu-byte aligned", kAlign);
  if (have < need) return exl3_fail(EXL3_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", have, need);
  return EXL3_OK;
}

template <typename T>
T *at(void *base, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(base) + off);
}

}  // namespace

// ================================================================== C ABI ==

extern "C" {

const char *exl3_last_error(void) { return g_last_error.c_str(); }

int exl3_version(void) { return 200; }

int exl3_set_weight_prefetch(int enable) { return g_weight_prefetch.exchange(enable ? 1 : 0); }

int exl3_set_row_invariant(int enable) { return g_row_invariant.exchange(enable ? 1 : 0); }

int exl3_copy_in(const void *src, void *dst, size_t bytes, exl3_stream_t stream) {
  g_last_error.clear();
  if (bytes == 0) return EXL3_OK;
  EXL3_TRY(check_ptr(src, "src"));
  EXL3_TRY(check_ptr(dst, "dst"));
  return exl3_cuda_check(exl3_launch_copy_in(src, dst, bytes, stream, true), "copy_in launch");
}

int exl3_workspace_clear(void *workspace, size_t ws_bytes, exl3_stream_t stream) {
  g_last_error.clear();
  if (!workspace || ws_bytes == 0) return EXL3_OK;
  return exl3_cuda_check(cudaMemsetAsync(workspace, 0, ws_bytes, stream), "cudaMemsetAsync(workspace)");
}

int exl3_check_device_error(void *workspace, size_t ws_bytes, exl3_stream_t stream, int *err_out) {
  g_last_error.clear();
  if (!err_out) return exl3_fail(EXL3_ERR_ARG, "err_out is NULL");
  *err_out = 0;
  EXL3_TRY(check_workspace(workspace, ws_bytes, kCtrlBytes));
  EXL3_TRY(exl3_cuda_check(cudaStreamSynchronize(stream), "cudaStreamSynchronize"));
  int v = 0;
  EXL3_TRY(exl3_cuda_check(cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost), "read error word"));
  EXL3_TRY(exl3_cuda_check(cudaMemset(workspace, 0, sizeof v), "clear error word"));
  *err_out = v;
  return EXL3_OK;
}

int exl3_decode_tile(const uint16_t *trellis, int k, int n, int K, int codebook, int tk0, int tk_cnt,
                     int tn0, int tn_cnt, uint16_t *w_out, int64_t ld, exl3_stream_t stream) {
  g_last_error.clear();
  EXL3_TRY(check_ptr(trellis, "trellis"));
  EXL3_TRY(check_ptr(w_out, "w_out"));
  EXL3_TRY(check_bits_codebook(K, codebook));
  if (k <= 0 || n <= 0 || k % 16 || n % 16)
    return exl3_fail(EXL3_ERR_SHAPE, "k = %d, n = %d must be positive multiples of 16", k, n);
  if (tk0 < 0 || tn0 < 0 || tk_cnt < 0 || tn_cnt < 0 || tk0 + tk_cnt > k / 16 || tn0 + tn_cnt > n / 16)
    return exl3_fail(EXL3_ERR_SHAPE, "tile range [%d,+%d) x [%d,+%d) outside the %d x %d tile grid", tk0,
                     tk_cnt, tn0, tn_cnt, k / 16, n / 16);
  if (ld < 16LL * tn_cnt || ld % 8)
    return exl3_fail(EXL3_ERR_SHAPE, "ld = %lld must be >= 16 * tn_cnt and a multiple of 8", (long long)ld);
  if (tk_cnt == 0 || tn_cnt == 0) return EXL3_OK;
  if (tk_cnt * 2 > 65535) return exl3_fail(EXL3_ERR_SHAPE, "tk_cnt = %d too large for one call", tk_cnt);
  return exl3_cuda_check(
      exl3_launch_decode_tile(trellis, n, K, tk0, tk_cnt, tn0, tn_cnt, w_out, ld, stream), "decode_tile launch");
}

int exl3_input_rht(const uint16_t *x, int M, int k, const uint16_t *suh, void *out, int out_dtype,
                   exl3_stream_t stream) {
  g_last_error.clear();
  EXL3_TRY(check_ptr(x, "x"));
  EXL3_TRY(check_ptr(suh, "suh"));
  EXL3_TRY(check_ptr(out, "out"));
  if (out_dtype != EXL3_OUT_F16 && out_dtype != EXL3_OUT_F32)
    return exl3_fail(EXL3_ERR_ARG, "out_dtype %d invalid", out_dtype);
  if (M < 1 || k <= 0 || k % 128) return exl3_fail(EXL3_ERR_SHAPE, "M = %d, k = %d (k multiple of 128)", M, k);
  return exl3_cuda_check(exl3_launch_input_rht(x, M, k, suh, out, out_dtype == EXL3_OUT_F32, stream),
                         "input_rht launch");
}

size_t exl3_linear_workspace_size(int M, int k, int n, int K) {
  if (M < 1 || k <= 0 || n <= 0 || k % 128 || n % 128 || K < 1 || K > 8) return 0;
  if ((size_t)(n / 128) > kMaxCounters || (M == 1 && k > kMaxGemvK)) return 0;
  // large enough in either mode, so the mode may change between the query
  // and the call
  const size_t a = linear_ws(M, k, n, K, false).total, b = linear_ws(M, k, n, K, true).total;
  return a > b ? a : b;
}

}  // extern "C"

namespace {

// exl3_linear with an optional output bias (NULL: none).
int linear_impl(const uint16_t *x, int M, int k, int n, const uint16_t *trellis, const uint16_t *suh,
                const uint16_t *svh, const uint16_t *bias, int K, int codebook, void *y, int out_dtype,
                void *workspace, size_t ws_bytes, exl3_stream_t stream) {
  g_last_error.clear();
  EXL3_TRY(check_ptr(x, "x"));
  EXL3_TRY(check_ptr(trellis, "trellis"));
  EXL3_TRY(check_ptr(suh, "suh"));
  EXL3_TRY(check_ptr(svh, "svh"));
  EXL3_TRY(check_ptr(bias, "bias", false));
  EXL3_TRY(check_ptr(y, "y"));
  EXL3_TRY(check_bits_codebook(K, codebook));
  EXL3_TRY(check_linear_shape(M, k, n));
  if (out_dtype != EXL3_OUT_F16 && out_dtype != EXL3_OUT_F32)
    return exl3_fail(EXL3_ERR_ARG, "out_dtype %d invalid", out_dtype);
  const bool inv = g_row_invariant.load() != 0;
  const LinearWs L = linear_ws(M, k, n, K, inv);
  EXL3_TRY(check_workspace(workspace, ws_bytes, L.total));
  const bool f32 = out_dtype == EXL3_OUT_F32;
  int *err = at<int>(workspace, L.ctrl);
  if (inv) {
    // Row-invariant mode: x' for every row, then the fused kernel at one
    // fixed MMA width over chunks of that many rows.  A row's x' depends on that row only,
    // the MMA width and the k splits (a function of k and n) are the same
    // for every chunk, and rows past the chunk's end read as zero, so y[m]
    // has the same bits whatever M is.
    uint16_t *xh = at<uint16_t>(workspace, L.xh);
    float *xsum = at<float>(workspace, L.xsum);
    const int xunits = (k + 255) / 256;
    EXL3_TRY(exl3_cuda_check(exl3_launch_input_rht(x, M, k, suh, xh, false, stream, xsum), "input_rht launch"));
    for (int m0 = 0; m0 < M; m0 += kRowInvChunk) {
      const int Mc = M - m0 < kRowInvChunk ? M - m0 : kRowInvChunk;
      void *yc = static_cast<uint8_t *>(y) + (size_t)m0 * n * (f32 ? 4 : 2);
      EXL3_TRY(exl3_launch_fused_tc(xh + (size_t)m0 * k, xsum + (size_t)m0 * xunits, trellis, svh, Mc, k, n, K, yc,
                                    f32, at<float>(workspace, L.partials), at<int>(workspace, L.counters), err,
                                    L.splits, stream, kRowInvChunk, bias));
    }
    return EXL3_OK;
  }
  // M = 1 runs the GEMV unless x' for this k does not fit beside its ring
  if (M == 1 && exl3_gemv_fits(k, n, K)) {
    return exl3_cuda_check(exl3_launch_gemv_m1_bias(x, trellis, suh, svh, bias, k, n, K, y, f32,
                                                    at<float>(workspace, L.partials), at<int>(workspace, L.counters),
                                                    err, L.grid, stream, g_weight_prefetch.load() != 0),
                           "gemv launch");
  }
  uint16_t *xh = at<uint16_t>(workspace, L.xh);
  if (M <= kFusedMaxM) {
    float *xsum = at<float>(workspace, L.xsum);
    EXL3_TRY(exl3_cuda_check(exl3_launch_input_rht(x, M, k, suh, xh, false, stream, xsum), "input_rht launch"));
    return exl3_launch_fused_tc(xh, xsum, trellis, svh, M, k, n, K, y, f32, at<float>(workspace, L.partials),
                                at<int>(workspace, L.counters), err, L.splits, stream, 0, bias);
  }
  EXL3_TRY(exl3_cuda_check(exl3_launch_input_rht(x, M, k, suh, xh, false, stream), "input_rht launch"));
  uint16_t *wt = at<uint16_t>(workspace, L.wt);
  EXL3_TRY(exl3_cuda_check(exl3_launch_reconstruct_t(trellis, k, n, K, wt, stream), "reconstruct launch"));
  return exl3_launch_gemm_tc(xh, wt, M, n, k, svh, y, f32, nullptr, 1.0f, err, stream, false, nullptr, bias);
}

// exl3_linear_int8 with an optional output bias (NULL: none).
int linear_int8_impl(const uint16_t *x, int M, int k, int n, const uint16_t *trellis, const uint16_t *suh,
                     const uint16_t *svh, const uint16_t *bias, int K, int codebook, float weight_scale,
                     uint16_t *y, int8_t *xq_out, float *row_scale_out, int32_t *acc_out, void *workspace,
                     size_t ws_bytes, exl3_stream_t stream) {
  g_last_error.clear();
  EXL3_TRY(check_ptr(x, "x"));
  EXL3_TRY(check_ptr(trellis, "trellis"));
  EXL3_TRY(check_ptr(suh, "suh"));
  EXL3_TRY(check_ptr(svh, "svh"));
  EXL3_TRY(check_ptr(bias, "bias", false));
  EXL3_TRY(check_ptr(y, "y"));
  EXL3_TRY(check_ptr(xq_out, "xq_out", false));
  EXL3_TRY(check_ptr(row_scale_out, "row_scale_out", false));
  EXL3_TRY(check_ptr(acc_out, "acc_out", false));
  EXL3_TRY(check_bits_codebook(K, codebook));
  EXL3_TRY(check_linear_shape(M, k, n));
  if (!(weight_scale > 0.0f) || weight_scale > 1e30f)
    return exl3_fail(EXL3_ERR_ARG, "weight_scale must be positive and finite");
  if (k > kMaxGemvK) return exl3_fail(EXL3_ERR_SHAPE, "k = %d too large for the int8 path (k <= %d)", k, kMaxGemvK);
  const LinearInt8Ws L = linear_int8_ws(M, k, n);
  EXL3_TRY(check_workspace(workspace, ws_bytes, L.total));
  uint16_t *qh = at<uint16_t>(workspace, L.qh);
  uint16_t *wq = at<uint16_t>(workspace, L.wq);
  float *rs = row_scale_out ? row_scale_out : at<float>(workspace, L.rs);
  int *err = at<int>(workspace, 0);
  EXL3_TRY(exl3_cuda_check(exl3_launch_quant_act(x, M, k, suh, qh, xq_out, rs, stream), "quant_act launch"));
  EXL3_TRY(exl3_cuda_check(exl3_launch_reconstruct_q8_t(trellis, k, n, K, wq, stream), "reconstruct_q8 launch"));
  return exl3_launch_gemm_tc(qh, wq, M, n, k, svh, y, false, rs, weight_scale, err, stream, true, acc_out, bias);
}

}  // namespace

extern "C" {

int exl3_linear(const uint16_t *x, int M, int k, int n, const uint16_t *trellis, const uint16_t *suh,
                const uint16_t *svh, int K, int codebook, void *y, int out_dtype, void *workspace,
                size_t ws_bytes, exl3_stream_t stream) {
  return linear_impl(x, M, k, n, trellis, suh, svh, nullptr, K, codebook, y, out_dtype, workspace, ws_bytes,
                     stream);
}

int exl3_linear_bias(const uint16_t *x, int M, int k, int n, const uint16_t *trellis, const uint16_t *suh,
                     const uint16_t *svh, const uint16_t *bias, int K, int codebook, void *y, int out_dtype,
                     void *workspace, size_t ws_bytes, exl3_stream_t stream) {
  if (!bias) {
    g_last_error.clear();
    return exl3_fail(EXL3_ERR_ARG, "bias is NULL (use exl3_linear for a linear without bias)");
  }
  return linear_impl(x, M, k, n, trellis, suh, svh, bias, K, codebook, y, out_dtype, workspace, ws_bytes, stream);
}

size_t exl3_linear_int8_workspace_size(int M, int k, int n, int K) {
  if (M < 1 || k <= 0 || n <= 0 || k % 128 || n % 128 || K < 1 || K > 8) return 0;
  return linear_int8_ws(M, k, n).total;
}

int exl3_linear_int8(const uint16_t *x, int M, int k, int n, const uint16_t *trellis, const uint16_t *suh,
                     const uint16_t *svh, int K, int codebook, float weight_scale, uint16_t *y, int8_t *xq_out,
                     float *row_scale_out, int32_t *acc_out, void *workspace, size_t ws_bytes,
                     exl3_stream_t stream) {
  return linear_int8_impl(x, M, k, n, trellis, suh, svh, nullptr, K, codebook, weight_scale, y, xq_out,
                          row_scale_out, acc_out, workspace, ws_bytes, stream);
}

int exl3_linear_int8_bias(const uint16_t *x, int M, int k, int n, const uint16_t *trellis, const uint16_t *suh,
                          const uint16_t *svh, const uint16_t *bias, int K, int codebook, float weight_scale,
                          uint16_t *y, int8_t *xq_out, float *row_scale_out, int32_t *acc_out, void *workspace,
                          size_t ws_bytes, exl3_stream_t stream) {
  if (!bias) {
    g_last_error.clear();
    return exl3_fail(EXL3_ERR_ARG, "bias is NULL (use exl3_linear_int8 for a linear without bias)");
  }
  return linear_int8_impl(x, M, k, n, trellis, suh, svh, bias, K, codebook, weight_scale, y, xq_out, row_scale_out,
                          acc_out, workspace, ws_bytes, stream);
}

size_t exl3_moe_workspace_size(int T, int topk, int E, const exl3_expert_proj *w13,
                               const exl3_expert_proj *w2) {
  if (!w13 || !w2 || T < 1 || topk < 1 || E < 1 || E > 1024) return 0;
  return moe_ws(T, topk, E, w13->k, w13->n, w13->K, w2->K).total;
}

int exl3_moe_grouped(const uint16_t *x, int T, int hidden, const int32_t *topk_ids, const float *topk_weights,
                     int topk, int E, const exl3_expert_proj *w13, const exl3_expert_proj *w2, void *y,
                     int out_dtype, void *workspace, size_t ws_bytes, exl3_stream_t stream) {
  g_last_error.clear();
  EXL3_TRY(check_ptr(x, "x"));
  EXL3_TRY(check_ptr(topk_ids, "topk_ids"));
  EXL3_TRY(check_ptr(topk_weights, "topk_weights"));
  EXL3_TRY(check_ptr(y, "y"));
  EXL3_TRY(check_moe(T, hidden, topk, E, w13, w2));
  if (out_dtype != EXL3_OUT_F16 && out_dtype != EXL3_OUT_F32)
    return exl3_fail(EXL3_ERR_ARG, "out_dtype %d invalid", out_dtype);
  const int inter = w13->n;
  const int U = T * topk;
  const MoeWs L = moe_ws(T, topk, E, hidden, inter, w13->K, w2->K);
  EXL3_TRY(check_workspace(workspace, ws_bytes, L.total));
  int *err = at<int>(workspace, 0);
  if (L.gemv) {
    // few routed rows: gate and up as U x 2 GEMVs, down as U GEMVs whose
    // input transform applies SiLU(gate) up (output times the routing
    // weight), combine; no sort, expert ids read in place
    float *y13 = at<float>(workspace, L.y13), *d = at<float>(workspace, L.d);
    int *pos = at<int>(workspace, L.pos);
    float *partials = at<float>(workspace, L.partials);
    int *counters = at<int>(workspace, kCounterOff);   // the fixed counter region, zero between calls
    EXL3_TRY(exl3_cuda_check(exl3_launch_moe_gemv(x, nullptr, nullptr, topk_ids, nullptr, U, topk, E, 2, hidden,
                                                  inter, w13->K, w13->trellis, w13->suh, w13->svh, y13, partials,
                                                  counters, err, stream),
                             "moe gate/up gemv launch"));
    EXL3_TRY(exl3_cuda_check(exl3_launch_moe_gemv(nullptr, y13, pos, topk_ids, topk_weights, U, topk, E, 1, inter,
                                                  hidden, w2->K, w2->trellis, w2->suh, w2->svh, d, partials,
                                                  counters, err, stream),
                             "moe down gemv launch"));
    return exl3_cuda_check(exl3_launch_moe_combine(d, pos, T, topk, hidden, y, out_dtype == EXL3_OUT_F32, stream),
                           "moe combine launch");
  }
  int *counts = at<int>(workspace, L.counts), *offsets = at<int>(workspace, L.offsets);
  int *pos = at<int>(workspace, L.pos), *perm = at<int>(workspace, L.perm);
  int *mtiles = at<int>(workspace, L.mtiles), *chunk_tab = at<int>(workspace, L.chunk);
  int *n_mtiles = at<int>(workspace, L.n_mtiles);
  uint16_t *xg = at<uint16_t>(workspace, L.xg), *xu = at<uint16_t>(workspace, L.xu);
  uint16_t *h = at<uint16_t>(workspace, L.h);
  float *d = at<float>(workspace, L.d);
  EXL3_TRY(exl3_cuda_check(exl3_launch_moe_remap(topk_ids, U, E, counts, offsets, perm, pos, mtiles,
                                                 n_mtiles, L.max_mtiles, L.cap, chunk_tab, err, stream),
                           "moe remap launch"));
  EXL3_TRY(exl3_cuda_check(exl3_launch_moe_gather(x, U, hidden, topk, perm, offsets, E, topk_ids, w13->suh, xg, xu,
                                                  stream),
                           "moe gather launch"));
  float *partials = L.splits > 1 ? at<float>(workspace, L.partials) : nullptr;
  int *counters = at<int>(workspace, kCounterOff);   // the fixed counter region, zero between calls
  EXL3_TRY(exl3_launch_moe_fused_gateup(xg, xu, U, hidden, inter, w13->K, E, w13->trellis, mtiles, n_mtiles,
                                        L.grid_mtiles, L.cap, w13->svh, w2->suh, h, L.splits, partials, counters, err,
                                        stream));
  EXL3_TRY(exl3_launch_moe_fused_down(h, U, hidden, inter, w2->K, E, w2->trellis, mtiles, n_mtiles, L.grid_mtiles, L.cap,
                                      w2->svh, topk_weights, perm, d, err, stream));
  return exl3_cuda_check(exl3_launch_moe_combine(d, pos, T, topk, hidden, y, out_dtype == EXL3_OUT_F32, stream),
                         "moe combine launch");
}

// The largest width of a mixed projection's experts (host array K[E]).
static int max_width(const exl3_expert_proj_mixed *p, int E) {
  int m = 1;
  for (int e = 0; p->K && e < E; ++e) m = p->K[e] > m ? p->K[e] : m;
  return m;
}

// The mixed-width call's workspace: the few-token grouped GEMVs, or the
// tile kernels.
MoeWs moe_mixed_ws(int T, int topk, int E, int hidden, int inter, const exl3_expert_proj_mixed *w13,
                   const exl3_expert_proj_mixed *w2) {
  const size_t U = (size_t)T * topk;
  size_t pf = 0;
  if (mixed_gemv_plan(U, E, hidden, inter, w13, w2, &pf)) return moe_gemv_layout(U, hidden, inter, pf);
  return moe_ws(T, topk, E, hidden, inter, max_width(w13, E), max_width(w2, E), false);
}

size_t exl3_moe_mixed_workspace_size(int T, int topk, int E, const exl3_expert_proj_mixed *w13,
                                     const exl3_expert_proj_mixed *w2) {
  if (!w13 || !w2 || !w13->K || !w2->K || T < 1 || topk < 1 || E < 1 || E > 1024) return 0;
  for (int e = 0; e < E; ++e)
    if (w13->K[e] < 1 || w13->K[e] > 8 || w2->K[e] < 1 || w2->K[e] > 8) return 0;
  return moe_mixed_ws(T, topk, E, w13->k, w13->n, w13, w2).total;
}

int exl3_moe_grouped_mixed(const uint16_t *x, int T, int hidden, const int32_t *topk_ids,
                           const float *topk_weights, int topk, int E, const exl3_expert_proj_mixed *w13,
                           const exl3_expert_proj_mixed *w2, void *y, int out_dtype, void *workspace,
                           size_t ws_bytes, exl3_stream_t stream) {
  g_last_error.clear();
  EXL3_TRY(check_ptr(x, "x"));
  EXL3_TRY(check_ptr(topk_ids, "topk_ids"));
  EXL3_TRY(check_ptr(topk_weights, "topk_weights"));
  EXL3_TRY(check_ptr(y, "y"));
  if (!w13 || !w2) return exl3_fail(EXL3_ERR_ARG, "w13 / w2 descriptor is NULL");
  if (T < 1 || topk < 1 || E < 1 || E > 1024 || (int64_t)T * topk > (1 << 24))
    return exl3_fail(EXL3_ERR_SHAPE, "T = %d, topk = %d, E = %d out of range (E <= 1024)", T, topk, E);
  const int inter = w13->n;
  if (hidden <= 0 || inter <= 0 || hidden % 256 || inter % 128)
    return exl3_fail(EXL3_ERR_SHAPE, "hidden = %d must be a multiple of 256 and inter = %d of 128", hidden, inter);
  EXL3_TRY(check_mixed_proj(w13, "w13", E, 2, hidden, inter));
  EXL3_TRY(check_mixed_proj(w2, "w2", E, 1, inter, hidden));
  if (out_dtype != EXL3_OUT_F16 && out_dtype != EXL3_OUT_F32)
    return exl3_fail(EXL3_ERR_ARG, "out_dtype %d invalid", out_dtype);
  const int U = T * topk;
  const MoeWs L = moe_mixed_ws(T, topk, E, hidden, inter, w13, w2);
  EXL3_TRY(check_workspace(workspace, ws_bytes, L.total));
  int *err = at<int>(workspace, 0);
  if (L.gemv) {
    // few routed rows: per projection, one grouped-GEMV launch over all its
    // runs of equal width, which finds on the device the units of each
    // width and splits its CTAs over the widths.  Gate and up write
    // [U][2][inter] fp32, down reads SiLU(gate) up of them and writes d
    // times the routing weight; the down launch streams its weights while
    // gate and up finish.
    float *y13 = at<float>(workspace, L.y13), *d = at<float>(workspace, L.d);
    int *pos = at<int>(workspace, L.pos);
    float *partials = at<float>(workspace, L.partials);
    int *counters = at<int>(workspace, kCounterOff);
    for (int proj = 0; proj < 2; ++proj) {
      const std::vector<WidthRun> runs = width_runs(proj == 0 ? w13 : w2, E);
      int K[8], lo[8], cnt[8];
      size_t words[8];
      const int nr = (int)runs.size();
      for (int r = 0; r < nr; ++r) {
        K[r] = runs[r].K;
        lo[r] = runs[r].e_lo;
        cnt[r] = runs[r].cnt;
        words[r] = runs[r].words;
      }
      cudaError_t e =
          proj == 0 ? exl3_launch_moe_gemv_widths(x, nullptr, nullptr, topk_ids, nullptr, U, topk, E, 2, hidden,
                                                  inter, nr, K, lo, cnt, words, w13->trellis, w13->suh, w13->svh, y13,
                                                  partials, counters, err, stream, false)
                    : exl3_launch_moe_gemv_widths(nullptr, y13, pos, topk_ids, topk_weights, U, topk, E, 1, inter,
                                                  hidden, nr, K, lo, cnt, words, w2->trellis, w2->suh, w2->svh, d,
                                                  partials, counters, err, stream, true);
      EXL3_TRY(exl3_cuda_check(e, proj == 0 ? "moe gate/up gemv launch" : "moe down gemv launch"));
    }
    return exl3_cuda_check(exl3_launch_moe_combine(d, pos, T, topk, hidden, y, out_dtype == EXL3_OUT_F32, stream),
                           "moe combine launch");
  }
  int *counts = at<int>(workspace, L.counts), *offsets = at<int>(workspace, L.offsets);
  int *pos = at<int>(workspace, L.pos), *perm = at<int>(workspace, L.perm);
  int *mtiles = at<int>(workspace, L.mtiles), *chunk_tab = at<int>(workspace, L.chunk);
  int *n_mtiles = at<int>(workspace, L.n_mtiles);
  uint16_t *xg = at<uint16_t>(workspace, L.xg), *xu = at<uint16_t>(workspace, L.xu);
  uint16_t *h = at<uint16_t>(workspace, L.h);
  float *d = at<float>(workspace, L.d);
  // routing, gather and combine as in exl3_moe_grouped; each projection runs
  // one grouped launch per run of equal width, over that run's experts only
  EXL3_TRY(exl3_cuda_check(exl3_launch_moe_remap(topk_ids, U, E, counts, offsets, perm, pos, mtiles,
                                                 n_mtiles, L.max_mtiles, L.cap, chunk_tab, err, stream),
                           "moe remap launch"));
  EXL3_TRY(exl3_cuda_check(exl3_launch_moe_gather(x, U, hidden, topk, perm, offsets, E, topk_ids, w13->suh, xg, xu,
                                                  stream),
                           "moe gather launch"));
  float *partials = L.splits > 1 ? at<float>(workspace, L.partials) : nullptr;
  int *counters = at<int>(workspace, kCounterOff);
  for (const WidthRun &r : width_runs(w13, E))
    EXL3_TRY(exl3_launch_moe_fused_gateup(xg, xu, U, hidden, inter, r.K, E, w13->trellis + r.words, mtiles, n_mtiles,
                                          L.grid_mtiles, L.cap, w13->svh, w2->suh, h, L.splits, partials, counters, err,
                                          stream, r.e_lo, r.cnt));
  for (const WidthRun &r : width_runs(w2, E))
    EXL3_TRY(exl3_launch_moe_fused_down(h, U, hidden, inter, r.K, E, w2->trellis + r.words, mtiles, n_mtiles,
                                        L.grid_mtiles, L.cap, w2->svh, topk_weights, perm, d, err, stream, r.e_lo, r.cnt));
  return exl3_cuda_check(exl3_launch_moe_combine(d, pos, T, topk, hidden, y, out_dtype == EXL3_OUT_F32, stream),
                         "moe combine launch");
}

// Fused shards: the one-launch plan at M = 1 (grid, partial floats), or
// false when the shards take one exl3_linear each.
static bool shards_one_launch(int M, int k, int n, int K, int S, size_t *floats) {
  int grid = 0, blocks = 0;
  size_t pf = 0;
  if (M != 1 || g_row_invariant.load() != 0) return false;
  if (!exl3_gemv_shards_plan(S, k, n, K, &grid, &pf, &blocks) || (size_t)blocks > kMaxCounters) return false;
  if (floats) *floats = pf;
  return true;
}

size_t exl3_linear_shards_workspace_size(int M, int k, int n, int K, int nshards) {
  if (nshards < 1 || nshards > 64) return 0;
  const size_t per = exl3_linear_workspace_size(M, k, n, K);
  if (per == 0) return 0;
  size_t pf = 0;
  int grid = 0, blocks = 0;
  size_t one = 0;
  if (M == 1 && exl3_gemv_shards_plan(nshards, k, n, K, &grid, &pf, &blocks))
    one = align_up(kDataOff + sizeof(float) * pf);
  return per > one ? per : one;
}

int exl3_linear_shards(const uint16_t *x, int M, int k, int n, int nshards, const uint16_t *trellis,
                       const uint16_t *suh, const uint16_t *svh, int K, int codebook, void *y, int out_dtype,
                       void *workspace, size_t ws_bytes, exl3_stream_t stream) {
  g_last_error.clear();
  EXL3_TRY(check_ptr(x, "x"));
  EXL3_TRY(check_ptr(trellis, "trellis"));
  EXL3_TRY(check_ptr(suh, "suh"));
  EXL3_TRY(check_ptr(svh, "svh"));
  EXL3_TRY(check_ptr(y, "y"));
  EXL3_TRY(check_bits_codebook(K, codebook));
  EXL3_TRY(check_linear_shape(M, k, n));
  if (nshards < 1 || nshards > 64) return exl3_fail(EXL3_ERR_SHAPE, "nshards = %d outside 1..64", nshards);
  if (out_dtype != EXL3_OUT_F16 && out_dtype != EXL3_OUT_F32)
    return exl3_fail(EXL3_ERR_ARG, "out_dtype %d invalid", out_dtype);
  const size_t need = exl3_linear_shards_workspace_size(M, k, n, K, nshards);
  EXL3_TRY(check_workspace(workspace, ws_bytes, need));
  const bool f32 = out_dtype == EXL3_OUT_F32;
  size_t pf = 0;
  if (shards_one_launch(M, k, n, K, nshards, &pf)) {
    return exl3_cuda_check(exl3_launch_gemv_shards(x, nshards, k, n, K, trellis, suh, svh, y, f32,
                                                   at<float>(workspace, kDataOff), at<int>(workspace, kCounterOff),
                                                   at<int>(workspace, 0), stream, g_weight_prefetch.load() != 0),
                           "gemv shards launch");
  }
  // one linear per shard, each into its own [M][n] block of y
  const size_t words = (size_t)(k / 16) * (n / 16) * 16 * K;
  const size_t ybytes = (size_t)M * n * (f32 ? 4 : 2);
  for (int sh = 0; sh < nshards; ++sh)
    EXL3_TRY(linear_impl(x, M, k, n, trellis + sh * words, suh + (size_t)sh * k, svh + (size_t)sh * n, nullptr, K,
                         codebook, static_cast<uint8_t *>(y) + sh * ybytes, out_dtype, workspace, ws_bytes,
                         stream));
  return EXL3_OK;
}

size_t exl3_linear_shards_var_workspace_size(int M, int k, int nshards, const int *n, int K) {
  if (nshards < 1 || nshards > 64 || !n) return 0;
  size_t need = 0;
  for (int i = 0; i < nshards; ++i) {
    const size_t w = exl3_linear_workspace_size(M, k, n[i], K);
    if (w == 0) return 0;
    if (w > need) need = w;
  }
  int grid = 0, blocks = 0;
  size_t pf = 0;
  if (M == 1 && exl3_gemv_shards_var_plan(nshards, k, n, K, &grid, &pf, &blocks)) {
    const size_t one = align_up(kDataOff + sizeof(float) * pf);
    if (one > need) need = one;
  }
  return need;
}

int exl3_linear_shards_var(const uint16_t *x, int M, int k, int nshards, const int *n, const uint16_t *trellis,
                           const uint16_t *suh, const uint16_t *svh, int K, int codebook, void *y, int out_dtype,
                           void *workspace, size_t ws_bytes, exl3_stream_t stream) {
  g_last_error.clear();
  EXL3_TRY(check_ptr(x, "x"));
  EXL3_TRY(check_ptr(trellis, "trellis"));
  EXL3_TRY(check_ptr(suh, "suh"));
  EXL3_TRY(check_ptr(svh, "svh"));
  EXL3_TRY(check_ptr(y, "y"));
  if (!n) return exl3_fail(EXL3_ERR_ARG, "n (host array of shard widths) is NULL");
  EXL3_TRY(check_bits_codebook(K, codebook));
  if (nshards < 1 || nshards > 64) return exl3_fail(EXL3_ERR_SHAPE, "nshards = %d outside 1..64", nshards);
  long long ntot = 0;
  for (int i = 0; i < nshards; ++i) {
    EXL3_TRY(check_linear_shape(M, k, n[i]));
    ntot += n[i];
  }
  if ((long long)M * ntot > INT32_MAX) return exl3_fail(EXL3_ERR_SHAPE, "M * sum of widths too large");
  if (out_dtype != EXL3_OUT_F16 && out_dtype != EXL3_OUT_F32)
    return exl3_fail(EXL3_ERR_ARG, "out_dtype %d invalid", out_dtype);
  const size_t need = exl3_linear_shards_var_workspace_size(M, k, nshards, n, K);
  EXL3_TRY(check_workspace(workspace, ws_bytes, need));
  const bool f32 = out_dtype == EXL3_OUT_F32;
  int grid = 0, blocks = 0;
  size_t pf = 0;
  if (M == 1 && g_row_invariant.load() == 0 && exl3_gemv_shards_var_plan(nshards, k, n, K, &grid, &pf, &blocks) &&
      (size_t)blocks <= kMaxCounters) {
    return exl3_cuda_check(exl3_launch_gemv_shards_var(x, nshards, k, n, K, trellis, suh, svh, y, f32,
                                                       at<float>(workspace, kDataOff),
                                                       at<int>(workspace, kCounterOff), at<int>(workspace, 0),
                                                       stream, g_weight_prefetch.load() != 0),
                           "gemv shards launch");
  }
  // one linear per shard, into its [M][n] block of the shard-major output
  size_t words = 0, col = 0;
  for (int i = 0; i < nshards; ++i) {
    EXL3_TRY(linear_impl(x, M, k, n[i], trellis + words, suh + (size_t)i * k, svh + col, nullptr, K, codebook,
                         static_cast<uint8_t *>(y) + (size_t)M * col * (f32 ? 4 : 2), out_dtype, workspace,
                         ws_bytes, stream));
    words += (size_t)(k / 16) * (n[i] / 16) * 16 * K;
    col += n[i];
  }
  return EXL3_OK;
}

}  // extern "C"
