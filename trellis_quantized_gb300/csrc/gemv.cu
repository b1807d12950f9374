// gemv.cu -- fused M = 1 EXL3 linear on CUDA cores (the decode GEMV; "dp4a
// GEMV" of "exl3xpu" README, "Layout"; the GEMM runs in the Hadamard domain,
// "exl3xpu" README, "Prefill: int8 linears and oneDNN fused attention").
//
//   y = RHT_out( sigma * sum_k x'_k (B_kn - 510) ) . svh,  x' = RHT_in(x . suh)
//
// The contraction uses the exact codebook value (B - 510) * sigma, of which
// the fp16 weight is the rounding (a difference below 2^-11 relative per
// term, inside the output tolerance), and x' in fp32.  DP4A yields the
// integer byte sum B, read as the bit pattern of the subnormal fp32 B 2^-149;
// with x' held as x' 2^100 the product is exact, and one fp32 FMA adds it to
// the column's accumulator: sum x' B.  The offset 510 * sum x' is removed once per column
// block from per-tile-row sums of x' kept beside x'.
//
// Lane work.  A lane owns G >= 4 consecutive rows of one tile: 16 G weights
// whose states come from CPL contiguous 16-byte chunks (128 CPL bits) plus
// the first 32 bits of the next row group (the last group of a tile wraps to
// the first).  LPT = 16 / G lanes cover a tile and a warp covers one tile row
// of the CTA's column block (128 or 256 columns).  Each window is cut out of
// byte-aligned (possibly pre-shifted) words with one LOP/SHR/PRMT where it
// can, hashed (IMAD), byte-summed by DP4A and accumulated by one fp32 FMA.
//
// Work split.  The work is the list of "rows" (column block c, tile row tk),
// c-major.  One CTA per SM takes an equal contiguous range of that list, so
// every SM gets the same amount of trellis.  Inside the CTA one thread loads
// the rows with 3-D tensor copies (8 tile rows of the column block each) into
// a ring of shared-memory stages, and NCW consumer warps decode every stage
// together (warp w takes rows w, w + NCW, ...).  Because all consumer warps
// share one ring, none can run more than the ring's depth ahead of the
// others, so they finish together; separate CTAs per SM did not (the warp
// schedulers favour the first-resident CTA, which left the SM's last CTA
// running alone at low issue rate).  Every wait is bounded; a wait that runs
// out sets the device error word.
//
// Column blocks.  A CTA's range crosses column blocks.  At each crossing
// the consumer warps leave their column sums in shared memory for a flusher
// warp and go straight on with the next block; the flusher adds the warps'
// sums in warp order and either finishes the block itself (its CTA owned all
// of it) or shares it with the neighbouring CTAs: the block's first CTA, for
// which it is the last segment, waits (bounded) until the others have
// published partial sums in slots fixed by (block, CTA), adds them in CTA
// order, applies the output transform and writes y.  The result does not
// depend on timing.
#include <cudaTypedefs.h>

#include <algorithm>

#include "exl3_common.cuh"
#include "gemv_core.cuh"
#include "tc_ptx.cuh"

namespace exl3 {

struct GemvArgs {
  const __half *x;          // [k]
  const __half *suh;        // [k]
  const __half *svh;        // [n]
  void *y;                  // [n] fp16 or fp32
  float *partials;          // [colblocks + grid][CTA_COLS]
  int *counters;            // [nops * colblocks]
  int *err;                 // device error word
  int k, n, tiles_k, colblocks, stages;
  int xops;                 // GROUPED: x' slots in shared memory (ops a CTA's range may touch)
  int pre_stages;           // stages the producer loads before x' is ready
  uint32_t total;           // nops * colblocks * tiles_k (grid * total < 2^32)
  // Routed-expert mode (GROUPED): the rows of op o = unit u * nslots + slot
  // follow those of op o - 1; op o multiplies x row (x_per_unit ? u : u / topk)
  // by expert e = ids[u]'s slot `slot` (trellis rows (e nslots + slot) k/16 of
  // one tensor over all experts, suh/svh [E][nslots][k or n]) into y[o][n]
  // (fp32, or fp16 when F32OUT is false), times weights[u] when weights is
  // set.  An id outside [0, E) sets the error word and makes the op's output
  // zero.  ids NULL: every unit uses expert 0 (the fused shards of one
  // input, op o = shard o).
  const int32_t *ids;
  const float *weights;
  int topk, nslots, E, x_per_unit, nops;
  uint32_t op_rows;         // colblocks * tiles_k
  // act_in set (down projection): unit u's input is SiLU(g) u of the gate and
  // up outputs act_in[u][0][k], act_in[u][1][k] (fp32) instead of x; pos_out
  // (if set) receives u, or -1 for an invalid expert id, for the combine
  const float *act_in;
  int *pos_out;
  // Output bias [n] fp16 added after svh (NULL: none; not GROUPED)
  const __half *bias;
  // Shards of different widths (GROUPED, var > 0 shards, no expert ids):
  // shard s has width vn[s], its column blocks are global blocks
  // vb[s] .. vb[s + 1] - 1, its svh and y start at column vo[s] of the
  // concatenated [sum of widths] vectors, suh at s k, and its trellis is
  // tensor map s.
  int var;
  int vn[8], vo[8], vb[9];
  // Routed experts of mixed widths (GROUPED, runs > 0, at most 512 units):
  // this launch serves the experts of runs [run_lo[r], run_hi[r]) of one
  // width (tensor map r, over run r's part of the packed arena from expert
  // run_lo[r]).  The units whose expert lies in one of them are the active
  // ones: compacted in unit order (op o = active unit o / nslots, slot
  // o % nslots) and counted on the device, so that the rows split evenly
  // over the CTAs whatever the routing; `total` is then found on the device.
  int runs, units;
  int wlist_off;            // byte offset of the unit list in dynamic shared memory (past every width's layout)
  int run_lo[8], run_hi[8], run_K[8];
  // per width K (index 1..8) of a launch over runs of several widths: column
  // blocks, ring stages, and the width's first arrival counter and partial
  // slot in the launch's arrays
  int wcolblocks[9], wstages[9], wcounter_base[9], wpartial_base[9];
};

// One CTA's share of a launch: its index and the number of CTAs sharing the
// rows, the rows (total, op_rows per op, column blocks per op), the active
// units (mixed widths), the ring depth, and the arrival counters and
// partial slots of its column blocks.
struct GemvPart {
  int me, grid;
  uint32_t total, op_rows;
  const int *ulist;         // mixed widths: this width's units in unit order (shared memory), else NULL
  int colblocks, stages;
  int *counters;
  float *partials;
};

constexpr int kGemvMinRows = 32;       // rows per CTA below which the M = 1 GEMV uses fewer CTAs
constexpr int kGemvMaxOps = 4;        // ops one CTA's range may touch in GROUPED mode (x' slots)
constexpr int kGemvMaxOpsMoe = 8;     // the routed-expert plan's limit, when x' for them fits
constexpr int kGemvMaxShards = 8;     // shards of different widths in one launch
constexpr int kGemvPrePartials = 2;   // partials a block's first CTA loads before its segment ends
constexpr int kGemvPreStages = 2;     // stages the producer loads before x' is ready

// The pointers of op o (one op, the linear itself, when not GROUPED).
struct GemvOp {
  const __half *x, *suh, *svh;
  void *y;
  float scale;
  int trow;                 // first trellis row of the op's weights
  bool bad;                 // invalid expert id
  int map;                  // tensor map of the op's trellis
  int unit;                 // routed unit (GROUPED)
};

// Mixed widths: whether expert e belongs to one of the launch's runs, and
// which (-1: none).
__device__ __forceinline__ int gemv_run_of(const GemvArgs &a, int e) {
  int r = -1;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < a.runs && e >= a.run_lo[i] && e < a.run_hi[i]) r = i;
  return r;
}

// The combine's row of each unit (-1 for an invalid expert id), when the
// launch has pos_out; threads tid of nthreads.
__device__ __forceinline__ void gemv_write_pos(const GemvArgs &a, int tid, int nthreads) {
  if (!a.pos_out) return;
  for (int u = tid; u < a.nops / a.nslots; u += nthreads) {
    const int e = a.ids[u];
    a.pos_out[u] = (e >= 0 && e < a.E) ? u : -1;
  }
}

template <bool GROUPED, bool F32OUT>
__device__ __forceinline__ GemvOp gemv_op(const GemvArgs &a, int o, const int *ulist = nullptr) {
  if constexpr (!GROUPED) {
    return GemvOp{a.x, a.suh, a.svh, a.y, 1.0f, 0, false, 0, 0};
  } else {
    if (a.var)   // shard o of different widths: its own map, column offset vo[o]
      return GemvOp{a.x, a.suh + (long)o * a.k, a.svh + a.vo[o],
                    static_cast<char *>(a.y) + (long)a.vo[o] * (F32OUT ? 4 : 2), 1.0f, 0, false, o, 0};
    int u = o / a.nslots;
    const int slot = o - u * a.nslots;
    if (a.runs) u = ulist[u];   // the u-th unit of this width
    int e = a.ids ? a.ids[u] : 0;   // no id list: every unit uses expert 0 (fused shards)
    const bool bad = e < 0 || e >= a.E;
    float scale = a.weights ? a.weights[u] : 1.0f;
    if (bad) {
      e = 0;
      scale = 0.0f;
    }
    const long es = (long)e * a.nslots + slot;
    const long xr = a.x_per_unit ? u : u / a.topk;
    int map = 0;
    long trow = es * a.tiles_k;
    if (a.runs) {   // the expert's run: its own map, experts counted from the run's first
      map = gemv_run_of(a, e);
      trow = ((long)(e - a.run_lo[map]) * a.nslots + slot) * a.tiles_k;
    }
    return GemvOp{a.x + xr * a.k, a.suh + es * a.k, a.svh + es * a.n,
                  static_cast<char *>(a.y) + (long)(u * a.nslots + slot) * a.n * (F32OUT ? 4 : 2), scale,
                  (int)trow, bad, map, u};
  }
}

// GROUPED mode: the op of global column block c, c's index inside that op,
// and the op's width.
__device__ __forceinline__ int op_of_block(const GemvArgs &a, const GemvPart &p, int c) {
  if (!a.var) return c / p.colblocks;
  int o = 0;
#pragma unroll
  for (int s = 1; s < kGemvMaxShards; ++s)
    if (s < a.var && c >= a.vb[s]) o = s;
  return o;
}
__device__ __forceinline__ int block_in_op(const GemvArgs &a, const GemvPart &p, int c, int op) {
  return a.var ? c - a.vb[op] : c - op * p.colblocks;
}
__device__ __forceinline__ int op_width(const GemvArgs &a, int op) { return a.var ? a.vn[op] : a.n; }

// Whether all `others` CTAs sharing column block c besides its first have
// published their partials (one acquire load, no waiting).
__device__ __forceinline__ bool gemv_all_arrived(const GemvArgs &a, const GemvPart &p, int c, int others,
                                                 int lane) {
  int got = 0;
  if (lane == 0) {
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(got) : "l"(p.counters + c) : "memory");
    if (got > others) set_device_error(a.err, kErrDirtyCounter);
  }
  got = __shfl_sync(0xffffffffu, got, 0);
  __threadfence();
  return got >= others;
}

// pre[j] = the partial of CTA i0 + 1 + j of column block c, for j below
// min(cnt, kGemvPrePartials) (lane l: columns 128 g + 4 l .. +3).
template <int NG>
__device__ __forceinline__ void gemv_load_partials(const GemvPart &p, int c, int i0, int cnt, int lane,
                                                   float (&pre)[kGemvPrePartials][NG][4]) {
#pragma unroll
  for (int j = 0; j < kGemvPrePartials; ++j)
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < cnt)
        r = __ldcg(reinterpret_cast<const float4 *>(p.partials + (long)(c + i0 + 1 + j) * (NG * 128) + g * 128 +
                                                    lane * 4));
      pre[j][g][0] = r.x;
      pre[j][g][1] = r.y;
      pre[j][g][2] = r.z;
      pre[j][g][3] = r.w;
    }
}

// p = the partial of CTA i of column block c.
template <int NG>
__device__ __forceinline__ void gemv_load_partial(const GemvPart &pt, int c, int i, int lane, float (&p)[NG][4]) {
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const float4 r = __ldcg(reinterpret_cast<const float4 *>(pt.partials + (long)(c + i) * (NG * 128) + g * 128 +
                                                             lane * 4));
    p[g][0] = r.x;
    p[g][1] = r.y;
    p[g][2] = r.z;
    p[g][3] = r.w;
  }
}

// v += the partial of CTA i of column block c.
template <int NG>
__device__ __forceinline__ void gemv_add_partial(const GemvPart &pt, int c, int i, int lane, float (&v)[NG][4]) {
  float p[NG][4];
  gemv_load_partial<NG>(pt, c, i, lane, p);
#pragma unroll
  for (int g = 0; g < NG; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) v[g][e] += p[g][e];
}

// The block's svh and output bias for lane l's columns (zero when not
// `load` or past the op's width).
template <int NG>
__device__ __forceinline__ void gemv_load_out_vectors(const __half *svh, const __half *bias, int col0, int nop,
                                                      int lane, bool load, uint2 (&svv)[NG], uint2 (&bvv)[NG]) {
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const bool mine = load && col0 + g * 128 < nop;
    svv[g] = mine ? *reinterpret_cast<const uint2 *>(svh + col0 + g * 128 + lane * 4) : make_uint2(0u, 0u);
    bvv[g] = mine && bias ? *reinterpret_cast<const uint2 *>(bias + col0 + g * 128 + lane * 4) : make_uint2(0u, 0u);
  }
}

// The kernel body; maps holds the trellis tensor map (one per shard for
// shards of different widths).
template <int K, bool F32OUT, bool GROUPED>
__device__ __forceinline__ void gemv_body(const CUtensorMap *maps, const GemvArgs &a, const GemvPart &p) {
  using S = GemvShape<K>;
  constexpr int NCW = S::NCW, NCT = NCW * 32;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int STAGES = p.stages;
  uint8_t *ring = smem_raw;                                            // [STAGES][R][ROWB]
  float *red = reinterpret_cast<float *>(smem_raw + (size_t)STAGES * S::STAGE_B);   // [NCW][CTA_COLS]
  volatile int *s_abort = reinterpret_cast<volatile int *>(red + NCW * S::CTA_COLS);   // a wait ran out
  uint64_t *full = reinterpret_cast<uint64_t *>(red + NCW * S::CTA_COLS + 4);    // [STAGES]
  uint64_t *empty = full + STAGES;                                     // [STAGES]
  uint64_t *seg_full = empty + STAGES;                                 // red holds a finished segment
  uint64_t *red_free = seg_full + 1;                                   // the flusher has read red
  uint64_t *xready = red_free + 1;                                     // the consumers' x' is ready
  const int NOPS = GROUPED ? a.xops : 1;
  float *xs = reinterpret_cast<float *>(xready + 2);                   // [NOPS][k] x' 2^100 (touched blocks)
  float *rsum = xs + NOPS * a.k;                                       // [NOPS][k/16] sum of x' per tile row

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int me = p.me, grid = p.grid;
  const int TK = a.tiles_k;
  // the kernel launched after this one on the stream may start as soon as
  // every CTA has begun (it only streams weights until this grid completes)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Row arithmetic is 32-bit (the host keeps grid * total below 2^32): a
  // 64-bit division is a long software sequence on every path's start.
  const uint32_t TKU = (uint32_t)TK;
  const uint32_t total = p.total;
  const int *ulist = p.ulist;
  const uint32_t t0 = me < grid ? range_start(me, total, grid) : 0;
  const uint32_t t1 = me < grid ? range_start(me + 1, total, grid) : 0;
  if (t0 >= t1) {
    // An empty share (mixed widths: fewer active rows than CTAs).  The
    // launch must still complete only after the kernel before it, which the
    // kernels after it rely on, so wait for it; the first CTA still writes
    // the combine's row of every unit.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (GROUPED && me == 0) gemv_write_pos(a, tid, (S::NCW + 2) * 32);
    return;
  }

  if (tid == 0) {
    for (int st = 0; st < STAGES; ++st) {
      tc::mbar_init(&full[st], 1);
      tc::mbar_init(&empty[st], NCW);
    }
    tc::mbar_init(seg_full, NCW);
    tc::mbar_init(red_free, 1);
    tc::mbar_init(xready, 1);
    *s_abort = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();

  if (warp == NCW) {
    // ---------------- producer: one thread loads the rows into the ring
    if (lane == 0) {
      for (int m = 0; m < (GROUPED && a.var ? a.var : 1); ++m) tc::prefetch_tmap(maps + m);
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      for (uint32_t t = t0; t < t1 && !*s_abort;) {
        const uint32_t c = t / TKU;   // block: op c / colblocks, column block c % colblocks
        const uint32_t seg_end = min(t1, (c + 1) * TKU);
        const int tk_first = (int)(t - c * TKU), nrows = (int)(seg_end - t);
        const int op = GROUPED ? op_of_block(a, p, (int)c) : 0;
        const int tn0 = (GROUPED ? block_in_op(a, p, (int)c, op) : (int)c) * (S::CTA_COLS / 16);
        const GemvOp Pp = gemv_op<GROUPED, F32OUT>(a, op, ulist);
        const int trow = Pp.trow + tk_first;
        const CUtensorMap *tmT = maps + Pp.map;
        for (int r0 = 0; r0 < nrows && !*s_abort; r0 += S::R) {
          const int cnt = min(S::R, nrows - r0);
          if (issued++ == a.pre_stages) {
            // The first stages are in flight.  Hold the rest until the
            // consumers have made x': with every SM's whole ring queued the
            // x loads (and the first stages) wait behind those copies.  The
            // hardware wait covers the preceding kernel, so the bounded wait
            // only spans the x' prologue.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            if (!tc::mbar_wait(xready, 0)) {
              set_device_error(a.err, kErrBounds);
              *s_abort = 1;
              break;
            }
          }
          if (!tc::mbar_wait(&empty[stage], phase ^ 1)) {
            set_device_error(a.err, kErrBounds);
            *s_abort = 1;
            break;
          }
          // whole 8-row copies: rows past the block's end are outside the
          // tensor (zero-filled, not read); rows past the range's end are
          // loaded and ignored
          const int nb = (cnt + kGemvBoxRows - 1) / kGemvBoxRows;
          tc::mbar_arrive_expect_tx(&full[stage], (uint32_t)(nb * kGemvBoxRows * S::ROWB));
          uint8_t *dst = ring + (size_t)stage * S::STAGE_B;
          for (int b = 0; b < nb; ++b)
            tc::tma_load_3d(dst + (size_t)b * kGemvBoxRows * S::ROWB, tmT, &full[stage], 0, tn0,
                            trow + r0 + b * kGemvBoxRows);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        t = seg_end;
      }
    }
    return;
  }

  // Bring x and suh into L2 (one 128-byte line per thread) while the
  // preceding kernel finishes.  L2 is the point of coherence, so a line that
  // kernel writes later is still read current after the wait below.
  if (!GROUPED && warp < NCW) {
    const int lines = a.k >> 6;   // 64 fp16 per line
    for (int i = tid; i < 2 * lines; i += NCT) {
      const __half *p = i < lines ? a.x + (i << 6) : a.suh + ((i - lines) << 6);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
  }

  // Under a programmatic dependent launch the producer above is already
  // streaming weights; everything below (x, the workspace, y) waits until
  // the preceding kernel on the stream has completed and its writes are
  // visible.  Without one the wait returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == NCW + 1) {
    // ---------------- flusher: finishes each column block the consumers hand
    // over while they go on decoding the next one.  Lane l holds columns
    // 128 g + 4 l .. +3 of every 128-column group g.
    uint32_t sp = 0;
    const int op0 = GROUPED ? op_of_block(a, p, (int)(t0 / TKU)) : 0;
    for (uint32_t t = t0; t < t1;) {
      const int c = (int)(t / TKU);   // block: op c / colblocks, column block c % colblocks
      const uint32_t seg_end = min(t1, (uint32_t)(c + 1) * TKU);
      const int op = GROUPED ? op_of_block(a, p, c) : 0;
      const GemvOp P = gemv_op<GROUPED, F32OUT>(a, op, ulist);
      const int nop = GROUPED ? op_width(a, op) : a.n;
      const float *rs = rsum + (op - op0) * (a.k / 16);
      const int col0 = (GROUPED ? block_in_op(a, p, c, op) : c) * S::CTA_COLS;
      const uint32_t blk_first = (uint32_t)c * TKU, blk_last = min((uint32_t)(c + 1) * TKU, total) - 1;
      const int i_first = range_owner(blk_first, total, grid), i_last = range_owner(blk_last, total, grid);
      // A block shared by several CTAs is finished by whichever of them
      // publishes its partial sum last: each stores its partial in the slot
      // of (block, CTA) and makes one acquire-release increment of the
      // block's counter, and the one that sees every other arrival adds all
      // partials in CTA order (its own from registers, the same bits as the
      // stored one), so the result does not depend on timing and no CTA ever
      // waits for another.  The block's first CTA, whose range ends in it
      // (for the others it is the first segment, done long before), looks at
      // the counter without waiting, before and after its own segment; when
      // every other CTA is in it adds their partials straight away (loaded
      // while its consumers still decode) and publishes nothing.
      const bool shared = i_first != i_last, first = shared && me == i_first;
      const int others = i_last - i_first;
      float pre[kGemvPrePartials][S::NG][4];
      bool all_in = false;
      if (first) {
        all_in = gemv_all_arrived(a, p, c, others, lane);
        if (all_in) gemv_load_partials<S::NG>(p, c, i_first, others, lane, pre);
      }
      uint2 svv[S::NG];   // the block's svh (and bias), loaded ahead where this CTA usually finishes
      uint2 bvv[S::NG];
      const bool has_bias = !GROUPED && a.bias != nullptr;
      gemv_load_out_vectors<S::NG>(P.svh, has_bias ? a.bias : nullptr, col0, nop, lane, !shared || first, svv, bvv);
      if (!*s_abort && !tc::mbar_wait(seg_full, sp)) {
        if (lane == 0) set_device_error(a.err, kErrBounds);
        *s_abort = 1;
      }
      float v[S::NG][4];
#pragma unroll
      for (int g = 0; g < S::NG; ++g) {
        v[g][0] = v[g][1] = v[g][2] = v[g][3] = 0.f;
        for (int w = 0; w < NCW; ++w) {   // fixed order: the result does not depend on timing
          const float4 r = *reinterpret_cast<const float4 *>(red + w * S::CTA_COLS + g * 128 + lane * 4);
          v[g][0] += r.x;
          v[g][1] += r.y;
          v[g][2] += r.z;
          v[g][3] += r.w;
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(red_free);
      // every column's sum is 2^-49 sum x' B: remove 510 * (the segment's sum of x')
      float sg = 0.f;
      {
        const int tk_first = (int)(t - (uint32_t)c * TKU), nrows = (int)(seg_end - t);
        for (int r = lane; r < nrows; r += 32) sg += rs[tk_first + r];
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) sg += __shfl_xor_sync(0xffffffffu, sg, m);
      }
#pragma unroll
      for (int g = 0; g < S::NG; ++g)
#pragma unroll
        for (int e = 0; e < 4; ++e) v[g][e] = fmaf(-510.0f, sg, v[g][e] * kAccUnscale) * kSigma;

      bool finish = true;
      if (shared) {
        if (first && !all_in) {   // a second look, now that the own segment is done
          all_in = gemv_all_arrived(a, p, c, others, lane);
          if (all_in) gemv_load_partials<S::NG>(p, c, i_first, others, lane, pre);
        }
        if (first && all_in) {
          // every other CTA is in: add their partials in CTA order
#pragma unroll
          for (int j = 0; j < kGemvPrePartials; ++j)
            if (j < others)
#pragma unroll
              for (int g = 0; g < S::NG; ++g)
#pragma unroll
                for (int e = 0; e < 4; ++e) v[g][e] += pre[j][g][e];
          for (int i = i_first + 1 + kGemvPrePartials; i <= i_last; ++i) gemv_add_partial<S::NG>(p, c, i, lane, v);
        } else {
          // publish this CTA's partial and arrive; the last to arrive finishes
#pragma unroll
          for (int g = 0; g < S::NG; ++g)
            __stcg(reinterpret_cast<float4 *>(p.partials + (long)(c + me) * S::CTA_COLS + g * 128 + lane * 4),
                   make_float4(v[g][0], v[g][1], v[g][2], v[g][3]));
          __threadfence();
          __syncwarp();
          int old = 0;
          if (lane == 0)
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p.counters + c) : "memory");
          old = __shfl_sync(0xffffffffu, old, 0);
          if (old > others && lane == 0) set_device_error(a.err, kErrDirtyCounter);
          finish = old >= others;
          if (finish) {
            __threadfence();
            float own[S::NG][4];
#pragma unroll
            for (int g = 0; g < S::NG; ++g)
#pragma unroll
              for (int e = 0; e < 4; ++e) own[g][e] = v[g][e];
            for (int i = i_first; i <= i_last; ++i) {   // CTA order: p[i_first] + p[i_first + 1] + ...
              float pq[S::NG][4];
              if (i == me) {
#pragma unroll
                for (int g = 0; g < S::NG; ++g)
#pragma unroll
                  for (int e = 0; e < 4; ++e) pq[g][e] = own[g][e];
              } else {
                gemv_load_partial<S::NG>(p, c, i, lane, pq);
              }
#pragma unroll
              for (int g = 0; g < S::NG; ++g)
#pragma unroll
                for (int e = 0; e < 4; ++e) v[g][e] = i == i_first ? pq[g][e] : v[g][e] + pq[g][e];
            }
            if (!first) gemv_load_out_vectors<S::NG>(P.svh, has_bias ? a.bias : nullptr, col0, nop, lane, true, svv, bvv);
          }
        }
        if (finish && lane == 0) p.counters[c] = 0;   // leave the workspace clean
      }
      if (finish) {
        // ---- output transform of the block's 128-column groups
#pragma unroll
        for (int g = 0; g < S::NG; ++g) {
          const int gc = col0 + g * 128 + lane * 4;
          if (col0 + g * 128 < nop) {
            fwht128_warp(v[g], lane);
            const __half2 *sh = reinterpret_cast<const __half2 *>(&svv[g]);
            float o0 = v[g][0] * kRhtScale * __low2float(sh[0]);
            float o1 = v[g][1] * kRhtScale * __high2float(sh[0]);
            float o2 = v[g][2] * kRhtScale * __low2float(sh[1]);
            float o3 = v[g][3] * kRhtScale * __high2float(sh[1]);
            if (GROUPED) {   // the routing weight (or zero for an invalid expert id)
              o0 *= P.scale;
              o1 *= P.scale;
              o2 *= P.scale;
              o3 *= P.scale;
            }
            if (has_bias) {   // the output bias, per output feature
              const __half2 *bh = reinterpret_cast<const __half2 *>(&bvv[g]);
              o0 = __fadd_rn(o0, __low2float(bh[0]));   // one rounding, never contracted
              o1 = __fadd_rn(o1, __high2float(bh[0]));
              o2 = __fadd_rn(o2, __low2float(bh[1]));
              o3 = __fadd_rn(o3, __high2float(bh[1]));
            }
            if (F32OUT) {
              *reinterpret_cast<float4 *>(static_cast<float *>(P.y) + gc) = make_float4(o0, o1, o2, o3);
            } else {
              __half2 o[2] = {__floats2half2_rn(o0, o1), __floats2half2_rn(o2, o3)};
              *reinterpret_cast<uint2 *>(static_cast<__half *>(P.y) + gc) = *reinterpret_cast<uint2 *>(o);
            }
          }
        }
      }
      sp ^= 1;
      t = seg_end;
    }
    return;
  }

  // ---------------- consumers (warps 0..NCW-1)
  // prologue: x' = 2^-3.5 H (x . suh) for the 512-element chunks (32 tile
  // rows) this range touches; a warp transforms four 128-blocks at once,
  // eight lanes per block and 16 contiguous elements per lane
  const int op0 = GROUPED ? op_of_block(a, p, (int)(t0 / TKU)) : 0;
  if (GROUPED && me == 0) gemv_write_pos(a, tid, NCT);
  {
    const int KC = (a.k + 511) >> 9;
    int c0 = 0, nc = KC;
    if (GROUPED) {          // every chunk of each op the range touches (ops op0 ..)
      nc = (op_of_block(a, p, (int)((t1 - 1) / TKU)) - op0 + 1) * KC;
    } else if (t1 - t0 < TK) {   // fewer rows than one block: at most two column blocks
      c0 = (int)(t0 % TKU) >> 5;
      const int c1 = (int)((t1 - 1) % TKU) >> 5;
      const bool wrap = (t0 / TKU) != ((t1 - 1) / TKU);
      nc = !wrap ? c1 - c0 + 1 : (c1 >= c0 ? KC : KC - c0 + c1 + 1);
    }
    for (int i = warp; i < nc; i += NCW) {
      const int jop = GROUPED ? i / KC : 0;               // op op0 + jop
      const GemvOp P = gemv_op<GROUPED, F32OUT>(a, op0 + jop, ulist);
      if (GROUPED && P.bad && lane == 0 && i % KC == 0) set_device_error(a.err, kErrExpertId);
      const int e0 = ((c0 + i - jop * KC) % KC) * 512 + lane * 16;
      const bool live = e0 < a.k;   // k is a multiple of 128: whole 8-lane groups
      float *xso = xs + jop * a.k;
      float *rso = rsum + jop * (a.k / 16);
      float v[16];
      if (live && GROUPED && a.act_in) {
        // h = SiLU(g) u of this unit (fp32, the gate and up outputs), times suh
        const int u = P.unit;
        const float *g = a.act_in + (long)(2 * u) * a.k + e0, *up = g + a.k;
        uint4 sv[2];
        sv[0] = *reinterpret_cast<const uint4 *>(P.suh + e0);
        sv[1] = *reinterpret_cast<const uint4 *>(P.suh + e0 + 8);
        const __half *sh = reinterpret_cast<const __half *>(sv);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const float4 gg = *reinterpret_cast<const float4 *>(g + j), uu = *reinterpret_cast<const float4 *>(up + j);
          v[j] = gg.x / (1.0f + expf(-gg.x)) * uu.x * __half2float(sh[j]);
          v[j + 1] = gg.y / (1.0f + expf(-gg.y)) * uu.y * __half2float(sh[j + 1]);
          v[j + 2] = gg.z / (1.0f + expf(-gg.z)) * uu.z * __half2float(sh[j + 2]);
          v[j + 3] = gg.w / (1.0f + expf(-gg.w)) * uu.w * __half2float(sh[j + 3]);
        }
      } else if (live) {
        uint4 xv[2], sv[2];
        xv[0] = *reinterpret_cast<const uint4 *>(P.x + e0);
        xv[1] = *reinterpret_cast<const uint4 *>(P.x + e0 + 8);
        sv[0] = *reinterpret_cast<const uint4 *>(P.suh + e0);
        sv[1] = *reinterpret_cast<const uint4 *>(P.suh + e0 + 8);
        const __half2 *xh = reinterpret_cast<const __half2 *>(xv);
        const __half2 *sh = reinterpret_cast<const __half2 *>(sv);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[2 * j] = __low2float(xh[j]) * __low2float(sh[j]);
          v[2 * j + 1] = __high2float(xh[j]) * __high2float(sh[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.f;
      }
      fwht128_x8(v, lane);
      if (live) {
        float rs = 0.f;   // the 16 elements are one tile row
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          v[j] *= kRhtScale * kXScale;   // x' 2^100: the same rounding as x', then an exact scale
          rs += v[j];
        }
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<float4 *>(xso + e0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        rso[e0 >> 4] = rs * (1.0f / kXScale);
      }
    }
  }
  consumer_sync(NCT);
  if (tid == 0) tc::mbar_arrive(xready);

  const int wk = warp;
  const int tile_in_warp = lane / S::LPT, q = lane % S::LPT;
  const int my_off = tile_in_warp * 32 * K + q * 16 * S::CPL;                  // byte offset in a row
  const int next_off = tile_in_warp * 32 * K + ((q + 1) % S::LPT) * 16 * S::CPL;  // next row group (wraps)
  int stage = 0;
  uint32_t phase = 0, sp = 0;
  // Row g of the range (counted across its segments) belongs to warp
  // g mod NCW, so the partial stages at segment ends do not always give
  // their rows to the same warps: every warp has the same number of rows,
  // to within one, and the assignment stays fixed.
  uint32_t gbase = 0;

  for (uint32_t t = t0; t < t1;) {
    const int c = (int)(t / TKU);
    const uint32_t seg_end = min(t1, (uint32_t)(c + 1) * TKU);
    const int tk_first = (int)(t - (uint32_t)c * TKU), nrows = (int)(seg_end - t);
    const float *xso = xs + (GROUPED ? op_of_block(a, p, c) - op0 : 0) * a.k;   // this op's x' 2^100

    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;

    for (int r0 = 0; r0 < nrows; r0 += S::R) {
      const int cnt = min(S::R, nrows - r0);
      if (!*s_abort && !tc::mbar_wait(&full[stage], phase)) {
        if (lane == 0) set_device_error(a.err, kErrBounds);
        *s_abort = 1;
      }
      const uint8_t *sbase = ring + (size_t)stage * S::STAGE_B;
      const int j0 = (wk - (int)(gbase % NCW) + NCW) % NCW;
      gbase += cnt;
#pragma unroll
      for (int jj = 0; jj < S::RPW; ++jj) {
        const int j = j0 + jj * NCW;
        if (j < cnt) {
          uint32_t w[S::NW + 1];
          const uint8_t *rowp = sbase + (size_t)j * S::ROWB;
#pragma unroll
          for (int cc = 0; cc < S::CPL; ++cc) {
            const uint4 v4 = *reinterpret_cast<const uint4 *>(rowp + my_off + 16 * cc);
            w[4 * cc + 0] = v4.x;
            w[4 * cc + 1] = v4.y;
            w[4 * cc + 2] = v4.z;
            w[4 * cc + 3] = v4.w;
          }
          w[S::NW] = *reinterpret_cast<const uint32_t *>(rowp + next_off);
          const int tk = tk_first + r0 + j;
          float xr[S::G];
#pragma unroll
          for (int i = 0; i < S::G; i += 4) {
            const float4 x4 = *reinterpret_cast<const float4 *>(xso + tk * 16 + S::G * q + i);
            xr[i] = x4.x;
            xr[i + 1] = x4.y;
            xr[i + 2] = x4.z;
            xr[i + 3] = x4.w;
          }
          decode_accumulate<K, 0>(w, xr, acc);
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[stage]);
      if (++stage == STAGES) { stage = 0; phase ^= 1; }
    }

    // ---- hand the block over: reduce over the LPT lanes of a tile, then
    // leave this warp's column sums in red for the flusher
    float accf[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) accf[i] = acc[i];
#pragma unroll
    for (int m = 1; m < S::LPT; m <<= 1)
#pragma unroll
      for (int i = 0; i < 16; ++i) accf[i] += __shfl_xor_sync(0xffffffffu, accf[i], m);
    if (!*s_abort && !tc::mbar_wait(red_free, sp ^ 1)) {
      if (lane == 0) set_device_error(a.err, kErrBounds);
      *s_abort = 1;
    }
    if (q == 0) {
      float4 *dst = reinterpret_cast<float4 *>(red + wk * S::CTA_COLS + tile_in_warp * 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_float4(accf[4 * i], accf[4 * i + 1], accf[4 * i + 2], accf[4 * i + 3]);
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(seg_full);
    sp ^= 1;
    t = seg_end;
  }
}

// The partition of a launch over one width: every CTA of the grid.
__device__ __forceinline__ GemvPart gemv_whole_grid(const GemvArgs &a) {
  return GemvPart{(int)blockIdx.x, (int)gridDim.x, a.total, a.op_rows, nullptr, a.colblocks, a.stages, a.counters,
                  a.partials};
}

template <int K, bool F32OUT, bool GROUPED>
__global__ void __launch_bounds__(GemvShape<K>::THREADS, 1)
    gemv_m1_kernel(const __grid_constant__ CUtensorMap tmT, GemvArgs a) {
  gemv_body<K, F32OUT, GROUPED>(&tmT, a, gemv_whole_grid(a));
}

// Shards of different widths: one trellis map per shard.
struct GemvShardMaps {
  CUtensorMap m[kGemvMaxShards];
};

template <int K, bool F32OUT>
__global__ void __launch_bounds__(GemvShape<K>::THREADS, 1)
    gemv_shards_kernel(const __grid_constant__ GemvShardMaps maps, GemvArgs a) {
  gemv_body<K, F32OUT, true>(maps.m, a, gemv_whole_grid(a));
}

constexpr int kGemvThreads = GemvShape<4>::THREADS;   // the same for every width
static_assert(GemvShape<1>::THREADS == kGemvThreads && GemvShape<3>::THREADS == kGemvThreads &&
                  GemvShape<8>::THREADS == kGemvThreads,
              "one block size for every width");

// Routed experts of mixed widths for a few tokens, one launch per
// projection: the runs (at most 8, their tensor maps in `maps`) have widths
// run_K[r].  Every CTA counts the units of each width (warp ballots, 32
// units at a time), splits the grid over the widths in proportion to their
// weights (at least one CTA each, as many for every column block, no more
// CTAs than rows), lists its width's units in shared memory and runs the
// decode of its width on its share; the widths' column blocks have their
// own arrival counters and partial slots.
template <bool F32OUT>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_widths_kernel(const __grid_constant__ GemvShardMaps maps, GemvArgs a) {
  const int lane = threadIdx.x & 31, me = blockIdx.x;
  // width of unit u's expert (0: no run of this launch)
  auto width_of = [&](int u) -> int {
    if (u >= a.units) return 0;
    const int r = gemv_run_of(a, a.ids[u]);
    return r >= 0 ? a.run_K[r] : 0;
  };
  uint32_t count[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};   // units of each width (every warp counts them all)
  for (int base = 0; base < a.units; base += 32) {
    const int ku = width_of(base + lane);
    if (me == 0 && threadIdx.x < 32 && base + lane < a.units) {
      const int e = a.ids[base + lane];
      if (e < 0 || e >= a.E) set_device_error(a.err, kErrExpertId);
    }
#pragma unroll
    for (int w = 1; w <= 8; ++w) count[w] += (uint32_t)__popc(__ballot_sync(0xffffffffu, ku == w));
  }
  // Rows of odd widths hold 256 columns, of even widths 128: the CTAs are
  // split in proportion to each width's weights, so that every CTA decodes
  // about as many weights whatever its width.
  constexpr uint32_t cols_of[9] = {0,
                                   GemvShape<1>::CTA_COLS, GemvShape<2>::CTA_COLS, GemvShape<3>::CTA_COLS,
                                   GemvShape<4>::CTA_COLS, GemvShape<5>::CTA_COLS, GemvShape<6>::CTA_COLS,
                                   GemvShape<7>::CTA_COLS, GemvShape<8>::CTA_COLS};
  uint32_t rows[9];
  unsigned long long weights[9], all = 0;
  int nw = 0;
#pragma unroll
  for (int w = 1; w <= 8; ++w) {
    rows[w] = count[w] * (uint32_t)a.nslots * (uint32_t)a.wcolblocks[w] * (uint32_t)a.tiles_k;
    weights[w] = (unsigned long long)rows[w] * cols_of[w];
    all += weights[w];
    nw += rows[w] > 0;
  }
  const int G = gridDim.x;
  int wsel = 0, first = 0, cnt = 0;
  for (int w = 1, start = 0; w <= 8; ++w) {   // width w takes CTAs [start, start + c)
    if (rows[w] == 0) continue;
    int c = 1 + (int)((unsigned long long)(G - nw) * weights[w] / all);
    // as many CTAs for every column block of the width (block boundaries
    // then fall on CTA boundaries), at least kGemvMinRows rows each
    const int wblocks = (int)(rows[w] / (uint32_t)a.tiles_k);
    if (c >= wblocks) {
      int per = c / wblocks;
      while (per > 1 && a.tiles_k / per < kGemvMinRows) --per;
      c = per * wblocks;
    }
    if (me >= start && me < start + c) {
      wsel = w;
      first = start;
      cnt = c;
    }
    start += c;
  }
  if (wsel == 0) {   // no share: still complete after the kernel before this one
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (me == 0) gemv_write_pos(a, threadIdx.x, kGemvThreads);
    return;
  }
  // this width's units in unit order, past every width's shared-memory layout
  extern __shared__ __align__(128) uint8_t gw_smem[];
  int *ulist = reinterpret_cast<int *>(gw_smem + a.wlist_off);
  if (threadIdx.x < 32) {
    int pos = 0;
    for (int base = 0; base < a.units; base += 32) {
      const bool mine = width_of(base + lane) == wsel;
      const uint32_t bal = __ballot_sync(0xffffffffu, mine);
      if (mine) ulist[pos + __popc(bal & ((1u << lane) - 1u))] = base + lane;
      pos += __popc(bal);
    }
  }
  __syncthreads();
  GemvPart p;
  p.me = me - first;
  p.grid = (uint32_t)cnt < rows[wsel] ? cnt : (int)rows[wsel];   // every CTA taking part owns a row
  p.total = rows[wsel];
  p.ulist = ulist;
  p.colblocks = a.wcolblocks[wsel];
  p.op_rows = (uint32_t)p.colblocks * (uint32_t)a.tiles_k;
  p.stages = a.wstages[wsel];
  p.counters = a.counters + a.wcounter_base[wsel];
  p.partials = a.partials + a.wpartial_base[wsel];
  switch (wsel) {
    case 1: gemv_body<1, F32OUT, true>(maps.m, a, p); break;
    case 2: gemv_body<2, F32OUT, true>(maps.m, a, p); break;
    case 3: gemv_body<3, F32OUT, true>(maps.m, a, p); break;
    case 4: gemv_body<4, F32OUT, true>(maps.m, a, p); break;
    case 5: gemv_body<5, F32OUT, true>(maps.m, a, p); break;
    case 6: gemv_body<6, F32OUT, true>(maps.m, a, p); break;
    case 7: gemv_body<7, F32OUT, true>(maps.m, a, p); break;
    default: gemv_body<8, F32OUT, true>(maps.m, a, p); break;
  }
}

static int gemv_sm_count() { return exl3_sm_count(); }

static PFN_cuTensorMapEncodeTiled_v12000 gemv_tmap_fn() { return exl3_tmap_encode_fn(); }

template <int K, bool F32, bool GROUPED = false>
struct Launcher {
  using S = GemvShape<K>;
  // ring stages that fit beside the reduction buffers, x' (4 bytes per k)
  // and its per-tile-row sums (4 bytes per 16 k), for xops ops in GROUPED
  // mode
  static size_t xbytes(int k, int xops = kGemvMaxOps) {
    return (GROUPED ? xops : 1) * (4 * (size_t)k + (size_t)k / 4);
  }
  static int stages(int k, int xops = kGemvMaxOps, size_t reserve = 0) {
    const long avail = (long)kGemvSmemMax - S::FIXED_B - (long)xbytes(k, xops) - (long)reserve;
    long st = avail / S::STAGE_B;
    if (st > kGemvMaxStages) st = kGemvMaxStages;
    return (int)st;
  }
  static size_t smem(int k, int st, int xops = kGemvMaxOps) {
    return (size_t)st * S::STAGE_B + S::FIXED_B + xbytes(k, xops);
  }
  static cudaError_t launch(const CUtensorMap &tm, const GemvArgs &a, int grid, cudaStream_t s, bool prefetch) {
    const size_t sm = smem(a.k, a.stages, GROUPED ? a.xops : 1);
    static std::atomic<size_t> attr[kMaxDevices];   // per device: the attribute is per device
    cudaError_t e = exl3_ensure_smem(reinterpret_cast<const void *>(gemv_m1_kernel<K, F32, GROUPED>), sm, attr);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(S::THREADS);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = s;
    // programmatic dependent launch: CTAs may become resident (and stream
    // weights) while the preceding kernel on the stream finishes
    cfg.attrs = prefetch ? attrs : nullptr;
    cfg.numAttrs = prefetch ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_m1_kernel<K, F32, GROUPED>, tm, a);
  }
};

}  // namespace exl3

using namespace exl3;

#define EXL3_K_SWITCH(K, ...)                         \
  switch (K) {                                        \
    case 1: { constexpr int KK = 1; __VA_ARGS__; } break; \
    case 2: { constexpr int KK = 2; __VA_ARGS__; } break; \
    case 3: { constexpr int KK = 3; __VA_ARGS__; } break; \
    case 4: { constexpr int KK = 4; __VA_ARGS__; } break; \
    case 5: { constexpr int KK = 5; __VA_ARGS__; } break; \
    case 6: { constexpr int KK = 6; __VA_ARGS__; } break; \
    case 7: { constexpr int KK = 7; __VA_ARGS__; } break; \
    default: { constexpr int KK = 8; __VA_ARGS__; } break; \
  }

// Columns covered by one column block for width K (128 or 256).
int exl3_gemv_cta_cols(int K) {
  int r = 128;
  EXL3_K_SWITCH(K, r = GemvShape<KK>::CTA_COLS);
  return r;
}

// Whether the GEMV holds x' for this k beside two ring stages (otherwise
// the caller takes the tensor-core path).
bool exl3_gemv_fits(int k, int n, int K) {
  int st = 0;
  EXL3_K_SWITCH(K, st = Launcher<KK, false>::stages(k));
  const int cc = exl3_gemv_cta_cols(K);
  const unsigned long long total = (unsigned long long)((n + cc - 1) / cc) * (unsigned long long)(k / 16);
  return st >= 2 && total * (unsigned long long)gemv_sm_count() < (1ull << 32);
}

// Grid size (one CTA per SM, at most one per row) and the partial-sum slots
// (floats) the GEMV needs.
// One CTA per SM, or, with fewer column blocks than SMs, the same number of
// CTAs for every block so that block boundaries fall on CTA boundaries (no
// block is then shared, or each is shared evenly): taken when it keeps at
// least 80% of the SMs busy (n = 17408 at k = 5120: 136 CTAs of one block
// each ran 7% faster than 152 sharing blocks), or when one CTA per SM would
// get fewer than kGemvMinRows rows (a small matrix on every SM leaves each
// block split over dozens of CTAs, whose partials the block's finisher then
// adds one after another).  The equal ranges of the partition put block
// boundaries on CTA boundaries: CTA b per + j of g = blocks per starts at
// b rows_per_block + floor(j rows_per_block / per).
static long long gemv_grid_for(long long blocks, long long rows_per_block, long long sms) {
  const long long total = blocks * rows_per_block;
  long long g = sms;
  if (blocks < sms) {
    long long per = sms / blocks;   // CTAs per block
    while (per > 1 && rows_per_block / per < kGemvMinRows) --per;
    const long long aligned = blocks * per;
    if (5 * aligned >= 4 * sms || total / sms < kGemvMinRows) g = aligned;
  }
  return g > total ? total : g;
}

void exl3_gemv_plan(int k, int n, int K, int *grid, size_t *partial_floats) {
  const int cc = exl3_gemv_cta_cols(K);
  const long long colblocks = (n + cc - 1) / cc;
  const int g = (int)gemv_grid_for(colblocks, k / 16, gemv_sm_count());
  *grid = g;
  *partial_floats = (size_t)(colblocks + g) * (size_t)cc;
}

// bias: [n] fp16 added to the output (NULL: none).
cudaError_t exl3_launch_gemv_m1_bias(const uint16_t *x, const uint16_t *trellis, const uint16_t *suh,
                                     const uint16_t *svh, const uint16_t *bias, int k, int n, int K, void *y,
                                     bool f32out, float *partials, int *counters, int *err, int grid,
                                     cudaStream_t s, bool prefetch) {
  auto fn = gemv_tmap_fn();
  if (!fn) return cudaErrorNotSupported;
  const int cc = exl3_gemv_cta_cols(K);
  // trellis [k/16][n/16][32K bytes] as u64 (4K per tile): one copy brings 8
  // tile rows of the CTA_COLS / 16 tiles of a column block
  CUtensorMap tm;
  {
    cuuint64_t dims[3] = {(cuuint64_t)4 * K, (cuuint64_t)(n / 16), (cuuint64_t)(k / 16)};
    cuuint64_t strides[2] = {(cuuint64_t)32 * K, (cuuint64_t)(n / 16) * 32 * K};
    cuuint32_t box[3] = {(cuuint32_t)(4 * K), (cuuint32_t)(cc / 16), (cuuint32_t)kGemvBoxRows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint16_t *>(trellis), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  GemvArgs a{};
  a.xops = kGemvMaxOps;
  a.x = reinterpret_cast<const __half *>(x);
  a.suh = reinterpret_cast<const __half *>(suh);
  a.svh = reinterpret_cast<const __half *>(svh);
  a.y = y;
  a.partials = partials;
  a.counters = counters;
  a.err = err;
  a.k = k;
  a.n = n;
  a.tiles_k = k / 16;
  a.colblocks = (n + cc - 1) / cc;
  if ((unsigned long long)a.colblocks * a.tiles_k * (unsigned long long)grid >= (1ull << 32))
    return cudaErrorInvalidValue;
  a.total = (uint32_t)a.colblocks * (uint32_t)a.tiles_k;
  a.ids = nullptr;
  a.weights = nullptr;
  a.topk = a.nslots = a.nops = 1;
  a.E = a.x_per_unit = 0;
  a.op_rows = a.total;
  a.act_in = nullptr;
  a.pos_out = nullptr;
  a.var = 0;
  a.bias = reinterpret_cast<const __half *>(bias);
  a.pre_stages = kGemvPreStages;
  a.stages = 0;
  EXL3_K_SWITCH(K, a.stages = Launcher<KK, false>::stages(k));
  if (a.stages < 2) return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  if (f32out) {
    EXL3_K_SWITCH(K, e = Launcher<KK, true>::launch(tm, a, grid, s, prefetch));
  } else {
    EXL3_K_SWITCH(K, e = Launcher<KK, false>::launch(tm, a, grid, s, prefetch));
  }
  return e;
}

cudaError_t exl3_launch_gemv_m1(const uint16_t *x, const uint16_t *trellis, const uint16_t *suh,
                                const uint16_t *svh, int k, int n, int K, void *y, bool f32out,
                                float *partials, int *counters, int *err, int grid, cudaStream_t s,
                                bool prefetch) {
  return exl3_launch_gemv_m1_bias(x, trellis, suh, svh, nullptr, k, n, K, y, f32out, partials, counters, err, grid,
                                  s, prefetch);
}

// ---- routed experts for a few tokens: U * nslots M = 1 GEMVs in one launch

// Grid, partial-sum floats and arrival counters for nops = U * nslots ops of
// [k] x [k][n]; false when a CTA's range would touch more than kGemvMaxOps
// ops or x' for them does not fit beside two ring stages.
bool exl3_moe_gemv_plan(int U, int nslots, int k, int n, int K, int *grid, size_t *partial_floats, int *blocks,
                        int *xops) {
  const int cc = exl3_gemv_cta_cols(K);
  const long long colblocks = (n + cc - 1) / cc, op_rows = colblocks * (k / 16);
  const long long total = (long long)U * nslots * op_rows;
  const long long g = gemv_grid_for((long long)U * nslots * colblocks, k / 16, gemv_sm_count());
  if (g < 1) return false;
  if ((unsigned long long)total * (unsigned long long)g >= (1ull << 32)) return false;
  const long long range = (total + g - 1) / g;
  // x' slots for the ops a CTA's range may touch (at least kGemvMaxOps, at
  // most kGemvMaxOpsMoe), with two ring stages beside them
  const long long need = (range + op_rows - 1) / op_rows + 1;
  if (need > kGemvMaxOpsMoe) return false;
  const int xo = need > kGemvMaxOps ? (int)need : kGemvMaxOps;
  int st = 0;
  EXL3_K_SWITCH(K, st = Launcher<KK, true, true>::stages(k, xo));
  if (st < 2) return false;
  *grid = (int)g;
  *blocks = (int)(U * nslots * colblocks);
  *partial_floats = (size_t)(*blocks + g) * (size_t)cc;
  if (xops) *xops = xo;
  return true;
}

// Input: x [T][k] fp16, row u / topk for unit u (gate and up), or act_in
// [U][2][k] fp32, SiLU(gate) up of unit u (down); trellis: all experts'
// slots [E][nslots][k/16][n/16][16K];
// suh [E][nslots][k], svh [E][nslots][n]; y: [U * nslots][n] fp32, times
// weights[u] when weights is not NULL.
cudaError_t exl3_launch_moe_gemv(const uint16_t *x, const float *act_in, int *pos_out, const int32_t *ids,
                                 const float *weights, int U, int topk, int E, int nslots, int k, int n, int K,
                                 const uint16_t *trellis, const uint16_t *suh, const uint16_t *svh, float *y,
                                 float *partials, int *counters, int *err, cudaStream_t s) {
  auto fn = gemv_tmap_fn();
  if (!fn) return cudaErrorNotSupported;
  int grid = 0, blocks = 0;
  size_t pf = 0;
  int xo = kGemvMaxOps;
  if (!exl3_moe_gemv_plan(U, nslots, k, n, K, &grid, &pf, &blocks, &xo)) return cudaErrorInvalidValue;
  const int cc = exl3_gemv_cta_cols(K);
  // all experts' trellis as u64 rows: row (e nslots + slot) k/16 + tk
  CUtensorMap tm;
  {
    cuuint64_t dims[3] = {(cuuint64_t)4 * K, (cuuint64_t)(n / 16), (cuuint64_t)E * nslots * (k / 16)};
    cuuint64_t strides[2] = {(cuuint64_t)32 * K, (cuuint64_t)(n / 16) * 32 * K};
    cuuint32_t box[3] = {(cuuint32_t)(4 * K), (cuuint32_t)(cc / 16), (cuuint32_t)kGemvBoxRows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint16_t *>(trellis), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  GemvArgs a{};
  a.xops = kGemvMaxOps;
  a.x = reinterpret_cast<const __half *>(x);
  a.suh = reinterpret_cast<const __half *>(suh);
  a.svh = reinterpret_cast<const __half *>(svh);
  a.y = y;
  a.partials = partials;
  a.counters = counters;
  a.err = err;
  a.k = k;
  a.n = n;
  a.tiles_k = k / 16;
  a.colblocks = (n + cc - 1) / cc;
  a.ids = ids;
  a.weights = weights;
  a.topk = topk;
  a.nslots = nslots;
  a.E = E;
  a.x_per_unit = 0;
  a.act_in = act_in;
  a.pos_out = pos_out;
  a.var = 0;
  a.bias = nullptr;
  a.pre_stages = kGemvPreStages;
  a.nops = U * nslots;
  if ((unsigned long long)a.colblocks * a.tiles_k * a.nops * (unsigned long long)grid >= (1ull << 32))
    return cudaErrorInvalidValue;
  a.op_rows = (uint32_t)a.colblocks * (uint32_t)a.tiles_k;
  a.total = (uint32_t)a.nops * a.op_rows;
  a.stages = 0;
  a.xops = xo;
  EXL3_K_SWITCH(K, a.stages = Launcher<KK, true, true>::stages(k, xo));
  cudaError_t e = cudaSuccess;
  // The down projection (act_in set) is a programmatic dependent of the gate
  // and up launch: it streams its experts' weights (the expert ids are final
  // before that launch began) while gate and up finish, and reads their
  // outputs after griddepcontrol.wait.
  EXL3_K_SWITCH(K, e = Launcher<KK, true, true>::launch(tm, a, grid, s, act_in != nullptr));
  return e;
}

// ---- routed experts of mixed widths for a few tokens: every routed unit
// whose expert lies in one of `runs` runs (run r: experts e_lo[r] ..
// e_lo[r] + cnt[r] - 1 of width K[r], their nslots tensors packed from
// trellis + words[r]) as grouped M = 1 GEMVs, all widths in one launch.
// Arguments otherwise as exl3_launch_moe_gemv (y [U * nslots][n] fp32).
// partial_floats / counters_needed (optional): the sizes it uses.
// Units the mixed-width kernel takes: its unit list lives in shared memory.
constexpr int kGemvWidthsMaxUnits = 512;
static size_t gemv_list_bytes(int U) { return ((size_t)U * sizeof(int) + 15) & ~(size_t)15; }

bool exl3_moe_gemv_widths_plan(int U, int nslots, int k, int n, int runs, const int *K, int *grid,
                               size_t *partial_floats, int *counters_needed, int *xops) {
  if (runs < 1 || runs > kGemvMaxShards || U < 1 || U > kGemvWidthsMaxUnits) return false;
  const long long g = gemv_sm_count();
  bool seen[9] = {};
  int nw = 0;
  long long max_rows = 0;
  for (int r = 0; r < runs; ++r) {
    if (K[r] < 1 || K[r] > 8) return false;
    if (!seen[K[r]]) ++nw;
    seen[K[r]] = true;
  }
  if (g <= nw) return false;
  size_t pf = 0;
  int cnt = 0;
  long long max_weights = 0;   // of one width, had every unit that width
  for (int w = 1; w <= 8; ++w) {
    if (!seen[w]) continue;
    const int cc = exl3_gemv_cta_cols(w);
    const long long colblocks = (n + cc - 1) / cc, op_rows = colblocks * (k / 16);
    const long long rows = (long long)U * nslots * op_rows;
    max_rows += rows;
    if (rows * cc > max_weights) max_weights = rows * cc;
    pf += (size_t)(U * nslots * colblocks + g) * (size_t)cc;
    cnt += (int)(U * nslots * colblocks);
  }
  // The device splits the CTAs over the widths in proportion to their
  // weights, so a CTA of width w gets at most about (all weights) / (cols(w)
  // (g - nw)) rows; all weights are at most max_weights (units of one
  // width's weights add up to at most what all U units would have at the
  // width with the most).  The x' slots cover the ops such a share touches
  // (at least kGemvMaxOps, at most kGemvMaxOpsMoe), with two ring stages
  // beside them and the unit list.
  int xo = kGemvMaxOps;
  for (int w = 1; w <= 8; ++w) {
    if (!seen[w]) continue;
    const int cc = exl3_gemv_cta_cols(w);
    const long long op_rows = ((n + cc - 1) / cc) * (k / 16);
    const long long range = (max_weights + (long long)cc * (g - nw) - 1) / ((long long)cc * (g - nw)) + 1;
    const long long need = (range + op_rows - 1) / op_rows + 1;
    if (need > kGemvMaxOpsMoe) return false;
    if (need > xo) xo = (int)need;
    if ((unsigned long long)max_rows * (unsigned long long)g >= (1ull << 32)) return false;
  }
  for (int w = 1; w <= 8; ++w) {
    if (!seen[w]) continue;
    int st = 0;
    EXL3_K_SWITCH(w, st = Launcher<KK, true, true>::stages(k, xo, gemv_list_bytes(U)));
    if (st < 2) return false;
  }
  if (xops) *xops = xo;
  *grid = (int)g;
  if (partial_floats) *partial_floats = pf;
  if (counters_needed) *counters_needed = cnt;
  return true;
}

cudaError_t exl3_launch_moe_gemv_widths(const uint16_t *x, const float *act_in, int *pos_out, const int32_t *ids,
                                        const float *weights, int U, int topk, int E, int nslots, int k, int n,
                                        int runs, const int *K, const int *e_lo, const int *cnt, const size_t *words,
                                        const uint16_t *trellis, const uint16_t *suh, const uint16_t *svh, float *y,
                                        float *partials, int *counters, int *err, cudaStream_t s, bool prefetch) {
  auto fn = gemv_tmap_fn();
  if (!fn) return cudaErrorNotSupported;
  int grid = 0, xo = kGemvMaxOps;
  if (!exl3_moe_gemv_widths_plan(U, nslots, k, n, runs, K, &grid, nullptr, nullptr, &xo)) return cudaErrorInvalidValue;
  GemvShardMaps maps;
  memset(&maps, 0, sizeof maps);
  GemvArgs a{};
  a.xops = kGemvMaxOps;
  for (int r = 0; r < runs; ++r) {   // run r's experts' trellis as u64 rows: row (e' nslots + slot) k/16 + tk
    const int cc = exl3_gemv_cta_cols(K[r]);
    cuuint64_t dims[3] = {(cuuint64_t)4 * K[r], (cuuint64_t)(n / 16), (cuuint64_t)cnt[r] * nslots * (k / 16)};
    cuuint64_t strides[2] = {(cuuint64_t)32 * K[r], (cuuint64_t)(n / 16) * 32 * K[r]};
    cuuint32_t box[3] = {(cuuint32_t)(4 * K[r]), (cuuint32_t)(cc / 16), (cuuint32_t)kGemvBoxRows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult rr = fn(&maps.m[r], CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint16_t *>(trellis) + words[r], dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (rr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    a.run_lo[r] = e_lo[r];
    a.run_hi[r] = e_lo[r] + cnt[r];
    a.run_K[r] = K[r];
  }
  // per width: column blocks, ring stages, and the first counter and
  // partial slot of its blocks; the shared memory is the largest width's,
  // then the unit list
  a.xops = xo;
  const size_t list = gemv_list_bytes(U);
  size_t sm = 0;
  int cbase = 0;
  size_t pbase = 0;
  bool seen[9] = {};
  for (int r = 0; r < runs; ++r) seen[K[r]] = true;
  for (int w = 1; w <= 8; ++w) {
    if (!seen[w]) continue;
    const int cc = exl3_gemv_cta_cols(w);
    a.wcolblocks[w] = (n + cc - 1) / cc;
    EXL3_K_SWITCH(w, a.wstages[w] = Launcher<KK, true, true>::stages(k, xo, list);
                  sm = std::max(sm, Launcher<KK, true, true>::smem(k, a.wstages[w], xo)));
    a.wcounter_base[w] = cbase;
    a.wpartial_base[w] = (int)pbase;
    cbase += U * nslots * a.wcolblocks[w];
    pbase += (size_t)(U * nslots * a.wcolblocks[w] + grid) * (size_t)cc;
  }
  a.wlist_off = (int)((sm + 15) & ~(size_t)15);
  sm = (size_t)a.wlist_off + list;
  a.runs = runs;
  a.units = U;
  a.x = reinterpret_cast<const __half *>(x);
  a.suh = reinterpret_cast<const __half *>(suh);
  a.svh = reinterpret_cast<const __half *>(svh);
  a.y = y;
  a.partials = partials;
  a.counters = counters;
  a.err = err;
  a.k = k;
  a.n = n;
  a.tiles_k = k / 16;
  a.ids = ids;
  a.weights = weights;
  a.topk = topk;
  a.nslots = nslots;
  a.E = E;
  a.act_in = act_in;
  a.pos_out = pos_out;
  a.pre_stages = kGemvPreStages;
  a.nops = U * nslots;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  cfg.attrs = prefetch ? attrs : nullptr;
  cfg.numAttrs = prefetch ? 1 : 0;
  static std::atomic<size_t> attr[kMaxDevices];
  cudaError_t e = exl3_ensure_smem(reinterpret_cast<const void *>(gemv_widths_kernel<true>), sm, attr);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, gemv_widths_kernel<true>, maps, a);
}

// ---- fused shards: S linears of one input row, [S][k/16][n/16][16K]
// trellis, suh [S][k], svh [S][n], y [S][n], in one launch of the grouped
// GEMV (one unit, S slots, no expert ids).  False when a CTA's range would
// touch more than kGemvMaxOps shards or x' for them does not fit.
bool exl3_gemv_shards_plan(int S, int k, int n, int K, int *grid, size_t *partial_floats, int *blocks) {
  int xo = kGemvMaxOps;
  if (!exl3_moe_gemv_plan(1, S, k, n, K, grid, partial_floats, blocks, &xo)) return false;
  return xo <= kGemvMaxOps;   // the shards' launch keeps kGemvMaxOps x' slots
}

cudaError_t exl3_launch_gemv_shards(const uint16_t *x, int S, int k, int n, int K, const uint16_t *trellis,
                                    const uint16_t *suh, const uint16_t *svh, void *y, bool f32out,
                                    float *partials, int *counters, int *err, cudaStream_t s, bool prefetch) {
  auto fn = gemv_tmap_fn();
  if (!fn) return cudaErrorNotSupported;
  int grid = 0, blocks = 0;
  size_t pf = 0;
  if (!exl3_gemv_shards_plan(S, k, n, K, &grid, &pf, &blocks)) return cudaErrorInvalidValue;
  const int cc = exl3_gemv_cta_cols(K);
  // the shards' trellis as u64 rows: row s k/16 + tk
  CUtensorMap tm;
  {
    cuuint64_t dims[3] = {(cuuint64_t)4 * K, (cuuint64_t)(n / 16), (cuuint64_t)S * (k / 16)};
    cuuint64_t strides[2] = {(cuuint64_t)32 * K, (cuuint64_t)(n / 16) * 32 * K};
    cuuint32_t box[3] = {(cuuint32_t)(4 * K), (cuuint32_t)(cc / 16), (cuuint32_t)kGemvBoxRows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint16_t *>(trellis), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  GemvArgs a{};
  a.xops = kGemvMaxOps;
  a.x = reinterpret_cast<const __half *>(x);
  a.suh = reinterpret_cast<const __half *>(suh);
  a.svh = reinterpret_cast<const __half *>(svh);
  a.y = y;
  a.partials = partials;
  a.counters = counters;
  a.err = err;
  a.k = k;
  a.n = n;
  a.tiles_k = k / 16;
  a.colblocks = (n + cc - 1) / cc;
  a.ids = nullptr;
  a.weights = nullptr;
  a.topk = 1;
  a.nslots = S;
  a.E = 1;
  a.x_per_unit = 0;
  a.act_in = nullptr;
  a.pos_out = nullptr;
  a.var = 0;
  a.bias = nullptr;
  a.pre_stages = kGemvPreStages;
  a.nops = S;
  if ((unsigned long long)a.colblocks * a.tiles_k * a.nops * (unsigned long long)grid >= (1ull << 32))
    return cudaErrorInvalidValue;
  a.op_rows = (uint32_t)a.colblocks * (uint32_t)a.tiles_k;
  a.total = (uint32_t)a.nops * a.op_rows;
  a.stages = 0;
  EXL3_K_SWITCH(K, a.stages = Launcher<KK, true, true>::stages(k));
  cudaError_t e = cudaSuccess;
  if (f32out) {
    EXL3_K_SWITCH(K, e = Launcher<KK, true, true>::launch(tm, a, grid, s, prefetch));
  } else {
    EXL3_K_SWITCH(K, e = Launcher<KK, false, true>::launch(tm, a, grid, s, prefetch));
  }
  return e;
}

// ---- shards of different widths: shard s has n[s] (host) output columns, its
// trellis [k/16][n[s]/16][16K] right after shard s-1's, suh [S][k], svh and y
// the concatenated [sum n] vectors; one launch with a tensor map per shard.
// False when S is outside 1..kGemvMaxShards, a CTA's range would touch more
// than kGemvMaxOps shards, or x' for them does not fit.
bool exl3_gemv_shards_var_plan(int S, int k, const int *n, int K, int *grid, size_t *partial_floats, int *blocks) {
  if (S < 1 || S > kGemvMaxShards) return false;
  const int cc = exl3_gemv_cta_cols(K);
  long long vb[kGemvMaxShards + 1];
  vb[0] = 0;
  for (int i = 0; i < S; ++i) vb[i + 1] = vb[i] + (n[i] + cc - 1) / cc;
  const long long TK = k / 16, total = vb[S] * TK;
  long long g = gemv_sm_count();
  if (g > total) g = total;
  if (g < 1 || (unsigned long long)total * (unsigned long long)g >= (1ull << 32)) return false;
  auto op_of = [&](long long c) {
    int o = 0;
    for (int i = 1; i < S; ++i)
      if (c >= vb[i]) o = i;
    return o;
  };
  for (long long i = 0; i < g; ++i) {   // the kernel's split: CTA i takes rows [i total / g, (i + 1) total / g)
    const long long r0 = i * total / g, r1 = (i + 1) * total / g;
    if (r1 > r0 && op_of((r1 - 1) / TK) - op_of(r0 / TK) + 1 > kGemvMaxOps) return false;
  }
  int st = 0;
  EXL3_K_SWITCH(K, st = Launcher<KK, true, true>::stages(k));
  if (st < 2) return false;
  *grid = (int)g;
  *blocks = (int)vb[S];
  *partial_floats = (size_t)(vb[S] + g) * (size_t)cc;
  return true;
}

cudaError_t exl3_launch_gemv_shards_var(const uint16_t *x, int S, int k, const int *n, int K, const uint16_t *trellis,
                                        const uint16_t *suh, const uint16_t *svh, void *y, bool f32out,
                                        float *partials, int *counters, int *err, cudaStream_t s, bool prefetch) {
  auto fn = gemv_tmap_fn();
  if (!fn) return cudaErrorNotSupported;
  int grid = 0, blocks = 0;
  size_t pf = 0;
  if (!exl3_gemv_shards_var_plan(S, k, n, K, &grid, &pf, &blocks)) return cudaErrorInvalidValue;
  const int cc = exl3_gemv_cta_cols(K);
  GemvShardMaps maps;
  memset(&maps, 0, sizeof maps);
  GemvArgs a{};
  memset(&a, 0, sizeof a);
  a.xops = kGemvMaxOps;
  size_t words = 0;
  int vo = 0, vb = 0;
  for (int i = 0; i < S; ++i) {
    cuuint64_t dims[3] = {(cuuint64_t)4 * K, (cuuint64_t)(n[i] / 16), (cuuint64_t)(k / 16)};
    cuuint64_t strides[2] = {(cuuint64_t)32 * K, (cuuint64_t)(n[i] / 16) * 32 * K};
    cuuint32_t box[3] = {(cuuint32_t)(4 * K), (cuuint32_t)(cc / 16), (cuuint32_t)kGemvBoxRows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(&maps.m[i], CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint16_t *>(trellis) + words, dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    words += (size_t)(k / 16) * (n[i] / 16) * 16 * K;
    a.vn[i] = n[i];
    a.vo[i] = vo;
    a.vb[i] = vb;
    vo += n[i];
    vb += (n[i] + cc - 1) / cc;
  }
  a.vb[S] = vb;
  a.var = S;
  a.x = reinterpret_cast<const __half *>(x);
  a.suh = reinterpret_cast<const __half *>(suh);
  a.svh = reinterpret_cast<const __half *>(svh);
  a.y = y;
  a.partials = partials;
  a.counters = counters;
  a.err = err;
  a.k = k;
  a.n = vo;
  a.tiles_k = k / 16;
  a.colblocks = vb;
  a.ids = nullptr;
  a.weights = nullptr;
  a.topk = 1;
  a.nslots = S;
  a.E = 1;
  a.nops = S;
  a.bias = nullptr;
  a.pre_stages = kGemvPreStages;
  a.total = (uint32_t)vb * (uint32_t)a.tiles_k;
  a.op_rows = a.total;
  EXL3_K_SWITCH(K, a.stages = Launcher<KK, true, true>::stages(k));
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.stream = s;
  cfg.attrs = prefetch ? attrs : nullptr;
  cfg.numAttrs = prefetch ? 1 : 0;
  cudaError_t e = cudaSuccess;
#define EXL3_GSV(KK, F32)                                                                                    \
  do {                                                                                                     \
    const size_t sm = Launcher<KK, F32, true>::smem(k, a.stages);                                          \
    static std::atomic<size_t> attr[kMaxDevices];                                                          \
    e = exl3_ensure_smem(reinterpret_cast<const void *>(gemv_shards_kernel<KK, F32>), sm, attr);           \
    if (e != cudaSuccess) break;                                                                           \
    cfg.blockDim = dim3(GemvShape<KK>::THREADS);                                                           \
    cfg.dynamicSmemBytes = sm;                                                                             \
    e = cudaLaunchKernelEx(&cfg, gemv_shards_kernel<KK, F32>, maps, a);                                    \
  } while (0)
  if (f32out) {
    EXL3_K_SWITCH(K, EXL3_GSV(KK, true));
  } else {
    EXL3_K_SWITCH(K, EXL3_GSV(KK, false));
  }
#undef EXL3_GSV
  return e;
}
