// moe_fused.cu -- the two grouped expert projections with the trellis decoded
// straight into tcgen05 operands ("Bringing EXL3 Trellis Quantization to 35B
// MoE on Intel Arc 140V", section 2.B: one grouped launch for gate+up with a
// shared input row, one for down; "exl3xpu" README, "MoE (routed experts)":
// routing weight on the down output, in fp32, and no fp16 expert weights
// anywhere).
//
// A CTA handles one (expert tile, 128-column output tile) pair of the
// device-side tile list.  A tile holds up to NMAX routed rows of one expert
// (NMAX = 32 when the call routes few rows per expert; 160 or 256 when it
// routes many (160 keeps three x' stages in shared memory, 256 holds more
// rows per expert) and the widths fit; else 128); the MMA
// computes the transposed product (decoded weights as the MN-major A operand,
// M = 128 output columns; the tile's x' rows as the K-major B operand, N =
// the tile's rows rounded up to 16).  Roles (2 + NISS + 16 warps):
//   warp 0         trellis producer: one tensor load per projection and stage
//                  over all experts' trellis (16 tile rows per stage)
//   warps 1..NISS  MMA issuers: pair P goes to issuer P mod NISS, into that
//                  issuer's own accumulators (summed in a fixed order by the
//                  epilogue); four issuers for 32-row tiles, two for 128, one
//                  for 256 (TMEM holds 512 columns)
//   next 16 warps  decoders in two groups of eight, taking alternate "pairs":
//                  phase 1 a pair is the gate and up weights of one k step,
//                  phase 2 two k steps of down; one fence and one signal per pair
//   last warp      x' producer: the pair's B operands in one or two loads
//
// Pair P uses weight slot P mod NPS and x' slot P mod XS; both ring sizes
// are multiples of NISS (and NPS of the two decoder groups), so every slot
// has one issuer and its waits on the slot's barriers are for consecutive
// phases (a waiter never sees an older phase of the same parity).
//
// Phase 1 (gate + up): per token row the epilogue forms
//   g = RHT_out(gate) . svh_gate, u = RHT_out(up) . svh_up, h = SiLU(g) u and
//   the down projection's input transform h' = 2^-3.5 H (h . suh_down).
// Phase 2 (down): d = RHT_out(h' Wdown) . svh_down * routing weight (fp32).
#include <cudaTypedefs.h>

#include "fused_decode.cuh"

namespace exl3 {
namespace mf {

using ftc::BK;
using ftc::BN;
using ftc::NDEC;
using ftc::NGRP;
using ftc::W_BYTES;

template <int NMAX>
struct Roles {
  static constexpr int NISS = NMAX <= 32 ? 4 : (NMAX <= 128 ? 2 : 1);   // MMA issuer warps
  static constexpr int DEC0 = 1 + NISS;                  // first decoder warp
  static constexpr int XWARP = DEC0 + NGRP * NDEC;       // the x' producer
  static constexpr int WARPS = XWARP + 1;
};

template <int K, int PHASE, int NMAX>
struct Cfg {
  static constexpr int NISS = Roles<NMAX>::NISS;
  static constexpr int XROWS = NMAX;                    // rows of a tile (largest MMA N)
  static constexpr int X_STEP = XROWS * BK * 2;         // B operand of one k step
  static constexpr int NP = PHASE == 1 ? 2 : 1;         // projections (accumulators per issuer)
  static constexpr int ROWB = (BN / 16) * 32 * K;       // one tile row of the CTA's 8 tiles
  static constexpr int T_STAGE = 16 * ROWB;             // two pairs
  static constexpr int X_STAGE = 2 * X_STEP;            // one pair
  static constexpr int BUDGET = 227 * 1024 - 2048;
  // pair slots of the weight ring: 4 where they fit beside two x' and two
  // trellis stages, else 2 (a multiple of the issuers and of the groups)
  static constexpr int NPS_FIT4 = (BUDGET - 8 * W_BYTES - 2 * X_STAGE - 2 * T_STAGE) >= 0;
  static constexpr int NPS = (NPS_FIT4 || NISS > 2) ? 4 : 2;
  // the epilogue transposes the accumulators into a scratch over the rings,
  // ECH rows at a time
  static constexpr int ECH = NMAX < 128 ? NMAX : 128;
  static constexpr int W_RING = 2 * NPS * W_BYTES;
  // x' ring: as deep as the budget allows after two trellis stages (the
  // loads come from L2 or HBM and must run several pairs ahead), a multiple
  // of the issuers
  static constexpr int XS_FIT = (BUDGET - W_RING - 2 * T_STAGE) / X_STAGE;
  static constexpr int XS = (XS_FIT >= 4 ? 4 : XS_FIT) / NISS * NISS;
  static constexpr int TS_FIT = (BUDGET - W_RING - XS * X_STAGE) / T_STAGE;
  static constexpr int TS = TS_FIT > 8 ? 8 : TS_FIT;
  static constexpr int SMEM_BYTES = XS * X_STAGE + W_RING + TS * T_STAGE + 2048;
  static constexpr int ITEMS = 32 * ftc::Shape<K, 32>::LPT;  // items per (k step, projection)
  // phase 2 may take several output tiles per CTA (one accumulator set
  // each): four with 32-row tiles, two otherwise (TMEM holds 512 columns)
  static constexpr int NTC = PHASE == 2 ? (NMAX <= 32 ? 4 : 2) : 1;
  static constexpr uint32_t TMEM_COLS = NISS * NP * XROWS * NTC;
  // the allocation: the next power of two (160-row tiles use 320 columns)
  static constexpr uint32_t TMEM_ALLOC = TMEM_COLS <= 32 ? 32 : TMEM_COLS <= 64 ? 64 : TMEM_COLS <= 128 ? 128
                                         : TMEM_COLS <= 256 ? 256 : 512;
  // whether this width and tile capacity fit (256-row tiles leave room for
  // K <= 4 only); the host launches only configurations that do
  static constexpr bool OK = TS >= 2 && XS >= NISS && NPS % NISS == 0 && NPS % NGRP == 0 && XS % NISS == 0 &&
                             NTC * NP * ECH * 128 * 4 <= XS * X_STAGE + W_RING && TMEM_COLS <= 512 &&
                             SMEM_BYTES <= 227 * 1024;
};

struct Args {
  const int4 *mtiles;       // (expert, first row, rows, 0)
  const int *n_mtiles;
  int NT, KB;               // output tiles per m-tile, k steps
  int tiles_k, nslots;      // trellis rows of one projection, projections per expert
  const __half *svh13;      // [E][2][inter]
  const __half *suh2;       // [E][inter]
  __half *hout;             // [U][inter]
  int inter;
  const __half *svh2;       // [E][hidden]
  const float *weights;     // [U] routing weight by unit
  const int *perm;          // sorted row -> unit
  float *dout;              // [U][hidden]
  int hidden;
  int *err;
  // phase 1 split over k (small token counts): CTA blockIdx.x takes split
  // blockIdx.x % splits of tile blockIdx.x / splits; the last CTA of a tile
  // to arrive adds the partial sums in split order
  int splits;
  int ntc;                  // output tiles per CTA (phase 2: 1, 2 or 4, at most Cfg::NTC)
  float *partials;          // [tiles][splits][2][NMAX][128] fp32 (splits > 1 only with NMAX <= 128)
  int *counters;            // [tiles], zero between calls
  // experts [e_lo, e_hi) only: the trellis map covers just their arena
  // (row 0 = expert e_lo) and tiles of other experts are left to other launches
  int e_lo, e_hi;
};

template <int K, int PHASE, int NMAX>
__global__ void __launch_bounds__(Roles<NMAX>::WARPS * 32, 1)
    moe_fused_kernel(const __grid_constant__ CUtensorMap tmX0, const __grid_constant__ CUtensorMap tmX1,
                     const __grid_constant__ CUtensorMap tmT, Args a) {
  using C = Cfg<K, PHASE, NMAX>;
  using S = ftc::Shape<K, 32>;
  static_assert(C::OK, "rings, TMEM and shared memory fit this width and tile capacity");
  constexpr int NP = C::NP, XS = C::XS, TS = C::TS, NPS = C::NPS, NISS = C::NISS, XROWS = C::XROWS;
  constexpr int kDec0 = Roles<NMAX>::DEC0, kXWarp = Roles<NMAX>::XWARP;
  const int tile = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
  // output tiles nt0 .. nt0 + nts - 1 (phase 2 may take several: their
  // pairs follow one another, tile j's pair Pt being pair j * nptile + Pt)
  pdl_trigger();   // the chain's kernels are programmatic dependents of one another
  pdl_wait();      // the tile list and x' come from the kernels before
  const int ntc = PHASE == 2 ? a.ntc : 1, NTG = (a.NT + ntc - 1) / ntc;
  if (tile >= *a.n_mtiles * NTG) return;   // uniform per CTA: the tile list is device-side
  const int4 mt = a.mtiles[tile / NTG];
  const int nt0 = (tile % NTG) * ntc, nts = min(ntc, a.NT - nt0), e = mt.x, row0 = mt.y, rows = mt.z;
  if (e < a.e_lo || e >= a.e_hi) return;   // uniform per CTA: another launch's expert
  const int et = e - a.e_lo;                // the expert's place in this launch's trellis map
  const int npad = (rows + 15) & ~15;       // MMA N: the tile's rows rounded up to 16
  const int KB = a.KB;
  // this CTA's pairs: absolute pair P0 + P for P < npairs (P0 even, so a
  // trellis stage still holds pairs 2j, 2j + 1 of the range; with two tiles
  // nptile is even, so no stage spans them)
  const int nptile = (PHASE == 1 ? KB : KB / 2) / a.splits;
  const int npairs = nptile * nts;
  const int P0 = split * npairs;
  const int ntst = (npairs + 1) / 2;                 // a trellis stage holds two pairs

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t *sX = smem;                                   // [XS][X_STAGE]
  uint8_t *sW = sX + XS * C::X_STAGE;                   // [2 NPS][W_BYTES]
  uint8_t *sT = sW + C::W_RING;                         // [TS][T_STAGE]
  uint64_t *tfull = reinterpret_cast<uint64_t *>(sT + TS * C::T_STAGE);
  uint64_t *tempty = tfull + TS;
  uint64_t *xfull = tempty + TS;
  uint64_t *xempty = xfull + XS;
  uint64_t *wfull = xempty + XS;
  uint64_t *wempty = wfull + NPS;
  uint64_t *accum = wempty + NPS;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *s_last = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < TS; ++st) {
      tc::mbar_init(&tfull[st], 1);
      tc::mbar_init(&tempty[st], NGRP * NDEC);   // every decoder warp, once per stage
    }
    for (int st = 0; st < XS; ++st) {
      tc::mbar_init(&xfull[st], 1);
      tc::mbar_init(&xempty[st], 1);             // the issuer of the stage's pair
    }
    for (int st = 0; st < NPS; ++st) {
      tc::mbar_init(&wfull[st], NDEC);           // one group's warps, once per pair
      tc::mbar_init(&wempty[st], 1);
    }
    tc::mbar_init(accum, NISS);
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmX0);
    if (PHASE == 1) tc::prefetch_tmap(&tmX1);
    tc::prefetch_tmap(&tmT);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::TMEM_ALLOC);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- trellis producer.  Phase 1: per projection 8 tile rows
    // (two k steps); phase 2: 16 tile rows (four k steps).
    if (lane == 0) {
      for (int j = 0; j < ntst && !*abort_flag; ++j) {
        const int st = j % TS;
        if (!tc::mbar_wait_backoff(&tempty[st], ((j / TS) & 1) ^ 1)) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&tfull[st], C::T_STAGE);
        if (PHASE == 1) {
#pragma unroll
          for (int p = 0; p < 2; ++p)
            tc::tma_load_2d(sT + st * C::T_STAGE + p * 8 * C::ROWB, &tmT, &tfull[st], nt0 * (BN / 16) * (4 * K),
                            (et * a.nslots + p) * a.tiles_k + 4 * P0 + 8 * j);
        } else {
          const int jt = (2 * j) / nptile, js = j - jt * (nptile / 2);   // tile, stage within its k
          tc::tma_load_2d(sT + st * C::T_STAGE, &tmT, &tfull[st], (nt0 + jt) * (BN / 16) * (4 * K),
                          et * a.tiles_k + 16 * js);
        }
      }
    }
  } else if (warp == kXWarp) {
    // ---------------- x' producer: the pair's two B operands (phase 1: x'g
    // and x'u of k step P; phase 2: h' of k steps 2P, 2P + 1), XROWS rows each
    if (lane == 0) {
      for (int P = 0; P < npairs && !*abort_flag; ++P) {
        const int st = P % XS;
        if (!tc::mbar_wait_backoff(&xempty[st], ((P / XS) & 1) ^ 1)) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&xfull[st], C::X_STAGE);
        if (PHASE == 1) {
          tc::tma_load_2d(sX + st * C::X_STAGE, &tmX0, &xfull[st], (P0 + P) * BK, row0);
          tc::tma_load_2d(sX + st * C::X_STAGE + C::X_STEP, &tmX1, &xfull[st], (P0 + P) * BK, row0);
        } else {
          tc::tma_load_3d(sX + st * C::X_STAGE, &tmX0, &xfull[st], 0, row0, 2 * (P % nptile));
        }
      }
    }
  } else if (warp <= NISS) {
    // ---------------- MMA issuers: warp 1 + g takes the pairs P = g, g + NISS,
    // ... into accumulators (jt NISS NP + g NP + p) * XROWS (phase 1: p =
    // gate, up; jt: the CTA's output tile).  The first pair of a tile that
    // an issuer sees is among the tile's first NISS pairs.  The whole warp
    // runs the loop (waits and descriptors stay warp-uniform); one elected
    // lane issues the MMAs and their commits.
    const int g = __shfl_sync(0xffffffffu, warp, 0) - 1;
    const uint32_t idesc = ftc::idesc_f16_amn(BN, npad);
    bool stop = false;
    for (int P = g; P < npairs; P += NISS) {
      const int xs = P % XS, ps = P % NPS;
      bool ok = tc::mbar_wait(&xfull[xs], (P / XS) & 1) && tc::mbar_wait(&wfull[ps], (P / NPS) & 1);
      ok = __all_sync(0xffffffffu, ok && !*abort_flag);
      if (!ok) {
        if (lane == 0) set_device_error(a.err, kErrBounds);
        *abort_flag = 1;
        stop = true;
        break;
      }
      tc::tc_fence_after();
      const int jt = P / nptile, Pt = P - jt * nptile;
      if (tc::elect_one()) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int p = PHASE == 1 ? h : 0;
          const uint32_t dcol = tmem_base + (uint32_t)(((jt * NISS + g) * NP + p) * XROWS);
          const uint64_t ad = ftc::sdesc_mn_sw128(sW + (2 * ps + h) * W_BYTES, 1024, 2048);
          const uint64_t bd = tc::sdesc_k_sw128(sX + xs * C::X_STAGE + h * C::X_STEP);
          const bool first = (Pt < NISS) && (PHASE == 1 || h == 0);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_f16(dcol, ad + (uint64_t)((2 * 2048 * kk) >> 4), bd + 2 * kk, idesc,
                        (!first || kk != 0) ? 1u : 0u);
        }
        tc::mma_commit(&wempty[ps]);
        tc::mma_commit(&xempty[xs]);
      }
      __syncwarp();
    }
    if (!stop && tc::elect_one()) tc::mma_commit(accum);
  } else {
    // ---------------- decoders: group g takes the pairs P = g, g + 2, ...
    const int dw = warp - kDec0;
    const int grp = dw / NDEC, dt = (dw % NDEC) * 32 + lane;
    // Epilogue operands, loaded now so that their latency hides behind the
    // decode: this lane's 4 columns of svh (gate, up) and suh (down), or of
    // svh (down, every output tile of the CTA) and the routing weights of
    // the warp's rows (lane q holds row dw + 16 q).
    const int col0 = nt0 * BN;
    float ep_a[4], ep_b[4], ep_c[4], row_w = 0.f;
    float ep_t[PHASE == 2 ? C::NTC : 1][4];
    {
      auto ld4 = [&](const __half *src, float (&o)[4]) {
        const uint2 r = __ldg(reinterpret_cast<const uint2 *>(src + col0 + 4 * lane));
        const __half2 *hh = reinterpret_cast<const __half2 *>(&r);
        o[0] = __low2float(hh[0]);
        o[1] = __high2float(hh[0]);
        o[2] = __low2float(hh[1]);
        o[3] = __high2float(hh[1]);
      };
      if (PHASE == 1) {
        ld4(a.svh13 + ((long)e * 2 + 0) * a.inter, ep_a);
        ld4(a.svh13 + ((long)e * 2 + 1) * a.inter, ep_b);
        ld4(a.suh2 + (long)e * a.inter, ep_c);
      } else {
#pragma unroll
        for (int jt = 0; jt < (PHASE == 2 ? C::NTC : 1); ++jt)
          if (jt < nts) ld4(a.svh2 + (long)e * a.hidden + jt * BN, ep_t[jt]);
        const int m = dw + NGRP * NDEC * lane;
        if (lane < XROWS / (NGRP * NDEC) && m < rows) row_w = a.weights[a.perm[row0 + m]];
      }
    }
    // this thread's items of a pair (the same every pair): half h = it2 /
    // ITEMS of item it, for it2 = dt + 256 j
    constexpr int NI = 2 * C::ITEMS / (NDEC * 32);
    static_assert(NI * NDEC * 32 == 2 * C::ITEMS, "whole items per decoder thread");
    ftc::ItemPlan plan[NI];
#pragma unroll
    for (int j = 0; j < NI; ++j) plan[j] = ftc::item_plan<K>((dt + NDEC * 32 * j) % C::ITEMS);
    for (int P = grp; P < npairs; P += NGRP) {
      const int tj = P / 2, ts = tj % TS, ps = P % NPS;
      const bool ok = (*abort_flag) || (tc::mbar_wait(&tfull[ts], (tj / TS) & 1) &&
                                        tc::mbar_wait(&wempty[ps], ((P / NPS) & 1) ^ 1));
      if (!ok) {
        if (lane == 0) set_device_error(a.err, kErrBounds);
        *abort_flag = 1;
      }
      // the pair's items
#pragma unroll
      for (int j = 0; j < NI; ++j) {
        const int h = (dt + NDEC * 32 * j) / C::ITEMS;
        // phase 1: projection h of k step P (stage rows h * 8 + (P % 2) * 4);
        // phase 2: k step 2P + h (stage rows ((2P + h) % 4) * 4)
        const int r0 = PHASE == 1 ? h * 8 + (P % 2) * 4 : ((2 * P + h) % 4) * 4;
        ftc::decode_planned<K, false>(sT + ts * C::T_STAGE + r0 * C::ROWB, sW + (2 * ps + h) * W_BYTES, plan[j]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic stores -> tensor-core reads
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&wfull[ps]);
        tc::mbar_arrive(&tempty[ts]);   // the group's only pair in the stage
      }
    }

    // ---------------- epilogue, ECH rows of the tile at a time
    // (1) four decoder warps (one per TMEM lane quarter = output columns)
    // write the sum of the issuers' accumulators of each projection (and
    // output tile), in issuer order, times sigma, transposed into a scratch
    // [tile][NP][ECH rows][128] over the x' and weight rings (idle once every
    // MMA has completed).
    constexpr int ECH = C::ECH;
    float *scratch = reinterpret_cast<float *>(smem);
    if (dw < 4) {
      bool okw = tc::mbar_wait(accum, 0);
      okw = __all_sync(0xffffffffu, okw) && !*abort_flag;
      if (!okw && lane == 0) set_device_error(a.err, kErrBounds);
      tc::tc_fence_after();
    }
    for (int mc = 0; mc < rows; mc += ECH) {
      const int mrows = min(ECH, rows - mc);
      if (dw < 4) {
        const int lane_base = 32 * (warp & 3);
        const int ncol = lane_base + lane;
        for (int jp = 0; jp < nts * NP; ++jp) {   // (tile, projection) jt NP + p
          const int jt = jp / NP, p = jp - jt * NP;
          for (int m0 = 0; m0 < mrows; m0 += 8) {
            float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int g = 0; g < NISS; ++g) {
              // issuer g's first pair of tile jt is Pt = (g - jt nptile) mod NISS;
              // without one its accumulator was never written
              if (((g - jt * nptile) % NISS + NISS) % NISS >= nptile) continue;
              uint32_t r[8];
              const uint32_t taddr = tmem_base + ((uint32_t)lane_base << 16) +
                                     (uint32_t)(((jt * NISS + g) * NP + p) * XROWS + mc + m0);
              asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                           : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                             "=r"(r[7])
                           : "r"(taddr));
              tc::tmem_ld_wait();
#pragma unroll
              for (int q = 0; q < 8; ++q) sum[q] += __uint_as_float(r[q]);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (m0 + q < mrows) scratch[(jp * ECH + m0 + q) * 128 + ncol] = sum[q] * kSigma;
          }
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(NGRP * NDEC * 32) : "memory");
      bool finish = true;
      if (PHASE == 1 && a.splits > 1) {
        // split over k (the host uses it with one chunk only, NMAX <= 128):
        // store this split's sums, count the arrival; the last CTA of the
        // tile adds all splits in order (no CTA waits for another)
        constexpr int TILE_F = 2 * XROWS * 128;
        float *part = a.partials + ((long)tile * a.splits + split) * TILE_F;
#pragma unroll
        for (int p = 0; p < 2; ++p)
          for (int m = dw; m < mrows; m += NGRP * NDEC)
            *reinterpret_cast<float4 *>(part + (p * XROWS + m) * 128 + 4 * lane) =
                *reinterpret_cast<const float4 *>(scratch + (p * ECH + m) * 128 + 4 * lane);
        __threadfence();
        asm volatile("bar.sync 1, %0;" ::"n"(NGRP * NDEC * 32) : "memory");
        if (dw == 0 && lane == 0) {
          const int old = atomicAdd(a.counters + tile, 1);
          if (old >= a.splits) set_device_error(a.err, kErrDirtyCounter);
          *s_last = (old == a.splits - 1);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(NGRP * NDEC * 32) : "memory");
        finish = *s_last != 0;
        if (finish) {
          __threadfence();
          const float *base = a.partials + (long)tile * a.splits * TILE_F;
#pragma unroll
          for (int p = 0; p < 2; ++p)
            for (int m = dw; m < mrows; m += NGRP * NDEC) {   // the rows this warp transforms below
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int sp = 0; sp < a.splits; ++sp) {
                const float4 t =
                    __ldcg(reinterpret_cast<const float4 *>(base + sp * TILE_F + (p * XROWS + m) * 128 + 4 * lane));
                acc.x += t.x;
                acc.y += t.y;
                acc.z += t.z;
                acc.w += t.w;
              }
              *reinterpret_cast<float4 *>(scratch + (p * ECH + m) * 128 + 4 * lane) = acc;
            }
          if (dw == 0 && lane == 0) a.counters[tile] = 0;   // leave the workspace clean
          __syncwarp();
        }
      }
      // (2) one warp per row of the chunk
      for (int ml = dw; finish && ml < mrows; ml += NGRP * NDEC) {
        const int m = mc + ml;
        const long row = (long)row0 + m;
        const float4 g4 = *reinterpret_cast<const float4 *>(scratch + ml * 128 + 4 * lane);
        float v[4] = {g4.x, g4.y, g4.z, g4.w};
        fwht128_warp(v, lane);
        if (PHASE == 1) {
          const float4 u4 = *reinterpret_cast<const float4 *>(scratch + (ECH + ml) * 128 + 4 * lane);
          float u[4] = {u4.x, u4.y, u4.z, u4.w};
          fwht128_warp(u, lane);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float gg = v[q] * kRhtScale * ep_a[q];
            const float uu = u[q] * kRhtScale * ep_b[q];
            v[q] = gg / (1.0f + expf(-gg)) * uu * ep_c[q];   // h . suh_down
          }
          fwht128_warp(v, lane);
          __half2 o[2] = {__floats2half2_rn(v[0] * kRhtScale, v[1] * kRhtScale),
                          __floats2half2_rn(v[2] * kRhtScale, v[3] * kRhtScale)};
          *reinterpret_cast<uint2 *>(a.hout + row * a.inter + col0 + 4 * lane) = *reinterpret_cast<uint2 *>(o);
        } else {
          const float w = __shfl_sync(0xffffffffu, row_w, m / (NGRP * NDEC));
          float4 o;
          o.x = v[0] * kRhtScale * ep_t[0][0] * w;
          o.y = v[1] * kRhtScale * ep_t[0][1] * w;
          o.z = v[2] * kRhtScale * ep_t[0][2] * w;
          o.w = v[3] * kRhtScale * ep_t[0][3] * w;
          *reinterpret_cast<float4 *>(a.dout + row * a.hidden + col0 + 4 * lane) = o;
#pragma unroll
          for (int jt = 1; jt < (PHASE == 2 ? C::NTC : 1); ++jt) {   // the CTA's further output tiles
            if (jt >= nts) break;
            const float4 h4 = *reinterpret_cast<const float4 *>(scratch + (jt * ECH + ml) * 128 + 4 * lane);
            float t[4] = {h4.x, h4.y, h4.z, h4.w};
            fwht128_warp(t, lane);
            o.x = t[0] * kRhtScale * ep_t[jt][0] * w;
            o.y = t[1] * kRhtScale * ep_t[jt][1] * w;
            o.z = t[2] * kRhtScale * ep_t[jt][2] * w;
            o.w = t[3] * kRhtScale * ep_t[jt][3] * w;
            *reinterpret_cast<float4 *>(a.dout + row * a.hidden + col0 + jt * BN + 4 * lane) = o;
          }
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(NGRP * NDEC * 32) : "memory");   // the scratch is reused
    }
    if (dw < 4) tc::tc_fence_before();
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, C::TMEM_ALLOC);
  }
}

}  // namespace mf
}  // namespace exl3

using namespace exl3;

static PFN_cuTensorMapEncodeTiled_v12000 mf_tmap_fn() { return exl3_tmap_encode_fn(); }

static int mf_encode(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base, const cuuint64_t *dims,
                     const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle sw, const char *what) {
  auto fn = mf_tmap_fn();
  if (!fn) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, rank, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled (%s) failed (%d)", what, (int)r);
  return EXL3_OK;
}

// rows x cols fp16 (cols contiguous), box `box_rows` rows x 64, 128-byte swizzle.
static int mf_xmap(CUtensorMap *m, const void *base, int rows, int cols, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  return mf_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "x'");
}

// All experts' trellis of one projection kind, [E * nslots * (k/16)][(n/16) * 32K bytes] as u64:
// one load brings box_rows tile rows of 8 tiles.
static int mf_tmap(CUtensorMap *m, const uint16_t *trellis, long rows, int n, int K, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)(n / 16) * 4 * K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(n / 16) * 32 * K};
  cuuint32_t box[2] = {(cuuint32_t)(8 * 4 * K), (cuuint32_t)box_rows};
  return mf_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, trellis, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                   "trellis");
}

template <int PHASE, int NMAX>
static int mf_launch(int K, const CUtensorMap &t0, const CUtensorMap &t1, const CUtensorMap &tt, const mf::Args &a,
                     int grid, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
#define EXL3_MF(KK)                                                                                              \
  case KK:                                                                                                       \
    if constexpr (mf::Cfg<KK, PHASE, NMAX>::OK) {                                                                \
      using CF = mf::Cfg<KK, PHASE, NMAX>;                                                                       \
      auto kfn = mf::moe_fused_kernel<KK, PHASE, NMAX>;                                                          \
      cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_BYTES);                    \
      e = launch_pdl(kfn, dim3(grid), dim3(mf::Roles<NMAX>::WARPS * 32), CF::SMEM_BYTES, s, t0, t1, tt, a);       \
    } else {                                                                                                     \
      return exl3_fail(EXL3_ERR_ARG, "tile capacity %d does not fit K = %d", NMAX, KK);                          \
    }                                                                                                            \
    break;
  switch (K) {
    EXL3_MF(1) EXL3_MF(2) EXL3_MF(3) EXL3_MF(4) EXL3_MF(5) EXL3_MF(6) EXL3_MF(7) EXL3_MF(8)
    default: return exl3_fail(EXL3_ERR_BITS, "K = %d", K);
  }
#undef EXL3_MF
  return exl3_cuda_check(e, "moe fused launch");
}

// Whether the grouped kernels have a configuration for tiles of `cap` rows
// at width K.
bool exl3_moe_fused_cap_fits(int cap, int K) {
  bool ok = false;
#define EXL3_MF_FIT(KK)                                                                                         \
  case KK:                                                                                                      \
    ok = cap == 32 ? (mf::Cfg<KK, 1, 32>::OK && mf::Cfg<KK, 2, 32>::OK)                                        \
                   : cap == 128 ? (mf::Cfg<KK, 1, 128>::OK && mf::Cfg<KK, 2, 128>::OK)                           \
                   : cap == 160 ? (mf::Cfg<KK, 1, 160>::OK && mf::Cfg<KK, 2, 160>::OK)                           \
                                : (mf::Cfg<KK, 1, 256>::OK && mf::Cfg<KK, 2, 256>::OK);                          \
    break;
  switch (K) {
    EXL3_MF_FIT(1) EXL3_MF_FIT(2) EXL3_MF_FIT(3) EXL3_MF_FIT(4) EXL3_MF_FIT(5) EXL3_MF_FIT(6) EXL3_MF_FIT(7)
    EXL3_MF_FIT(8)
    default: break;
  }
#undef EXL3_MF_FIT
  return ok;
}

// Phase 1: xg, xu [U][hidden] fp16 sorted rows; w13 trellis [E][2][hidden/16][inter/16][16K];
// the tile list holds tiles of at most cap (32, 128, 160 or 256) rows.
// splits > 1 (k split of the gate+up projection): partials [max_mtiles * inter/128][splits][2][cap][128]
// fp32 and counters [max_mtiles * inter/128], zero on entry and left zero.
// e_lo, e_cnt: only experts [e_lo, e_lo + e_cnt), whose trellis starts at
// w13_trellis (e_cnt < 0: all E experts from 0).
int exl3_launch_moe_fused_gateup(const uint16_t *xg, const uint16_t *xu, int U, int hidden, int inter, int K, int E,
                                 const uint16_t *w13_trellis, const int *mtiles, const int *n_mtiles, int max_mtiles,
                                 int cap, const uint16_t *svh13, const uint16_t *suh2, uint16_t *hout, int splits,
                                 float *partials, int *counters, int *err, cudaStream_t s, int e_lo, int e_cnt) {
  if (e_cnt < 0) {
    e_lo = 0;
    e_cnt = E;
  }
  CUtensorMap t0, t1, tt;
  if (cap != 32 && cap != 128 && cap != 160 && cap != 256) return exl3_fail(EXL3_ERR_ARG, "tile capacity %d", cap);
  int rc = mf_xmap(&t0, xg, U, hidden, cap);
  if (!rc) rc = mf_xmap(&t1, xu, U, hidden, cap);
  if (!rc) rc = mf_tmap(&tt, w13_trellis, (long)e_cnt * 2 * (hidden / 16), inter, K, 8);
  if (rc) return rc;
  mf::Args a{};
  a.e_lo = e_lo;
  a.e_hi = e_lo + e_cnt;
  a.mtiles = reinterpret_cast<const int4 *>(mtiles);
  a.n_mtiles = n_mtiles;
  a.NT = inter / 128;
  a.KB = hidden / 64;
  a.tiles_k = hidden / 16;
  a.nslots = 2;
  a.svh13 = reinterpret_cast<const __half *>(svh13);
  a.suh2 = reinterpret_cast<const __half *>(suh2);
  a.hout = reinterpret_cast<__half *>(hout);
  a.inter = inter;
  a.err = err;
  a.splits = splits;
  a.ntc = 1;
  a.partials = partials;
  a.counters = counters;
  const int grid = max_mtiles * a.NT * splits;
  if (cap == 32) return mf_launch<1, 32>(K, t0, t1, tt, a, grid, s);
  if (cap == 128) return mf_launch<1, 128>(K, t0, t1, tt, a, grid, s);
  if (splits > 1) return exl3_fail(EXL3_ERR_ARG, "no k split with tiles of more than 128 rows");
  if (cap == 160) return mf_launch<1, 160>(K, t0, t1, tt, a, grid, s);
  return mf_launch<1, 256>(K, t0, t1, tt, a, grid, s);
}

// Phase 2: h' [U][inter] fp16 sorted rows; w2 trellis [E][1][inter/16][hidden/16][16K]; d [U][hidden] fp32.
// e_lo, e_cnt as for the gate+up launch.
int exl3_launch_moe_fused_down(const uint16_t *hin, int U, int hidden, int inter, int K, int E,
                               const uint16_t *w2_trellis, const int *mtiles, const int *n_mtiles, int max_mtiles,
                               int cap, const uint16_t *svh2, const float *weights, const int *perm, float *dout,
                               int *err, cudaStream_t s, int e_lo, int e_cnt) {
  if (cap != 32 && cap != 128 && cap != 160 && cap != 256) return exl3_fail(EXL3_ERR_ARG, "tile capacity %d", cap);
  if (e_cnt < 0) {
    e_lo = 0;
    e_cnt = E;
  }
  CUtensorMap t0, tt;
  // h' as (64 k, U rows, inter/64 blocks): one load brings two k steps of the tile's rows
  cuuint64_t dims[3] = {64, (cuuint64_t)U, (cuuint64_t)(inter / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)inter * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)cap, 2};
  int rc = mf_encode(&t0, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, hin, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                     "h'");
  if (!rc) rc = mf_tmap(&tt, w2_trellis, (long)e_cnt * (inter / 16), hidden, K, 16);
  if (rc) return rc;
  mf::Args a{};
  a.e_lo = e_lo;
  a.e_hi = e_lo + e_cnt;
  a.mtiles = reinterpret_cast<const int4 *>(mtiles);
  a.n_mtiles = n_mtiles;
  a.NT = hidden / 128;
  a.KB = inter / 64;
  a.tiles_k = inter / 16;
  a.nslots = 1;
  a.svh2 = reinterpret_cast<const __half *>(svh2);
  a.weights = weights;
  a.perm = perm;
  a.dout = dout;
  a.hidden = hidden;
  a.err = err;
  a.splits = 1;
  // several output tiles per CTA (one fill and one epilogue for all: four
  // with 32-row tiles, else two) when each tile's pairs fill whole trellis
  // stages and the grid still covers the SMs twice over; few routed rows
  // keep fewer tiles per CTA for parallelism
  const int sms = exl3_sm_count();
  a.ntc = 1;
  if ((a.KB / 2) % 2 == 0)
    for (int c = cap == 32 ? 4 : 2; c >= 2; c /= 2)
      if ((long)max_mtiles * (a.NT / c) >= 2L * sms) {
        a.ntc = c;
        break;
      }
  const int grid = max_mtiles * ((a.NT + a.ntc - 1) / a.ntc);
  if (cap == 32) return mf_launch<2, 32>(K, t0, t0, tt, a, grid, s);
  if (cap == 128) return mf_launch<2, 128>(K, t0, t0, tt, a, grid, s);
  if (cap == 160) return mf_launch<2, 160>(K, t0, t0, tt, a, grid, s);
  return mf_launch<2, 256>(K, t0, t0, tt, a, grid, s);
}
