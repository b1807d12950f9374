// fused_tc.cu -- small-M EXL3 linear (2 <= M <= 128 tokens) with the trellis
// decoded straight into tensor-core operands: no reconstructed weights in
// HBM ("exl3xpu" README, "Layout": fused GEMM for M <= 128; "Prefill: int8
// linears and oneDNN fused attention": the GEMM runs in the Hadamard domain).
//
//   y[m, :] = RHT_out( sigma * x'[m, :] (B - 510) ) . svh      per 128-column tile
//
// The MMA computes the transposed product D[n][m] = sum_k W[k][n] x'[m][k]:
// the decoded weights are the A operand (M = 128 output columns, MN-major)
// and x' is the narrow B operand (N = M rounded up to 16, K-major), so an
// operand slot stays small and many fit in shared memory.
//
// Per CTA: one 128-column tile of y and one k-range (k splits over CTAs).
//   warp 0       trellis producer: one tensor load per stage of 16 tile rows
//                (8 tiles each, four 64-deep k steps) into a ring
//   warps 1-4    MMA issuers, one per SM sub-partition, taking every fourth
//                pair of k steps: 4 x tcgen05.mma M128 N(M) K16 per step
//                into the issuer's own TMEM accumulator (an issuer thread
//                shares its sub-partition's issue slots with four decoder
//                warps; fewer issuers could not keep up with the decoders)
//   warp 21      operand producer: one tensor load of the x' tiles of 2-4 k
//                steps (M rows x 64 k each, 128-byte swizzled)
//   warps 5-20   decoders, two groups of eight taking alternate pairs of k
//                steps (one fence and one signal per pair): each
//                lane cuts 16 G trellis states out of its chunk, hashes them
//                (IMAD + DP4A seeded with 0x6400 gives the fp16 value
//                1024 + B) and stores these integers (exact in fp16) as the
//                MN-major, 128-byte-swizzled fp16 operand; the epilogue
//                removes 1534 sum x' per token, from per-256 sums of x'
//                that the input transform writes (row k, 64 n per 128-byte
//                row of the operand; 8-row k groups 2 KB
//                apart, 64-wide n atoms 1 KB apart); an item's rows share
//                one 8-row k group, so its store slots are one XOR each.  The
//                decoders then run the epilogue: the TMEM accumulator
//                (lane = output column, column = token) transposed into a
//                shared scratch, the fixed-order split-k combine (last CTA to
//                arrive, no waiting) and a warp-level FWHT-128 per token row.
// Every wait is bounded and reports through the device error word.
#include <cudaTypedefs.h>

#include "exl3_common.cuh"
#include "tc_ptx.cuh"
#include "fused_decode.cuh"

namespace exl3 {
namespace ftc {

// Warp roles.  Every weight slot pair and x' slot is used by one issuer only
// (NPS and the x' stage-to-slot map are multiples of NISS), so an issuer's
// waits on a slot's barrier are for consecutive phases.
template <int NMAX>
struct Roles {
  static constexpr int NISS = NMAX <= 32 ? 4 : 2;   // MMA issuer warps
  static constexpr int DEC0 = 1 + NISS;              // first decoder warp
  static constexpr int XWARP = DEC0 + NGRP * NDEC;   // the x' producer follows the decoder warps
  static constexpr int WARPS = XWARP + 1;
};

struct Args {
  const uint16_t *trellis;
  const float *xsum;   // [M][xunits] sums of x' over 256-element units of k
  const __half *svh;
  void *y;
  float *partials;     // [splits][M][n]
  int *counters;       // [n / 128]
  int *err;
  int M, k, n, tiles_n, kb_per_split, splits, xunits;
  int npad;            // MMA N: tokens rounded up to 16, or 128 for every M (row-invariant mode)
  const __half *bias;  // [n] fp16 added after svh, or NULL
};

template <int K, bool F32OUT, int NMAX>
__global__ void __launch_bounds__(Roles<NMAX>::WARPS * 32, 1) fused_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                  const __grid_constant__ CUtensorMap tmT, Args a) {
  using S = Shape<K, NMAX>;
  constexpr int WS = S::WS, XS = S::XS, TS = S::TS;
  constexpr int NISS = Roles<NMAX>::NISS, kDec0 = Roles<NMAX>::DEC0, kXWarp = Roles<NMAX>::XWARP;
  static_assert((WS / 2) % NISS == 0 && (WS / 2) % NGRP == 0, "one issuer and one decoder group per weight slot");
  static_assert((XS * (S::XSTEPS / 2)) % NISS == 0, "the same issuers on every use of an x' slot");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t *sW = smem;                                   // [WS][W_BYTES] decoded weights (A operand)
  uint8_t *sX = smem + WS * W_BYTES;                    // [XS][X_STAGE] x' rows (B operand)
  uint8_t *sT = sX + XS * S::X_STAGE;                   // [TS][T_STAGE]
  uint64_t *tfull = reinterpret_cast<uint64_t *>(sT + TS * S::T_STAGE);   // [TS] trellis landed
  uint64_t *tempty = tfull + TS;                        // [TS] trellis decoded
  uint64_t *xfull = tempty + TS;                        // [XS] x' tile landed
  uint64_t *xempty = xfull + XS;                        // [XS] MMA done with the x' slot
  uint64_t *wfull = xempty + XS;                        // [WS / 2] a pair of weight slots decoded
  uint64_t *wempty = wfull + WS;                        // [WS / 2] MMA done with the pair of slots
  uint64_t *accum = wempty + WS;                        // accumulator complete
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_last = const_cast<int *>(abort_flag + 1);
  float *s_sx = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(s_last + 1) + 15) & ~(uintptr_t)15);   // [128] sum of x' over this split's k, 16-byte aligned

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x, split = blockIdx.y;
  // k range of this split: whole trellis stages (the last stage of the
  // tensor may hold only two steps; k is a multiple of 128, so nkb is even)
  const int kbt = a.k / BK, kst = (kbt + S::TSTEPS - 1) / S::TSTEPS;
  const int kb0 = (int)((long)split * kst / a.splits) * S::TSTEPS;
  const int nkb = min(kbt, (int)((long)(split + 1) * kst / a.splits) * S::TSTEPS) - kb0;
  const int ntst = (nkb + S::TSTEPS - 1) / S::TSTEPS;   // trellis stages
  const int nxst = (nkb + S::XSTEPS - 1) / S::XSTEPS;   // x' stages
  // Work is handed over in pairs of k steps: pair P = steps 2P, 2P + 1 (half
  // a trellis stage), decoder group and MMA issuer P mod 2, weight slots
  // 2 (P mod NPS) and 2 (P mod NPS) + 1.
  constexpr int NPS = WS / 2;
  const int npairs = nkb / 2;
  const int tn0 = nt * (BN / 16);
  const int npad = a.npad;                              // MMA N (x' rows past M read as zero)

  if (threadIdx.x == 0) {
    for (int s = 0; s < TS; ++s) {
      tc::mbar_init(&tfull[s], 1);
      tc::mbar_init(&tempty[s], NGRP * NDEC);   // every decoder warp, once per stage
    }
    for (int s = 0; s < XS; ++s) {
      tc::mbar_init(&xfull[s], 1);
      tc::mbar_init(&xempty[s], S::XSTEPS / 2);  // the issuers of the stage's pairs
    }
    for (int s = 0; s < NPS; ++s) {
      tc::mbar_init(&wfull[s], NDEC);            // one group's warps, once per pair
      tc::mbar_init(&wempty[s], 1);
    }
    tc::mbar_init(accum, NISS);
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmX);
    tc::prefetch_tmap(&tmT);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, NISS * NMAX);   // one accumulator per issuer
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- trellis producer: one tensor load per stage (16 tile
    // rows x the CTA's 8 tiles)
    if (lane == 0) {
      for (int j = 0; j < ntst && !*abort_flag; ++j) {
        const int st = j % TS;
        if (!tc::mbar_wait_backoff(&tempty[st], ((j / TS) & 1) ^ 1)) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&tfull[st], S::T_STAGE);
        tc::tma_load_2d(sT + st * S::T_STAGE, &tmT, &tfull[st], tn0 * (4 * K), (kb0 + j * S::TSTEPS) * 4);
      }
    }
  } else if (warp == kXWarp) {
    // ---------------- x' producer: XSTEPS k blocks of every token per tensor load
    // This kernel is a programmatic dependent of the input transform that
    // writes x' and its sums: everything before this wait (set-up, trellis
    // loads, decoding) overlaps that kernel; x' and the workspace are read
    // after it.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (lane == 0) {
      const uint32_t xbytes = (uint32_t)S::XSTEPS * npad * BK * 2;
      for (int j = 0; j < nxst && !*abort_flag; ++j) {
        const int st = j % XS;
        if (!tc::mbar_wait_backoff(&xempty[st], ((j / XS) & 1) ^ 1)) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&xfull[st], xbytes);
        tc::tma_load_3d(sX + st * S::X_STAGE, &tmX, &xfull[st], 0, 0, kb0 + j * S::XSTEPS);
      }
    }
  } else if (warp <= NISS) {
    // ---------------- MMA issuers: warp 1 + g takes the pairs P = g, g + 4,
    // ... (8 MMAs after one wait) into its own accumulator (TMEM columns
    // g * NMAX ...).  One issuer per SM sub-partition: an issuer shares its
    // sub-partition's issue slots with four decoder warps, and two issuers
    // could not keep up with the decoders.  The whole warp runs the loop
    // (waits and descriptors stay warp-uniform); one elected lane issues
    // the MMAs and their commits.
    const int g = __shfl_sync(0xffffffffu, warp, 0) - 1;
    const uint32_t dcol = tmem_base + (uint32_t)(g * NMAX);
    const uint32_t idesc = idesc_f16_amn(BN, npad);
    int xwaited = -1;
    bool stop = false;
    for (int P = g; P < npairs; P += NISS) {
      const int xj = (2 * P) / S::XSTEPS, xs = xj % XS, ps = P % NPS;
      bool ok = true;
      if (xj != xwaited) {            // once per x' stage
        ok = tc::mbar_wait(&xfull[xs], (xj / XS) & 1);
        xwaited = xj;
      }
      ok = ok && tc::mbar_wait(&wfull[ps], (P / NPS) & 1);
      ok = __all_sync(0xffffffffu, ok && !*abort_flag);
      if (!ok) {
        if (lane == 0) set_device_error(a.err, kErrBounds);
        *abort_flag = 1;
        stop = true;
        break;
      }
      tc::tc_fence_after();
      if (tc::elect_one()) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = 2 * P + h;
          const uint64_t ad = sdesc_mn_sw128(sW + (2 * ps + h) * W_BYTES, 1024, 2048);
          const uint64_t bd = tc::sdesc_k_sw128(sX + xs * S::X_STAGE + (i % S::XSTEPS) * npad * (BK * 2));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_f16(dcol, ad + (uint64_t)((2 * 2048 * kk) >> 4), bd + 2 * kk, idesc,
                        (P != g || h != 0 || kk != 0) ? 1u : 0u);
        }
        tc::mma_commit(&wempty[ps]);
        tc::mma_commit(&xempty[xs]);    // each issuer uses an x' stage for one pair
      }
      __syncwarp();
    }
    if (!stop && tc::elect_one()) tc::mma_commit(accum);
  } else {
    // ---------------- decoders: group g takes k steps i = g, g + 2, ...
    const int dw = warp - kDec0;             // 0..15
    const int grp = dw / NDEC, dt = (dw % NDEC) * 32 + lane;
    // this thread's items of a pair (the same every pair): k step 2P + h of
    // item it, for it2 = dt + 256 j, h = it2 / ITEMS
    constexpr int NI = 2 * S::ITEMS / (NDEC * 32);
    static_assert(NI * NDEC * 32 == 2 * S::ITEMS, "whole items per decoder thread");
    ItemPlan plan[NI];
#pragma unroll
    for (int j = 0; j < NI; ++j) plan[j] = item_plan<K>((dt + NDEC * 32 * j) % S::ITEMS);
    for (int P = grp; P < npairs; P += NGRP) {
      const int tj = P / 2, ts = tj % TS, ps = P % NPS;   // a trellis stage holds two pairs
      const bool ok = (*abort_flag) || (tc::mbar_wait(&tfull[ts], (tj / TS) & 1) &&
                                        tc::mbar_wait(&wempty[ps], ((P / NPS) & 1) ^ 1));
      if (!ok) {
        if (lane == 0) set_device_error(a.err, kErrBounds);
        *abort_flag = 1;
      }
      // the pair's items: k step 2P + h (the operand keeps 1024 + B)
#pragma unroll
      for (int j = 0; j < NI; ++j) {
        const int h = (dt + NDEC * 32 * j) / S::ITEMS;
        const int i = 2 * P + h;
        decode_planned<K, true>(sT + ts * S::T_STAGE + (i % S::TSTEPS) * S::T_BYTES, sW + (2 * ps + h) * W_BYTES,
                                plan[j]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic stores -> tensor-core reads
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&wfull[ps]);
        tc::mbar_arrive(&tempty[ts]);   // the group's only pair in the stage
      }
    }

    // ---------------- epilogue
    // (1) the first four decoder warps (one per TMEM lane quarter = output
    // columns) write the sum of the issuers' accumulators (issuer 0 + 1 + 2 +
    // 3, in that order), times sigma, transposed into a scratch [M][128] fp32
    // that reuses the operand ring (free once every MMA has completed).
    float *scratch = reinterpret_cast<float *>(smem);
    asm volatile("griddepcontrol.wait;" ::: "memory");   // x' sums, workspace and y (see the x' producer)
    // (0) each token's sum of x' over this split's k (256-element units of
    // four k steps; the last stage may hold two): the accumulators hold
    // sum x' (1024 + B), and 1534 sum x' is removed below
    {
      const int dtid = dw * 32 + lane;
      if (dtid < a.M) {
        const int u0 = kb0 / S::TSTEPS, u1 = (kb0 + nkb + S::TSTEPS - 1) / S::TSTEPS;
        float sx = 0.f;
#pragma unroll 8
        for (int u = u0; u < u1; ++u) sx += a.xsum[(long)dtid * a.xunits + u];
        s_sx[dtid] = sx;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(NGRP * NDEC * 32) : "memory");   // all decoder warps
    }
    if (dw < 4) {
      bool ok = tc::mbar_wait(accum, 0);
      ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
      if (!ok && lane == 0) set_device_error(a.err, kErrBounds);
      tc::tc_fence_after();
      const int lane_base = 32 * (warp & 3);
      const int ncol = lane_base + lane;
      for (int m0 = 0; m0 < a.M; m0 += 8) {
        // the tokens' x' sums, read before the TMEM loads so that their
        // latency overlaps them
        const float4 sa = *reinterpret_cast<const float4 *>(s_sx + m0);
        const float4 sb = *reinterpret_cast<const float4 *>(s_sx + m0 + 4);
        const float sxv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
        float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int g = 0; g < NISS; ++g) {
          if (g >= npairs) break;        // issuer g had no pair: its accumulator was never written
          uint32_t r[8];
          const uint32_t taddr = tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)(g * NMAX + m0);
          asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                       : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                         "=r"(r[7])
                       : "r"(taddr));
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j) sum[j] += __uint_as_float(r[j]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (m0 + j < a.M) scratch[(m0 + j) * 128 + ncol] = fmaf(-1534.0f, sxv[j], sum[j]) * kSigma;
      }
      tc::tc_fence_before();
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NGRP * NDEC * 32) : "memory");   // all decoder warps
    const int col0 = nt * BN;
    const int ew = dw;                                // 0..15
    constexpr int NEW = NGRP * NDEC;
    bool finish = true;
    if (a.splits > 1) {
      // (2) partial sums of this split; the last CTA of the column tile adds all
      // splits in order.
      for (int m = ew; m < a.M; m += NEW) {
        const float4 v = *reinterpret_cast<const float4 *>(scratch + m * 128 + 4 * lane);
        *reinterpret_cast<float4 *>(a.partials + ((long)split * a.M + m) * a.n + col0 + 4 * lane) = v;
      }
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"n"(NEW * 32) : "memory");
      if (dw == 0 && lane == 0) {
        const int old = atomicAdd(a.counters + nt, 1);
        if (old >= a.splits) set_device_error(a.err, kErrDirtyCounter);
        *s_last = (old == a.splits - 1);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(NEW * 32) : "memory");
      finish = *s_last != 0;
      if (finish) __threadfence();
    }
    // (3) one warp per token row: sum the splits, FWHT-128, 2^-3.5, svh, store
    if (finish) {
      for (int m = ew; m < a.M; m += NEW) {
        float v[4];
        if (a.splits > 1) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int sp = 0; sp < a.splits; ++sp) {
            const float4 p =
                __ldcg(reinterpret_cast<const float4 *>(a.partials + ((long)sp * a.M + m) * a.n + col0 + 4 * lane));
            acc.x += p.x;
            acc.y += p.y;
            acc.z += p.z;
            acc.w += p.w;
          }
          v[0] = acc.x; v[1] = acc.y; v[2] = acc.z; v[3] = acc.w;
        } else {
          const float4 p = *reinterpret_cast<const float4 *>(scratch + m * 128 + 4 * lane);
          v[0] = p.x; v[1] = p.y; v[2] = p.z; v[3] = p.w;
        }
        fwht128_warp(v, lane);
        const int gc = col0 + 4 * lane;
        const uint2 sv = *reinterpret_cast<const uint2 *>(a.svh + gc);
        const __half2 *sh = reinterpret_cast<const __half2 *>(&sv);
        v[0] = v[0] * kRhtScale * __low2float(sh[0]);
        v[1] = v[1] * kRhtScale * __high2float(sh[0]);
        v[2] = v[2] * kRhtScale * __low2float(sh[1]);
        v[3] = v[3] * kRhtScale * __high2float(sh[1]);
        if (a.bias) {   // the output bias, per output feature
          const uint2 bv = *reinterpret_cast<const uint2 *>(a.bias + gc);
          const __half2 *bh = reinterpret_cast<const __half2 *>(&bv);
          v[0] = __fadd_rn(v[0], __low2float(bh[0]));   // one rounding, never contracted
          v[1] = __fadd_rn(v[1], __high2float(bh[0]));
          v[2] = __fadd_rn(v[2], __low2float(bh[1]));
          v[3] = __fadd_rn(v[3], __high2float(bh[1]));
        }
        if (F32OUT) {
          *reinterpret_cast<float4 *>(static_cast<float *>(a.y) + (long)m * a.n + gc) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
          __half2 o[2] = {__floats2half2_rn(v[0], v[1]), __floats2half2_rn(v[2], v[3])};
          *reinterpret_cast<uint2 *>(static_cast<__half *>(a.y) + (long)m * a.n + gc) = *reinterpret_cast<uint2 *>(o);
        }
      }
      if (a.splits > 1 && dw == 0 && lane == 0) a.counters[nt] = 0;   // leave the workspace clean
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, NISS * NMAX);
  }
}

}  // namespace ftc
}  // namespace exl3

using namespace exl3;

static PFN_cuTensorMapEncodeTiled_v12000 ftc_tmap_fn() { return exl3_tmap_encode_fn(); }

// Number of k splits (one CTA per SM): the split count whose CTAs fill whole
// waves best, keeping at least 4 trellis stages (16 k steps of 64) per CTA
// (fewer splits on ties).  Splits fall on stage boundaries.
int exl3_fused_tc_splits(int k, int n) {
  const int sms = exl3_sm_count();
  const int kst = (k / 64 + 3) / 4, tiles = n / 128;
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= kst && (s == 1 || kst / s >= 4); ++s) {
    const long ctas = (long)tiles * s;
    const long waves = (ctas + sms - 1) / sms;
    const double eff = (double)ctas / (double)(waves * sms);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

// xh: x' fp16 [M][k] (M <= 128); partials: [splits][M][n] fp32 (unused when splits == 1).
// bias: [n] fp16 added to the output, or NULL.
// npad_fixed (32 or 128, at least M): the MMA is that many tokens wide
// whatever M is, so that a token's result does not depend on how many tokens
// share the call; 0: M rounded up to 16.
int exl3_launch_fused_tc(const uint16_t *xh, const float *xsum, const uint16_t *trellis, const uint16_t *svh, int M,
                         int k, int n, int K, void *y, bool f32out, float *partials, int *counters, int *err,
                         int splits, cudaStream_t s, int npad_fixed, const uint16_t *bias) {
  auto fn = ftc_tmap_fn();
  if (!fn) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  // x' [M][k] as (64 k, M rows, k/64 blocks): one load brings XSTEPS k blocks
  // of every token, each block a 128-byte-swizzled K-major operand.
  const int npad = npad_fixed ? npad_fixed : (M + 15) & ~15;
  if (npad < M || (npad_fixed && npad_fixed != 32 && npad_fixed != 128))
    return exl3_fail(EXL3_ERR_ARG, "MMA width %d for M = %d", npad, M);
  const int xsteps = npad <= 32 ? ftc::Shape<1, 32>::XSTEPS : ftc::Shape<1, 128>::XSTEPS;
  CUtensorMap ta, tt;
  {
    cuuint64_t dims[3] = {64, (cuuint64_t)M, (cuuint64_t)(k / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)k * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)npad, (cuuint32_t)xsteps};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t *>(xh), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled (x') failed (%d)", (int)r);
  }
  // trellis [k/16][n/16 * 32K bytes] as u64: one load brings 16 tile rows of
  // the CTA's 8 tiles (4K u64 per tile).
  {
    cuuint64_t dims[2] = {(cuuint64_t)(n / 16) * 4 * K, (cuuint64_t)(k / 16)};
    cuuint64_t strides[1] = {(cuuint64_t)(n / 16) * 32 * K};
    cuuint32_t box[2] = {(cuuint32_t)(8 * 4 * K), 16};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(&tt, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint16_t *>(trellis), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled (trellis) failed (%d)", (int)r);
  }
  ftc::Args a{trellis, xsum, reinterpret_cast<const __half *>(svh), y, partials, counters, err, M, k, n, n / 16,
              0, splits, (k + 255) / 256, npad, reinterpret_cast<const __half *>(bias)};
  dim3 grid(n / 128, splits);
  cudaError_t e = cudaSuccess;
#define EXL3_FTC(KK, F32, NM)                                                                                \
  do {                                                                                                      \
    auto kfn = ftc::fused_tc_kernel<KK, F32, NM>;                                                           \
    cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, ftc::Shape<KK, NM>::SMEM_BYTES);  \
    /* a programmatic dependent of the input transform: CTAs start while it finishes */                  \
    e = launch_pdl(kfn, grid, dim3(ftc::Roles<NM>::WARPS * 32), ftc::Shape<KK, NM>::SMEM_BYTES, s, ta, tt, a); \
  } while (0)
#define EXL3_FTC_K(KK)                                          \
  case KK:                                                      \
    if (npad <= 32) {                                           \
      if (f32out) EXL3_FTC(KK, true, 32); else EXL3_FTC(KK, false, 32); \
    } else {                                                    \
      if (f32out) EXL3_FTC(KK, true, 128); else EXL3_FTC(KK, false, 128); \
    }                                                           \
    break;
  switch (K) {
    EXL3_FTC_K(1) EXL3_FTC_K(2) EXL3_FTC_K(3) EXL3_FTC_K(4) EXL3_FTC_K(5) EXL3_FTC_K(6) EXL3_FTC_K(7)
    EXL3_FTC_K(8)
    default: return exl3_fail(EXL3_ERR_BITS, "K = %d", K);
  }
#undef EXL3_FTC_K
#undef EXL3_FTC
  return exl3_cuda_check(e, "fused_tc launch");
}
