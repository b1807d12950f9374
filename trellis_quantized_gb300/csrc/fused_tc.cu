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
//   warp 0       trellis producer: bulk copies of the four trellis rows (8
//                tiles each) of every 64-deep k step into a deep ring
//   warp 1       MMA issuer: 4 x tcgen05.mma M128 N(M) K16 per step into TMEM
//   warp 2       operand producer: TMA of the x' tile (M rows x 64 k) into the
//                operand ring
//   warps 3-18   decoders, two groups of eight taking alternate k steps: each
//                lane cuts 16 G trellis states out of its chunk, hashes them
//                (IMAD + DP4A seeded with 0x6400 gives the fp16 value
//                1024 + B), subtracts 1534 in half2 (exact) and stores the
//                integers B - 510 as the MN-major, 128-byte-swizzled fp16
//                operand (row k, 64 n per 128-byte row; 8-row k groups 2 KB
//                apart, 64-wide n atoms 1 KB apart).  The lane-to-chunk
//                mapping keeps both the 16-byte chunk loads and the swizzled
//                stores free of bank conflicts where the width allows.  The
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

struct Args {
  const uint16_t *trellis;
  const __half *svh;
  void *y;
  float *partials;     // [splits][M][n]
  int *counters;       // [n / 128]
  int *err;
  int M, k, n, tiles_n, kb_per_split, splits;
};

template <int K, bool F32OUT, int NMAX>
__global__ void __launch_bounds__(NWARPS * 32, 1) fused_tc_kernel(const __grid_constant__ CUtensorMap tmX, Args a) {
  using S = Shape<K, NMAX>;
  constexpr int WS = S::WS, XS = S::XS, TS = S::TS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t *sW = smem;                                   // [WS][W_BYTES] decoded weights (A operand)
  uint8_t *sX = smem + WS * W_BYTES;                    // [XS][X_BYTES] x' rows (B operand)
  uint8_t *sT = sX + XS * S::X_BYTES;                   // [TS][T_BYTES]
  uint64_t *tfull = reinterpret_cast<uint64_t *>(sT + TS * S::T_BYTES);   // [TS] trellis landed
  uint64_t *tempty = tfull + TS;                        // [TS] trellis decoded
  uint64_t *xfull = tempty + TS;                        // [XS] x' tile landed
  uint64_t *xempty = xfull + XS;                        // [XS] MMA done with the x' slot
  uint64_t *wfull = xempty + XS;                        // [WS] weights decoded
  uint64_t *wempty = wfull + WS;                        // [WS] MMA done with the weight slot
  uint64_t *accum = wempty + WS;                        // accumulator complete
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_last = const_cast<int *>(abort_flag + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x, split = blockIdx.y;
  const int kb0 = (int)((long)split * (a.k / BK) / a.splits);
  const int nkb = (int)((long)(split + 1) * (a.k / BK) / a.splits) - kb0;
  const int tn0 = nt * (BN / 16);
  const int npad = (a.M + 15) & ~15;                    // MMA N: tokens rounded up to 16

  if (threadIdx.x == 0) {
    for (int s = 0; s < TS; ++s) {
      tc::mbar_init(&tfull[s], 1);
      tc::mbar_init(&tempty[s], NDEC);
    }
    for (int s = 0; s < XS; ++s) {
      tc::mbar_init(&xfull[s], 1);
      tc::mbar_init(&xempty[s], 1);
    }
    for (int s = 0; s < WS; ++s) {
      tc::mbar_init(&wfull[s], NDEC);
      tc::mbar_init(&wempty[s], 1);
    }
    tc::mbar_init(accum, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, NMAX);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- trellis producer
    if (lane == 0) {
      for (int i = 0; i < nkb && !*abort_flag; ++i) {
        const int st = i % TS;
        if (!tc::mbar_wait(&tempty[st], ((i / TS) & 1) ^ 1)) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&tfull[st], S::T_BYTES);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const long tk = (long)(kb0 + i) * 4 + j;
          bulk_copy(sT + st * S::T_BYTES + j * S::ROWB, a.trellis + (tk * a.tiles_n + tn0) * 16 * K, S::ROWB,
                    &tfull[st]);
        }
      }
    }
  } else if (warp == 2) {
    // ---------------- x' operand producer
    if (lane == 0) {
      for (int i = 0; i < nkb && !*abort_flag; ++i) {
        const int st = i % XS;
        if (!tc::mbar_wait(&xempty[st], ((i / XS) & 1) ^ 1)) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&xfull[st], (uint32_t)npad * BK * 2);
        tc::tma_load_2d(sX + st * S::X_BYTES, &tmX, &xfull[st], (kb0 + i) * BK, 0);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      for (int i = 0; i < nkb; ++i) {
        const int xs = i % XS, ws = i % WS;
        const bool ok = tc::mbar_wait(&xfull[xs], (i / XS) & 1) && tc::mbar_wait(&wfull[ws], (i / WS) & 1);
        if (!ok || *abort_flag) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        const uint64_t ad = sdesc_mn_sw128(sW + ws * W_BYTES, 1024, 2048);
        const uint64_t bd = tc::sdesc_k_sw128(sX + xs * S::X_BYTES);
        const uint32_t idesc = idesc_f16_amn(BN, npad);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc::mma_f16(tmem_base, ad + (uint64_t)((2 * 2048 * kk) >> 4), bd + 2 * kk, idesc, (i | kk) != 0 ? 1u : 0u);
        tc::mma_commit(&wempty[ws]);
        tc::mma_commit(&xempty[xs]);
      }
      tc::mma_commit(accum);
    }
  } else {
    // ---------------- decoders: group g takes k steps i = g, g + 2, ...
    const int dw = warp - 3;                 // 0..15
    const int grp = dw / NDEC, dt = (dw % NDEC) * 32 + lane;
    for (int i = grp; i < nkb; i += NGRP) {
      const int ts = i % TS, bs = i % WS;
      const bool ok = (*abort_flag) || (tc::mbar_wait(&tfull[ts], (i / TS) & 1) &&
                                        tc::mbar_wait(&wempty[bs], ((i / WS) & 1) ^ 1));
      if (!ok) {
        if (lane == 0) set_device_error(a.err, kErrBounds);
        *abort_flag = 1;
      }
      const uint8_t *tst = sT + ts * S::T_BYTES;
      uint8_t *bst = sW + bs * W_BYTES;
      for (int it = dt; it < S::ITEMS; it += NDEC * 32) {
        int ti, q, swp;
        item_map<K>(it, ti, q, swp);
        const int tkl = ti >> 3, tnl = ti & 7;
        const uint8_t *tile = tst + tkl * S::ROWB + tnl * 32 * K;
        uint32_t w[S::NW + 1];
#pragma unroll
        for (int cc = 0; cc < S::CPL; ++cc) {
          const uint4 v4 = *reinterpret_cast<const uint4 *>(tile + q * 16 * S::CPL + 16 * cc);
          w[4 * cc + 0] = v4.x;
          w[4 * cc + 1] = v4.y;
          w[4 * cc + 2] = v4.z;
          w[4 * cc + 3] = v4.w;
        }
        w[S::NW] = *reinterpret_cast<const uint32_t *>(tile + ((q + 1) % S::LPT) * 16 * S::CPL);
        decode_rows<K, 0>(w, bst, tkl * 16 + S::G * q, tnl * 16, swp);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic stores -> tensor-core reads
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&wfull[bs]);
        tc::mbar_arrive(&tempty[ts]);
      }
    }

    // ---------------- epilogue
    // (1) warps 3..6 (TMEM lanes 96-127, 0-31, 32-63, 64-95 = output columns)
    // write the accumulator, times sigma, transposed into a scratch [M][128]
    // fp32 that reuses the operand ring (free once every MMA has completed).
    float *scratch = reinterpret_cast<float *>(smem);
    if (warp < 7) {
      bool ok = tc::mbar_wait(accum, 0);
      ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
      if (!ok && lane == 0) set_device_error(a.err, kErrBounds);
      tc::tc_fence_after();
      const int lane_base = 32 * (warp & 3);
      const int ncol = lane_base + lane;
      for (int m0 = 0; m0 < a.M; m0 += 8) {
        uint32_t r[8];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "r"(tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)m0));
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (m0 + j < a.M) scratch[(m0 + j) * 128 + ncol] = __uint_as_float(r[j]) * kSigma;
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
    tc::tmem_dealloc(tmem_base, NMAX);
  }
}

}  // namespace ftc
}  // namespace exl3

using namespace exl3;

static PFN_cuTensorMapEncodeTiled_v12000 ftc_tmap_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Number of k splits (one CTA per SM): the split count whose CTAs fill whole
// waves best, keeping at least 16 k steps of 64 per CTA (fewer on ties).
int exl3_fused_tc_splits(int k, int n) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
    cudaGetLastError();
  }
  const int kb = k / 64, tiles = n / 128;
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= kb && (s == 1 || kb / s >= 16); ++s) {
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
int exl3_launch_fused_tc(const uint16_t *xh, const uint16_t *trellis, const uint16_t *svh, int M, int k, int n,
                         int K, void *y, bool f32out, float *partials, int *counters, int *err, int splits,
                         cudaStream_t s) {
  auto fn = ftc_tmap_fn();
  if (!fn) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  CUtensorMap ta;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)k * 2};
  const int npad = (M + 15) & ~15;
  cuuint32_t box[2] = {64, (cuuint32_t)npad};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(xh), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  ftc::Args a{trellis, reinterpret_cast<const __half *>(svh), y, partials, counters, err, M, k, n, n / 16,
              0, splits};
  dim3 grid(n / 128, splits);
  cudaError_t e = cudaSuccess;
#define EXL3_FTC(KK, F32, NM)                                                                                \
  do {                                                                                                      \
    auto kfn = ftc::fused_tc_kernel<KK, F32, NM>;                                                           \
    cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, ftc::Shape<KK, NM>::SMEM_BYTES);  \
    kfn<<<grid, ftc::NWARPS * 32, ftc::Shape<KK, NM>::SMEM_BYTES, s>>>(ta, a);                              \
    e = cudaGetLastError();                                                                                 \
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
