// moe_fused.cu -- the two grouped expert projections with the trellis decoded
// straight into tcgen05 operands ("Bringing EXL3 Trellis Quantization to 35B
// MoE on Intel Arc 140V", section 2.B: one grouped launch for gate+up with a
// shared input row, one for down; "exl3xpu" README, "MoE (routed experts)":
// routing weight on the down output, in fp32, and no fp16 expert weights
// anywhere).
//
// A CTA handles one (128-row expert tile, 128-column output tile) pair of the
// device-side tile list; the MMA computes the transposed product (decoded
// weights as the MN-major A operand, M = 128 output columns; the tile's x'
// rows as the K-major B operand, N = 128), with the warp roles of the
// small-M linear: trellis producer, MMA issuer, x' producer, two groups of
// eight decoder warps on alternate k steps.
//
// Phase 1 (gate + up): both projections of the expert are decoded per k step
//   into two accumulators; per token row the epilogue forms
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
using ftc::NWARPS;
using ftc::W_BYTES;

constexpr int XROWS = 128;
constexpr int X_BYTES = XROWS * BK * 2;

template <int K, int PHASE>
struct Cfg {
  static constexpr int NP = PHASE == 1 ? 2 : 1;                 // projections decoded per k step
  static constexpr int T_ONE = 4 * (BN / 16) * 32 * K;          // trellis of one projection per k step
  static constexpr int T_BYTES = NP * T_ONE;
  static constexpr int XS = PHASE == 1 ? 3 : 4;
  static constexpr int WS = PHASE == 1 ? 2 : 4;
  static constexpr int TS_FIT = (220 * 1024 - XS * NP * X_BYTES - WS * NP * W_BYTES) / T_BYTES;
  static constexpr int TS = TS_FIT > 24 ? 24 : TS_FIT;
  static constexpr int SMEM_BYTES = XS * NP * X_BYTES + WS * NP * W_BYTES + TS * T_BYTES + 1024 + 1024;
  static constexpr int ITEMS = NP * 32 * ftc::Shape<K, 32>::LPT;
  static constexpr uint32_t TMEM_COLS = NP == 2 ? 256 : 128;
  static_assert(TS >= 2, "trellis ring too shallow");
  static_assert(NP * XROWS * 128 * 4 <= XS * NP * X_BYTES + WS * NP * W_BYTES, "epilogue scratch overlaps the trellis ring");
};

struct Args {
  const int4 *mtiles;       // (expert, first row, rows, 0)
  const int *n_mtiles;
  int NT, KB;               // output tiles per m-tile, k steps
  const uint16_t *trellis;  // [E][nslots][k/16][n/16][16K]
  int tiles_n;              // n / 16 of one projection
  long slot_words;          // words of one (expert, slot) trellis
  int nslots;
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
};

template <int K, int PHASE>
__global__ void __launch_bounds__(NWARPS * 32, 1) moe_fused_kernel(const __grid_constant__ CUtensorMap tmX0,
                                                                   const __grid_constant__ CUtensorMap tmX1,
                                                                   Args a) {
  using C = Cfg<K, PHASE>;
  using S = ftc::Shape<K, 32>;
  constexpr int NP = C::NP, XS = C::XS, WS = C::WS, TS = C::TS;
  const int tile = blockIdx.x;
  if (tile >= *a.n_mtiles * a.NT) return;   // uniform per CTA: the tile list is device-side
  const int4 mt = a.mtiles[tile / a.NT];
  const int nt = tile % a.NT, e = mt.x, row0 = mt.y, rows = mt.z;
  const int tn0 = nt * (BN / 16);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t *sX = smem;                                   // [XS][NP][X_BYTES]
  uint8_t *sW = sX + XS * NP * X_BYTES;                 // [WS][NP][W_BYTES]
  uint8_t *sT = sW + WS * NP * W_BYTES;                 // [TS][T_BYTES]
  uint64_t *tfull = reinterpret_cast<uint64_t *>(sT + TS * C::T_BYTES);
  uint64_t *tempty = tfull + TS;
  uint64_t *xfull = tempty + TS;
  uint64_t *xempty = xfull + XS;
  uint64_t *wfull = xempty + XS;
  uint64_t *wempty = wfull + WS;
  uint64_t *accum = wempty + WS;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = a.KB;

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
    tc::prefetch_tmap(&tmX0);
    if (NP == 2) tc::prefetch_tmap(&tmX1);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- trellis producer
    if (lane == 0) {
      for (int i = 0; i < KB && !*abort_flag; ++i) {
        const int st = i % TS;
        if (!tc::mbar_wait(&tempty[st], ((i / TS) & 1) ^ 1)) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&tfull[st], C::T_BYTES);
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          const uint16_t *tr = a.trellis + ((long)e * a.nslots + p) * a.slot_words;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const long tk = (long)i * 4 + j;
            ftc::bulk_copy(sT + st * C::T_BYTES + p * C::T_ONE + j * S::ROWB, tr + (tk * a.tiles_n + tn0) * 16 * K,
                           S::ROWB, &tfull[st]);
          }
        }
      }
    }
  } else if (warp == 2) {
    // ---------------- x' producer: the tile's sorted rows
    if (lane == 0) {
      for (int i = 0; i < KB && !*abort_flag; ++i) {
        const int st = i % XS;
        if (!tc::mbar_wait(&xempty[st], ((i / XS) & 1) ^ 1)) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&xfull[st], NP * X_BYTES);
        tc::tma_load_2d(sX + st * NP * X_BYTES, &tmX0, &xfull[st], i * BK, row0);
        if (NP == 2) tc::tma_load_2d(sX + st * NP * X_BYTES + X_BYTES, &tmX1, &xfull[st], i * BK, row0);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ftc::idesc_f16_amn(BN, XROWS);
      for (int i = 0; i < KB; ++i) {
        const int xs = i % XS, ws = i % WS;
        const bool ok = tc::mbar_wait(&xfull[xs], (i / XS) & 1) && tc::mbar_wait(&wfull[ws], (i / WS) & 1);
        if (!ok || *abort_flag) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          const uint64_t ad = ftc::sdesc_mn_sw128(sW + (ws * NP + p) * W_BYTES, 1024, 2048);
          const uint64_t bd = tc::sdesc_k_sw128(sX + (xs * NP + p) * X_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_f16(tmem_base + p * XROWS, ad + (uint64_t)((2 * 2048 * kk) >> 4), bd + 2 * kk, idesc,
                        (i | kk) != 0 ? 1u : 0u);
        }
        tc::mma_commit(&wempty[ws]);
        tc::mma_commit(&xempty[xs]);
      }
      tc::mma_commit(accum);
    }
  } else {
    // ---------------- decoders: group g takes k steps i = g, g + 2, ...
    const int dw = warp - 3;
    const int grp = dw / NDEC, dt = (dw % NDEC) * 32 + lane;
    constexpr int PER_P = 32 * S::LPT;
    // Epilogue operands, loaded now so that their latency hides behind the
    // decode: this lane's 4 columns of svh (gate, up) and suh (down), or of
    // svh (down) and the routing weights of the warp's rows (lane q holds
    // row dw + 16 q).
    const int col0 = nt * BN;
    float ep_a[4], ep_b[4], ep_c[4], row_w = 0.f;
    {
      auto ld4 = [&](const __half *src, float (&o)[4]) {
        const uint2 r = __ldg(reinterpret_cast<const uint2 *>(src + col0 + 4 * lane));
        const __half2 *h = reinterpret_cast<const __half2 *>(&r);
        o[0] = __low2float(h[0]);
        o[1] = __high2float(h[0]);
        o[2] = __low2float(h[1]);
        o[3] = __high2float(h[1]);
      };
      if (PHASE == 1) {
        ld4(a.svh13 + ((long)e * 2 + 0) * a.inter, ep_a);
        ld4(a.svh13 + ((long)e * 2 + 1) * a.inter, ep_b);
        ld4(a.suh2 + (long)e * a.inter, ep_c);
      } else {
        ld4(a.svh2 + (long)e * a.hidden, ep_a);
        const int m = dw + NGRP * NDEC * lane;
        if (lane < XROWS / (NGRP * NDEC) && m < rows) row_w = a.weights[a.perm[row0 + m]];
      }
    }
    for (int i = grp; i < KB; i += NGRP) {
      const int ts = i % TS, bs = i % WS;
      const bool ok = (*abort_flag) || (tc::mbar_wait(&tfull[ts], (i / TS) & 1) &&
                                        tc::mbar_wait(&wempty[bs], ((i / WS) & 1) ^ 1));
      if (!ok) {
        if (lane == 0) set_device_error(a.err, kErrBounds);
        *abort_flag = 1;
      }
      for (int it = dt; it < C::ITEMS; it += NDEC * 32) {
        const int p = it / PER_P;
        int ti, q, swp;
        ftc::item_map<K>(it % PER_P, ti, q, swp);
        const int tkl = ti >> 3, tnl = ti & 7;
        const uint8_t *tilep = sT + ts * C::T_BYTES + p * C::T_ONE + tkl * S::ROWB + tnl * 32 * K;
        uint32_t w[S::NW + 1];
        ftc::load_item<K>(tilep, q, w);
        ftc::decode_rows<K, 0>(w, sW + (bs * NP + p) * W_BYTES, tkl * 16 + S::G * q, tnl * 16, swp);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&wfull[bs]);
        tc::mbar_arrive(&tempty[ts]);
      }
    }

    // ---------------- epilogue
    // (1) accumulators (lane = output column, column = row of the tile),
    // times sigma, transposed into scratch [NP][rows][128] over the rings.
    float *scratch = reinterpret_cast<float *>(smem);
    if (warp < 7) {
      bool ok = tc::mbar_wait(accum, 0);
      ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
      if (!ok && lane == 0) set_device_error(a.err, kErrBounds);
      tc::tc_fence_after();
      const int lane_base = 32 * (warp & 3);
      const int ncol = lane_base + lane;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        for (int m0 = 0; m0 < rows; m0 += 8) {
          uint32_t r[8];
          asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                       : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                         "=r"(r[7])
                       : "r"(tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)(p * XROWS + m0)));
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (m0 + j < rows) scratch[(p * XROWS + m0 + j) * 128 + ncol] = __uint_as_float(r[j]) * kSigma;
        }
      }
      tc::tc_fence_before();
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NGRP * NDEC * 32) : "memory");
    // (2) one warp per row of the tile
    for (int m = dw; m < rows; m += NGRP * NDEC) {
      const long row = (long)row0 + m;
      const float4 g4 = *reinterpret_cast<const float4 *>(scratch + m * 128 + 4 * lane);
      float v[4] = {g4.x, g4.y, g4.z, g4.w};
      fwht128_warp(v, lane);
      if (PHASE == 1) {
        const float4 u4 = *reinterpret_cast<const float4 *>(scratch + (XROWS + m) * 128 + 4 * lane);
        float u[4] = {u4.x, u4.y, u4.z, u4.w};
        fwht128_warp(u, lane);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float g = v[q] * kRhtScale * ep_a[q];
          const float uu = u[q] * kRhtScale * ep_b[q];
          v[q] = g / (1.0f + expf(-g)) * uu * ep_c[q];   // h . suh_down
        }
        fwht128_warp(v, lane);
        __half2 o[2] = {__floats2half2_rn(v[0] * kRhtScale, v[1] * kRhtScale),
                        __floats2half2_rn(v[2] * kRhtScale, v[3] * kRhtScale)};
        *reinterpret_cast<uint2 *>(a.hout + row * a.inter + col0 + 4 * lane) = *reinterpret_cast<uint2 *>(o);
      } else {
        const float w = __shfl_sync(0xffffffffu, row_w, m / (NGRP * NDEC));
        float4 o;
        o.x = v[0] * kRhtScale * ep_a[0] * w;
        o.y = v[1] * kRhtScale * ep_a[1] * w;
        o.z = v[2] * kRhtScale * ep_a[2] * w;
        o.w = v[3] * kRhtScale * ep_a[3] * w;
        *reinterpret_cast<float4 *>(a.dout + row * a.hidden + col0 + 4 * lane) = o;
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace mf
}  // namespace exl3

using namespace exl3;

static PFN_cuTensorMapEncodeTiled_v12000 mf_tmap_fn() {
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

// rows x cols fp16 (cols contiguous), box 128 rows x 64, 128-byte swizzle.
static int mf_tmap(CUtensorMap *m, const void *base, int rows, int cols) {
  auto fn = mf_tmap_fn();
  if (!fn) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)mf::XROWS};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return EXL3_OK;
}

template <int PHASE>
static int mf_launch(int K, const CUtensorMap &t0, const CUtensorMap &t1, const mf::Args &a, int grid,
                     cudaStream_t s) {
  cudaError_t e = cudaSuccess;
#define EXL3_MF(KK)                                                                                      \
  case KK: {                                                                                             \
    auto kfn = mf::moe_fused_kernel<KK, PHASE>;                                                          \
    cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, mf::Cfg<KK, PHASE>::SMEM_BYTES); \
    kfn<<<grid, mf::NWARPS * 32, mf::Cfg<KK, PHASE>::SMEM_BYTES, s>>>(t0, t1, a);                        \
    e = cudaGetLastError();                                                                              \
  } break;
  switch (K) {
    EXL3_MF(1) EXL3_MF(2) EXL3_MF(3) EXL3_MF(4) EXL3_MF(5) EXL3_MF(6) EXL3_MF(7) EXL3_MF(8)
    default: return exl3_fail(EXL3_ERR_BITS, "K = %d", K);
  }
#undef EXL3_MF
  return exl3_cuda_check(e, "moe fused launch");
}

// Phase 1: xg, xu [U][hidden] fp16 sorted rows; w13 trellis [E][2][hidden/16][inter/16][16K].
int exl3_launch_moe_fused_gateup(const uint16_t *xg, const uint16_t *xu, int U, int hidden, int inter, int K,
                                 const uint16_t *w13_trellis, const int *mtiles, const int *n_mtiles, int max_mtiles,
                                 const uint16_t *svh13, const uint16_t *suh2, uint16_t *hout, int *err,
                                 cudaStream_t s) {
  CUtensorMap t0, t1;
  int rc = mf_tmap(&t0, xg, U, hidden);
  if (rc) return rc;
  rc = mf_tmap(&t1, xu, U, hidden);
  if (rc) return rc;
  mf::Args a{};
  a.mtiles = reinterpret_cast<const int4 *>(mtiles);
  a.n_mtiles = n_mtiles;
  a.NT = inter / 128;
  a.KB = hidden / 64;
  a.trellis = w13_trellis;
  a.tiles_n = inter / 16;
  a.slot_words = (long)(hidden / 16) * (inter / 16) * 16 * K;
  a.nslots = 2;
  a.svh13 = reinterpret_cast<const __half *>(svh13);
  a.suh2 = reinterpret_cast<const __half *>(suh2);
  a.hout = reinterpret_cast<__half *>(hout);
  a.inter = inter;
  a.err = err;
  return mf_launch<1>(K, t0, t1, a, max_mtiles * a.NT, s);
}

// Phase 2: h' [U][inter] fp16 sorted rows; w2 trellis [E][1][inter/16][hidden/16][16K]; d [U][hidden] fp32.
int exl3_launch_moe_fused_down(const uint16_t *hin, int U, int hidden, int inter, int K, const uint16_t *w2_trellis,
                               const int *mtiles, const int *n_mtiles, int max_mtiles, const uint16_t *svh2,
                               const float *weights, const int *perm, float *dout, int *err, cudaStream_t s) {
  CUtensorMap t0;
  int rc = mf_tmap(&t0, hin, U, inter);
  if (rc) return rc;
  mf::Args a{};
  a.mtiles = reinterpret_cast<const int4 *>(mtiles);
  a.n_mtiles = n_mtiles;
  a.NT = hidden / 128;
  a.KB = inter / 64;
  a.trellis = w2_trellis;
  a.tiles_n = hidden / 16;
  a.slot_words = (long)(inter / 16) * (hidden / 16) * 16 * K;
  a.nslots = 1;
  a.svh2 = reinterpret_cast<const __half *>(svh2);
  a.weights = weights;
  a.perm = perm;
  a.dout = dout;
  a.hidden = hidden;
  a.err = err;
  return mf_launch<2>(K, t0, t0, a, max_mtiles * a.NT, s);
}
