// fused_tc.cu -- small-M EXL3 linear (2 <= M <= 128 tokens) with the trellis
// decoded straight into tensor-core operands: no reconstructed weights in
// HBM ("exl3xpu" README, "Layout": fused GEMM for M <= 128; "Prefill: int8
// linears and oneDNN fused attention": the GEMM runs in the Hadamard domain).
//
//   y[m, :] = RHT_out( sigma * x'[m, :] (B - 510) ) . svh      per 128-column tile
//
// Per CTA: one 128-column tile of y and one k-range (k splits over CTAs).
//   warp 0     producer: TMA of the x' tile (128 rows x 64 k, rows >= M read as
//              zero) and bulk copies of the four trellis rows (8 tiles each) of
//              every 64-deep k step into a ring of shared-memory stages
//   warp 1     MMA issuer: 4 x tcgen05.mma M128 N128 K16 per stage into TMEM
//   warps 2-9  decoders: each lane cuts 16 G trellis states out of its stage
//              chunk, hashes them (IMAD + DP4A seeded with 0x6400 gives the
//              fp16 value 1024 + B), subtracts 1534 in half2 (exact) and stores
//              the integers B - 510 as the MN-major, 128-byte-swizzled fp16
//              operand (row k, 64 n per 128-byte row; 8-row k groups 2 KB
//              apart, 64-wide n atoms 1 KB apart).  They then run the
//              epilogue: TMEM rows to a shared scratch, the fixed-order split-k
//              combine (last CTA to arrive, no waiting) and a warp-level
//              FWHT-128 per token row.
// Every wait is bounded and reports through the device error word.
#include <cudaTypedefs.h>

#include "exl3_common.cuh"
#include "tc_ptx.cuh"
#include "trellis_window.cuh"

namespace exl3 {
namespace ftc {

constexpr int BM = 128, BN = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BK * BN * 2;
constexpr int NDEC = 8;   // decoder warps

template <int K>
struct Shape {
  static constexpr int G = 8 / gcd_c(K, 8);      // rows per lane item
  static constexpr int CPL = K / gcd_c(K, 8);    // 16-byte chunks per item
  static constexpr int LPT = 16 / G;             // items per tile
  static constexpr int ROWB = (BN / 16) * 32 * K;   // one tile row of the CTA: 8 tiles
  static constexpr int T_BYTES = 4 * ROWB;          // 4 tile rows per 64-deep k step
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + T_BYTES;
  static constexpr int STAGES = 3;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024;
  static constexpr int ITEMS = 32 * LPT;         // (tile, group) items per stage
  static constexpr int NW = 4 * CPL;
};

// MN-major 128B-swizzle descriptor: LBO = n-atom stride, SBO = k-group stride.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(const void *base, uint32_t lbo, uint32_t sbo) {
  const uint64_t addr = tc::smem_u32(base);
  uint64_t d = 0;
  d |= (addr >> 4) & 0x3FFFull;
  d |= (uint64_t)(lbo >> 4) << 16;
  d |= (uint64_t)(sbo >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__host__ __device__ constexpr uint32_t idesc_f16_bmn(int M, int N) {
  return tc::idesc_f16(M, N) | (1u << 16);   // B is MN-major
}

struct Args {
  const uint16_t *trellis;
  const __half *svh;
  void *y;
  float *partials;     // [splits][M][n]
  int *counters;       // [n / 128]
  int *err;
  int M, k, n, tiles_n, kb_per_split, splits;
};

__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   tc::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
               : "memory");
}

// Two adjacent weights (columns C, C + 1 of row R) as the half2 (B0 - 510, B1 - 510):
// DP4A seeded with 0x6400 gives the fp16 bits of 1024 + B; 1024 + B - 1534 is exact.
template <int K, int R, int C>
__device__ __forceinline__ uint32_t decode_pair(const uint32_t (&w)[Shape<K>::NW + 1]) {
  const uint32_t s0 = window_at<(16 * R + C) * K>(w), s1 = window_at<(16 * R + C + 1) * K>(w);
  const uint32_t h0 = __dp4a(s0 * kMul1, 0x01010101u, 0x6400u);
  const uint32_t h1 = __dp4a(s1 * kMul1, 0x01010101u, 0x6400u);
  const uint32_t pr = __byte_perm(h0, h1, 0x5410);
  const __half2 d = __hsub2(*reinterpret_cast<const __half2 *>(&pr), __half2half2(__ushort_as_half(0x65FE)));
  return *reinterpret_cast<const uint32_t *>(&d);
}

// Decode one (tile, row group) item: rows G q .. G q + G - 1 of the tile,
// 16 columns each, into the operand stage.
template <int K, int R>
__device__ __forceinline__ void decode_rows(const uint32_t (&w)[Shape<K>::NW + 1], uint8_t *bstage, int k0,
                                            int nn0) {
  if constexpr (R < Shape<K>::G) {
    const uint4 lo = make_uint4(decode_pair<K, R, 0>(w), decode_pair<K, R, 2>(w), decode_pair<K, R, 4>(w),
                                decode_pair<K, R, 6>(w));
    const uint4 hi = make_uint4(decode_pair<K, R, 8>(w), decode_pair<K, R, 10>(w), decode_pair<K, R, 12>(w),
                                decode_pair<K, R, 14>(w));
    const int kk = k0 + R;                         // k within the 64-deep step
    const int kg = kk >> 3, kr = kk & 7;
    const int na = nn0 >> 6, ch = (nn0 & 63) >> 3;  // 16 columns = chunks ch, ch + 1 of a 64-wide atom
    uint8_t *row = bstage + kg * 2048 + na * 1024 + kr * 128;
    *reinterpret_cast<uint4 *>(row + ((ch ^ kr) << 4)) = lo;
    *reinterpret_cast<uint4 *>(row + (((ch + 1) ^ kr) << 4)) = hi;
    decode_rows<K, R + 1>(w, bstage, k0, nn0);
  }
}

template <int K, bool F32OUT>
__global__ void __launch_bounds__(320, 2) fused_tc_kernel(const __grid_constant__ CUtensorMap tmA, Args a) {
  using S = Shape<K>;
  constexpr int STAGES = S::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t *sA = smem;                                   // [STAGES][A_BYTES]
  uint8_t *sB = smem + STAGES * A_BYTES;                // [STAGES][B_BYTES]
  uint8_t *sT = sB + STAGES * B_BYTES;                  // [STAGES][T_BYTES]
  uint64_t *full = reinterpret_cast<uint64_t *>(sT + STAGES * S::T_BYTES);
  uint64_t *bfull = full + STAGES;
  uint64_t *empty = bfull + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tfull + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_last = const_cast<int *>(abort_flag + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x, split = blockIdx.y;
  const int kb0 = split * a.kb_per_split, nkb = a.kb_per_split;
  const int tn0 = nt * (BN / 16);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&bfull[s], NDEC);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(tfull, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmA);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 128);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int i = 0; i < nkb && !*abort_flag; ++i) {
        const int kb = kb0 + i;
        if (!tc::mbar_wait(&empty[stage], phase ^ 1)) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&full[stage], A_BYTES + S::T_BYTES);
        tc::tma_load_2d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, 0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const long tk = (long)kb * 4 + j;
          bulk_copy(sT + stage * S::T_BYTES + j * S::ROWB, a.trellis + (tk * a.tiles_n + tn0) * 16 * K, S::ROWB,
                    &full[stage]);
        }
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; i < nkb && ok; ++i) {
        ok = tc::mbar_wait(&full[stage], phase) && tc::mbar_wait(&bfull[stage], phase);
        if (!ok || *abort_flag) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        const uint64_t ad = tc::sdesc_k_sw128(sA + stage * A_BYTES);
        const uint64_t bd = sdesc_mn_sw128(sB + stage * B_BYTES, 1024, 2048);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc::mma_f16(tmem_base, ad + 2 * kk, bd + (uint64_t)((2 * 2048 * kk) >> 4), idesc_f16_bmn(BM, BN),
                      (i | kk) != 0 ? 1u : 0u);
        tc::mma_commit(&empty[stage]);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
      tc::mma_commit(tfull);
    }
  } else {
    // ---------------- decoders (warps 2..9)
    const int dt = threadIdx.x - 64;   // 0..255
    int stage = 0;
    uint32_t phase = 0;
    for (int i = 0; i < nkb; ++i) {
      if (!*abort_flag && !tc::mbar_wait(&full[stage], phase)) {
        if (lane == 0) set_device_error(a.err, kErrBounds);
        *abort_flag = 1;
      }
      const uint8_t *tst = sT + stage * S::T_BYTES;
      uint8_t *bst = sB + stage * B_BYTES;
      for (int it = dt; it < S::ITEMS; it += NDEC * 32) {
        const int ti = it / S::LPT, q = it % S::LPT;
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
        decode_rows<K, 0>(w, bst, tkl * 16 + S::G * q, tnl * 16);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic stores -> tensor-core reads
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bfull[stage]);
      if (++stage == STAGES) { stage = 0; phase ^= 1; }
    }

    // ---------------- epilogue
    // (1) warps 2..5 (TMEM lanes 64-95, 96-127, 0-31, 32-63) copy the valid
    // token rows, times sigma, into a scratch [M][128] fp32 that reuses the
    // operand ring (free once every MMA has completed).
    float *scratch = reinterpret_cast<float *>(smem);
    {
      bool ok = true;
      if (warp < 6) {
        ok = tc::mbar_wait(tfull, 0);
        ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
        if (!ok && lane == 0) set_device_error(a.err, kErrBounds);
        tc::tc_fence_after();
        const int lane_base = 32 * (warp & 3);
        const int m = lane_base + lane;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float t[32];
          tc::tmem_ld32(tmem_base + ((uint32_t)lane_base << 16) + 32 * c, t);
          tc::tmem_ld_wait();
          if (m < a.M) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4 *>(scratch + m * 128 + 32 * c + j) =
                  make_float4(t[j] * kSigma, t[j + 1] * kSigma, t[j + 2] * kSigma, t[j + 3] * kSigma);
          }
        }
        tc::tc_fence_before();
      }
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");   // the eight decoder warps
    const int col0 = nt * BN;
    const int ew = warp - 2;                          // 0..7
    bool finish = true;
    if (a.splits > 1) {
      // (2) partial sums of this split; the last CTA of the column tile adds all
      // splits in order.
      for (int m = ew; m < a.M; m += NDEC) {
        const float4 v = *reinterpret_cast<const float4 *>(scratch + m * 128 + 4 * lane);
        *reinterpret_cast<float4 *>(a.partials + ((long)split * a.M + m) * a.n + col0 + 4 * lane) = v;
      }
      __threadfence();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (threadIdx.x == 64) {
        const int old = atomicAdd(a.counters + nt, 1);
        if (old >= a.splits) set_device_error(a.err, kErrDirtyCounter);
        *s_last = (old == a.splits - 1);
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      finish = *s_last != 0;
      if (finish) __threadfence();
    }
    // (3) one warp per token row: sum the splits, FWHT-128, 2^-3.5, svh, store
    if (finish) {
      for (int m = ew; m < a.M; m += NDEC) {
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
      if (a.splits > 1 && threadIdx.x == 64) a.counters[nt] = 0;   // leave the workspace clean
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, 128);
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

// Number of k splits: the smallest divisor of k/64 giving at least 2 CTAs per SM.
int exl3_fused_tc_splits(int k, int n) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
    cudaGetLastError();
  }
  const int kb = k / 64, tiles = n / 128;
  int best = kb;
  for (int s = 1; s <= kb; ++s) {
    if (kb % s) continue;
    best = s;
    if (tiles * s >= 2 * sms) break;
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
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(xh), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  ftc::Args a{trellis, reinterpret_cast<const __half *>(svh), y, partials, counters, err, M, k, n, n / 16,
              (k / 64) / splits, splits};
  dim3 grid(n / 128, splits);
  cudaError_t e = cudaSuccess;
#define EXL3_FTC(KK, F32)                                                                                    \
  do {                                                                                                      \
    auto kfn = ftc::fused_tc_kernel<KK, F32>;                                                               \
    cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, ftc::Shape<KK>::SMEM_BYTES);      \
    kfn<<<grid, 320, ftc::Shape<KK>::SMEM_BYTES, s>>>(ta, a);                                               \
    e = cudaGetLastError();                                                                                 \
  } while (0)
#define EXL3_FTC_K(KK) \
  case KK: if (f32out) EXL3_FTC(KK, true); else EXL3_FTC(KK, false); break;
  switch (K) {
    EXL3_FTC_K(1) EXL3_FTC_K(2) EXL3_FTC_K(3) EXL3_FTC_K(4) EXL3_FTC_K(5) EXL3_FTC_K(6) EXL3_FTC_K(7)
    EXL3_FTC_K(8)
    default: return exl3_fail(EXL3_ERR_BITS, "K = %d", K);
  }
#undef EXL3_FTC_K
#undef EXL3_FTC
  return exl3_cuda_check(e, "fused_tc launch");
}
