// gemm_tc.cu -- prefill contraction on the 5th-generation tensor cores
// (tcgen05 MMA, TMEM accumulators, TMA operand staging), with the output
// Hadamard transform fused into the epilogue.
//
//   y[m, :] = ( 2^-3.5 H (pre * rs[m] * (x' W)[m, :]) per 128-block ) . svh
//
// x' fp16 [M][k] (K-major) and Wt fp16 [n][k] (the transposed reconstruct,
// K-major) are read by TMA in 128-byte-swizzled boxes.  This is the
// reconstruct-then-GEMM form of the prefill linear ("exl3xpu" README,
// "Layout": large M goes through reconstruct + a dense GEMM; "Prefill: int8
// linears and oneDNN fused attention": the GEMM runs in the Hadamard domain).
//
// Persistent kernel, one CTA per SM, 6 warps:
//   warp 0     TMA producer (one thread): A box 128 x 64, B box 256 x 64 per stage
//   warp 1     TMEM owner and MMA issuer (one thread): 4 x (M128 N256 K16) per stage
//   warps 2-5  epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31, one output
//              row per thread, two 128-column FWHTs in registers per tile
//              (integer mode with 256-column tiles: warps 2-9, see below)
// TMEM holds two 128 x BN fp32 accumulators so the epilogue of one tile
// overlaps the MMAs of the next.
//
// Integer mode (the int8 variant of "exl3xpu" README, "Prefill: int8
// linears and oneDNN fused attention").  GB300's tcgen05 has no int8 kind
// (kind::i8 does not assemble for sm_103a), so the s8 x s8 -> s32 product is
// computed exactly on the f16 kind: both operands hold integers in
// [-127, 127] as fp16, every k-chunk of 512 accumulates in a fresh fp32
// accumulator (|partial sum| <= 512 * 127^2 < 2^23, so every sum is exact),
// and the epilogue converts each chunk to int32 and adds them in registers.
// With 256-column tiles the epilogue has 8 warps (two per TMEM lane quarter,
// 128 columns each), so the MMA reads 48 KB of operands per 512 tensor cycles
// rather than 32 KB per 256 (the 128-column tile needed more shared-memory
// bandwidth than the SM has).
// The output is y = RHT_out(acc * row_scale[m] * weight_scale) . svh.
#include <cudaTypedefs.h>

#include "exl3_common.cuh"
#include "tc_ptx.cuh"

namespace exl3 {
namespace gtc {

constexpr int BM = 128, BK = 64;

// BN = 256: 4 stages of 48 KB; BN = 128: 6 stages of 32 KB.
template <int BN>
struct Cfg {
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*barriers*/ + 1024 /*alignment*/;
  static constexpr uint32_t IDESC = tc::idesc_f16(BM, BN);
  static constexpr uint32_t TMEM_COLS = 2 * BN;
};

constexpr int Q8_CHUNK_KB = 8;   // k-blocks of 64 per exact fp32 chunk (512 elements)

// Epilogue warps: the integer mode with 256-column tiles keeps each row's 256
// running int32 sums in two warps of 128 registers (two warps per TMEM lane
// quarter); otherwise four warps, one per lane quarter.
template <int BN, bool Q8>
constexpr int epi_warps() { return (Q8 && BN == 256) ? 8 : 4; }

struct Args {
  int M, n, k;
  const __half *svh;     // [n]
  void *y;               // [M][n]
  const float *row_scale;  // [M] or null
  float pre;
  int *err;
  int32_t *acc_out;      // integer mode: optional [M][n] copy of the accumulators
  const __half *bias;    // [n] fp16 added after svh, or null
};

__device__ __forceinline__ void fwht128_regs(float (&v)[128]) {
#pragma unroll
  for (int h = 1; h < 128; h <<= 1)
#pragma unroll
    for (int i = 0; i < 128; i += 2 * h)
#pragma unroll
      for (int j = i; j < i + h; ++j) {
        const float a = v[j], b = v[j + h];
        v[j] = a + b;
        v[j + h] = a - b;
      }
}

// y[row][col0 .. col0+127] = v * 2^-3.5 * svh (+ bias) (v already transformed).
template <bool F32OUT>
__device__ __forceinline__ void store_row(const float (&v)[128], const Args &a, int row, int col0) {
  if (row >= a.M) return;
#pragma unroll
  for (int c8 = 0; c8 < 16; ++c8) {
    const uint4 sv = __ldg(reinterpret_cast<const uint4 *>(a.svh + col0 + 8 * c8));
    const __half2 *sh = reinterpret_cast<const __half2 *>(&sv);
    float o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      o[2 * j] = v[8 * c8 + 2 * j] * kRhtScale * __low2float(sh[j]);
      o[2 * j + 1] = v[8 * c8 + 2 * j + 1] * kRhtScale * __high2float(sh[j]);
    }
    if (a.bias) {   // the output bias, per output feature
      const uint4 bv = __ldg(reinterpret_cast<const uint4 *>(a.bias + col0 + 8 * c8));
      const __half2 *bh = reinterpret_cast<const __half2 *>(&bv);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        o[2 * j] = __fadd_rn(o[2 * j], __low2float(bh[j]));   // one rounding, never contracted
        o[2 * j + 1] = __fadd_rn(o[2 * j + 1], __high2float(bh[j]));
      }
    }
    if (F32OUT) {
      float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.y) + (long)row * a.n + col0 + 8 * c8);
      dst[0] = make_float4(o[0], o[1], o[2], o[3]);
      dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    } else {
      __half2 h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = __floats2half2_rn(o[2 * j], o[2 * j + 1]);
      *reinterpret_cast<uint4 *>(static_cast<__half *>(a.y) + (long)row * a.n + col0 + 8 * c8) =
          *reinterpret_cast<uint4 *>(h);
    }
  }
}

template <int BN, bool F32OUT, bool Q8>
__global__ void __launch_bounds__((2 + epi_warps<BN, Q8>()) * 32, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                                                         const __grid_constant__ CUtensorMap tmB, Args a) {
  using C = Cfg<BN>;
  constexpr int STAGES = C::STAGES, A_BYTES = C::A_BYTES, B_BYTES = C::B_BYTES, STAGE_BYTES = C::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t *sA = smem;                                   // [STAGES][A_BYTES]
  uint8_t *sB = smem + STAGES * A_BYTES;                // [STAGES][B_BYTES]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int MT = (a.M + BM - 1) / BM, NT = a.n / BN, KB = a.k / BK;
  const int num_tiles = MT * NT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], epi_warps<BN, Q8>());
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // a programmatic dependent of the reconstruct, whose completion implies
  // the activation transform's: operands, y and the error word after this
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x) {
        const int mt = tile % MT, nt = tile / MT;
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait(&empty[stage], phase ^ 1)) {
            set_device_error(a.err, kErrBounds);
            *abort_flag = 1;
            break;
          }
          tc::mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          tc::tma_load_2d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, mt * BM);
          tc::tma_load_2d(sB + stage * B_BYTES, &tmB, &full[stage], kb * BK, nt * BN);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    // MMA issuer: the whole warp runs the loop (waits and descriptors stay
    // warp-uniform); one elected lane issues the MMAs and their commits.
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    const int CH = Q8 ? Q8_CHUNK_KB : KB;       // k-blocks per accumulator hand-off
    bool stop = __any_sync(0xffffffffu, *abort_flag != 0);
    for (int tile = blockIdx.x; tile < num_tiles && !stop; tile += gridDim.x) {
      for (int kb0 = 0; kb0 < KB && !stop; kb0 += CH) {
        const bool okt = __all_sync(0xffffffffu, tc::mbar_wait(&tempty[acc], acc_phase ^ 1));
        if (!okt) {
          if (lane == 0) set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          stop = true;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        const int kb1 = min(KB, kb0 + CH);
        for (int kb = kb0; kb < kb1; ++kb) {
          const bool okf = __all_sync(0xffffffffu, tc::mbar_wait(&full[stage], phase));
          if (!okf) {
            if (lane == 0) set_device_error(a.err, kErrBounds);
            *abort_flag = 1;
            stop = true;
            break;
          }
          tc::tc_fence_after();
          const uint64_t ad = tc::sdesc_k_sw128(sA + stage * A_BYTES);
          const uint64_t bd = tc::sdesc_k_sw128(sB + stage * B_BYTES);
          if (tc::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc::mma_f16(d, ad + 2 * kk, bd + 2 * kk, C::IDESC, (kb != kb0 || kk != 0) ? 1u : 0u);
            tc::mma_commit(&empty[stage]);
          }
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (tc::elect_one()) tc::mma_commit(&tfull[acc]);
        __syncwarp();
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        stop = stop || __any_sync(0xffffffffu, *abort_flag != 0);
      }
    }
  } else {
    // epilogue warps 2 .. 2 + epi_warps - 1
    const int lane_base = 32 * (warp & 3);
    const int half = (Q8 && BN == 256) ? (warp - 2) / 4 : 0;   // integer mode: 128-column half
    int acc = 0;
    uint32_t acc_phase = 0;
    const int CH = Q8 ? Q8_CHUNK_KB : KB;
    const int nchunks = (KB + CH - 1) / CH;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int mt = tile % MT, nt = tile / MT;
      const int row = mt * BM + lane_base + lane;
      float rs = a.pre;
      if (a.row_scale && row < a.M) rs *= a.row_scale[row];
      bool failed = false;
      if constexpr (Q8) {
        // One 128-column block per warp (BN == 256: two warps per row),
        // integer accumulation per chunk.  The int32 sums live in the same
        // registers that later hold the float row (bit patterns), keeping one
        // 128-entry array alive.
        float v[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) v[i] = __int_as_float(0);
        for (int ch = 0; ch < nchunks; ++ch) {
          bool ok = tc::mbar_wait(&tfull[acc], acc_phase);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok || *abort_flag) { failed = true; break; }
          tc::tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float t[32];
            tc::tmem_ld32(tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)(acc * BN + half * 128 + 32 * c), t);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              v[32 * c + i] = __int_as_float(__float_as_int(v[32 * c + i]) + __float2int_rn(t[i]));
          }
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&tempty[acc]);
          if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        if (failed) {
          if (lane == 0) set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        const int col0 = nt * BN + half * 128;
        if (a.acc_out && row < a.M) {
#pragma unroll
          for (int c4 = 0; c4 < 32; ++c4)
            *reinterpret_cast<int4 *>(a.acc_out + (long)row * a.n + col0 + 4 * c4) =
                make_int4(__float_as_int(v[4 * c4]), __float_as_int(v[4 * c4 + 1]), __float_as_int(v[4 * c4 + 2]),
                          __float_as_int(v[4 * c4 + 3]));
        }
#pragma unroll
        for (int i = 0; i < 128; ++i) v[i] = (float)__float_as_int(v[i]) * rs;
        fwht128_regs(v);
        store_row<F32OUT>(v, a, row, col0);
      } else {
        bool ok = tc::mbar_wait(&tfull[acc], acc_phase);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok || *abort_flag) {
          if (lane == 0) set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
#pragma unroll 1
        for (int blk = 0; blk < BN / 128; ++blk) {
          float v[128];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float t[32];
            tc::tmem_ld32(tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)(acc * BN + blk * 128 + 32 * c), t);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[32 * c + i] = t[i];
          }
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 128; ++i) v[i] *= rs;
          fwht128_regs(v);
          store_row<F32OUT>(v, a, row, nt * BN + blk * 128);
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&tempty[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
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

}  // namespace gtc
}  // namespace exl3

using namespace exl3;

static PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() { return exl3_tmap_encode_fn(); }

// 2-D fp16 tensor [rows][cols] (cols contiguous), box [box_rows][64], 128-byte swizzle.
static int make_tmap_f16(CUtensorMap *m, const void *base, int rows, int cols, int box_rows) {
  auto fn = tmap_encode_fn();
  if (!fn) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return EXL3_OK;
}

// n must be a multiple of 128 and k of 64; rows of x' beyond M read as zero.
// q8: integer mode (operands integer-valued fp16, exact int32 accumulation).
// bias: [n] fp16 added to the output, or null.
int exl3_launch_gemm_tc(const uint16_t *xh, const uint16_t *wt, int M, int n, int k, const uint16_t *svh,
                        void *y, bool f32out, const float *row_scale, float pre, int *err, cudaStream_t s,
                        bool q8 = false, int32_t *acc_out = nullptr, const uint16_t *bias = nullptr) {
  CUtensorMap ta, tb;
  int rc = make_tmap_f16(&ta, xh, M, k, gtc::BM);
  if (rc) return rc;
  const bool wide = (n % 256) == 0;
  rc = make_tmap_f16(&tb, wt, n, k, wide ? 256 : 128);
  if (rc) return rc;
  const int sms = exl3_sm_count();
  gtc::Args a{M, n, k, reinterpret_cast<const __half *>(svh), y, row_scale, pre, err, acc_out,
              reinterpret_cast<const __half *>(bias)};
  const int tiles = ((M + gtc::BM - 1) / gtc::BM) * (n / (wide ? 256 : 128));
  const int grid = tiles < sms ? tiles : sms;
  cudaError_t e = cudaSuccess;
#define EXL3_GTC(BNV, F32, Q)                                                                           \
  do {                                                                                                \
    auto kfn = gtc::gemm_tc_kernel<BNV, F32, Q>;                                                      \
    cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, gtc::Cfg<BNV>::SMEM_BYTES); \
    e = launch_pdl(kfn, dim3(grid), dim3((2 + gtc::epi_warps<BNV, Q>()) * 32), gtc::Cfg<BNV>::SMEM_BYTES, s, ta, \
                   tb, a);                                                                            \
  } while (0)
  if (q8 && wide) {
    if (f32out) EXL3_GTC(256, true, true); else EXL3_GTC(256, false, true);
  } else if (q8) {
    if (f32out) EXL3_GTC(128, true, true); else EXL3_GTC(128, false, true);
  } else if (wide) {
    if (f32out) EXL3_GTC(256, true, false); else EXL3_GTC(256, false, false);
  } else {
    if (f32out) EXL3_GTC(128, true, false); else EXL3_GTC(128, false, false);
  }
#undef EXL3_GTC
  return exl3_cuda_check(e, "gemm_tc launch");
}
