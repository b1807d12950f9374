// moe_gemm.cu -- the two grouped expert projections on the tensor cores
// (tcgen05 MMA, TMEM accumulators, TMA staging), one launch each, driven by
// the device-side tile list of the routing step ("Bringing EXL3 Trellis
// Quantization to 35B MoE on Intel Arc 140V", section 2.B: one grouped launch
// for gate+up with a shared input row, one for down; "exl3xpu" README, "MoE
// (routed experts)": routing weight on the down output, in fp32).
//
// Rows are the (token, slot) units sorted by expert; a 128-row m-tile never
// spans two experts (the routing step cuts tiles per expert), rows past the
// expert's count are computed and discarded.
//
// Phase 1 (gate + up, n-tile j = 128 columns of each):
//   TMEM[0:128)   += xg_tile * Wgate_e[j]^T      (xg = RHT(x . suh_gate_e))
//   TMEM[128:256) += xu_tile * Wup_e[j]^T        (xu = RHT(x . suh_up_e))
//   epilogue per row: g = RHT_out(gate) . svh_gate, u = RHT_out(up) . svh_up,
//   h = SiLU(g) u, and the down projection's input transform applied at once:
//   h' = 2^-3.5 H (h . suh_down) -> fp16 rows of the down GEMM's operand.
// Phase 2 (down, n-tile = 256 columns):
//   d = RHT_out(h' Wdown_e^T) . svh_down * routing weight -> fp32 rows.
#include <cudaTypedefs.h>

#include "exl3_common.cuh"
#include "tc_ptx.cuh"

namespace exl3 {
namespace mg {

constexpr int BM = 128, BK = 64, BN = 256;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;

template <int PHASE>
struct Cfg {
  static constexpr int NA = PHASE == 1 ? 2 : 1;
  static constexpr int STAGES = PHASE == 1 ? 3 : 4;
  static constexpr int STAGE_BYTES = NA * A_BYTES + B_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024;
  static constexpr uint32_t IDESC = PHASE == 1 ? tc::idesc_f16(BM, 128) : tc::idesc_f16(BM, 256);
};

struct Args {
  const int4 *mtiles;      // (expert, first row, rows, 0)
  const int *n_mtiles;
  int NT, KB;              // n-tiles per m-tile, k-blocks
  const __half *svh13;     // [E][2][inter]
  const __half *suh2;      // [E][inter]
  __half *hout;            // [U][inter]
  int inter;
  const __half *svh2;      // [E][hidden]
  const float *weights;    // [U] routing weight by unit
  const int *perm;         // sorted row -> unit
  float *dout;             // [U][hidden]
  int hidden;
  int *err;
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

__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float t[32];
    tc::tmem_ld32(taddr + 32 * c, t);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[32 * c + i] = t[i];
  }
  tc::tmem_ld_wait();
}

// v = (2^-3.5 H v) . s (s: 128 fp16 values): the output-side transform.
__device__ __forceinline__ void rht_scale(float (&v)[128], const __half *s) {
  fwht128_regs(v);
#pragma unroll
  for (int c8 = 0; c8 < 16; ++c8) {
    const uint4 sv = __ldg(reinterpret_cast<const uint4 *>(s + 8 * c8));
    const __half2 *sh = reinterpret_cast<const __half2 *>(&sv);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * c8 + 2 * j] = v[8 * c8 + 2 * j] * kRhtScale * __low2float(sh[j]);
      v[8 * c8 + 2 * j + 1] = v[8 * c8 + 2 * j + 1] * kRhtScale * __high2float(sh[j]);
    }
  }
}

// v = 2^-3.5 H (v . s): the input-side transform (sign flip before H).
__device__ __forceinline__ void rht_in(float (&v)[128], const __half *s) {
#pragma unroll
  for (int c8 = 0; c8 < 16; ++c8) {
    const uint4 sv = __ldg(reinterpret_cast<const uint4 *>(s + 8 * c8));
    const __half2 *sh = reinterpret_cast<const __half2 *>(&sv);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * c8 + 2 * j] *= __low2float(sh[j]);
      v[8 * c8 + 2 * j + 1] *= __high2float(sh[j]);
    }
  }
  fwht128_regs(v);
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] *= kRhtScale;
}

template <int PHASE>
__global__ void __launch_bounds__(192, 1) moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA0,
                                                          const __grid_constant__ CUtensorMap tmA1,
                                                          const __grid_constant__ CUtensorMap tmB, Args a) {
  using C = Cfg<PHASE>;
  constexpr int STAGES = C::STAGES, STAGE_BYTES = C::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = *a.n_mtiles * a.NT;
  const int KB = a.KB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], 4);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmA0);
    if (PHASE == 1) tc::prefetch_tmap(&tmA1);
    tc::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
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
      for (int tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x) {
        const int4 mt = a.mtiles[tile / a.NT];
        const int ni = tile % a.NT;
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait(&empty[stage], phase ^ 1)) {
            set_device_error(a.err, kErrBounds);
            *abort_flag = 1;
            break;
          }
          uint8_t *st = smem + stage * STAGE_BYTES;
          tc::mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          tc::tma_load_2d(st, &tmA0, &full[stage], kb * BK, mt.y);
          if (PHASE == 1) tc::tma_load_2d(st + A_BYTES, &tmA1, &full[stage], kb * BK, mt.y);
          tc::tma_load_3d(st + C::NA * A_BYTES, &tmB, &full[stage], kb * BK, ni * BN, mt.x);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x) {
        if (!tc::mbar_wait(&tempty[acc], acc_phase ^ 1)) {
          set_device_error(a.err, kErrBounds);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * 256);
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait(&full[stage], phase)) {
            set_device_error(a.err, kErrBounds);
            *abort_flag = 1;
            break;
          }
          tc::tc_fence_after();
          uint8_t *st = smem + stage * STAGE_BYTES;
          const uint64_t bd = tc::sdesc_k_sw128(st + C::NA * A_BYTES);
          const uint64_t a0 = tc::sdesc_k_sw128(st);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t accum = (kb | kk) != 0;
            if (PHASE == 1) {
              const uint64_t a1 = tc::sdesc_k_sw128(st + A_BYTES);
              // gate: rows 0..127 of B; up: rows 128..255 (16 KB further)
              tc::mma_f16(d, a0 + 2 * kk, bd + 2 * kk, C::IDESC, accum);
              tc::mma_f16(d + 128, a1 + 2 * kk, bd + (16384 >> 4) + 2 * kk, C::IDESC, accum);
            } else {
              tc::mma_f16(d, a0 + 2 * kk, bd + 2 * kk, C::IDESC, accum);
            }
          }
          tc::mma_commit(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        tc::mma_commit(&tfull[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
    }
  } else {
    const int lane_base = 32 * (warp & 3);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int4 mt = a.mtiles[tile / a.NT];
      const int ni = tile % a.NT;
      bool ok = tc::mbar_wait(&tfull[acc], acc_phase);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok || *abort_flag) {
        if (lane == 0) set_device_error(a.err, kErrBounds);
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      const int r = lane_base + lane;              // row within the tile
      const bool valid = r < mt.z;
      const long row = (long)mt.y + r;             // sorted row
      const int e = mt.x;
      const uint32_t tbase = tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)(acc * 256);
      if (PHASE == 1) {
        const int col0 = ni * 128;
        float v[128];
        // gate half: transform, keep in TMEM
        tmem_ld128(tbase, v);
        rht_scale(v, a.svh13 + ((long)e * 2 + 0) * a.inter + col0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float t[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) t[i] = v[32 * c + i];
          tc::tmem_st32(tbase + 32 * c, t);
        }
        tc::tmem_st_wait();
        // up half, then h = SiLU(g) * u
        tmem_ld128(tbase + 128, v);
        rht_scale(v, a.svh13 + ((long)e * 2 + 1) * a.inter + col0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float g[32];
          tc::tmem_ld32(tbase + 32 * c, g);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * c + i] *= g[i] / (1.0f + expf(-g[i]));
        }
        // the down projection's input transform of this 128-block
        rht_in(v, a.suh2 + (long)e * a.inter + col0);
        if (valid) {
          __half *dst = a.hout + row * a.inter + col0;
#pragma unroll
          for (int c8 = 0; c8 < 16; ++c8) {
            __half2 h[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) h[j] = __floats2half2_rn(v[8 * c8 + 2 * j], v[8 * c8 + 2 * j + 1]);
            *reinterpret_cast<uint4 *>(dst + 8 * c8) = *reinterpret_cast<uint4 *>(h);
          }
        }
      } else {
        const float w = valid ? a.weights[a.perm[row]] : 0.f;
#pragma unroll 1
        for (int blk = 0; blk < 2; ++blk) {
          const int col0 = ni * BN + blk * 128;
          float v[128];
          tmem_ld128(tbase + blk * 128, v);
          rht_scale(v, a.svh2 + (long)e * a.hidden + col0);
          if (valid) {
            float *dst = a.dout + row * a.hidden + col0;
#pragma unroll
            for (int c4 = 0; c4 < 32; ++c4)
              *reinterpret_cast<float4 *>(dst + 4 * c4) =
                  make_float4(v[4 * c4] * w, v[4 * c4 + 1] * w, v[4 * c4 + 2] * w, v[4 * c4 + 3] * w);
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace mg
}  // namespace exl3

using namespace exl3;

static PFN_cuTensorMapEncodeTiled_v12000 moe_tmap_fn() {
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

// fp16 tensor [d2][d1][d0] (d0 contiguous), box [b2][b1][64], 128-byte swizzle.
static int moe_tmap(CUtensorMap *m, const void *base, int rank, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1) {
  auto fn = moe_tmap_fn();
  if (!fn) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {64, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return exl3_fail(EXL3_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return EXL3_OK;
}

static int moe_grid(int max_tiles) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  return max_tiles < sms ? (max_tiles > 0 ? max_tiles : 1) : sms;
}

// Phase 1: xg, xu [U][hidden] fp16 (sorted rows); w13 arena [E][2 inter][hidden].
int exl3_launch_moe_gateup(const uint16_t *xg, const uint16_t *xu, int U, int hidden, int inter, int E,
                           const uint16_t *w13_arena, const int *mtiles, const int *n_mtiles, int max_mtiles,
                           const uint16_t *svh13, const uint16_t *suh2, uint16_t *hout, int *err, cudaStream_t s) {
  CUtensorMap ta0, ta1, tb;
  int rc = moe_tmap(&ta0, xg, 2, hidden, U, 1, 128);
  if (rc) return rc;
  rc = moe_tmap(&ta1, xu, 2, hidden, U, 1, 128);
  if (rc) return rc;
  rc = moe_tmap(&tb, w13_arena, 3, hidden, 2 * inter, E, 256);
  if (rc) return rc;
  mg::Args a{};
  a.mtiles = reinterpret_cast<const int4 *>(mtiles);
  a.n_mtiles = n_mtiles;
  a.NT = inter / 128;
  a.KB = hidden / 64;
  a.svh13 = reinterpret_cast<const __half *>(svh13);
  a.suh2 = reinterpret_cast<const __half *>(suh2);
  a.hout = reinterpret_cast<__half *>(hout);
  a.inter = inter;
  a.err = err;
  auto kfn = mg::moe_gemm_kernel<1>;
  cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, mg::Cfg<1>::SMEM_BYTES);
  kfn<<<moe_grid(max_mtiles * a.NT), 192, mg::Cfg<1>::SMEM_BYTES, s>>>(ta0, ta1, tb, a);
  return exl3_cuda_check(cudaGetLastError(), "moe gate/up launch");
}

// Phase 2: h' [U][inter] fp16; w2 arena [E][hidden][inter]; d [U][hidden] fp32.
int exl3_launch_moe_down(const uint16_t *hin, int U, int hidden, int inter, int E, const uint16_t *w2_arena,
                         const int *mtiles, const int *n_mtiles, int max_mtiles, const uint16_t *svh2,
                         const float *weights, const int *perm, float *dout, int *err, cudaStream_t s) {
  CUtensorMap ta, tb;
  int rc = moe_tmap(&ta, hin, 2, inter, U, 1, 128);
  if (rc) return rc;
  rc = moe_tmap(&tb, w2_arena, 3, inter, hidden, E, 256);
  if (rc) return rc;
  mg::Args a{};
  a.mtiles = reinterpret_cast<const int4 *>(mtiles);
  a.n_mtiles = n_mtiles;
  a.NT = hidden / 256;
  a.KB = inter / 64;
  a.svh2 = reinterpret_cast<const __half *>(svh2);
  a.weights = weights;
  a.perm = perm;
  a.dout = dout;
  a.hidden = hidden;
  a.err = err;
  auto kfn = mg::moe_gemm_kernel<2>;
  cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, mg::Cfg<2>::SMEM_BYTES);
  kfn<<<moe_grid(max_mtiles * a.NT), 192, mg::Cfg<2>::SMEM_BYTES, s>>>(ta, ta, tb, a);
  return exl3_cuda_check(cudaGetLastError(), "moe down launch");
}
