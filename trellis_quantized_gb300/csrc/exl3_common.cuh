// exl3_common.cuh -- device helpers shared by the libexl3 kernels.
//
// Format facts used here (this library's reading of the pages; sources by
// page title and section):
//  * trellis tensor [k/16][n/16][16K] ("Bringing EXL3 Trellis Quantization to
//    35B MoE on Intel Arc 140V", section 2.A); tile bit i = bit (i % 16) of
//    word i / 16; weight p = 16 r + c of a tile takes the 16-bit window of
//    stream bits p*K .. p*K + 15, wrapping around the tile's 256 K bits.
//  * mul1 codebook bounded by 3.453125 ("exl3xpu" README, "Prefill: int8
//    linears and oneDNN fused attention"): B(s) = byte sum of
//    (s * 0x9E3779B1) mod 2^32 (one IMAD and one DP4A), value =
//    fp16_RNE((B - 510) * 1775 * 2^-18).
//  * block Hadamard in and out ("exl3xpu" README, "Layout"): Sylvester order,
//    scale 2^-3.5 per side, butterfly stages 1, 2, ..., 64 of (a+b, a-b).
#pragma once

#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/exl3.h"

namespace exl3 {

constexpr uint32_t kMul1 = 0x9E3779B1u;      // the mul1 multiplier
constexpr float kSigma = 0x1.bbcp-8f;        // 1775 * 2^-18, an fp16 value
constexpr float kRhtScale = 0x1.6a09e6p-4f;  // fp32 nearest 2^-3.5
constexpr float kMagic = 8388608.0f;         // 2^23: float bits 0x4B000000
constexpr float kBsumBias = 8389118.0f;      // 2^23 + 510

// Device error word bits (workspace offset 0).
constexpr int kErrDirtyCounter = 1;   // arrival counter found above its target
constexpr int kErrExpertId = 2;       // routed expert id outside [0, E)
constexpr int kErrBounds = 4;         // an index check failed

// ---------------------------------------------------------------- codebook --

// Byte sum B(s) of the mul1 hash of a 16-bit state (s must be < 2^16).
__device__ __forceinline__ uint32_t mul1_bsum(uint32_t s) {
  return __dp4a(s * kMul1, 0x01010101u, 0u);
}

// Exact fp16 codebook value: (B - 510) * 1775 is an integer below 2^24, so
// the fp32 product is exact and __float2half_rn rounds it once.
__device__ __forceinline__ __half mul1_half(uint32_t s) {
  return __float2half_rn((float)((int)mul1_bsum(s) - 510) * kSigma);
}

// (B - 510) as an exact fp32 value, via the DP4A accumulator seeded with the
// bit pattern of 2^23: the result's bits are those of the float 2^23 + B.
__device__ __forceinline__ float mul1_centered(uint32_t s) {
  return __int_as_float((int)__dp4a(s * kMul1, 0x01010101u, 0x4B000000u)) - kBsumBias;
}

// 16-bit window starting at bit `sh` (0..31) of the 64-bit pair (hi:lo).
__device__ __forceinline__ uint32_t window16(uint32_t lo, uint32_t hi, uint32_t sh) {
  return __funnelshift_r(lo, hi, sh) & 0xFFFFu;
}

// ------------------------------------------------------------------ FWHT-128 --

// 128-point Sylvester Hadamard over one warp, lane l holding elements
// 4l .. 4l+3.  Same per-element operation order as the definition: stage h,
// pair (i, i+h) -> (a+b, a-b) with a the lower index.  Stages 1 and 2 are in
// registers, stages 4..64 exchange with lane l ^ (h / 4).
__device__ __forceinline__ void fwht128_warp(float v[4], int lane) {
  float a, b;
  // h = 1: pairs (0,1), (2,3)
  a = v[0]; b = v[1]; v[0] = a + b; v[1] = a - b;
  a = v[2]; b = v[3]; v[2] = a + b; v[3] = a - b;
  // h = 2: pairs (0,2), (1,3)
  a = v[0]; b = v[2]; v[0] = a + b; v[2] = a - b;
  a = v[1]; b = v[3]; v[1] = a + b; v[3] = a - b;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    // lower lane: v + other; upper lane: other - v; both one rounding of
    // fma(+-1, v, other), with no select between two results
    const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float other = __shfl_xor_sync(0xffffffffu, v[j], m);
      v[j] = fmaf(sgn, v[j], other);
    }
  }
}

// The same transform with 16 contiguous values per lane: lanes 8j .. 8j + 7
// of the warp hold one 128-block (lane l: elements 16 (l mod 8) + i), so a
// warp transforms four blocks at once.  Stages h = 1, 2, 4, 8 stay in
// registers, h = 16, 32, 64 exchange with lane l ^ 1, ^ 2, ^ 4 (three shuffle
// stages instead of five).  The stage order and every rounding are those of
// fwht128_warp: fma(+-1, v, partner) is the single-rounded sum or difference.
__device__ __forceinline__ void fwht128_x8(float (&v)[16], int lane) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1)
#pragma unroll
    for (int i = 0; i < 16; i += 2 * h)
#pragma unroll
      for (int j = i; j < i + h; ++j) {
        const float a = v[j], b = v[j + h];
        v[j] = a + b;
        v[j + h] = a - b;
      }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {
    const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float other = __shfl_xor_sync(0xffffffffu, v[j], m);
      v[j] = fmaf(sgn, v[j], other);
    }
  }
}

// FWHT-128 that exchanges half of the values per cross-lane stage (8
// shuffles instead of 16), on packed pairs of fp32 lanes.  Eight lanes hold a
// block as in fwht128_x8 (p[i] = elements 2i, 2i + 1 of the lane's 16),
// except that a lane with l & 1 set holds its two 8-element halves swapped
// (p[0..3] = elements 16 (l mod 8) + 8 ..15, loaded that way).  In each stage
// h = 16, 32, 64 a lane keeps p[0..3], sends p[4..7] to its partner, and
// computes the sum and the difference of eight of the sixteen pairs; the next
// stage's lane bit decides which of p[0..3] / p[4..7] takes which, so no value
// is ever selected.  A lane whose kept operand is the upper one of its pairs
// computes b - a in place of a - b, so values carry a sign per lane;
// fwht128_xh_signs gives the factors that restore them.  Stages h >= 2 run two
// butterflies per packed instruction (add.rn.f32x2, or fma.rn.f32x2 with a
// factor of +-1: one rounding of the sum or difference).  Every result is the
// single rounding of fwht128_x8's (negation is exact), so the transform equals
// fwht128_x8's except possibly for the sign of a zero.  On return lane l holds
// block elements 8 (l mod 8) + 2i, +1 in p[i] and 64 + 8 (l mod 8) + 2i, +1
// in p[4 + i] (i < 4), before the sign factors.
__device__ __forceinline__ void fwht128_xh(float2 (&p)[8], int lane) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {                  // h = 1, inside each pair
    const float a = p[i].x, b = p[i].y;
    p[i] = make_float2(a + b, a - b);
  }
  const float2 neg = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int h = 1; h < 4; h <<= 1)                // h = 2, 4 (1, 2 pairs apart)
#pragma unroll
    for (int i = 0; i < 8; i += 2 * h)
#pragma unroll
      for (int j = i; j < i + h; ++j) {
        const float2 a = p[j], b = p[j + h];
        p[j] = __fadd2_rn(a, b);
        p[j + h] = __ffma2_rn(neg, b, a);
      }
  {                                              // h = 8 on the swapped halves
    const float s0 = (lane & 1) ? -1.0f : 1.0f;
    const float2 sp = make_float2(s0, s0), sn = make_float2(-s0, -s0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 lo = p[i], hi = p[i + 4];
      p[i] = __ffma2_rn(sp, lo, hi);
      p[i + 4] = __ffma2_rn(sn, hi, lo);
    }
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {              // h = 16, 32, 64 with lane l ^ m
    // where the results go: by the next stage's lane bit (the last stage puts
    // the sum first)
    const float c = (m < 4 && (lane & (2 * m))) ? -1.0f : 1.0f;
    const float2 cp = make_float2(c, c), cn = make_float2(-c, -c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 r = make_float2(__shfl_xor_sync(0xffffffffu, p[i + 4].x, m),
                                   __shfl_xor_sync(0xffffffffu, p[i + 4].y, m));
      const float2 k = p[i];
      p[i] = __ffma2_rn(cp, r, k);
      p[i + 4] = __ffma2_rn(cn, r, k);
    }
  }
}

// Sign factors of fwht128_xh's p[0..3] (lo) and p[4..7] (hi) on this lane.
__device__ __forceinline__ void fwht128_xh_signs(int lane, float &lo, float &hi) {
  const float s0 = (lane & 1) ? -1.0f : 1.0f, s1 = (lane & 2) ? -1.0f : 1.0f, s2 = (lane & 4) ? -1.0f : 1.0f;
  lo = ((lane & 2) ? s0 : 1.0f) * ((lane & 4) ? s1 : 1.0f);
  hi = lo * s2;
}

// The exact fp32 products of two pairs of binary16 values (a 22-bit product
// always fits): one mixed-precision FMA per value, with a -0 addend so that a
// zero product keeps its sign.
__device__ __forceinline__ float2 mul_f16x2_exact(uint32_t x, uint32_t s) {
  float lo, hi;
  asm("{\n.reg .f16 xl, xh, sl, sh;\n.reg .b16 b0, b1, b2, b3;\n"
      "mov.b32 {b0, b1}, %2;\nmov.b32 {b2, b3}, %3;\n"
      "mov.b16 xl, b0;\nmov.b16 xh, b1;\nmov.b16 sl, b2;\nmov.b16 sh, b3;\n"
      "fma.rn.f32.f16 %0, xl, sl, 0f80000000;\nfma.rn.f32.f16 %1, xh, sh, 0f80000000;\n}\n"
      : "=f"(lo), "=f"(hi)
      : "r"(x), "r"(s));
  return make_float2(lo, hi);
}

// ------------------------------------------------------------ small helpers --

__device__ __forceinline__ void set_device_error(int *err, int bit) {
  if (err) atomicOr(err, bit);
}

// Programmatic dependent launch.  pdl_trigger lets the kernel launched after
// this one on the stream start its CTAs; pdl_wait blocks until the kernel
// launched before it has completed and its writes are visible (both return at
// once when the launch had no programmatic dependency).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch kfn as a programmatic dependent of the preceding kernel on s.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kfn)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       const Args &...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kfn, args...);
}

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

__host__ __device__ constexpr int gcd_c(int a, int b) { return b == 0 ? a : gcd_c(b, a % b); }

}  // namespace exl3

// ------------------------------------------------------------ host helpers --
// Defined in api.cu: thread-local error message and CUDA error capture.
int exl3_fail(int code, const char *fmt, ...);
int exl3_cuda_check(cudaError_t e, const char *what);

// Device-dependent host state (SM counts, kernel attributes) is cached per
// device ordinal, for ordinals below kMaxDevices (larger ones query each
// time); the caches are safe to use from several host threads.
constexpr int kMaxDevices = 64;
// SM count of the current device (152 if the query fails).
int exl3_sm_count();
// Raise kfn's dynamic shared-memory limit on the current device to at least
// `bytes` (cudaFuncSetAttribute applies per device); `per_dev` caches what
// each device was given, one array per kernel.
cudaError_t exl3_ensure_smem(const void *kfn, size_t bytes, std::atomic<size_t> *per_dev);
// The driver's cuTensorMapEncodeTiled (NULL if unavailable), looked up once.
PFN_cuTensorMapEncodeTiled_v12000 exl3_tmap_encode_fn();
