// gemv_core.cuh -- the CUDA-core M = 1 decode shared by the linear GEMV and
// the few-token routed-expert GEMV: lane items, the per-weight decode and
// accumulate, and the balanced contiguous split of rows over CTAs.  See
// gemv.cu for the kernel design ("dp4a GEMV" of "exl3xpu" README, "Layout").
#pragma once

#include "exl3_common.cuh"
#include "trellis_window.cuh"

namespace exl3 {

constexpr int kGemvBoxRows = 8;                 // tile rows per tensor copy
constexpr int kGemvSmemMax = 232448;            // opt-in shared memory per CTA (227 KB; no static smem)
constexpr int kGemvMaxStages = 8;

template <int K>
struct GemvShape {
  // rows per lane item: a whole number of 16-byte chunks, and at least four
  // rows so that per-item costs (loads, x', loop) are shared by 64+ weights
  static constexpr int G0 = 8 / gcd_c(K, 8);
  static constexpr int G = G0 < 4 ? 4 : G0;
  static constexpr int CPL = K * G / 8;          // 16-byte chunks per lane
  static constexpr int LPT = 16 / G;             // lanes per tile
  static constexpr int TPW = 32 / LPT;           // tiles per warp
  static constexpr int CTA_COLS = TPW * 16;      // 128 or 256 columns per block
  static constexpr int NW = 4 * CPL;             // 32-bit stream words per lane
  static constexpr int ROWB = CTA_COLS * 2 * K;  // bytes of one row (CTA_COLS/16 tiles of 32K bytes)
  // consumer warps (16 measured faster than 8, 12, 20 or 24: more
  // registers per thread and a shorter spread of warp finishing times), and
  // rows per consumer warp per stage (stages of 16-56 KB)
  static constexpr int NCW = 16;
  static constexpr int RPW = ROWB >= 1536 ? 1 : 2;
  static constexpr int R = RPW * NCW;            // rows per stage
  static constexpr int STAGE_B = R * ROWB;
  static constexpr int NG = CTA_COLS / 128;      // 128-column groups per block
  static constexpr int THREADS = (NCW + 2) * 32; // + the producer and the flusher warp
  static constexpr int FIXED_B = 4 * NCW * CTA_COLS + 256;   // red, flags, barriers
  static_assert(R % kGemvBoxRows == 0, "stages hold whole tensor copies");
  static_assert(ROWB % 128 == 0, "tensor copies land on 128-byte boundaries");
};


// acc += x * h, x and h binary16 (h = low half of r), acc binary32.
__device__ __forceinline__ float fma_f16_f32(unsigned short x, uint32_t r, float acc) {
  asm("{\n.reg .f16 hx, hh;\n.reg .b16 lo, hi;\nmov.b32 {lo, hi}, %1;\nmov.b16 hh, lo;\nmov.b16 hx, %2;\n"
      "fma.rn.f32.f16 %0, hx, hh, %0;\n}\n"
      : "+f"(acc)
      : "r"(r), "h"(x));
  return acc;
}

__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Decode the lane's 16 G weights and accumulate x'_row * (1024 + B) into the
// 16 column accumulators.
template <int K, int J>
__device__ __forceinline__ void decode_accumulate(const uint32_t (&w)[GemvShape<K>::NW + 1],
                                                  const unsigned short (&xr)[GemvShape<K>::G],
                                                  float (&acc)[16]) {
  if constexpr (J < 16 * GemvShape<K>::G) {
    const uint32_t s = window_at<J * K>(w);
    const uint32_t h = __dp4a(s * kMul1, 0x01010101u, 0x6400u);   // fp16 bits of 1024 + B
    acc[J & 15] = fma_f16_f32(xr[J >> 4], h, acc[J & 15]);
    decode_accumulate<K, J + 1>(w, xr, acc);
  }
}

// Start of CTA i's rows (grid * total < 2^32).
__device__ __forceinline__ uint32_t range_start(int i, uint32_t total, int grid) {
  return (uint32_t)i * total / (uint32_t)grid;
}

// Index of the CTA whose range holds row r.
__device__ __forceinline__ int range_owner(uint32_t r, uint32_t total, int grid) {
  int i = (int)((r * (uint32_t)grid) / total);
  while (i + 1 < grid && range_start(i + 1, total, grid) <= r) ++i;
  while (i > 0 && range_start(i, total, grid) > r) --i;
  return i;
}

}  // namespace exl3
