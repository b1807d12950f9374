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


__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// x' is held scaled by 2^100 (kXScale) and the byte sum B of a weight, an
// integer below 2^10, is read as the bit pattern of the fp32 value B * 2^-149
// (a subnormal, exact): their product is x' B 2^-49, exact in fp32, so one
// fp32 FMA accumulates a weight with fp32 rounding of the sums only.  The
// column sums carry 510 * sum x', removed once per column block from
// per-tile-row sums of x'.
constexpr float kXScale = 0x1p100f;      // x' scale in shared memory
constexpr float kAccUnscale = 0x1p49f;   // accumulator scale back to x' B

// Decode the lane's 16 G weights and accumulate x'_row * B into the 16
// column accumulators.
template <int K, int J>
__device__ __forceinline__ void decode_accumulate(const uint32_t (&w)[GemvShape<K>::NW + 1],
                                                  const float (&xr)[GemvShape<K>::G], float (&acc)[16]) {
  if constexpr (J < 16 * GemvShape<K>::G) {
    const uint32_t b = __dp4a(window_at<J * K>(w) * kMul1, 0x01010101u, 0u);
    acc[J & 15] = fmaf(xr[J >> 4], __uint_as_float(b), acc[J & 15]);
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
