// gemv.cu -- fused M = 1 EXL3 linear on CUDA cores (the decode GEMV; "dp4a
// GEMV" of "exl3xpu" README, "Layout"; the GEMM runs in the Hadamard domain,
// "exl3xpu" README, "Prefill: int8 linears and oneDNN fused attention").
//
//   y = RHT_out( sigma * sum_k x'_k (B_kn - 510) ) . svh,  x' = RHT_in(x . suh)
//
// The contraction uses the exact codebook value (B - 510) * sigma, of which
// the fp16 weight is the rounding, and x' rounded to fp16 (as the tensor-core
// paths do); both differences (< 2^-11 relative per term) stay inside the
// output tolerance.  DP4A seeded with 0x6400 yields the fp16 value 1024 + B
// in the low half of its result, which a mixed-precision FMA multiplies by
// the fp16 x' into an fp32 accumulator: sum x' (1024 + B).  The offset is
// removed once per lane, 1534 * sum x' (1024 + 510 = 1534), at the end.
//
// Lane work.  A lane owns G = 8 / gcd(K, 8) consecutive rows of one tile:
// 16 G weights whose states come from CPL = K / gcd(K, 8) contiguous 16-byte
// chunks (128 CPL bits) plus the first 32 bits of the next row group (one
// warp shuffle; the last group of a tile wraps to the first).  LPT = 16 / G
// lanes cover a tile and a warp covers 2 G consecutive tiles along n.  Each
// window is cut out of byte-aligned (possibly pre-shifted) words with one
// LOP/SHR/PRMT where it can, hashed (IMAD), byte-summed by DP4A and
// accumulated by one mixed-precision FMA.
//
// Staging.  One producer warp streams the CTA's rows (the tiles of one
// column block at one tile row, 0.5-3.5 KB of contiguous trellis each) into
// a ring of shared-memory stages with bulk asynchronous copies completing on
// mbarriers; eight consumer warps decode out of shared memory.  Every wait is
// bounded; a wait that runs out sets the device error word.
//
// Work split.  The work is the list of "rows" (column block c, tile row tk),
// c-major; a column block is 128 (or 256) output columns.  A persistent grid
// sized to the resident CTA slots takes equal contiguous ranges of that list,
// so every SM gets the same amount of trellis.  A CTA's range crosses column
// blocks; at each crossing it reduces its accumulators and either finishes
// the block itself (it owned all of it) or stores a partial sum in a slot
// fixed by (block, CTA).  The last CTA to arrive at a block (atomic counter,
// no waiting) adds the partials in CTA order, applies the output transform
// and writes y: the result does not depend on timing.
#include "exl3_common.cuh"
#include "trellis_window.cuh"

namespace exl3 {

template <int K>
struct GemvShape {
  // rows per lane item: a whole number of 16-byte chunks, and at least four
  // rows so that per-item costs (loads, x', loop) are shared by 64+ weights
  static constexpr int G0 = 8 / gcd_c(K, 8);
  static constexpr int G = G0 < 4 ? 4 : G0;
  static constexpr int CPL = K * G / 8;          // 16-byte chunks per lane
  static constexpr int LPT = 16 / G;             // lanes per tile
  static constexpr int TPW = 32 / LPT;           // tiles per warp
  static constexpr int COLW = TPW * 16;          // columns per warp
  static constexpr int WC = COLW >= 128 ? 1 : 128 / COLW;  // column warps per CTA
  static constexpr int WK = 8 / WC;              // k warps per CTA
  static constexpr int CTA_COLS = WC * COLW;     // 128 or 256
  static constexpr int NW = 4 * CPL;             // 32-bit stream words per lane
  static constexpr int ROWB = CTA_COLS * 2 * K;  // bytes of one row (CTA_COLS/16 tiles of 32K bytes)
  // rows per stage: each k-warp takes RPW rows per wait, aiming at 16 KB
  // stages (at least the one or two rows of a wide or narrow row, at most 4)
  static constexpr int RPW_MIN = ROWB >= 2048 ? 1 : 2;
  static constexpr int RPW_FIT = 16384 / (WK * ROWB);
  static constexpr int RPW = RPW_FIT > 4 ? 4 : (RPW_FIT < RPW_MIN ? RPW_MIN : RPW_FIT);
  static constexpr int R = RPW * WK;
  static constexpr int STAGE_B = R * ROWB;
  static constexpr int STAGES = (48 * 1024) / STAGE_B < 2 ? 2 : (48 * 1024) / STAGE_B;
  static constexpr int RING_B = STAGES * STAGE_B;
};

struct GemvArgs {
  const __half *x;          // [k]
  const uint16_t *trellis;  // [k/16][n/16][16K]
  const __half *suh;        // [k]
  const __half *svh;        // [n]
  void *y;                  // [n] fp16 or fp32
  float *partials;          // [colblocks + grid][CTA_COLS]
  int *counters;            // [colblocks]
  int *err;                 // device error word
  int k, n, tiles_k, colblocks;
  long long total;          // colblocks * tiles_k
};

// acc += x * h, x and h binary16 (h = low half of r), acc binary32.
__device__ __forceinline__ float fma_f16_f32(unsigned short x, uint32_t r, float acc) {
  asm("{\n.reg .f16 hx, hh;\n.reg .b16 lo, hi;\nmov.b32 {lo, hi}, %1;\nmov.b16 hh, lo;\nmov.b16 hx, %2;\n"
      "fma.rn.f32.f16 %0, hx, hh, %0;\n}\n"
      : "+f"(acc)
      : "r"(r), "h"(x));
  return acc;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(n));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}
// Bounded wait for the phase of the given parity; false if it ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *b, uint32_t parity) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    // the suspend-time hint (ns) lets the thread sleep until the phase
    // completes instead of spinning through issue slots
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 10000;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok)
                 : "r"(smem_addr(b)), "r"(parity)
                 : "memory");
    if (ok) return true;
    if (clock64() - t0 > 2000000000LL) return false;
  }
}
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

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

__device__ __forceinline__ long long range_start(int i, long long total, int grid) {
  return (long long)i * total / grid;
}

// Index of the CTA whose range holds row r.
__device__ __forceinline__ int range_owner(long long r, long long total, int grid) {
  int i = (int)((r * grid) / total);
  while (i + 1 < grid && range_start(i + 1, total, grid) <= r) ++i;
  while (i > 0 && range_start(i, total, grid) > r) --i;
  return i;
}

template <int K, bool F32OUT>
__global__ void __launch_bounds__(288) gemv_m1_kernel(GemvArgs a) {
  using S = GemvShape<K>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t *ring = smem_raw;                                         // [STAGES][R][ROWB]
  float *red = reinterpret_cast<float *>(smem_raw + S::RING_B);    // [WK][CTA_COLS]
  float *ys = red + S::WK * S::CTA_COLS;                           // [CTA_COLS]
  uint64_t *full = reinterpret_cast<uint64_t *>(ys + S::CTA_COLS); // [STAGES]
  uint64_t *empty = full + S::STAGES;                              // [STAGES]
  __half *xs = reinterpret_cast<__half *>(empty + S::STAGES);      // [k] fp16 x' (touched blocks)
  __shared__ int s_last;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grid = gridDim.x, me = blockIdx.x;
  const int TK = a.tiles_k, tiles_n = a.n >> 4;
  const long long t0 = range_start(me, a.total, grid), t1 = range_start(me + 1, a.total, grid);
  if (t0 >= t1) return;

  if (tid == 0) {
    for (int st = 0; st < S::STAGES; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 8);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == 8) {
    // ---------------- producer: one thread streams the rows into the ring
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (long long t = t0; t < t1 && !s_abort;) {
        const int c = (int)(t / TK);
        const long long seg_end = min(t1, (long long)(c + 1) * TK);
        const int tk_first = (int)(t - (long long)c * TK), nrows = (int)(seg_end - t);
        const int tn0 = c * (S::CTA_COLS / 16);
        const int tiles_valid = min(S::CTA_COLS / 16, tiles_n - tn0);
        const uint32_t bytes = (uint32_t)tiles_valid * 32u * K;
        for (int r0 = 0; r0 < nrows && !s_abort; r0 += S::R) {
          const int cnt = min(S::R, nrows - r0);
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1)) {
            set_device_error(a.err, kErrBounds);
            s_abort = 1;
            break;
          }
          mbar_expect_tx(&full[stage], bytes * cnt);
          for (int j = 0; j < cnt; ++j) {
            const long tk = tk_first + r0 + j;
            const uint16_t *src = a.trellis + ((long)tk * tiles_n + tn0) * 16 * K;
            bulk_copy(ring + (size_t)stage * S::STAGE_B + (size_t)j * S::ROWB, src, bytes, &full[stage]);
          }
          if (++stage == S::STAGES) { stage = 0; phase ^= 1; }
        }
        t = seg_end;
      }
    }
    return;
  }

  // ---------------- consumers (warps 0..7)
  // prologue: x' = 2^-3.5 H (x . suh) for the 128-blocks this range touches
  {
    const int KB = a.k >> 7;
    int b0 = 0, nb = KB;
    if (t1 - t0 < TK) {   // fewer rows than one block: at most two column blocks
      b0 = (int)(t0 % TK) >> 3;
      const int b1 = (int)((t1 - 1) % TK) >> 3;
      const bool wrap = (t0 / TK) != ((t1 - 1) / TK);
      nb = !wrap ? b1 - b0 + 1 : (b1 >= b0 ? KB : KB - b0 + b1 + 1);
    }
    for (int i = warp; i < nb; i += 8) {
      const int b = (b0 + i) % KB;
      const int col = b * 128 + lane * 4;
      const uint2 xv = *reinterpret_cast<const uint2 *>(a.x + col);
      const uint2 sv = *reinterpret_cast<const uint2 *>(a.suh + col);
      const __half2 *xh = reinterpret_cast<const __half2 *>(&xv);
      const __half2 *sh = reinterpret_cast<const __half2 *>(&sv);
      float v[4] = {__low2float(xh[0]) * __low2float(sh[0]), __high2float(xh[0]) * __high2float(sh[0]),
                    __low2float(xh[1]) * __low2float(sh[1]), __high2float(xh[1]) * __high2float(sh[1])};
      fwht128_warp(v, lane);
      __half2 o[2] = {__floats2half2_rn(v[0] * kRhtScale, v[1] * kRhtScale),
                      __floats2half2_rn(v[2] * kRhtScale, v[3] * kRhtScale)};
      *reinterpret_cast<uint2 *>(xs + col) = *reinterpret_cast<uint2 *>(o);
    }
  }
  consumer_sync();

  const int wc = warp % S::WC, wk = warp / S::WC;
  const int tile_in_warp = lane / S::LPT, q = lane % S::LPT;
  const int tile_local = wc * S::TPW + tile_in_warp;                 // tile within the row
  const int my_off = tile_local * 32 * K + q * 16 * S::CPL;          // byte offset in a row
  const int next_off = tile_local * 32 * K + ((q + 1) % S::LPT) * 16 * S::CPL;  // next row group (wraps)
  int stage = 0;
  uint32_t phase = 0;

  for (long long t = t0; t < t1;) {
    const int c = (int)(t / TK);
    const long long seg_end = min(t1, (long long)(c + 1) * TK);
    const int tk_first = (int)(t - (long long)c * TK), nrows = (int)(seg_end - t);
    const bool valid = c * (S::CTA_COLS / 16) + tile_local < tiles_n;

    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    float sx = 0.f;   // sum of the x' this lane used (for the 1024 + 510 offset)

    for (int r0 = 0; r0 < nrows; r0 += S::R) {
      const int cnt = min(S::R, nrows - r0);
      if (!s_abort && !mbar_wait_bounded(&full[stage], phase)) {
        if (lane == 0) set_device_error(a.err, kErrBounds);
        s_abort = 1;
      }
      const uint8_t *sbase = ring + (size_t)stage * S::STAGE_B;
#pragma unroll
      for (int jj = 0; jj < S::R / S::WK; ++jj) {
        const int j = wk + jj * S::WK;
        if (j < cnt) {
          uint32_t w[S::NW + 1];
          const uint8_t *rowp = sbase + (size_t)j * S::ROWB;
          if (valid) {
#pragma unroll
            for (int cc = 0; cc < S::CPL; ++cc) {
              const uint4 v4 = *reinterpret_cast<const uint4 *>(rowp + my_off + 16 * cc);
              w[4 * cc + 0] = v4.x;
              w[4 * cc + 1] = v4.y;
              w[4 * cc + 2] = v4.z;
              w[4 * cc + 3] = v4.w;
            }
            w[S::NW] = *reinterpret_cast<const uint32_t *>(rowp + next_off);
          } else {
#pragma unroll
            for (int i = 0; i <= S::NW; ++i) w[i] = 0u;
          }
          const int tk = tk_first + r0 + j;
          unsigned short xr[S::G];
#pragma unroll
          for (int i = 0; i < S::G; ++i) {
            const __half xv = xs[tk * 16 + S::G * q + i];
            xr[i] = __half_as_ushort(xv);
            sx += __half2float(xv);
          }
          decode_accumulate<K, 0>(w, xr, acc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive1(&empty[stage]);
      if (++stage == S::STAGES) { stage = 0; phase ^= 1; }
    }

    // ---- reduce: LPT lanes of a tile, then the k-warps of the CTA
    float accf[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) accf[i] = fmaf(-1534.0f, sx, acc[i]);
#pragma unroll
    for (int m = 1; m < S::LPT; m <<= 1)
#pragma unroll
      for (int i = 0; i < 16; ++i) accf[i] += __shfl_xor_sync(0xffffffffu, accf[i], m);
    if (q == 0) {
#pragma unroll
      for (int i = 0; i < 16; ++i) red[wk * S::CTA_COLS + wc * S::COLW + tile_in_warp * 16 + i] = accf[i];
    }
    consumer_sync();
    const int col0 = c * S::CTA_COLS;
    float part = 0.f;
    if (tid < S::CTA_COLS) {
#pragma unroll
      for (int w = 0; w < S::WK; ++w) part += red[w * S::CTA_COLS + tid];
      part *= kSigma;
    }
    const long long blk_first = (long long)c * TK, blk_last = min((long long)(c + 1) * TK, a.total) - 1;
    const int i_first = range_owner(blk_first, a.total, grid), i_last = range_owner(blk_last, a.total, grid);
    bool finish;
    if (i_first == i_last) {
      if (tid < S::CTA_COLS) ys[tid] = part;
      finish = true;
    } else {
      if (tid < S::CTA_COLS) {
        a.partials[(long)(c + me) * S::CTA_COLS + tid] = part;
        __threadfence();
      }
      consumer_sync();
      if (tid == 0) {
        const int expected = i_last - i_first + 1;
        const int old = atomicAdd(a.counters + c, 1);
        if (old >= expected) set_device_error(a.err, kErrDirtyCounter);
        s_last = (old == expected - 1);
      }
      consumer_sync();
      finish = s_last != 0;
      if (finish) {
        __threadfence();
        if (tid < S::CTA_COLS) {
          float sum = 0.f;
          for (int i = i_first; i <= i_last; ++i) sum += __ldcg(a.partials + (long)(c + i) * S::CTA_COLS + tid);
          ys[tid] = sum;
        }
        if (tid == 0) a.counters[c] = 0;   // leave the workspace clean
      }
    }
    consumer_sync();

    // ---- output transform of the block's 128-column groups
    if (finish && warp < S::CTA_COLS / 128 && col0 + warp * 128 < a.n) {
      const int cc = warp * 128 + lane * 4;
      float v[4] = {ys[cc], ys[cc + 1], ys[cc + 2], ys[cc + 3]};
      fwht128_warp(v, lane);
      const int gc = col0 + cc;
      const uint2 sv = *reinterpret_cast<const uint2 *>(a.svh + gc);
      const __half2 *sh = reinterpret_cast<const __half2 *>(&sv);
      v[0] = v[0] * kRhtScale * __low2float(sh[0]);
      v[1] = v[1] * kRhtScale * __high2float(sh[0]);
      v[2] = v[2] * kRhtScale * __low2float(sh[1]);
      v[3] = v[3] * kRhtScale * __high2float(sh[1]);
      if (F32OUT) {
        *reinterpret_cast<float4 *>(static_cast<float *>(a.y) + gc) = make_float4(v[0], v[1], v[2], v[3]);
      } else {
        __half2 o[2] = {__floats2half2_rn(v[0], v[1]), __floats2half2_rn(v[2], v[3])};
        *reinterpret_cast<uint2 *>(static_cast<__half *>(a.y) + gc) = *reinterpret_cast<uint2 *>(o);
      }
    }
    consumer_sync();   // red / ys are reused by the next segment
    t = seg_end;
  }
}

template <int K, bool F32>
struct Launcher {
  static size_t smem(int k) {
    using S = GemvShape<K>;
    return (size_t)S::RING_B + sizeof(float) * ((size_t)S::WK * S::CTA_COLS + S::CTA_COLS) +
           sizeof(uint64_t) * 2 * S::STAGES + sizeof(__half) * (size_t)k;
  }
  static int grid(int k) {
    static int cached_k = -1, cached = 0;
    if (cached_k == k) return cached;
    int dev = 0, sms = 0, occ = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t sm = smem(k);
    cudaFuncSetAttribute(gemv_m1_kernel<K, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_m1_kernel<K, F32>, 288, sm);
    cudaGetLastError();
    if (sms <= 0) sms = 152;
    if (occ <= 0) occ = 1;
    // three resident CTAs per SM: more rows per CTA between column-block
    // flushes, still enough warps to hide the decode latencies (measured
    // faster than four at k = 5120, n = 5120 ... 25600)
    if (occ > 3) occ = 3;
    cached_k = k;
    cached = sms * occ;
    return cached;
  }
  static cudaError_t launch(const GemvArgs &a, int grid, cudaStream_t s) {
    static int attr_k = -1;
    const size_t sm = smem(a.k);
    if (attr_k != a.k) {
      cudaFuncSetAttribute(gemv_m1_kernel<K, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      attr_k = a.k;
    }
    gemv_m1_kernel<K, F32><<<grid, 288, sm, s>>>(a);
    return cudaGetLastError();
  }
};

}  // namespace exl3

using namespace exl3;

#define EXL3_K_SWITCH(K, ...)                         \
  switch (K) {                                        \
    case 1: { constexpr int KK = 1; __VA_ARGS__; } break; \
    case 2: { constexpr int KK = 2; __VA_ARGS__; } break; \
    case 3: { constexpr int KK = 3; __VA_ARGS__; } break; \
    case 4: { constexpr int KK = 4; __VA_ARGS__; } break; \
    case 5: { constexpr int KK = 5; __VA_ARGS__; } break; \
    case 6: { constexpr int KK = 6; __VA_ARGS__; } break; \
    case 7: { constexpr int KK = 7; __VA_ARGS__; } break; \
    default: { constexpr int KK = 8; __VA_ARGS__; } break; \
  }

// Columns covered by one column block for width K (128 or 256).
int exl3_gemv_cta_cols(int K) {
  int r = 128;
  EXL3_K_SWITCH(K, r = GemvShape<KK>::CTA_COLS);
  return r;
}

// Persistent grid size and the partial-sum slots (floats) the GEMV needs.
void exl3_gemv_plan(int k, int n, int K, int *grid, size_t *partial_floats) {
  int g = 0, cc = 128;
  EXL3_K_SWITCH(K, (g = Launcher<KK, false>::grid(k), cc = GemvShape<KK>::CTA_COLS));
  const long long colblocks = (n + cc - 1) / cc;
  const long long total = colblocks * (k / 16);
  if (g > total) g = (int)total;
  *grid = g;
  *partial_floats = (size_t)(colblocks + g) * (size_t)cc;
}

cudaError_t exl3_launch_gemv_m1(const uint16_t *x, const uint16_t *trellis, const uint16_t *suh,
                                const uint16_t *svh, int k, int n, int K, void *y, bool f32out,
                                float *partials, int *counters, int *err, int grid, cudaStream_t s) {
  GemvArgs a;
  a.x = reinterpret_cast<const __half *>(x);
  a.trellis = trellis;
  a.suh = reinterpret_cast<const __half *>(suh);
  a.svh = reinterpret_cast<const __half *>(svh);
  a.y = y;
  a.partials = partials;
  a.counters = counters;
  a.err = err;
  a.k = k;
  a.n = n;
  a.tiles_k = k / 16;
  const int cc = exl3_gemv_cta_cols(K);
  a.colblocks = (n + cc - 1) / cc;
  a.total = (long long)a.colblocks * a.tiles_k;
  cudaError_t e = cudaSuccess;
  if (f32out) {
    EXL3_K_SWITCH(K, e = Launcher<KK, true>::launch(a, grid, s));
  } else {
    EXL3_K_SWITCH(K, e = Launcher<KK, false>::launch(a, grid, s));
  }
  return e;
}
