// gemv.cu -- fused M = 1 EXL3 linear on CUDA cores (the decode GEMV; "dp4a
// GEMV" of "exl3xpu" README, "Layout"; the GEMM runs in the Hadamard domain,
// "exl3xpu" README, "Prefill: int8 linears and oneDNN fused attention").
//
//   y = RHT_out( sigma * sum_k x'_k (B_kn - 510) ) . svh,  x' = RHT_in(x . suh)
//
// The contraction uses the exact codebook value (B - 510) * sigma, of which
// the fp16 weight is the rounding; the difference (< 2^-11 relative per
// weight) stays inside the output tolerance.
//
// Work split.  A lane owns G = 8 / gcd(K, 8) consecutive rows of one tile:
// 16 G weights whose states come from CPL = K / gcd(K, 8) contiguous 16-byte
// chunks (128 CPL bits) plus the first 32 bits of the next row group (one
// warp shuffle; the last group of a tile wraps to the first).  LPT = 16 / G
// lanes cover a tile, a warp covers 2 G consecutive tiles along n, and the
// lane keeps 16 column accumulators while the warp walks down k.  A CTA of 8
// warps spans 128 (or 256) output columns and one k-range; CTAs on the same
// columns split k.  The last CTA to arrive for a column block (atomic
// counter, no waiting) sums the k-split partials in a fixed order, applies
// the output transform and writes y, so results are deterministic.
#include "exl3_common.cuh"

namespace exl3 {

template <int K>
struct GemvShape {
  static constexpr int G = 8 / gcd_c(K, 8);      // rows per lane
  static constexpr int CPL = K / gcd_c(K, 8);    // 16-byte chunks per lane
  static constexpr int LPT = 16 / G;             // lanes per tile
  static constexpr int TPW = 32 / LPT;           // tiles per warp
  static constexpr int COLW = TPW * 16;          // columns per warp
  static constexpr int WC = COLW >= 128 ? 1 : 128 / COLW;  // column warps per CTA
  static constexpr int WK = 8 / WC;              // k warps per CTA
  static constexpr int CTA_COLS = WC * COLW;     // 128 or 256
  static constexpr int NW = 4 * CPL;             // 32-bit stream words per lane
  static constexpr int DEPTH = CPL == 1 ? 4 : (CPL == 3 ? 2 : 1);  // loads in flight
};

struct GemvArgs {
  const __half *x;         // [k]
  const uint16_t *trellis; // [k/16][n/16][16K]
  const __half *suh;       // [k]
  const __half *svh;       // [n]
  void *y;                 // [n] fp16 or fp32
  float *partials;         // [splits][n]
  int *counters;           // [n / CTA_COLS]
  int *err;                // device error word
  int k, n, tk_per_split, splits;
};

template <int K>
__device__ __forceinline__ void load_chunks(const uint4 *src, bool valid, uint32_t (&w)[GemvShape<K>::NW]) {
  constexpr int CPL = GemvShape<K>::CPL;
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    uint4 t = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    w[4 * c + 0] = t.x;
    w[4 * c + 1] = t.y;
    w[4 * c + 2] = t.z;
    w[4 * c + 3] = t.w;
  }
}

template <int K, bool F32OUT>
__global__ void __launch_bounds__(256) gemv_m1_kernel(GemvArgs a) {
  using S = GemvShape<K>;
  extern __shared__ __align__(16) float smem[];
  const int kr = a.tk_per_split * 16;
  float *xs = smem;                           // [kr] transformed input slice
  float *red = xs + kr;                       // [WK][CTA_COLS]
  float *ys = red + S::WK * S::CTA_COLS;      // [CTA_COLS]
  __shared__ int s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.y;
  const int tk_begin = split * a.tk_per_split;
  const int tiles_n = a.n >> 4;

  // ---- prologue: x' = 2^-3.5 H (x . suh) for this CTA's k-range
  for (int b = warp; b < kr / 128; b += 8) {
    const int col = tk_begin * 16 + b * 128 + lane * 4;
    const uint2 xv = *reinterpret_cast<const uint2 *>(a.x + col);
    const uint2 sv = *reinterpret_cast<const uint2 *>(a.suh + col);
    const __half2 *xh = reinterpret_cast<const __half2 *>(&xv);
    const __half2 *sh = reinterpret_cast<const __half2 *>(&sv);
    float v[4] = {__low2float(xh[0]) * __low2float(sh[0]), __high2float(xh[0]) * __high2float(sh[0]),
                  __low2float(xh[1]) * __low2float(sh[1]), __high2float(xh[1]) * __high2float(sh[1])};
    fwht128_warp(v, lane);
    *reinterpret_cast<float4 *>(xs + b * 128 + lane * 4) =
        make_float4(v[0] * kRhtScale, v[1] * kRhtScale, v[2] * kRhtScale, v[3] * kRhtScale);
  }
  __syncthreads();

  // ---- main loop
  const int wc = warp % S::WC, wk = warp / S::WC;
  const int tile_in_warp = lane / S::LPT, q = lane % S::LPT;
  const int tn = blockIdx.x * (S::CTA_COLS / 16) + wc * S::TPW + tile_in_warp;
  const bool valid = tn < tiles_n;
  const int src_lane = (q == S::LPT - 1) ? lane - (S::LPT - 1) : lane + 1;
  const long tile_stride = (long)tiles_n * 16 * K / 8;   // uint4 units per tk row
  const uint4 *base = reinterpret_cast<const uint4 *>(a.trellis) +
                      ((long)tk_begin * tiles_n + tn) * (2 * K) + q * S::CPL;

  float acc[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) acc[c] = 0.f;

  const int iters = (a.tk_per_split - wk + S::WK - 1) / S::WK;   // tk = wk, wk + WK, ...
  uint32_t buf[S::DEPTH][S::NW];
#pragma unroll
  for (int d = 0; d < S::DEPTH; ++d)
    if (d < iters) load_chunks<K>(base + (long)(wk + d * S::WK) * tile_stride, valid, buf[d]);

  for (int it0 = 0; it0 < iters; it0 += S::DEPTH) {
#pragma unroll
    for (int d = 0; d < S::DEPTH; ++d) {
      const int it = it0 + d;
      if (it < iters) {
        uint32_t w[S::NW + 1];
#pragma unroll
        for (int i = 0; i < S::NW; ++i) w[i] = buf[d][i];
        w[S::NW] = __shfl_sync(0xffffffffu, w[0], src_lane);
        const int nxt = it + S::DEPTH;
        if (nxt < iters) load_chunks<K>(base + (long)(wk + nxt * S::WK) * tile_stride, valid, buf[d]);
        const int tkl = wk + it * S::WK;                       // tk - tk_begin
        float xr[S::G];
#pragma unroll
        for (int i = 0; i < S::G; ++i) xr[i] = xs[tkl * 16 + S::G * q + i];
#pragma unroll
        for (int j = 0; j < 16 * S::G; ++j) {
          const int bit = j * K;
          const uint32_t s = window16(w[bit >> 5], w[(bit >> 5) + 1], bit & 31);
          acc[j & 15] = fmaf(xr[j >> 4], mul1_centered(s), acc[j & 15]);
        }
      }
    }
  }

  // ---- reduce the LPT lanes of each tile, then the k-warps of the CTA
#pragma unroll
  for (int m = 1; m < S::LPT; m <<= 1)
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], m);
  if (q == 0) {
#pragma unroll
    for (int c = 0; c < 16; ++c) red[wk * S::CTA_COLS + wc * S::COLW + tile_in_warp * 16 + c] = acc[c];
  }
  __syncthreads();
  const int col0 = blockIdx.x * S::CTA_COLS;
  float part = 0.f;
  if (tid < S::CTA_COLS) {
#pragma unroll
    for (int w = 0; w < S::WK; ++w) part += red[w * S::CTA_COLS + tid];
    part *= kSigma;
  }

  if (a.splits == 1) {
    if (tid < S::CTA_COLS) ys[tid] = part;
  } else {
    if (tid < S::CTA_COLS && col0 + tid < a.n) a.partials[(long)split * a.n + col0 + tid] = part;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const int old = atomicAdd(a.counters + blockIdx.x, 1);
      if (old >= a.splits) set_device_error(a.err, kErrDirtyCounter);
      s_last = (old == a.splits - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid < S::CTA_COLS) {
      float sum = 0.f;
      if (col0 + tid < a.n)
        for (int s = 0; s < a.splits; ++s) sum += __ldcg(a.partials + (long)s * a.n + col0 + tid);
      ys[tid] = sum;
    }
    if (tid == 0) a.counters[blockIdx.x] = 0;   // leave the workspace clean
  }
  __syncthreads();

  // ---- output transform of the CTA's 128-column blocks
  if (warp < S::CTA_COLS / 128 && col0 + warp * 128 < a.n) {
    const int c = warp * 128 + lane * 4;
    float v[4] = {ys[c], ys[c + 1], ys[c + 2], ys[c + 3]};
    fwht128_warp(v, lane);
    const int gc = col0 + c;
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
}

template <int K>
int cta_cols() { return GemvShape<K>::CTA_COLS; }

template <int K>
size_t smem_bytes(int kr) {
  return sizeof(float) * ((size_t)kr + (size_t)GemvShape<K>::WK * GemvShape<K>::CTA_COLS +
                          GemvShape<K>::CTA_COLS);
}

}  // namespace exl3

using namespace exl3;

// Columns covered by one CTA for width K (128 or 256).
int exl3_gemv_cta_cols(int K) {
  switch (K) {
    case 1: return cta_cols<1>();
    case 2: return cta_cols<2>();
    case 3: return cta_cols<3>();
    case 4: return cta_cols<4>();
    case 5: return cta_cols<5>();
    case 6: return cta_cols<6>();
    case 7: return cta_cols<7>();
    case 8: return cta_cols<8>();
    default: return 128;
  }
}

// Number of k-splits: the smallest divisor of k/128 that gives at least
// `target_ctas` CTAs, with at most 8192 k-elements of x' per CTA.
int exl3_gemv_splits(int k, int n, int K, int target_ctas) {
  const int kb = k / 128;
  const int colblocks = ceil_div(n, exl3_gemv_cta_cols(K));
  int best = kb;
  for (int s = 1; s <= kb; ++s) {
    if (kb % s) continue;
    if ((kb / s) * 128 > 8192) continue;
    best = s;
    if (colblocks * s >= target_ctas) break;
  }
  return best;
}

size_t exl3_gemv_smem_bytes(int k, int K, int splits) {
  const int kr = k / splits;
  switch (K) {
    case 1: return smem_bytes<1>(kr);
    case 2: return smem_bytes<2>(kr);
    case 3: return smem_bytes<3>(kr);
    case 4: return smem_bytes<4>(kr);
    case 5: return smem_bytes<5>(kr);
    case 6: return smem_bytes<6>(kr);
    case 7: return smem_bytes<7>(kr);
    default: return smem_bytes<8>(kr);
  }
}

cudaError_t exl3_launch_gemv_m1(const uint16_t *x, const uint16_t *trellis, const uint16_t *suh,
                                const uint16_t *svh, int k, int n, int K, void *y, bool f32out,
                                float *partials, int *counters, int *err, int splits,
                                cudaStream_t s) {
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
  a.splits = splits;
  a.tk_per_split = (k / 16) / splits;
  const dim3 grid(ceil_div(n, exl3_gemv_cta_cols(K)), splits);
  const size_t smem = exl3_gemv_smem_bytes(k, K, splits);
  switch (K) {
#define EXL3_CASE(KK)                                                                          \
  case KK:                                                                                     \
    if (f32out) {                                                                              \
      cudaFuncSetAttribute(gemv_m1_kernel<KK, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           (int)smem);                                                         \
      gemv_m1_kernel<KK, true><<<grid, 256, smem, s>>>(a);                                     \
    } else {                                                                                   \
      cudaFuncSetAttribute(gemv_m1_kernel<KK, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           (int)smem);                                                         \
      gemv_m1_kernel<KK, false><<<grid, 256, smem, s>>>(a);                                    \
    }                                                                                          \
    break;
    EXL3_CASE(1) EXL3_CASE(2) EXL3_CASE(3) EXL3_CASE(4) EXL3_CASE(5) EXL3_CASE(6) EXL3_CASE(7)
    EXL3_CASE(8)
#undef EXL3_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}
