// decode.cu -- trellis dequantisation ("reconstruct", "exl3xpu" README,
// "Layout"; dequantised weights bit-exact, "exl3xpu" README, "Correctness").
//
// One thread decodes one row r of one 16x16 tile: 16 consecutive weights
// p = 16 r .. 16 r + 15, whose windows start at stream bits 16 r K + c K.
// Those windows read words r K .. r K + K of the tile (the last one wraps to
// word 0 for r = 15).  The words are packed into 32-bit registers and every
// window is one funnel shift and a mask at a compile-time offset.
#include "exl3_common.cuh"

namespace exl3 {

// Gather the stream words of tile row r into 32-bit registers:
// a[i] = word(rK + 2i) | word(rK + 2i + 1) << 16 (words taken mod 16K).
template <int K>
__device__ __forceinline__ void load_row_words(const uint16_t *__restrict__ tile, int r,
                                               uint32_t (&a)[(K + 2) / 2 + 1]) {
  constexpr int NW = 16 * K;
#pragma unroll
  for (int i = 0; i < (K + 2) / 2 + 1; ++i) {
    int w0 = r * K + 2 * i, w1 = w0 + 1;
    uint32_t lo = (2 * i <= K) ? (uint32_t)__ldg(tile + (w0 % NW)) : 0u;
    uint32_t hi = (2 * i + 1 <= K) ? (uint32_t)__ldg(tile + (w1 % NW)) : 0u;
    a[i] = lo | (hi << 16);
  }
}

// Decode the 16 weights of tile row r as fp16 values.
template <int K>
__device__ __forceinline__ void decode_row(const uint16_t *__restrict__ tile, int r, __half (&v)[16]) {
  uint32_t a[(K + 2) / 2 + 1];
  load_row_words<K>(tile, r, a);
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const int bit = c * K;
    const uint32_t s = window16(a[bit >> 5], a[(bit >> 5) + 1], bit & 31);
    v[c] = mul1_half(s);
  }
}

// w_out[(16 (tk - tk0) + r) * ld + 16 (tn - tn0) + c] for the tile range.
// Block: 256 threads = 8 tile rows x 32 consecutive tiles along n.
template <int K>
__global__ void __launch_bounds__(256) decode_tile_kernel(const uint16_t *__restrict__ trellis,
                                                          int tiles_n, int tk0, int tk_cnt, int tn0,
                                                          int tn_cnt, uint16_t *__restrict__ w_out,
                                                          int64_t ld) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.y * 8 + warp;          // row within the requested range
  const int tnl = blockIdx.x * 32 + lane;
  if (row >= tk_cnt * 16 || tnl >= tn_cnt) return;
  const int tkl = row >> 4, r = row & 15;
  const long tile = (long)(tk0 + tkl) * tiles_n + (tn0 + tnl);
  __align__(16) __half v[16];
  decode_row<K>(trellis + tile * 16 * K, r, v);
  uint4 *dst = reinterpret_cast<uint4 *>(w_out + (int64_t)row * ld + 16 * tnl);
  dst[0] = *reinterpret_cast<uint4 *>(&v[0]);
  dst[1] = *reinterpret_cast<uint4 *>(&v[8]);
}

// Transposed full reconstruct for the tensor-core GEMM: Wt[n][k] (K-major
// operand), Wt[16 tn + c][16 tk + r] = W[16 tk + r][16 tn + c].
// Block: 256 threads decode 8 tk x 2 tn tiles (16 rows each) into shared
// memory as [32 n][128 k], then write 32 rows of 256 contiguous bytes.
template <int K>
__global__ void __launch_bounds__(256) reconstruct_t_kernel(const uint16_t *__restrict__ trellis,
                                                            int tiles_k, int tiles_n,
                                                            uint16_t *__restrict__ wt, int k) {
  // A programmatic dependent of the input transform: it reads only the
  // trellis, so it runs beside that kernel, and it waits for it at the end so
  // that its own completion (which the GEMM waits for) implies both.
  pdl_trigger();
  __shared__ __align__(16) __half sm[32][128 + 8];
  const int t = threadIdx.x;
  const int tile_local = t >> 4, r = t & 15;       // 16 tiles per block
  const int tkl = tile_local & 7, tnl = tile_local >> 3;
  const int tk = blockIdx.y * 8 + tkl, tn = blockIdx.x * 2 + tnl;
  if (tk < tiles_k && tn < tiles_n) {
    __align__(16) __half v[16];
    decode_row<K>(trellis + ((long)tk * tiles_n + tn) * 16 * K, r, v);
#pragma unroll
    for (int c = 0; c < 16; ++c) sm[tnl * 16 + c][tkl * 16 + r] = v[c];
  }
  __syncthreads();
  // 32 rows x 128 halves = 512 chunks of 16 B, two per thread
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    int chunk = t + i * 256;
    int nrow = chunk >> 4, kc = (chunk & 15) * 8;
    int ng = blockIdx.x * 32 + nrow, kg = blockIdx.y * 128 + kc;
    if (ng < tiles_n * 16 && kg < k)
      *reinterpret_cast<uint4 *>(wt + (long)ng * k + kg) = *reinterpret_cast<const uint4 *>(&sm[nrow][kc]);
  }
  pdl_wait();
}

// int8 weights ("exl3xpu" README, "Prefill: int8 linears and oneDNN fused
// attention": one static weight scale, fused into reconstruct):
// q_w = RNE(v * 127 / 3.453125) of the decoded fp16 weight v, an exact
// rational.  One fp32 product v * fp32(127 / 3.453125) rounded to nearest
// even gives that integer for every one of the 1021 codebook values (checked
// exhaustively against exact rational arithmetic), so no table is needed.
constexpr float kQ8Scale = 127.0f / 3.453125f;

__device__ __forceinline__ __half mul1_q8(uint32_t s) {
  return __int2half_rn(__float2int_rn(__half2float(mul1_half(s)) * kQ8Scale));
}

// Transposed reconstruct of q_w as integer-valued fp16: Wq[16 tn + c][16 tk + r].
template <int K>
__global__ void __launch_bounds__(256) reconstruct_q8_t_kernel(const uint16_t *__restrict__ trellis,
                                                               int tiles_k, int tiles_n,
                                                               uint16_t *__restrict__ wq, int k) {
  pdl_trigger();   // beside the activation quantiser, as reconstruct_t_kernel
  __shared__ __align__(16) __half sm[32][128 + 8];
  const int t = threadIdx.x;
  const int tile_local = t >> 4, r = t & 15;
  const int tkl = tile_local & 7, tnl = tile_local >> 3;
  const int tk = blockIdx.y * 8 + tkl, tn = blockIdx.x * 2 + tnl;
  if (tk < tiles_k && tn < tiles_n) {
    uint32_t a[(K + 2) / 2 + 1];
    load_row_words<K>(trellis + ((long)tk * tiles_n + tn) * 16 * K, r, a);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int bit = c * K;
      sm[tnl * 16 + c][tkl * 16 + r] = mul1_q8(window16(a[bit >> 5], a[(bit >> 5) + 1], bit & 31));
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    int chunk = t + i * 256;
    int nrow = chunk >> 4, kc = (chunk & 15) * 8;
    int ng = blockIdx.x * 32 + nrow, kg = blockIdx.y * 128 + kc;
    if (ng < tiles_n * 16 && kg < k)
      *reinterpret_cast<uint4 *>(wq + (long)ng * k + kg) = *reinterpret_cast<const uint4 *>(&sm[nrow][kc]);
  }
  pdl_wait();
}

}  // namespace exl3

using namespace exl3;

cudaError_t exl3_launch_reconstruct_q8_t(const uint16_t *trellis, int k, int n, int K, uint16_t *wq,
                                         cudaStream_t s) {
  dim3 grid(ceil_div(n / 16, 2), ceil_div(k / 16, 8));
  switch (K) {
#define EXL3_CASE(KK) \
  case KK: return launch_pdl(reconstruct_q8_t_kernel<KK>, grid, dim3(256), 0, s, trellis, k / 16, n / 16, wq, k);
    EXL3_CASE(1) EXL3_CASE(2) EXL3_CASE(3) EXL3_CASE(4) EXL3_CASE(5) EXL3_CASE(6) EXL3_CASE(7)
    EXL3_CASE(8)
#undef EXL3_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// Launch helpers, called from api.cu after argument validation.
cudaError_t exl3_launch_decode_tile(const uint16_t *trellis, int n, int K, int tk0, int tk_cnt,
                                    int tn0, int tn_cnt, uint16_t *w_out, int64_t ld,
                                    cudaStream_t s) {
  dim3 grid(ceil_div(tn_cnt, 32), tk_cnt * 2);
  const int tiles_n = n / 16;
  switch (K) {
#define EXL3_CASE(KK)                                                                       \
  case KK:                                                                                  \
    decode_tile_kernel<KK><<<grid, 256, 0, s>>>(trellis, tiles_n, tk0, tk_cnt, tn0, tn_cnt, \
                                                w_out, ld);                                 \
    break;
    EXL3_CASE(1) EXL3_CASE(2) EXL3_CASE(3) EXL3_CASE(4) EXL3_CASE(5) EXL3_CASE(6) EXL3_CASE(7)
    EXL3_CASE(8)
#undef EXL3_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t exl3_launch_reconstruct_t(const uint16_t *trellis, int k, int n, int K, uint16_t *wt,
                                      cudaStream_t s) {
  dim3 grid(ceil_div(n / 16, 2), ceil_div(k / 16, 8));
  switch (K) {
#define EXL3_CASE(KK) \
  case KK: return launch_pdl(reconstruct_t_kernel<KK>, grid, dim3(256), 0, s, trellis, k / 16, n / 16, wt, k);
    EXL3_CASE(1) EXL3_CASE(2) EXL3_CASE(3) EXL3_CASE(4) EXL3_CASE(5) EXL3_CASE(6) EXL3_CASE(7)
    EXL3_CASE(8)
#undef EXL3_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}
