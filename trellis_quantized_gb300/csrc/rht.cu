// rht.cu -- the randomized block Hadamard transforms on activations and
// outputs ("Hadamard in/out", "exl3xpu" README, "Layout"; randomized Hadamard
// transforms, "Bringing EXL3 Trellis Quantization to 35B MoE on Intel Arc
// 140V", section 1).
//
// One warp transforms one aligned 128-element block held as 4 elements per
// lane (fwht128_warp): x' = 2^-3.5 H (x . suh).  The output side is fused
// into the epilogues of the GEMV and GEMM kernels.
#include "exl3_common.cuh"

namespace exl3 {

// x [M][k] fp16 -> out [M][k] fp32 (OUT_F32) or fp16.  One warp per group of
// four 128-blocks of a row (512 elements, 16 contiguous per lane: the
// fwht128_x8 layout).  With fp16 output, xsum (optional) receives the sum of
// each 256-element unit of the fp16 x' row, [M][ceil(k / 256)] fp32: 16
// values per lane in order, then lanes 0-15 (or 16-31) by halving.

template <bool F32OUT>
__global__ void __launch_bounds__(256) input_rht_kernel(const __half *__restrict__ x,
                                                        const __half *__restrict__ suh, int M, int k,
                                                        void *__restrict__ out, float *__restrict__ xsum) {
  // a dependent kernel (the small-M linear) may start its set-up and
  // weight loads now; it reads x' only after this grid completes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long wid = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int groups = (k + 511) / 512;
  if (wid >= (long)M * groups) return;            // uniform per warp
  const long row = wid / groups;
  const int col = (int)(wid % groups) * 512 + 16 * lane;
  const bool in = col < k;                        // whole 128-blocks are in or out
  uint4 xv[2] = {}, sv[2] = {};
  if (in) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      xv[q] = *reinterpret_cast<const uint4 *>(x + row * k + col + 8 * q);
      sv[q] = __ldg(reinterpret_cast<const uint4 *>(suh + col + 8 * q));
    }
  }
  const __half *xh = reinterpret_cast<const __half *>(xv);
  const __half *sh = reinterpret_cast<const __half *>(sv);
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __half2float(xh[j]) * __half2float(sh[j]);   // exact
  fwht128_x8(v, lane);
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], kRhtScale);
  if (F32OUT) {
    if (!in) return;
    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(out) + row * k + col);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  } else {
    __align__(16) __half2 o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
    if (in) {
      uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__half *>(out) + row * k + col);
      dst[0] = reinterpret_cast<const uint4 *>(o)[0];
      dst[1] = reinterpret_cast<const uint4 *>(o)[1];
    }
    if (xsum) {   // uniform per launch; lanes outside k hold zeros
      float t = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) t += __low2float(o[j]) + __high2float(o[j]);
#pragma unroll
      for (int m = 8; m >= 1; m >>= 1) t += __shfl_xor_sync(0xffffffffu, t, m);
      if ((lane & 15) == 0 && in) xsum[row * ((k + 255) / 256) + col / 256] = t;
    }
  }
}

}  // namespace exl3

using namespace exl3;

cudaError_t exl3_launch_input_rht(const uint16_t *x, int M, int k, const uint16_t *suh, void *out,
                                  bool f32out, cudaStream_t s, float *xsum) {
  const long warps = (long)M * ((k + 511) / 512);
  const unsigned grid = (unsigned)((warps + 7) / 8);
  if (grid == 0) return cudaSuccess;
  const __half *xh = reinterpret_cast<const __half *>(x);
  const __half *sh = reinterpret_cast<const __half *>(suh);
  if (f32out) input_rht_kernel<true><<<grid, 256, 0, s>>>(xh, sh, M, k, out, nullptr);
  else input_rht_kernel<false><<<grid, 256, 0, s>>>(xh, sh, M, k, out, xsum);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// int8 activations ("exl3xpu" README, "Prefill: int8 linears and oneDNN fused
// attention": one int8 scale per activation row, fused into the input
// Hadamard).  One CTA per row: x' in fp32 with the butterfly order above,
// amax over the row, inv = 127 / amax (IEEE division), q = clamp(RNE(x' inv),
// -127, 127), a = amax / 127; an all-zero row gives q = 0, a = 0.
// q is written as integer-valued fp16 (the tensor-core operand) and, if
// requested, as int8.
namespace exl3 {

__global__ void __launch_bounds__(256) quant_act_kernel(const __half *__restrict__ x,
                                                        const __half *__restrict__ suh, int k,
                                                        __half *__restrict__ qh, int8_t *__restrict__ q8,
                                                        float *__restrict__ row_scale) {
  extern __shared__ __align__(16) float xr[];   // [k]
  __shared__ float wmax[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long row = blockIdx.x;
  float m = 0.f;
  // warp w takes the 512-element groups w, w + 8, ... (fwht128_x8 layout)
  for (int c0 = warp * 512; c0 < k; c0 += 8 * 512) {
    const int col = c0 + 16 * lane;
    const bool in = col < k;
    uint4 xv[2] = {}, sv[2] = {};
    if (in) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        xv[q] = *reinterpret_cast<const uint4 *>(x + row * k + col + 8 * q);
        sv[q] = __ldg(reinterpret_cast<const uint4 *>(suh + col + 8 * q));
      }
    }
    const __half *xh = reinterpret_cast<const __half *>(xv);
    const __half *sh = reinterpret_cast<const __half *>(sv);
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __half2float(xh[j]) * __half2float(sh[j]);
    fwht128_x8(v, lane);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      v[j] = __fmul_rn(v[j], kRhtScale);
      m = fmaxf(m, fabsf(v[j]));
    }
    if (in) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<float4 *>(xr + col + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  float amax = wmax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, wmax[w]);
  const float inv = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
  if (threadIdx.x == 0 && row_scale) row_scale[row] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
  for (int i = threadIdx.x * 4; i < k; i += 256 * 4) {
    const float4 v = *reinterpret_cast<const float4 *>(xr + i);
    const float vv[4] = {v.x, v.y, v.z, v.w};
    int q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int t = amax > 0.f ? __float2int_rn(__fmul_rn(vv[j], inv)) : 0;
      q[j] = t > 127 ? 127 : (t < -127 ? -127 : t);
    }
    __half2 h[2] = {__floats2half2_rn((float)q[0], (float)q[1]), __floats2half2_rn((float)q[2], (float)q[3])};
    *reinterpret_cast<uint2 *>(qh + row * k + i) = *reinterpret_cast<uint2 *>(h);
    if (q8) {
      const uint32_t packed = (uint32_t)(q[0] & 255) | ((uint32_t)(q[1] & 255) << 8) |
                              ((uint32_t)(q[2] & 255) << 16) | ((uint32_t)(q[3] & 255) << 24);
      *reinterpret_cast<uint32_t *>(q8 + row * k + i) = packed;
    }
  }
}

}  // namespace exl3

cudaError_t exl3_launch_quant_act(const uint16_t *x, int M, int k, const uint16_t *suh, uint16_t *qh,
                                  int8_t *q8, float *row_scale, cudaStream_t s) {
  const size_t smem = sizeof(float) * (size_t)k;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(exl3::quant_act_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  exl3::quant_act_kernel<<<M, 256, smem, s>>>(reinterpret_cast<const __half *>(x),
                                              reinterpret_cast<const __half *>(suh), k,
                                              reinterpret_cast<__half *>(qh), q8, row_scale);
  return cudaGetLastError();
}
