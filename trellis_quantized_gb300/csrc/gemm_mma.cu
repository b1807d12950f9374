// gemm_mma.cu -- dense Hadamard-domain contraction y' = x' W on the legacy
// warp-level tensor-core path (mma.sync m16n8k16, fp16 in, fp32 out).
//
// Operands: x' fp16 [M][k] (row-major, K-major) and Wt fp16 [n][k] (the
// transposed reconstruct, K-major); output y' fp32 [M][n].  This is the
// "reconstruct, then dense GEMM" form of the prefill linear ("exl3xpu"
// README, "Layout": ops.py dispatches large M to reconstruct + a library
// GEMM).  CTA tile 128 x 128 x 32, 8 warps as 2 (M) x 4 (N), 3-stage
// cp.async pipeline, ldmatrix fragments.
#include "exl3_common.cuh"

namespace exl3 {
namespace mma {

constexpr int BM = 128, BN = 128, BK = 32, STAGES = 3, PITCH = BK + 8;  // halves

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool pred) {
  const int n = pred ? 16 : 0;   // zero-fill when out of range
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(n));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(256) gemm_kernel(const __half *__restrict__ A,   // [M][k]
                                                   const __half *__restrict__ B,   // [n][k]
                                                   float *__restrict__ C,          // [M][n]
                                                   int M, int n, int k) {
  extern __shared__ __align__(16) __half sm[];
  __half *As = sm;                               // [STAGES][BM][PITCH]
  __half *Bs = sm + STAGES * BM * PITCH;         // [STAGES][BN][PITCH]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 2, wn = warp & 3;       // warp tile 64 x 32
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int ktiles = k / BK;

  auto load_stage = [&](int stage, int kt) {
    const int kk = kt * BK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {                // 128 rows x 4 chunks = 512 chunks per operand
      const int c = tid + i * 256, row = c >> 2, ch = (c & 3) * 8;
      const int gm = m0 + row;
      cp_async16(As + (stage * BM + row) * PITCH + ch, A + (long)min(gm, M - 1) * k + kk + ch, gm < M);
      const int gn = n0 + row;
      cp_async16(Bs + (stage * BN + row) * PITCH + ch, B + (long)min(gn, n - 1) * k + kk + ch, gn < n);
    }
  };

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.f;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < ktiles) load_stage(s, s);
    asm volatile("cp.async.commit_group;\n");
  }

  for (int kt = 0; kt < ktiles; ++kt) {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(STAGES - 2));
    __syncthreads();
    const int nk = kt + STAGES - 1;
    if (nk < ktiles) load_stage(nk % STAGES, nk);
    asm volatile("cp.async.commit_group;\n");
    const int st = kt % STAGES;
#pragma unroll
    for (int ks = 0; ks < BK; ks += 16) {
      uint32_t af[4][4], bf[2][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = wm * 64 + i * 16 + (lane & 15), col = ks + (lane >> 4) * 8;
        ldmatrix_x4(af[i], As + (st * BM + row) * PITCH + col);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int row = wn * 32 + j * 16 + (lane & 7) + ((lane >> 4) << 3), col = ks + ((lane >> 3) & 1) * 8;
        ldmatrix_x4(bf[j], Bs + (st * BN + row) * PITCH + col);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma16816(acc[i][j], af[i], bf[j >> 1][(j & 1) * 2], bf[j >> 1][(j & 1) * 2 + 1]);
    }
  }
  asm volatile("cp.async.wait_group 0;\n");

#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int row = m0 + wm * 64 + i * 16 + (lane >> 2);
      const int col = n0 + wn * 32 + j * 8 + (lane & 3) * 2;
      if (col < n) {
        if (row < M) *reinterpret_cast<float2 *>(C + (long)row * n + col) = make_float2(acc[i][j][0], acc[i][j][1]);
        if (row + 8 < M)
          *reinterpret_cast<float2 *>(C + (long)(row + 8) * n + col) = make_float2(acc[i][j][2], acc[i][j][3]);
      }
    }
}

}  // namespace mma
}  // namespace exl3

cudaError_t exl3_launch_gemm_mma(const uint16_t *xh, const uint16_t *wt, float *yp, int M, int n, int k,
                                 cudaStream_t s) {
  using namespace exl3::mma;
  const size_t smem = sizeof(__half) * STAGES * (BM + BN) * PITCH;
  cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid(exl3::ceil_div(n, BN), exl3::ceil_div(M, BM));
  gemm_kernel<<<grid, 256, smem, s>>>(reinterpret_cast<const __half *>(xh), reinterpret_cast<const __half *>(wt),
                                      yp, M, n, k);
  return cudaGetLastError();
}
