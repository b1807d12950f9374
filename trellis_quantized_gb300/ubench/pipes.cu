// pipes.cu -- instruction-throughput microbenchmark behind the M = 1 decode
// ceiling ("dp4a GEMV" of "exl3xpu" README, "Layout").
//
// Every mul1 weight costs one 32-bit multiply (the hash s * 0x9E3779B1), one
// byte sum (DP4A) and its share of the accumulate; a window cut out of the
// packed stream costs one or two ALU instructions.  Each kernel here runs one
// fixed mix of those instructions in 8 independent chains per thread, with
// 1024 threads per SM, and measures SM cycles with clock64, so the result is
// lane-operations (or decoded weights) per clock per SM, independent of the
// SM clock the box happens to run at.
//
// Mixes (lane-ops per chain and iteration in brackets):
//   0 IMAD                    (1)   mad.lo.u32
//   1 DP4A                    (1)   dp4a.u32.u32
//   2 IMAD + DP4A             (2)   the hash and byte sum of one weight
//   3 FHFMA                   (1)   fma.rn.f32.f16 (mixed fp16 x fp16 -> fp32)
//   4 FFMA2                   (1)   fma.rn.f32x2 (two fp32 FMAs)
//   5 FFMA                    (1)   fma.rn.f32
//   6 decode, FHFMA accumulate       (3 per weight): IMAD, DP4A, FHFMA
//   7 decode, FFMA2 accumulate       (2.5 per weight): IMAD, DP4A, half an FFMA2
//   8 ALU                     (1)   funnel shift / byte permute / logic op
//   9 full K = 4 decode, FFMA2       (31 per 8 weights): 11 window ops, 8 IMAD,
//                                    8 DP4A, 4 FFMA2
//  10 full K = 4 decode, FHFMA       (35 per 8 weights): 11 window ops, 8 IMAD,
//                                    8 DP4A, 8 FHFMA
//  11 HMMA                    (1)   mma.sync.m16n8k16 f16 x f16 -> f32 (warp-wide)
//  12 full K = 4 decode, HMMA        (16 weights): 22 window ops, 16 IMAD,
//                                    16 DP4A and 4 lane-shares of an HMMA: each
//                                    DP4A result (fp16 1024 + B beside a zero
//                                    half) is one A element of an MMA whose odd
//                                    k columns are zero
//  13 decode, FFMA accumulate        (3 per weight): IMAD, DP4A, FFMA of x' and
//                                    the byte sum read as a subnormal fp32
//  14 full K = 4 decode, FFMA        (35 per 8 weights): 11 window ops, 8 IMAD,
//                                    8 DP4A, 8 FFMA
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint32_t kMul = 0x9E3779B1u;

__device__ __forceinline__ uint32_t imad(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t dp4a(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ float fhfma(uint32_t xh, uint32_t wh, float acc) {
  asm("{\n.reg .f16 a, b;\n.reg .b16 l0, h0, l1, h1;\nmov.b32 {l0, h0}, %1;\nmov.b32 {l1, h1}, %2;\n"
      "mov.b16 a, l0;\nmov.b16 b, l1;\nfma.rn.f32.f16 %0, a, b, %0;\n}\n"
      : "+f"(acc)
      : "r"(xh), "r"(wh));
  return acc;
}
__device__ __forceinline__ void ffma2(float &c0, float &c1, float a0, float a1, uint32_t b0, uint32_t b1) {
  asm("{\n.reg .b64 A, B, C;\nmov.b64 A, {%2, %3};\nmov.b64 B, {%4, %5};\nmov.b64 C, {%0, %1};\n"
      "fma.rn.f32x2 C, A, B, C;\nmov.b64 {%0, %1}, C;\n}\n"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t shf(uint32_t lo, uint32_t hi, uint32_t sh) {
  uint32_t d;
  asm("shf.r.wrap.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(lo), "r"(hi), "r"(sh));
  return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t land(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("and.b32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t shr(uint32_t a, uint32_t s) {
  uint32_t d;
  asm("shr.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(s));
  return d;
}

// K = 4: the eight windows of one 32-bit stream word w (next word n), each
// hashed, byte-summed (DP4A seeded with `seed`) into b[0..8).
__device__ __forceinline__ void decode8(uint32_t w, uint32_t n, uint32_t seed, uint32_t mask, uint32_t (&b)[8]) {
  const uint32_t w4 = shf(w, n, 4u);                       // window residues 4, 12, 20
  uint32_t s[8];
  s[0] = land(w, mask);                                    // residue 0
  s[2] = prmt(w, 0u, 0x4421u);                             // residue 8
  s[4] = shr(w, 16u);                                      // residue 16
  s[1] = land(w4, mask);
  s[3] = prmt(w4, 0u, 0x4421u);
  s[5] = shr(w4, 16u);
  s[6] = land(shf(w, n, 24u), mask);                       // residue 24
  s[7] = land(shf(w, n, 28u), mask);                       // residue 28
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = dp4a(imad(s[i], kMul, 0u), 0x01010101u, seed);
}

// D += A B, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void hmma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                     uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int MIX>
__global__ void __launch_bounds__(1024, 1) pipes_kernel(uint32_t seed, int iters, unsigned long long *cycles,
                                                        uint32_t *sink) {
  uint32_t u[8];
  float f[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    u[i] = seed * (threadIdx.x + 7u * i + 1u);
    f[i] = (float)(u[i] & 0xFFu) * 0.001f;
  }
  const uint32_t mask = seed >> 16;   // 0xFFFF at run time (seed is 0xFFFFxxxx)
  const float xa = __uint_as_float(seed & 0x3Fu) + 1.0f, xb = 0.5f + (float)(seed & 1u);
  __syncthreads();
  const unsigned long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    if constexpr (MIX == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = imad(u[i], kMul, 0x1234u);
    } else if constexpr (MIX == 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = dp4a(u[i], 0x01010101u, u[i]);
    } else if constexpr (MIX == 2) {
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = dp4a(imad(u[i], kMul, 0u), 0x01010101u, u[i]);
    } else if constexpr (MIX == 3) {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = fhfma(0x3C003C00u, u[i], f[i]);
    } else if constexpr (MIX == 4) {
#pragma unroll
      for (int i = 0; i < 8; i += 2) ffma2(f[i], f[i + 1], xa, xb, u[i], u[i + 1]);
#pragma unroll
      for (int i = 0; i < 8; i += 2) ffma2(f[i], f[i + 1], xb, xa, u[i + 1], u[i]);
    } else if constexpr (MIX == 5) {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = fmaf(xa, f[i], xb);
    } else if constexpr (MIX == 6) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        u[i] = dp4a(imad(u[i], kMul, 0u), 0x01010101u, 0x6400u);
        f[i] = fhfma(0x3C003C00u, u[i], f[i]);
      }
    } else if constexpr (MIX == 7) {
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = dp4a(imad(u[i], kMul, 0u), 0x01010101u, 0u);
#pragma unroll
      for (int i = 0; i < 8; i += 2) ffma2(f[i], f[i + 1], xa, xa, u[i], u[i + 1]);
    } else if constexpr (MIX == 8) {
#pragma unroll
      for (int i = 0; i < 8; i += 4) {
        u[i] = shf(u[i], u[i + 1], 4u);
        u[i + 1] = prmt(u[i + 1], u[i + 2], 0x4421u);
        u[i + 2] = land(u[i + 2], u[i + 3] | 1u);
        u[i + 3] = shr(u[i + 3], 3u) + u[i];
      }
    } else if constexpr (MIX == 9 || MIX == 10) {
      uint32_t b[8];
      decode8(u[0], u[1], MIX == 9 ? 0u : 0x6400u, mask, b);
      if constexpr (MIX == 9) {
#pragma unroll
        for (int i = 0; i < 8; i += 2) ffma2(f[i], f[i + 1], xa, xa, b[i], b[i + 1]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = fhfma(0x3C003C00u, b[i], f[i]);
      }
      u[0] ^= b[7];
      u[1] += b[3];
    } else if constexpr (MIX == 13) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        u[i] = dp4a(imad(u[i], kMul, 0u), 0x01010101u, 0u);
        f[i] = fmaf(xa, __uint_as_float(u[i]), f[i]);
      }
    } else if constexpr (MIX == 14) {
      uint32_t b[8];
      decode8(u[0], u[1], 0u, mask, b);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = fmaf(xa, __uint_as_float(b[i]), f[i]);
      u[0] ^= b[7];
      u[1] += b[3];
    } else if constexpr (MIX == 11) {
      float d[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = f[i];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i) hmma(d[i], u[i], u[i + 1], u[i + 2], u[i + 3], u[4], u[5]);
#pragma unroll
      for (int i = 0; i < 4; ++i) f[i] = d[i][0] + d[i][3];
    } else if constexpr (MIX == 12) {
      uint32_t b[16];
      decode8(u[0], u[1], 0x6400u, mask, *reinterpret_cast<uint32_t(*)[8]>(&b[0]));
      decode8(u[2], u[3], 0x6400u, mask, *reinterpret_cast<uint32_t(*)[8]>(&b[8]));
      float d[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = f[i];
#pragma unroll
      for (int i = 0; i < 4; ++i) hmma(d[i], b[4 * i], b[4 * i + 1], b[4 * i + 2], b[4 * i + 3], u[4], u[5]);
#pragma unroll
      for (int i = 0; i < 4; ++i) f[i] = d[i][0] + d[i][2];
      u[0] ^= b[7];
      u[1] += b[3];
      u[2] ^= b[15];
      u[3] += b[11];
    }
  }
  const unsigned long long t1 = clock64();
  uint32_t acc = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc ^= u[i] ^ __float_as_uint(f[i]);
  if (acc == 0x7FFFFFFFu) sink[threadIdx.x] = acc;   // practically never: keeps the chains live
  __syncthreads();
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int MIX>
cudaError_t launch(int grid, uint32_t seed, int iters, unsigned long long *cycles, uint32_t *sink, cudaStream_t s) {
  pipes_kernel<MIX><<<grid, 1024, 0, s>>>(seed, iters, cycles, sink);
  return cudaGetLastError();
}

}  // namespace

// Runs mix `mix` (0..14) on `grid` CTAs of 1024 threads (one per SM), each
// thread `iters` iterations; cycles[grid] (device) receives each CTA's SM
// cycles, sink[1024] (device) is a write target that keeps the results live.
// Returns a cudaError_t value (0 on success).  Lane-operations per iteration
// and thread are listed in the header comment.
extern "C" int exl3_ubench_pipes(int mix, int grid, int iters, unsigned long long *cycles, unsigned int *sink,
                                 void *stream) {
  const uint32_t seed = 0xFFFF1357u;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (mix) {
    case 0: return launch<0>(grid, seed, iters, cycles, sink, s);
    case 1: return launch<1>(grid, seed, iters, cycles, sink, s);
    case 2: return launch<2>(grid, seed, iters, cycles, sink, s);
    case 3: return launch<3>(grid, seed, iters, cycles, sink, s);
    case 4: return launch<4>(grid, seed, iters, cycles, sink, s);
    case 5: return launch<5>(grid, seed, iters, cycles, sink, s);
    case 6: return launch<6>(grid, seed, iters, cycles, sink, s);
    case 7: return launch<7>(grid, seed, iters, cycles, sink, s);
    case 8: return launch<8>(grid, seed, iters, cycles, sink, s);
    case 9: return launch<9>(grid, seed, iters, cycles, sink, s);
    case 10: return launch<10>(grid, seed, iters, cycles, sink, s);
    case 11: return launch<11>(grid, seed, iters, cycles, sink, s);
    case 12: return launch<12>(grid, seed, iters, cycles, sink, s);
    case 13: return launch<13>(grid, seed, iters, cycles, sink, s);
    case 14: return launch<14>(grid, seed, iters, cycles, sink, s);
    default: return (int)cudaErrorInvalidValue;
  }
}
