// moe.cu -- routed experts ("exl3xpu" README, "MoE (routed experts)";
// "Bringing EXL3 Trellis Quantization to 35B MoE on Intel Arc 140V",
// sections 2.A-2.D): device-side token-to-expert binning, the gather and
// input transform of the routed rows, and the final weighted combine.  The
// two grouped projections, with the trellis decoded on the fly, are in
// moe_fused.cu.
//
// Units are (token t, slot s) pairs, u = t * topk + s.  Every step runs on the
// device; the host never waits for routing results.
#include "exl3_common.cuh"

namespace exl3 {
namespace moe {

struct Plan {       // device-side routing results (workspace)
  int *counts;      // [E]
  int *offsets;     // [E + 1] exclusive scan of counts (rows in sorted order)
  int *perm;        // [U] sorted row -> unit
  int *pos;         // [U] unit -> sorted row (-1 for an invalid expert id)
  int4 *mtiles;     // [max_mtiles]: (expert, first row, rows, 0) per 128-row tile
  int *n_mtiles;    // [1]
};

// Counts, offsets and the 128-row tile list.
// One CTA of 1024 threads; E <= 1024.
__global__ void __launch_bounds__(1024) remap_count_kernel(const int32_t *__restrict__ ids, int U, int E,
                                                           Plan p, int max_mtiles, int *err) {
  extern __shared__ int sh[];   // cnt[E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  for (int u = threadIdx.x; u < U; u += blockDim.x) {
    const int e = ids[u];
    if (e >= 0 && e < E) {
      atomicAdd(&sh[e], 1);
    } else {
      set_device_error(err, kErrExpertId);
      p.pos[u] = -1;   // skipped: contributes nothing
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0, nt = 0;
    for (int e = 0; e < E; ++e) {
      const int c = sh[e];
      p.counts[e] = c;
      p.offsets[e] = off;
      if (c > 0) {
        for (int r = 0; r < c; r += 128) {
          if (nt < max_mtiles) p.mtiles[nt] = make_int4(e, off + r, min(128, c - r), 0);
          ++nt;
        }
      }
      off += c;
    }
    p.offsets[E] = off;
    if (nt > max_mtiles) set_device_error(err, kErrBounds);
    *p.n_mtiles = min(nt, max_mtiles);
  }
}

// Stable placement: warp e scans all units in order with ballots; the unit's
// row is offsets[e] + (number of earlier units routed to e).
__global__ void __launch_bounds__(256) remap_place_kernel(const int32_t *__restrict__ ids, int U, int E,
                                                          Plan p) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (e >= E || p.counts[e] == 0) return;
  int base = p.offsets[e];
  for (int u0 = 0; u0 < U; u0 += 32) {
    const int u = u0 + lane;
    const int id = u < U ? ids[u] : -1;
    const unsigned m = __ballot_sync(0xffffffffu, id == e);
    if (id == e) {
      const int r = base + __popc(m & ((1u << lane) - 1u));
      p.perm[r] = u;
      p.pos[u] = r;
    }
    base += __popc(m);
  }
}

// Sorted rows of the transformed token inputs for gate and up:
// xg[i] = RHT(x_t . suh_gate[e]), xu[i] = RHT(x_t . suh_up[e]), t = perm[i] / topk.
__global__ void __launch_bounds__(256) gather_rht_kernel(const __half *__restrict__ x, int hidden, int topk,
                                                         const int *__restrict__ perm,
                                                         const int *__restrict__ offsets, int E,
                                                         const int32_t *__restrict__ ids,
                                                         const __half *__restrict__ suh13,  // [E][2][hidden]
                                                         __half *__restrict__ xg, __half *__restrict__ xu) {
  const int lane = threadIdx.x & 31;
  const int blocks = hidden >> 7;
  const long wid = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int U = offsets[E];
  if (wid >= (long)U * blocks * 2) return;
  const int slot = (int)(wid & 1);
  const long rb = wid >> 1;
  const int i = (int)(rb / blocks), b = (int)(rb % blocks);
  const int u = perm[i];
  const int t = u / topk, e = ids[u];
  const int col = b * 128 + lane * 4;
  const uint2 xv = *reinterpret_cast<const uint2 *>(x + (long)t * hidden + col);
  const uint2 sv = *reinterpret_cast<const uint2 *>(suh13 + ((long)e * 2 + slot) * hidden + col);
  const __half2 *xh = reinterpret_cast<const __half2 *>(&xv);
  const __half2 *sh = reinterpret_cast<const __half2 *>(&sv);
  float v[4] = {__low2float(xh[0]) * __low2float(sh[0]), __high2float(xh[0]) * __high2float(sh[0]),
                __low2float(xh[1]) * __low2float(sh[1]), __high2float(xh[1]) * __high2float(sh[1])};
  fwht128_warp(v, lane);
  __half2 o[2] = {__floats2half2_rn(v[0] * kRhtScale, v[1] * kRhtScale),
                  __floats2half2_rn(v[2] * kRhtScale, v[3] * kRhtScale)};
  __half *dst = (slot == 0 ? xg : xu) + (long)i * hidden + col;
  *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<uint2 *>(o);
}

// y_t = sum over slots s (in order) of d[pos(t, s)]; d already carries the
// routing weight.  Invalid units (pos = -1) contribute nothing.
template <bool F32OUT>
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ d, const int *__restrict__ pos,
                                                      int T, int topk, int hidden, void *__restrict__ y) {
  const long idx = ((long)blockIdx.x * 256 + threadIdx.x) * 4;
  if (idx >= (long)T * hidden) return;
  const int t = (int)(idx / hidden), c = (int)(idx % hidden);
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < topk; ++j) {
    const int r = pos[t * topk + j];
    if (r < 0) continue;
    const float4 v = *reinterpret_cast<const float4 *>(d + (long)r * hidden + c);
    s.x += v.x;
    s.y += v.y;
    s.z += v.z;
    s.w += v.w;
  }
  if (F32OUT) {
    *reinterpret_cast<float4 *>(static_cast<float *>(y) + idx) = s;
  } else {
    __half2 o[2] = {__floats2half2_rn(s.x, s.y), __floats2half2_rn(s.z, s.w)};
    *reinterpret_cast<uint2 *>(static_cast<__half *>(y) + idx) = *reinterpret_cast<uint2 *>(o);
  }
}

}  // namespace moe
}  // namespace exl3

using namespace exl3;

cudaError_t exl3_launch_moe_remap(const int32_t *ids, int U, int E, int *counts, int *offsets, int *perm, int *pos,
                                  int *mtiles, int *n_mtiles, int max_mtiles, int *err,
                                  cudaStream_t s) {
  moe::Plan p{counts, offsets, perm, pos, reinterpret_cast<int4 *>(mtiles), n_mtiles};
  moe::remap_count_kernel<<<1, 1024, sizeof(int) * E, s>>>(ids, U, E, p, max_mtiles, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  moe::remap_place_kernel<<<(E + 7) / 8, 256, 0, s>>>(ids, U, E, p);
  return cudaGetLastError();
}

cudaError_t exl3_launch_moe_gather(const uint16_t *x, int U, int hidden, int topk, const int *perm,
                                   const int *offsets, int E, const int32_t *ids, const uint16_t *suh13,
                                   uint16_t *xg, uint16_t *xu, cudaStream_t s) {
  const long warps = (long)U * (hidden / 128) * 2;   // upper bound: all units valid
  const unsigned grid = (unsigned)((warps + 7) / 8);
  if (grid == 0) return cudaSuccess;
  moe::gather_rht_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const __half *>(x), hidden, topk, perm, offsets, E,
                                               ids, reinterpret_cast<const __half *>(suh13),
                                               reinterpret_cast<__half *>(xg), reinterpret_cast<__half *>(xu));
  return cudaGetLastError();
}

cudaError_t exl3_launch_moe_combine(const float *d, const int *pos, int T, int topk, int hidden, void *y,
                                    bool f32out, cudaStream_t s) {
  const long quads = (long)T * hidden / 4;
  const unsigned grid = (unsigned)((quads + 255) / 256);
  if (grid == 0) return cudaSuccess;
  if (f32out) moe::combine_kernel<true><<<grid, 256, 0, s>>>(d, pos, T, topk, hidden, y);
  else moe::combine_kernel<false><<<grid, 256, 0, s>>>(d, pos, T, topk, hidden, y);
  return cudaGetLastError();
}
