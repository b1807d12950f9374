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
  int4 *mtiles;     // [max_mtiles]: (expert, first row, rows, 0) per tile of at most `cap` rows
  int *n_mtiles;    // [1]
  int *chunk;       // [nchunks][E]: units of each expert per chunk, then the
                    // expert's rows before the chunk (exclusive scan over chunks)
};

// Units are binned in chunks of 32 W consecutive units (one CTA, W warps);
// W is chosen on the host so that a [W][E] int table fits 32 KB.
__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// (1) per-chunk histogram.  Lanes holding the same expert id elect one
// leader, which adds the group size: one shared atomic per distinct id per
// warp.  Invalid ids are reported, their unit gets pos = -1.
__global__ void remap_hist_kernel(const int32_t *__restrict__ ids, int U, int E, Plan p, int *err) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int hist[];   // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  const int id = u < U ? ids[u] : -1;
  const bool valid = id >= 0 && id < E;
  if (u < U && !valid) {
    set_device_error(err, kErrExpertId);
    p.pos[u] = -1;
  }
  const unsigned peers = __match_any_sync(0xffffffffu, valid ? id : -1);
  if (valid && (peers & lanemask_lt()) == 0) atomicAdd(&hist[id], __popc(peers));
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) p.chunk[(long)blockIdx.x * E + e] = hist[e];
}

// Block-wide exclusive scan of one int per thread (1024 threads); returns
// the prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sums[w] = incl;
  __syncthreads();
  if (w == 0) {
    int ws = warp_sums[lane];
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    warp_sums[lane] = wi - ws;   // exclusive prefix of the warps
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int r = warp_sums[w] + incl - v;
  __syncthreads();   // warp_sums may be reused by the caller
  return r;
}

// (2) one CTA of 1024 threads, thread e = expert e (E <= 1024): per-chunk
// counts become the expert's rows before each chunk; counts, offsets and the
// tile list (tiles of at most cap rows) follow from two
// block scans.
__global__ void __launch_bounds__(1024) remap_scan_kernel(int E, int nchunks, Plan p, int max_mtiles, int cap,
                                                          int *err) {
  pdl_trigger();
  pdl_wait();
  __shared__ int warp_sums[32];
  __shared__ int total;
  const int e = threadIdx.x;
  int c = 0;
  if (e < E) {
    int *col = p.chunk + e;
    int ch = 0;
    for (; ch + 8 <= nchunks; ch += 8) {
      int v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = col[(long)(ch + j) * E];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        col[(long)(ch + j) * E] = c;
        c += v[j];
      }
    }
    for (; ch < nchunks; ++ch) {
      const int v = col[(long)ch * E];
      col[(long)ch * E] = c;
      c += v;
    }
    p.counts[e] = c;
  }
  const int off = block_exclusive_scan(c, warp_sums, &total);
  if (e < E) p.offsets[e] = off;
  if (e == 0) p.offsets[E] = total;
  const int nt = (c + cap - 1) / cap;
  const int tb = block_exclusive_scan(nt, warp_sums, &total);
  for (int j = 0; j < nt; ++j)
    if (tb + j < max_mtiles) p.mtiles[tb + j] = make_int4(e, off + cap * j, min(cap, c - cap * j), 0);
  if (e == 0) {
    if (total > max_mtiles) set_device_error(err, kErrBounds);
    *p.n_mtiles = min(total, max_mtiles);
  }
}

// (3) stable placement: the unit's row is offsets[e] + (rows of e before the
// chunk) + (units of e in earlier warps of the chunk) + (earlier lanes of
// the same warp with e), so rows of an expert follow unit order.
__global__ void remap_place_kernel(const int32_t *__restrict__ ids, int U, int E, Plan p) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int wc[];   // [W][E]
  const int W = blockDim.x >> 5, w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < W * E; i += blockDim.x) wc[i] = 0;
  __syncthreads();
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  const int id = u < U ? ids[u] : -1;
  const bool valid = id >= 0 && id < E;
  const unsigned peers = __match_any_sync(0xffffffffu, valid ? id : -1);
  const unsigned lt = lanemask_lt();
  if (valid && (peers & lt) == 0) wc[w * E + id] = __popc(peers);
  __syncthreads();
  if (!valid) return;
  int r = p.offsets[id] + p.chunk[(long)blockIdx.x * E + id] + __popc(peers & lt);
  for (int j = 0; j < w; ++j) r += wc[j * E + id];
  p.perm[r] = u;
  p.pos[u] = r;
}

// Few units (U <= 1024, E <= 256): the three steps above in one CTA of 1024
// threads, thread u = unit u, with the per-warp counts [32][E] in shared
// memory (the same stable order: expert, then unit).
constexpr int kSmallU = 1024, kSmallE = 256;

__global__ void __launch_bounds__(1024) remap_small_kernel(const int32_t *__restrict__ ids, int U, int E, Plan p,
                                                           int max_mtiles, int cap, int *err) {
  __shared__ int wc[32][kSmallE];
  __shared__ int base[kSmallE];
  __shared__ int warp_sums[32];
  __shared__ int total;
  pdl_trigger();
  pdl_wait();
  const int t = threadIdx.x, w = t >> 5;
  for (int i = t; i < 32 * kSmallE; i += 1024) (&wc[0][0])[i] = 0;
  __syncthreads();
  const int id = t < U ? ids[t] : -1;
  const bool valid = id >= 0 && id < E;
  if (t < U && !valid) {
    set_device_error(err, kErrExpertId);
    p.pos[t] = -1;
  }
  const unsigned peers = __match_any_sync(0xffffffffu, valid ? id : -1);
  const unsigned lt = lanemask_lt();
  if (valid && (peers & lt) == 0) wc[w][id] = __popc(peers);
  __syncthreads();
  // thread e: the expert's units per warp become the units of earlier warps
  int c = 0;
  if (t < E) {
    for (int j = 0; j < 32; ++j) {
      const int v = wc[j][t];
      wc[j][t] = c;
      c += v;
    }
    p.counts[t] = c;
  }
  const int off = block_exclusive_scan(c, warp_sums, &total);
  if (t < E) {
    p.offsets[t] = off;
    base[t] = off;
  }
  if (t == 0) p.offsets[E] = total;
  const int nt = (c + cap - 1) / cap;
  const int tb = block_exclusive_scan(nt, warp_sums, &total);
  for (int j = 0; j < nt; ++j)
    if (tb + j < max_mtiles) p.mtiles[tb + j] = make_int4(t, off + cap * j, min(cap, c - cap * j), 0);
  if (t == 0) {
    if (total > max_mtiles) set_device_error(err, kErrBounds);
    *p.n_mtiles = min(total, max_mtiles);
  }
  __syncthreads();
  if (valid) {
    const int r = base[id] + wc[w][id] + __popc(peers & lt);
    p.perm[r] = t;
    p.pos[t] = r;
  }
}

// Sorted rows of the transformed token inputs for gate and up:
// xg[i] = RHT(x_t . suh_gate[e]), xu[i] = RHT(x_t . suh_up[e]), t = perm[i] / topk.
// One warp per sorted row: the row's unit and expert are looked up once, and
// the row's 512-element chunks follow one another with the loads of chunk
// c + 1 issued before chunk c is transformed.  Lane l loads 16 contiguous
// elements of a chunk, its two halves swapped on odd lanes, for fwht128_xh,
// and stores the two 8-element runs that the transform leaves it.
struct GatherIn {
  uint4 x[2], g[2], u[2];
};

// half q of the lane's 16 elements comes from col + 8 (q ^ sw)
__device__ __forceinline__ void gather_load(GatherIn &in, const __half *xr, const __half *sg, const __half *su,
                                            int col, int sw, bool live) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int c = col + 8 * (q ^ sw);
    in.x[q] = live ? *reinterpret_cast<const uint4 *>(xr + c) : make_uint4(0u, 0u, 0u, 0u);
    in.g[q] = live ? __ldg(reinterpret_cast<const uint4 *>(sg + c)) : make_uint4(0u, 0u, 0u, 0u);
    in.u[q] = live ? __ldg(reinterpret_cast<const uint4 *>(su + c)) : make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void __launch_bounds__(256) gather_rht_kernel(const __half *__restrict__ x, int hidden, int topk,
                                                         const int *__restrict__ perm,
                                                         const int *__restrict__ offsets, int E,
                                                         const int32_t *__restrict__ ids,
                                                         const __half *__restrict__ suh13,  // [E][2][hidden]
                                                         __half *__restrict__ xg, __half *__restrict__ xu) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long i = (long)blockIdx.x * 8 + (threadIdx.x >> 5);   // sorted row
  if (i >= offsets[E]) return;                                // uniform per warp
  const int u = perm[i];
  const int t = u / topk, e = ids[u];
  const __half *xr = x + (long)t * hidden;
  const __half *sg = suh13 + (long)e * 2 * hidden, *su = sg + hidden;
  __half *dg = xg + i * hidden, *du = xu + i * hidden;
  const int chunks = (hidden + 511) / 512;
  const int sw = lane & 1;
  float slo, shi;
  fwht128_xh_signs(lane, slo, shi);
  const float2 klo = make_float2(slo * kRhtScale, slo * kRhtScale);   // the output scale with the sign factors
  const float2 khi = make_float2(shi * kRhtScale, shi * kRhtScale);
  const int olo = 128 * (lane >> 3) + 8 * (lane & 7);   // the lane's output runs in a chunk: olo, olo + 64
  GatherIn cur, nxt;
  gather_load(cur, xr, sg, su, 16 * lane, sw, 16 * lane < hidden);
#pragma unroll 1
  for (int c = 0; c < chunks; ++c) {
    const int col = c * 512 + 16 * lane;
    const bool in = col < hidden;      // whole 128-blocks are in or out (hidden % 128 == 0)
    if (c + 1 < chunks) gather_load(nxt, xr, sg, su, col + 512, sw, col + 512 < hidden);
    const uint32_t *xw = reinterpret_cast<const uint32_t *>(cur.x);
    const uint32_t *gw = reinterpret_cast<const uint32_t *>(cur.g);
    const uint32_t *uw = reinterpret_cast<const uint32_t *>(cur.u);
    float2 a[8], b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      a[j] = mul_f16x2_exact(xw[j], gw[j]);
      b[j] = mul_f16x2_exact(xw[j], uw[j]);
    }
    fwht128_xh(a, lane);
    fwht128_xh(b, lane);
    if (in) {
      __align__(16) __half2 og[8], ou[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 k = j < 4 ? klo : khi;
        og[j] = __float22half2_rn(__fmul2_rn(a[j], k));
        ou[j] = __float22half2_rn(__fmul2_rn(b[j], k));
      }
      const long o = (long)c * 512 + olo;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        *reinterpret_cast<uint4 *>(dg + o + 64 * q) = reinterpret_cast<const uint4 *>(og)[q];
        *reinterpret_cast<uint4 *>(du + o + 64 * q) = reinterpret_cast<const uint4 *>(ou)[q];
      }
    }
    cur = nxt;
  }
}

template <bool F32OUT>
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ d, const int *__restrict__ pos,
                                                      int T, int topk, int hidden, void *__restrict__ y) {
  pdl_trigger();
  pdl_wait();
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

// Units per binning chunk: 32 W with W warps, the [W][E] placement table
// within 32 KB of shared memory (E <= 1024 gives W >= 8).
int exl3_moe_remap_chunk(int E) {
  const int W = E > 0 ? 8192 / E : 32;
  return 32 * (W > 32 ? 32 : W);
}

// chunk_tab: [ceil(U / exl3_moe_remap_chunk(E))][E] ints of workspace.
// cap: rows per tile (32, 128, 160 or 256) of the tile list the grouped kernels read.
cudaError_t exl3_launch_moe_remap(const int32_t *ids, int U, int E, int *counts, int *offsets, int *perm, int *pos,
                                  int *mtiles, int *n_mtiles, int max_mtiles, int cap, int *chunk_tab, int *err,
                                  cudaStream_t s) {
  if (E < 1 || E > 1024 || (cap != 32 && cap != 128 && cap != 160 && cap != 256)) return cudaErrorInvalidValue;
  moe::Plan p{counts, offsets, perm, pos, reinterpret_cast<int4 *>(mtiles), n_mtiles, chunk_tab};
  if (U <= moe::kSmallU && E <= moe::kSmallE) {
    return launch_pdl(moe::remap_small_kernel, dim3(1), dim3(1024), 0, s, ids, U, E, p, max_mtiles, cap, err);
  }
  const int CH = exl3_moe_remap_chunk(E);
  const int nchunks = (U + CH - 1) / CH;
  if (nchunks > 0) {
    cudaError_t e = launch_pdl(moe::remap_hist_kernel, dim3(nchunks), dim3(CH), sizeof(int) * E, s, ids, U, E, p, err);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_pdl(moe::remap_scan_kernel, dim3(1), dim3(1024), 0, s, E, nchunks, p, max_mtiles, cap, err);
  if (e != cudaSuccess || nchunks == 0) return e;
  return launch_pdl(moe::remap_place_kernel, dim3(nchunks), dim3(CH), sizeof(int) * (CH / 32) * E, s, ids, U, E, p);
}

cudaError_t exl3_launch_moe_gather(const uint16_t *x, int U, int hidden, int topk, const int *perm,
                                   const int *offsets, int E, const int32_t *ids, const uint16_t *suh13,
                                   uint16_t *xg, uint16_t *xu, cudaStream_t s) {
  const unsigned grid = (unsigned)(((long)U + 7) / 8);       // one warp per sorted row; rows <= U
  if (grid == 0) return cudaSuccess;
  return launch_pdl(moe::gather_rht_kernel, dim3(grid), dim3(256), 0, s, reinterpret_cast<const __half *>(x), hidden,
                    topk, perm, offsets, E, ids, reinterpret_cast<const __half *>(suh13),
                    reinterpret_cast<__half *>(xg), reinterpret_cast<__half *>(xu));
}

cudaError_t exl3_launch_moe_combine(const float *d, const int *pos, int T, int topk, int hidden, void *y,
                                    bool f32out, cudaStream_t s) {
  const long quads = (long)T * hidden / 4;
  const unsigned grid = (unsigned)((quads + 255) / 256);
  if (grid == 0) return cudaSuccess;
  if (f32out) return launch_pdl(moe::combine_kernel<true>, dim3(grid), dim3(256), 0, s, d, pos, T, topk, hidden, y);
  return launch_pdl(moe::combine_kernel<false>, dim3(grid), dim3(256), 0, s, d, pos, T, topk, hidden, y);
}
