// copy_in.cu -- a decode step's activations from pinned host memory to the
// device, copied by SM loads instead of a copy-engine transfer.
//
// On GB300 the GPU addresses pinned host memory directly over NVLink-C2C.  A
// copy-engine transfer of a few kilobytes costs several microseconds of
// latency and, inside a chain of programmatic dependent launches, breaks the
// chain: the next linear cannot start streaming its weights until the copy
// is done.  This kernel keeps the chain: it lets the next kernel launch at
// once, waits for the kernels ahead of it to complete (so it never
// overwrites an input they still read, and reads a source they may have
// written), then copies with 16-byte loads, four per thread in flight.
#include "exl3_common.cuh"

namespace {

constexpr int kCopyThreads = 128;
constexpr int kCopyPerThread = 4;   // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kCopyThreads) copy_in_kernel(const uint4 *__restrict__ src,
                                                               uint4 *__restrict__ dst, size_t n16,
                                                               const unsigned char *__restrict__ src_tail,
                                                               unsigned char *__restrict__ dst_tail, int tail) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const size_t stride = (size_t)gridDim.x * kCopyThreads * kCopyPerThread;
  for (size_t base = (size_t)blockIdx.x * kCopyThreads * kCopyPerThread + threadIdx.x; base < n16;
       base += stride) {
    uint4 v[kCopyPerThread];
#pragma unroll
    for (int j = 0; j < kCopyPerThread; ++j) {
      const size_t i = base + (size_t)j * kCopyThreads;
      if (i < n16) v[j] = src[i];
    }
#pragma unroll
    for (int j = 0; j < kCopyPerThread; ++j) {
      const size_t i = base + (size_t)j * kCopyThreads;
      if (i < n16) dst[i] = v[j];
    }
  }
  if (blockIdx.x == 0 && (int)threadIdx.x < tail) dst_tail[threadIdx.x] = src_tail[threadIdx.x];
}

}  // namespace

cudaError_t exl3_launch_copy_in(const void *src, void *dst, size_t bytes, cudaStream_t s, bool chained) {
  const size_t n16 = bytes / 16;
  const int tail = (int)(bytes % 16);
  const size_t per_cta = (size_t)kCopyThreads * kCopyPerThread;
  size_t grid = (n16 + per_cta - 1) / per_cta;
  const size_t cap = (size_t)4 * exl3_sm_count();
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kCopyThreads);
  cfg.stream = s;
  cfg.attrs = chained ? attrs : nullptr;
  cfg.numAttrs = chained ? 1 : 0;
  const unsigned char *sb = static_cast<const unsigned char *>(src);
  unsigned char *db = static_cast<unsigned char *>(dst);
  return cudaLaunchKernelEx(&cfg, copy_in_kernel, reinterpret_cast<const uint4 *>(src), reinterpret_cast<uint4 *>(dst),
                            n16, sb + n16 * 16, db + n16 * 16, tail);
}
