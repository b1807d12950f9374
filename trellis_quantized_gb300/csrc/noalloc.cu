// noalloc.cu -- the M = 1 linear for callers that cannot allocate device
// memory.
//
// Some callers of this library are not allowed to call cudaMalloc: plugin
// hosts whose framework owns the device memory pool, and latency-critical
// decode loops that reserve every byte at start-up (cudaMalloc can
// synchronise the device and take milliseconds).  exl3_linear_gemv_noalloc
// serves them: the same fused GEMV as exl3_linear with M = 1, but its scratch
// (the device error word, the arrival counters and the k-split partial sums)
// lives in one fixed array that belongs to the library, so the caller passes
// only inputs and outputs.
//
// The array is kNoAllocScratchBytes (2 MiB) of device memory on every GPU
// that loads the library, held until the process exits.  A call first
// clears the error word and the arrival counters it uses with a one-CTA
// kernel and launches the GEMV as its programmatic dependent, so the GEMV
// streams its weights while the clear runs (the clear itself waits for all
// earlier work on the stream) and touches the scratch only after the clear
// has completed.  In host code its
// name is only a host-side stand-in, not a device address, so the first call
// on each device (with that device current) looks the address up with
// cudaGetSymbolAddress and caches it; that first call should come before any
// stream capture.  All calls share the array and it keeps the last call's
// contents: each call clears the error word and the counters it uses, and
// calls that overlap on the GPU (different streams, or several host threads)
// race on it.  exl3_noalloc_device_error reads (and clears) the error word,
// which a call sets when one of its bounded waits runs out or an index check
// fails; such a call's y is incomplete.
#include <mutex>

#include "exl3_common.cuh"

cudaError_t exl3_launch_gemv_m1(const uint16_t *x, const uint16_t *trellis, const uint16_t *suh,
                                const uint16_t *svh, int k, int n, int K, void *y, bool f32out,
                                float *partials, int *counters, int *err, int grid, cudaStream_t s,
                                bool prefetch = false);
int exl3_gemv_cta_cols(int K);
void exl3_gemv_plan(int k, int n, int K, int *grid, size_t *partial_floats);
bool exl3_gemv_fits(int k, int n, int K);

namespace {

constexpr size_t kNoAllocScratchBytes = 2u << 20;   // the stated maximum
constexpr size_t kCtrl = 256;                        // error word
constexpr size_t kCounterBytes = 8192 * sizeof(int); // up to n / 128 = 8192 column blocks
constexpr size_t kPartialsOff = kCtrl + kCounterBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};
// Device address of the scratch array on the current device (looked up once).
int scratch_for_current_device(void **ptr) {
  int dev = 0;
  int rc = exl3_cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= kMaxDevices) return exl3_fail(EXL3_ERR_ARG, "device ordinal %d not supported", dev);
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    rc = exl3_cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress(scratch)");
    if (rc) return rc;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return EXL3_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

__global__ void __launch_bounds__(256) clear_words_kernel(int *words, int n) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = threadIdx.x; i < n; i += blockDim.x) words[i] = 0;
}

}  // namespace

extern "C" int exl3_linear_gemv_noalloc(const uint16_t *x, int k, int n, const uint16_t *trellis,
                                        const uint16_t *suh, const uint16_t *svh, int K, int codebook, void *y,
                                        int out_dtype, exl3_stream_t stream) {
  const void *ptrs[] = {x, trellis, suh, svh, y};
  const char *names[] = {"x", "trellis", "suh", "svh", "y"};
  for (int i = 0; i < 5; ++i) {
    if (!ptrs[i]) return exl3_fail(EXL3_ERR_ARG, "%s is NULL", names[i]);
    if (!aligned16(ptrs[i])) return exl3_fail(EXL3_ERR_ARG, "%s is not 16-byte aligned", names[i]);
  }
  if (codebook != EXL3_CB_MUL1)
    return exl3_fail(EXL3_ERR_CODEBOOK, "codebook %d is not implemented (only mul1 = %d); refusing rather than guessing",
                     codebook, EXL3_CB_MUL1);
  if (K < 1 || K > 8) return exl3_fail(EXL3_ERR_BITS, "K = %d outside 1..8", K);
  if (k <= 0 || n <= 0 || k % 128 || n % 128)
    return exl3_fail(EXL3_ERR_SHAPE, "k = %d and n = %d must be positive multiples of 128", k, n);
  if (out_dtype != EXL3_OUT_F16 && out_dtype != EXL3_OUT_F32)
    return exl3_fail(EXL3_ERR_ARG, "out_dtype %d invalid", out_dtype);

  if (k > 49152 || !exl3_gemv_fits(k, n, K))
    return exl3_fail(EXL3_ERR_SHAPE, "k = %d, n = %d too large for the M = 1 GEMV at K = %d", k, n, K);
  void *scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;

  int grid = 0;
  size_t partial_floats = 0;
  exl3_gemv_plan(k, n, K, &grid, &partial_floats);
  const size_t colblocks = (size_t)((n + exl3_gemv_cta_cols(K) - 1) / exl3_gemv_cta_cols(K));
  const size_t need = kPartialsOff + sizeof(float) * partial_floats;
  if (colblocks * sizeof(int) > kCounterBytes || need > kNoAllocScratchBytes)
    return exl3_fail(EXL3_ERR_SHAPE,
                     "k = %d, n = %d needs %zu bytes of the fixed scratch; its limit is %zu bytes "
                     "(use exl3_linear with a caller workspace)",
                     k, n, need, kNoAllocScratchBytes);

  char *base = static_cast<char *>(scratch);
  int *err = reinterpret_cast<int *>(base);
  int *counters = reinterpret_cast<int *>(base + kCtrl);
  float *partials = reinterpret_cast<float *>(base + kPartialsOff);
  // The error word and the counters must start at zero; a previous call that
  // did not finish cleanly could have left them set.
  clear_words_kernel<<<1, 256, 0, stream>>>(reinterpret_cast<int *>(base),
                                            (int)((kCtrl + colblocks * sizeof(int)) / sizeof(int)));
  rc = exl3_cuda_check(cudaGetLastError(), "clear scratch");
  if (rc) return rc;
  return exl3_cuda_check(exl3_launch_gemv_m1(x, trellis, suh, svh, k, n, K, y, out_dtype == EXL3_OUT_F32,
                                             partials, counters, err, grid, stream, /*prefetch=*/true),
                         "gemv launch");
}

extern "C" int exl3_noalloc_device_error(exl3_stream_t stream, int *err_out) {
  if (!err_out) return exl3_fail(EXL3_ERR_ARG, "err_out is NULL");
  void *scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  rc = exl3_cuda_check(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
  if (rc) return rc;
  int v = 0;
  rc = exl3_cuda_check(cudaMemcpy(&v, scratch, sizeof v, cudaMemcpyDeviceToHost), "read the error word");
  if (rc) return rc;
  rc = exl3_cuda_check(cudaMemset(scratch, 0, sizeof v), "clear the error word");
  if (rc) return rc;
  *err_out = v;
  return EXL3_OK;
}
