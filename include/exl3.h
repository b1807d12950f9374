/*
 * exl3.h -- C ABI of libexl3, the EXL3 trellis-quantized linear layer on one
 * NVIDIA GB300 (sm_103a).
 *
 * What the layer computes (sources by page title and section):
 *   - "exl3xpu" README, "Prefill: int8 linears and oneDNN fused attention":
 *     the GEMM runs in the Hadamard domain; every mul1 codebook value is
 *     bounded by 3.453125; the int8 variant has one activation scale per row
 *     (fused into the input Hadamard) and one static weight scale (fused into
 *     reconstruct), an s8 GEMM writing fp16.
 *   - "exl3xpu" README, "Layout": Hadamard in/out, GEMV, reconstruct kernels.
 *   - "exl3xpu" README, "MoE (routed experts)": the routed contribution in
 *     fp32 with the routing weight on the down-projection output; codebook
 *     ids (1 = MCG, 2 = mul1); unsupported width/codebook raises.
 *   - "Bringing EXL3 Trellis Quantization to 35B MoE on Intel Arc 140V",
 *     sections 1 and 2.A-2.D: trellis tensor [k/16, n/16, 16K]; packed expert
 *     arenas [E, nslots, k/16, n/16, 16K]; one grouped launch for gate+up
 *     (nslots = 2, shared input row) and one for down; device-side binning.
 *   - "exl3xpu" README, "Adding a model": all dims multiples of 128.
 *   - "EXL3 checkpoints on the native engine (tracker) #832": widths 1..8 per
 *     tensor; fp32-output projections.
 *
 * Format (this library's reading where the pages are silent):
 *   trellis  uint16 [k/16][n/16][16*K], tiles along n innermost.  Tile bit i
 *            is bit (i mod 16) of word i/16.  Weight p = 16*r + c of a tile
 *            (r along k, c along n) has the 16-bit state formed by stream bits
 *            p*K .. p*K+15 (LSB first), wrapping around the tile's 256*K bits.
 *   mul1     v(s) = fp16_RNE((B(s) - 510) * sigma), B(s) = sum of the bytes of
 *            (s * 0x9E3779B1) mod 2^32, sigma = 1775 * 2^-18 (= fp16 of
 *            3.453125/510).  |v| <= 3.453125, attained at s = 0.
 *   RHT      x' = 2^-3.5 * H (x . suh) per aligned 128-block, H the Sylvester
 *            Hadamard in natural order; y = (2^-3.5 * H y') . svh per block.
 *   linear   y = RHT_out( RHT_in(x . suh) @ W ) . svh, W = decoded weights.
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless stated; the caller owns every
 *     buffer.  The library allocates nothing and never synchronises the
 *     stream; every call only enqueues work on `stream` (asynchronous).
 *   - fp16 tensors are IEEE binary16 passed as uint16_t bits.
 *   - Device buffers must be 16-byte aligned; row-major, densely packed.
 *   - Return: EXL3_OK, or an error code with nothing enqueued (argument
 *     errors) or with the CUDA launch error captured (EXL3_ERR_CUDA).
 *     exl3_last_error() gives a message for the calling thread.
 *   - Workspaces: size from the matching *_workspace_size(); must be zero
 *     filled once before first use (exl3_workspace_clear); each call leaves
 *     its counters at zero again.  One workspace must not be used by calls
 *     that can run concurrently.
 */
#ifndef EXL3_H
#define EXL3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EXL3_OK 0
#define EXL3_ERR_ARG 1        /* null or misaligned pointer, bad enum value */
#define EXL3_ERR_SHAPE 2      /* k or n not a multiple of 128, M < 1, bad tile range */
#define EXL3_ERR_BITS 3       /* K outside 1..8 */
#define EXL3_ERR_CODEBOOK 4   /* codebook other than mul1: fail closed, never guess */
#define EXL3_ERR_WORKSPACE 5  /* workspace missing or too small */
#define EXL3_ERR_CUDA 6       /* a CUDA call failed; message holds the CUDA error */
#define EXL3_ERR_DEVICE 7     /* a kernel reported a violation in the error word */

typedef enum { EXL3_CB_MCG = 1, EXL3_CB_MUL1 = 2, EXL3_CB_3INST = 3 } exl3_codebook;
typedef enum { EXL3_OUT_F16 = 0, EXL3_OUT_F32 = 1 } exl3_out_dtype;

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *exl3_stream_t;

/* Message for the last failed call on this thread ("" if none). */
const char *exl3_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int exl3_version(void);

/*
 * exl3_copy_in -- copy `bytes` from pinned host memory to device memory with
 * a kernel on `stream` (no counterpart on the source pages; an addition of
 * this library for decode loops that take their inputs from the host).
 *   src   HOST memory the device can address: pinned (cudaHostAlloc,
 *         cudaMallocHost, cudaHostRegister'ed or a pinned tensor), 16-byte
 *         aligned.  dst: device memory, 16-byte aligned.  bytes: any size;
 *         0 enqueues nothing.
 *   The kernel reads src with 16-byte SM loads (over NVLink-C2C on GB300)
 *   instead of a copy-engine transfer.  It is a programmatic dependent
 *   launch: it reads src and writes dst only after the kernels ahead of it
 *   on the stream have completed, and it lets the kernel after it launch at
 *   once, so an M = 1 exl3_linear issued next with weight prefetch on
 *   streams its weights while the copy runs.
 *   Errors: EXL3_ERR_ARG for a NULL or misaligned pointer; a src the device
 *   cannot address is a device fault, as for any bad pointer.
 */
int exl3_copy_in(const void *src, void *dst, size_t bytes, exl3_stream_t stream);

/* Enqueue a zero fill of a workspace (cudaMemsetAsync; needed once before a
 * workspace is first used). */
int exl3_workspace_clear(void *workspace, size_t ws_bytes, exl3_stream_t stream);

/* Test helper: waits for `stream`, then copies the device error word of a
 * workspace to *err_out (0 = no violation recorded) and clears it. */
int exl3_check_device_error(void *workspace, size_t ws_bytes, exl3_stream_t stream, int *err_out);

/*
 * exl3_decode_tile -- dequantise ("reconstruct", "exl3xpu" README, "Layout";
 * bit-exact dequantised weights, "exl3xpu" README, "Correctness").
 *   trellis  [k/16][n/16][16*K] uint16 (whole tensor)
 *   tiles    [tk0, tk0+tk_cnt) x [tn0, tn0+tn_cnt) of the tile grid
 *   w_out    fp16 bits; weight (16*tk + r, 16*tn + c) of the requested range
 *            is written to w_out[(16*(tk-tk0) + r) * ld + 16*(tn-tn0) + c],
 *            ld >= 16*tn_cnt elements, ld a multiple of 8.
 *   Only k, n multiples of 16 are required here.  No workspace.
 */
int exl3_decode_tile(const uint16_t *trellis, int k, int n, int K, int codebook,
                     int tk0, int tk_cnt, int tn0, int tn_cnt,
                     uint16_t *w_out, int64_t ld, exl3_stream_t stream);

/*
 * exl3_input_rht -- the input transform alone (the "Hadamard in" kernel of
 * "exl3xpu" README, "Layout"): x' = 2^-3.5 H (x . suh) per 128-block.
 *   x [M][k] fp16, suh [k] fp16; out [M][k] as fp32 (out_dtype = EXL3_OUT_F32)
 *   or fp16 (EXL3_OUT_F16).  fp32 results are bit-identical to the stated
 *   butterfly order (stages 1, 2, ..., 64 of (a+b, a-b), then one multiply by
 *   fp32(2^-3.5)).
 */
int exl3_input_rht(const uint16_t *x, int M, int k, const uint16_t *suh,
                   void *out, int out_dtype, exl3_stream_t stream);

/*
 * exl3_linear -- y = RHT_out( RHT_in(x . suh) @ W ) . svh
 * ("exl3xpu" README, "Prefill: int8 linears..." and "Layout"; fp32 outputs
 * as the tracker #832 "decodeF32/promptF32" projections).
 *   x        [M][k] fp16          trellis [k/16][n/16][16K] uint16
 *   suh [k], svh [n] fp16         K in 1..8, codebook = EXL3_CB_MUL1
 *   y        [M][n], fp16 (EXL3_OUT_F16) or fp32 (EXL3_OUT_F32)
 *   workspace of exl3_linear_workspace_size(M, k, n, K) bytes.
 *   M = 1 runs the fused CUDA-core GEMV (or, for a k whose fp32 x' does not
 *   fit beside two stages of its ring, k > 23680 at K = 7 and k > 37248 at
 *   K = 4, the small-M tensor-core path); larger M runs the tensor-core
 *   paths.
 *   At M = 1, y may instead be pinned HOST memory the device can address
 *   (16-byte aligned): every M = 1 path writes y with plain stores, so the
 *   result lands in host memory (over NVLink-C2C on GB300) when the call's
 *   kernels complete, with no device-to-host copy.  x must stay in device
 *   memory (every CTA of the GEMV reads all of it; exl3_copy_in brings it
 *   over).
 */
size_t exl3_linear_workspace_size(int M, int k, int n, int K);
int exl3_linear(const uint16_t *x, int M, int k, int n,
                const uint16_t *trellis, const uint16_t *suh, const uint16_t *svh,
                int K, int codebook, void *y, int out_dtype,
                void *workspace, size_t ws_bytes, exl3_stream_t stream);

/*
 * exl3_linear_bias -- exl3_linear plus an output bias:
 *   y = RHT_out( RHT_in(x . suh) @ W ) . svh + bias
 * ("EXL3 checkpoints on the native engine (tracker) #832", "What is left": a
 * checkpoint's EXL3 group holds a bias beside trellis, suh and svh).  The
 * pages do not say where it enters; this library adds it as the bias of the
 * original linear: one fp16 value per output feature, added in fp32 after
 * svh, in the epilogue of every path (M = 1 GEMV, small-M and prefill
 * tensor-core kernels, row-invariant mode), before the output is rounded.
 *   bias [n] fp16 (device, 16-byte aligned; NULL is rejected with
 *   EXL3_ERR_ARG: use exl3_linear).  Everything else as exl3_linear, with the
 *   same workspace size.
 */
int exl3_linear_bias(const uint16_t *x, int M, int k, int n,
                     const uint16_t *trellis, const uint16_t *suh, const uint16_t *svh,
                     const uint16_t *bias, int K, int codebook, void *y, int out_dtype,
                     void *workspace, size_t ws_bytes, exl3_stream_t stream);

/*
 * exl3_linear_shards -- several linears over one input in one call: the
 * fused shards of a layer ("exl3xpu" README, "Layout": the vLLM linear
 * method handles fused shards), such as gate and up, or q, k and v when they
 * have one width and shape.  The pages do not describe the fusion; here the
 * shards keep their own suh and svh:
 *   y[s] = RHT_out( RHT_in(x . suh[s]) @ W[s] ) . svh[s]   for s < nshards
 *   x        [M][k] fp16
 *   trellis  [nshards][k/16][n/16][16K] uint16 (the shards stacked)
 *   suh      [nshards][k] fp16, svh [nshards][n] fp16
 *   y        [nshards][M][n], fp16 (EXL3_OUT_F16) or fp32 (EXL3_OUT_F32):
 *            shard-major, so at M = 1 the shards' outputs lie side by side
 *   nshards  1..64; K, codebook as for exl3_linear
 *   workspace of exl3_linear_shards_workspace_size(M, k, n, K, nshards) bytes.
 * At M = 1 all shards run in one launch of the CUDA-core GEMV (each CTA
 * takes an equal share of all shards' tile rows), unless a CTA's share would
 * span more than four shards or the row-invariant mode is on; otherwise, and
 * for M > 1, each shard runs as exl3_linear into its block of y.  Results
 * are within the library's tolerance of exl3_linear on each shard; the
 * one-launch GEMV splits the sums differently, so bits may differ.
 */
size_t exl3_linear_shards_workspace_size(int M, int k, int n, int K, int nshards);
int exl3_linear_shards(const uint16_t *x, int M, int k, int n, int nshards,
                       const uint16_t *trellis, const uint16_t *suh, const uint16_t *svh,
                       int K, int codebook, void *y, int out_dtype,
                       void *workspace, size_t ws_bytes, exl3_stream_t stream);

/*
 * exl3_linear_shards_var -- fused shards of different widths over one input,
 * such as q, k and v under grouped-query attention.  Same computation as
 * exl3_linear_shards, with shard s of width n[s]:
 *   n        HOST array of nshards widths (multiples of 128), read during
 *            the call only; nshards 1..64
 *   trellis  shard s as its own [k/16][n[s]/16][16K] tensor, right after
 *            shard s-1's (every shard starts on a 16-byte boundary)
 *   suh      [nshards][k] fp16; svh the shards' svh side by side [sum n]
 *   y        shard-major: shard s is an [M][n[s]] block starting at element
 *            M * (n[0] + ... + n[s-1]); at M = 1 the outputs side by side
 *   workspace of exl3_linear_shards_var_workspace_size(M, k, nshards, n, K).
 * At M = 1, for up to 8 shards whose CTA shares each span at most four
 * shards, one launch of the CUDA-core GEMV with a trellis map per shard;
 * otherwise (and in row-invariant mode) one exl3_linear per shard.
 */
size_t exl3_linear_shards_var_workspace_size(int M, int k, int nshards, const int *n, int K);
int exl3_linear_shards_var(const uint16_t *x, int M, int k, int nshards, const int *n,
                           const uint16_t *trellis, const uint16_t *suh, const uint16_t *svh,
                           int K, int codebook, void *y, int out_dtype,
                           void *workspace, size_t ws_bytes, exl3_stream_t stream);

/*
 * exl3_set_weight_prefetch -- let M = 1 calls of exl3_linear stream their
 * weights before the kernel launched ahead of them on the stream has
 * finished (CUDA programmatic dependent launch).  The source pages have no
 * counterpart: this is an addition of this library for decode loops, where
 * consecutive linears otherwise pay the start-up of each kernel in series.
 *   enable = 0 (the default) or 1; returns the previous setting.  Applies to
 *   calls made after it, from any host thread.
 *   When on, an M = 1 call may read trellis while earlier kernels on the
 *   stream are still running; it reads x, suh, svh and the workspace and
 *   writes y only once those kernels have completed and their writes are
 *   visible.  The caller must therefore not write a trellis buffer with
 *   kernels that can still be in flight when a call reading it is launched
 *   (write weights, then synchronise, then run the linears).
 */
int exl3_set_weight_prefetch(int enable);

/*
 * exl3_set_row_invariant -- make every row of an exl3_linear result
 * independent of the other rows in the call: y[m] has the same bits for any
 * M and any neighbouring rows ("EXL3 checkpoints on the native engine
 * (tracker) #832", opening paragraph: a row-invariant linear; "The gate":
 * rows keep one arithmetic at every row count).
 *   enable = 0 (the default) or 1; returns the previous setting.  Applies to
 *   calls made after it, from any host thread.
 *   When on, exl3_linear runs the input transform for all M rows and then the
 *   small-M tensor-core kernel with a 32-token MMA width over chunks of 32
 *   rows, for every M, so the k splits and the per-token reduction order
 *   depend on k and n only.  Up to 32 rows cost what the small-M path costs
 *   (M = 1 a little more than the GEMV); larger M costs one small-M call per
 *   32 rows, far more than the reconstruct + GEMM path at prefill sizes.
 *   exl3_linear_workspace_size covers both modes.
 *   exl3_linear_int8 is row-invariant in either mode (per-row activation
 *   scales and exact integer accumulation); exl3_linear_gemv_noalloc is not
 *   affected by this setting.
 */
int exl3_set_row_invariant(int enable);

/*
 * exl3_linear_int8 -- the int8 prefill variant ("exl3xpu" README, "Prefill:
 * int8 linears and oneDNN fused attention").
 *   a_r  = max_j |x'_rj| / 127 (fp32), x' the fp32 input transform above;
 *   q_x  = clamp(RNE(x' * (127 / max|x'_r|)), -127, 127), int8;
 *   q_w  = RNE(v * 127 / 3.453125) of each decoded weight v, int8;
 *   acc  = sum_j q_x * q_w, exact int32;
 *   y    = RHT_out(acc * a_r * weight_scale) . svh, fp16.
 *   weight_scale must be 3.453125f/127 (the static weight scale) or > 0.
 *   xq_out [M][k] int8, row_scale_out [M] fp32 and acc_out [M][n] int32 are
 *   optional (NULL to skip) copies of the intermediate results.
 */
size_t exl3_linear_int8_workspace_size(int M, int k, int n, int K);
int exl3_linear_int8(const uint16_t *x, int M, int k, int n,
                     const uint16_t *trellis, const uint16_t *suh, const uint16_t *svh,
                     int K, int codebook, float weight_scale, uint16_t *y,
                     int8_t *xq_out, float *row_scale_out, int32_t *acc_out,
                     void *workspace, size_t ws_bytes, exl3_stream_t stream);

/*
 * exl3_linear_int8_bias -- exl3_linear_int8 plus an output bias (the same
 * reading as exl3_linear_bias):
 *   y = fp16( RHT_out(acc * a_r * weight_scale) . svh + bias )
 *   bias [n] fp16 (device, 16-byte aligned; NULL is rejected with
 *   EXL3_ERR_ARG).  The intermediate results (xq_out, row_scale_out,
 *   acc_out) do not depend on the bias.
 */
int exl3_linear_int8_bias(const uint16_t *x, int M, int k, int n,
                          const uint16_t *trellis, const uint16_t *suh, const uint16_t *svh,
                          const uint16_t *bias, int K, int codebook, float weight_scale, uint16_t *y,
                          int8_t *xq_out, float *row_scale_out, int32_t *acc_out,
                          void *workspace, size_t ws_bytes, exl3_stream_t stream);

/*
 * Routed experts ("exl3xpu" README, "MoE (routed experts)"; Arc 140V MoE
 * post, sections 2.A, 2.B and 2.D).
 *   One descriptor per projection kind, all E experts in contiguous arenas:
 *   w13 (nslots = 2: slot 0 gate, slot 1 up; k = hidden, n = inter) and
 *   w2 (nslots = 1; k = inter, n = hidden).  Per token t and slot s:
 *     e = topk_ids[t][s]; g = lin(x_t; gate_e); u = lin(x_t; up_e);
 *     h = SiLU(g) * u; y_t += topk_weights[t][s] * lin(h; down_e)
 *   with the routing weight applied to the down output, in fp32.  Token to
 *   expert binning happens on the device; there is no host synchronisation.
 *   Expert ids outside [0, E) are recorded in the device error word and the
 *   unit is skipped.  Expert weights are decoded from the trellis inside the
 *   two grouped tensor-core launches; the workspace holds only routing
 *   tables and per-row activations (T * topk rows of hidden and inter).
 */
typedef struct {
  const uint16_t *trellis;  /* [E][nslots][k/16][n/16][16*K] */
  const uint16_t *suh;      /* [E][nslots][k] fp16 */
  const uint16_t *svh;      /* [E][nslots][n] fp16 */
  int k, n, K, codebook, nslots;
} exl3_expert_proj;

size_t exl3_moe_workspace_size(int T, int topk, int E, const exl3_expert_proj *w13,
                               const exl3_expert_proj *w2);
int exl3_moe_grouped(const uint16_t *x, int T, int hidden,
                     const int32_t *topk_ids, const float *topk_weights, int topk, int E,
                     const exl3_expert_proj *w13, const exl3_expert_proj *w2,
                     void *y, int out_dtype,
                     void *workspace, size_t ws_bytes, exl3_stream_t stream);

/*
 * Routed experts with a width per expert ("EXL3 checkpoints on the native
 * engine (tracker) #832": widths 1..8 per tensor, and the Oct 17 comment keeps
 * each expert's own width in the format).  Same computation as exl3_moe_grouped; each
 * projection kind has one width per expert instead of one for all.
 *   trellis  one packed arena per projection kind: expert e's nslots tensors
 *            ([k/16][n/16][16*K[e]] uint16 each) follow expert e-1's, so
 *            expert e starts sum_{e' < e} nslots*(k/16)*(n/16)*16*K[e'] words
 *            in (always a multiple of 16 bytes);
 *   suh, svh [E][nslots][k], [E][nslots][n] fp16 as for exl3_moe_grouped;
 *   K        HOST array of E widths (1..8), read during the call only.
 * Each maximal run of consecutive experts with one width gets its own
 * grouped launch per projection (over that run's experts; tiles of other
 * experts are skipped), so the call costs about one launch per run on top of
 * the work: number the experts so that equal widths are consecutive (the
 * arena order is the caller's; router ids index it).  Every token count runs
 * the tile kernels (the few-token GEMV path of exl3_moe_grouped is not used).
 * Routing, invalid ids, workspace rules and the output are as for
 * exl3_moe_grouped; the workspace size comes from
 * exl3_moe_mixed_workspace_size.
 */
typedef struct {
  const uint16_t *trellis;  /* packed arena, expert e right after expert e-1 */
  const uint16_t *suh;      /* [E][nslots][k] fp16 */
  const uint16_t *svh;      /* [E][nslots][n] fp16 */
  const int32_t *K;         /* HOST [E] widths */
  int k, n, codebook, nslots;
} exl3_expert_proj_mixed;

size_t exl3_moe_mixed_workspace_size(int T, int topk, int E, const exl3_expert_proj_mixed *w13,
                                     const exl3_expert_proj_mixed *w2);
int exl3_moe_grouped_mixed(const uint16_t *x, int T, int hidden,
                           const int32_t *topk_ids, const float *topk_weights, int topk, int E,
                           const exl3_expert_proj_mixed *w13, const exl3_expert_proj_mixed *w2,
                           void *y, int out_dtype,
                           void *workspace, size_t ws_bytes, exl3_stream_t stream);

/*
 * exl3_linear_gemv_noalloc -- the M = 1 linear (the same fused GEMV, with
 * the same result, as exl3_linear with M = 1) for callers that cannot
 * allocate device memory.  The source pages have no counterpart: this is an
 * addition of this library.
 *   Who needs it: plugin hosts whose framework owns the device memory pool
 *   and does not let a library call cudaMalloc, and latency-critical decode
 *   loops that reserve all memory at start-up (cudaMalloc can synchronise the
 *   device).  They pass only inputs and outputs; no workspace.
 *   x [k] fp16 (one row), trellis [k/16][n/16][16K], suh [k], svh [n] fp16,
 *   y [n] fp16 (EXL3_OUT_F16) or fp32 (EXL3_OUT_F32); K, codebook as above.
 *   Scratch: one fixed 2 MiB array of library device memory per GPU that
 *   loads the library, held until the process exits.  A shape whose k-split
 *   partial sums do not fit, or whose k is too large for the GEMV (see
 *   exl3_linear), is rejected with EXL3_ERR_SHAPE (use exl3_linear with a
 *   workspace instead).  The first call on a device looks up the
 *   array's device address (cudaGetSymbolAddress) with that device current;
 *   make that first call before any stream capture.  Each call enqueues two
 *   kernels: a one-CTA kernel that clears the parts of the array that must
 *   start at zero, and the GEMV as its programmatic dependent (it streams
 *   its weights while the clear runs; the clear waits for all earlier work
 *   on the stream).  All calls share the array:
 *   calls that can overlap on the GPU (other streams, other host threads)
 *   race with each other.  No cudaMalloc or cudaFree is ever called.
 */
int exl3_linear_gemv_noalloc(const uint16_t *x, int k, int n, const uint16_t *trellis,
                             const uint16_t *suh, const uint16_t *svh, int K, int codebook,
                             void *y, int out_dtype, exl3_stream_t stream);

/*
 * exl3_noalloc_device_error -- the device error word of the fixed scratch
 * array that exl3_linear_gemv_noalloc uses on the current device (no
 * counterpart on the source pages; a companion of that entry point).
 *   Waits for `stream` (cudaStreamSynchronize), copies the word to
 *   *err_out with a plain cudaMemcpy and clears it; allocates nothing.
 *   Each call clears the word first, so nonzero means the most recent call
 *   on this device hit a device-side check (a bounded wait that ran out, an
 *   index out of range): that call's y is incomplete.  The bits are those of exl3_check_device_error.  Returns
 *   EXL3_ERR_ARG for a NULL err_out, EXL3_ERR_CUDA if a CUDA call fails.
 */
int exl3_noalloc_device_error(exl3_stream_t stream, int *err_out);

#ifdef __cplusplus
}
#endif

#endif /* EXL3_H */
