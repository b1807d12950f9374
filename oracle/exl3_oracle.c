/*
 * exl3_oracle.c -- plain scalar CPU oracle for the EXL3 trellis-quantized linear.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product library never links, calls or falls back to it.  It shares no code,
 * header, table or constant generator with the CUDA sources.
 *
 * All floating arithmetic is IEEE binary64 unless a step is defined in
 * binary32 (the int8 activation path, whose fp32 butterfly order is part of
 * the definition).  Integer work (trellis states, codebook hash, int8
 * accumulators) is exact.  Build with -ffp-contract=off and without
 * -ffast-math so that every float operation rounds exactly once.
 *
 * Sources (page title, section):
 *   [README-int8]  "exl3xpu" README, "Prefill: int8 linears and oneDNN fused
 *                  attention": the GEMM runs in the Hadamard domain; every mul1
 *                  codebook value is bounded by 3.453125; one int8 scale per
 *                  activation row fused into the input Hadamard and one static
 *                  weight scale fused into reconstruct; s8 GEMM writes fp16.
 *   [README-moe]   "exl3xpu" README, "MoE (routed experts)": only the routed
 *                  contribution, in fp32, with the routing weight applied to
 *                  the down-projection output, never to the input; mul1 is
 *                  codebook id 2, MCG id 1.
 *   [README-layout] "exl3xpu" README, "Layout": Hadamard in/out kernels,
 *                  reconstruct, dp4a GEMV.
 *   [README-model] "exl3xpu" README, "Adding a model": linear dims are
 *                  multiples of 128.
 *   [ARC-1]        "Bringing EXL3 Trellis Quantization to 35B MoE on Intel Arc
 *                  140V", section 1: randomized Hadamard transforms and trellis
 *                  codebook decoding; trellis tensor [k/16, n/16, 16K].
 *   [ARC-2B]       same post, section 2.B: gate+up share one input row
 *                  (nslots=2), down has nslots=1, SiLU on device.
 *   [TF-832]       "EXL3 checkpoints on the native engine (tracker) #832":
 *                  widths 1..8 per tensor; trellis, suh/su, svh/sv groups.
 *
 * Where the pages are silent this file takes one plain reading, stated at the
 * step (bit order, window direction, intra-tile order, the mul1 multiplier and
 * scale, Hadamard order and normalisation, int8 rounding).  Parity with real
 * EXL3 checkpoints is unpinned: no checkpoint or decoder source is available.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_SHAPE 2
#define OR_ERR_BITS 3
#define OR_ERR_OVERFLOW 8

/* ------------------------------------------------------------------------- */
/* IEEE binary16 <-> binary64, written from the format definition.           */
/* ------------------------------------------------------------------------- */

/* binary16 bits -> exact double. */
double or_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* double -> binary16 bits, round to nearest, ties to even (one rounding). */
uint16_t or_f64_to_f16(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double a = fabs(x);
  if (isnan(x)) return 0x7e00u;
  if (a >= 65520.0) return sign | 0x7c00u;     /* at or past the midpoint to 2^16 */
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: quantum 2^-24; scaling by a power of two is exact */
    double q = nearbyint(ldexp(a, 24));        /* default mode: ties to even */
    return sign | (uint16_t)q;                 /* q == 1024 is the smallest normal */
  }
  int e;
  double m = frexp(a, &e);                     /* a = m * 2^e, m in [0.5, 1) */
  double q = nearbyint(ldexp(m, 11));          /* 11 significant bits */
  if (q == 2048.0) { q = 1024.0; e += 1; }
  int E = e - 1 + 15;
  if (E >= 31) return sign | 0x7c00u;
  return sign | (uint16_t)(E << 10) | (uint16_t)(q - 1024.0);
}

/* ------------------------------------------------------------------------- */
/* mul1 computed codebook ([README-int8], [README-moe]; constants chosen here) */
/* ------------------------------------------------------------------------- */

/*
 * Reading: "mul1" is one 32-bit multiply of the 16-bit state whose four bytes
 * are summed (the byte sum the "dp4a GEMV" of [README-layout] suggests):
 *   B(s) = sum of the four bytes of (s * OR_MUL1) mod 2^32,  B in [0, 1020]
 *   v(s) = fp16_RNE( (B(s) - 510) * sigma ),  sigma = fp16_RNE(3.453125 / 510)
 * 510 is the mean of B.  The multiplier is not printed on the pages; this
 * library uses Knuth's golden-ratio multiplicative-hash constant.  State 0
 * gives B = 0, so v(0) = fp16(-510 * sigma) = -3.453125 for any multiplier:
 * the bound [README-int8] prints is attained, and it fixes sigma to the fp16
 * value nearest 3.453125/510 (= 1775 * 2^-18).
 */
#define OR_MUL1 0x9E3779B1u

uint32_t or_mul1_bytesum(uint32_t state) {
  uint32_t p = (uint32_t)((uint64_t)(state & 0xFFFFu) * (uint64_t)OR_MUL1);  /* mod 2^32 */
  return (p & 255u) + ((p >> 8) & 255u) + ((p >> 16) & 255u) + ((p >> 24) & 255u);
}

double or_mul1_sigma(void) {
  return or_f16_to_f64(or_f64_to_f16(3.453125 / 510.0));
}

uint16_t or_mul1_value(uint32_t state) {
  double b = (double)or_mul1_bytesum(state);
  return or_f64_to_f16((b - 510.0) * or_mul1_sigma());
}

/* ------------------------------------------------------------------------- */
/* Bitshift trellis ([ARC-1]: tensor [k/16, n/16, 16K]; [TF-832]: K = 1..8)    */
/* ------------------------------------------------------------------------- */

/*
 * Readings (the pages fix the tensor shape only):
 *  - Tile (tk, tn) is trellis[tk][tn][0 .. 16K): a bitstream of L = 256K bits.
 *    Stream bit i is bit (i mod 16) of word floor(i / 16): LSB first, words in
 *    index order.
 *  - Weight p in [0, 256) of a tile has the 16-bit state whose bit j is stream
 *    bit (p*K + j) mod L: a window starting at bit p*K that wraps around the
 *    end of the tile (tail-biting).  Consecutive states therefore overlap in
 *    16 - K bits, the shift-register property of a bitshift trellis.
 *  - p = 16*r + c is row-major: r runs along the input (k) dimension and c
 *    along the output (n) dimension, so W[16 tk + r][16 tn + c] = v(s_p).
 */
static int stream_bit(const uint16_t *words, int K, long i) {
  long L = 256L * K;
  i %= L;
  return (words[i >> 4] >> (i & 15)) & 1;
}

void or_tile_states(const uint16_t *words, int K, uint16_t *states) {
  for (int p = 0; p < 256; ++p) {
    uint32_t s = 0;
    for (int j = 0; j < 16; ++j)
      s |= (uint32_t)stream_bit(words, K, (long)p * K + j) << j;
    states[p] = (uint16_t)s;
  }
}

/* Full dequantisation: W fp16 bits, row-major [k][n] (Hadamard domain). */
int or_reconstruct(const uint16_t *trellis, int k, int n, int K, uint16_t *W) {
  if (K < 1 || K > 8) return OR_ERR_BITS;
  if (k <= 0 || n <= 0 || k % 16 || n % 16) return OR_ERR_SHAPE;
  int tiles_n = n / 16;
  long tiles = (long)(k / 16) * tiles_n;
#pragma omp parallel for schedule(static)
  for (long t = 0; t < tiles; ++t) {
    int tk = (int)(t / tiles_n), tn = (int)(t % tiles_n);
    uint16_t st[256];
    or_tile_states(trellis + t * 16L * K, K, st);
    for (int p = 0; p < 256; ++p) {
      int r = p / 16, c = p % 16;
      W[(long)(16 * tk + r) * n + 16 * tn + c] = or_mul1_value(st[p]);
    }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Block Hadamard (Sylvester order) and the randomized transforms             */
/* ------------------------------------------------------------------------- */

/*
 * H is the 128 x 128 Sylvester Hadamard, H[i][j] = (-1)^popcount(i & j), in
 * natural (not sequency) order.  Readings: blocks are aligned 128-element
 * slices; each side is normalised by 2^-3.5 so the transform is orthonormal;
 * the input side flips signs before H and the output side applies svh after H:
 *     x' = 2^-3.5 H (x . suh)  per block,   y = (2^-3.5 H y') . svh  per block,
 * so the effective dense weight is diag(suh) Hn W Hn diag(svh), Hn = H/sqrt(128).
 */
void or_fwht128_f64(double *v) {
  for (int h = 1; h < 128; h <<= 1)
    for (int i = 0; i < 128; i += 2 * h)
      for (int j = i; j < i + h; ++j) {
        double a = v[j], b = v[j + h];
        v[j] = a + b;
        v[j + h] = a - b;
      }
}

/* Same butterfly tree in binary32: stages h = 1, 2, ..., 64, each (a+b, a-b). */
void or_fwht128_f32(float *v) {
  for (int h = 1; h < 128; h <<= 1)
    for (int i = 0; i < 128; i += 2 * h)
      for (int j = i; j < i + h; ++j) {
        float a = v[j], b = v[j + h];
        v[j] = a + b;
        v[j + h] = a - b;
      }
}

/* x' = RHT(x . suh) in float64; x fp16 [M][k], xr [M][k]. */
int or_rht_in_f64(const uint16_t *x, const uint16_t *suh, int M, int k, double *xr) {
  if (k <= 0 || k % 128 || M < 0) return OR_ERR_SHAPE;
  double scale = ldexp(1.0, -3) / sqrt(2.0);   /* 2^-3.5 */
#pragma omp parallel for schedule(static)
  for (long r = 0; r < M; ++r) {
    for (int b = 0; b < k; b += 128) {
      double v[128];
      for (int i = 0; i < 128; ++i)
        v[i] = or_f16_to_f64(x[r * k + b + i]) * or_f16_to_f64(suh[b + i]);
      or_fwht128_f64(v);
      for (int i = 0; i < 128; ++i) xr[r * k + b + i] = v[i] * scale;
    }
  }
  return OR_OK;
}

/* The binary32 input transform of the int8 path: fp32(x)*fp32(suh) (exact),
 * the butterfly tree above, then one multiply by fp32(2^-3.5). */
int or_rht_in_f32(const uint16_t *x, const uint16_t *suh, int M, int k, float *xr) {
  if (k <= 0 || k % 128 || M < 0) return OR_ERR_SHAPE;
  float scale = (float)(ldexp(1.0, -3) / sqrt(2.0));
#pragma omp parallel for schedule(static)
  for (long r = 0; r < M; ++r) {
    for (int b = 0; b < k; b += 128) {
      float v[128];
      for (int i = 0; i < 128; ++i)
        v[i] = (float)or_f16_to_f64(x[r * k + b + i]) * (float)or_f16_to_f64(suh[b + i]);
      or_fwht128_f32(v);
      for (int i = 0; i < 128; ++i) xr[r * k + b + i] = v[i] * scale;
    }
  }
  return OR_OK;
}

/* y = RHT_out(y') . svh in float64, in place on y [M][n]. */
int or_rht_out_f64(double *y, const uint16_t *svh, int M, int n) {
  if (n <= 0 || n % 128 || M < 0) return OR_ERR_SHAPE;
  double scale = ldexp(1.0, -3) / sqrt(2.0);
#pragma omp parallel for schedule(static)
  for (long r = 0; r < M; ++r) {
    for (int b = 0; b < n; b += 128) {
      double v[128];
      for (int i = 0; i < 128; ++i) v[i] = y[r * n + b + i];
      or_fwht128_f64(v);
      for (int i = 0; i < 128; ++i) y[r * n + b + i] = v[i] * scale * or_f16_to_f64(svh[b + i]);
    }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* The linear: y = RHT_out( RHT_in(x . suh) @ W ) . svh   ([README-int8])      */
/* ------------------------------------------------------------------------- */

static int check_linear(int M, int k, int n, int K) {
  if (K < 1 || K > 8) return OR_ERR_BITS;
  if (M < 0 || k <= 0 || n <= 0 || k % 128 || n % 128) return OR_ERR_SHAPE;
  return OR_OK;
}

/* y' = x' @ W in float64, W given as fp16 bits [k][n]. */
static void contract_f64(const double *xr, const uint16_t *W, int M, int k, int n, double *y) {
#pragma omp parallel for schedule(static)
  for (long r = 0; r < M; ++r) {
    double *yr = y + r * n;
    for (int j = 0; j < n; ++j) yr[j] = 0.0;
    for (int i = 0; i < k; ++i) {
      double a = xr[r * k + i];
      const uint16_t *wr = W + (long)i * n;
      for (int j = 0; j < n; ++j) yr[j] += a * or_f16_to_f64(wr[j]);
    }
  }
}

/* Linear from already-dequantised weights (so a caller can reuse W). */
int or_linear_w(const uint16_t *x, int M, int k, int n, const uint16_t *W,
                const uint16_t *suh, const uint16_t *svh, double *y) {
  int rc = check_linear(M, k, n, 1);
  if (rc) return rc;
  double *xr = (double *)malloc(sizeof(double) * (size_t)M * k + 8);
  if (!xr) return OR_ERR_SHAPE;
  or_rht_in_f64(x, suh, M, k, xr);
  contract_f64(xr, W, M, k, n, y);
  or_rht_out_f64(y, svh, M, n);
  free(xr);
  return OR_OK;
}

int or_linear(const uint16_t *x, int M, int k, int n, const uint16_t *trellis,
              const uint16_t *suh, const uint16_t *svh, int K, double *y) {
  int rc = check_linear(M, k, n, K);
  if (rc) return rc;
  uint16_t *W = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)k * n);
  if (!W) return OR_ERR_SHAPE;
  or_reconstruct(trellis, k, n, K, W);
  rc = or_linear_w(x, M, k, n, W, suh, svh, y);
  free(W);
  return rc;
}

/*
 * Output bias ([TF-832], "What is left": a checkpoint's EXL3 group holds a
 * bias beside trellis, suh and svh).  The pages do not place it; this file
 * reads it as the bias of the original linear, one fp16 value per output
 * feature added after the output transform and svh:
 *   y[r][j] += bias[j]   (float64, in place on y [M][n]).
 */
int or_add_bias(double *y, const uint16_t *bias, int M, int n) {
  if (M < 0 || n <= 0) return OR_ERR_SHAPE;
  for (long r = 0; r < M; ++r)
    for (int j = 0; j < n; ++j) y[r * n + j] += or_f16_to_f64(bias[j]);
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* int8 variant ([README-int8]; rounding details are this library's reading)   */
/* ------------------------------------------------------------------------- */

/*
 * Activations: x' from or_rht_in_f32; amax_r = max_j |x'_rj| (fp32);
 *   inv = fp32(127 / amax_r); q = clamp(RNE(fp32(x' * inv)), -127, 127);
 *   a_r = fp32(amax_r / 127); a row with amax_r = 0 gives q = 0, a_r = 0.
 * Weights: q_w = RNE(v * 127 / 3.453125) of the exact rational (v is the fp16
 *   weight); |q_w| <= 127 by the codebook bound and v(0) -> -127.
 * Accumulate: acc = sum_j q_x * q_w exactly (int64, must fit int32).
 * Output: y' = acc * a_r * (3.453125 / 127), then the output transform.
 */
int or_quant_act(const uint16_t *x, const uint16_t *suh, int M, int k,
                 int8_t *qx, float *row_scale) {
  if (k <= 0 || k % 128 || M < 0) return OR_ERR_SHAPE;
  float *xr = (float *)malloc(sizeof(float) * (size_t)M * k + 8);
  if (!xr) return OR_ERR_SHAPE;
  or_rht_in_f32(x, suh, M, k, xr);
#pragma omp parallel for schedule(static)
  for (long r = 0; r < M; ++r) {
    float amax = 0.0f;
    for (int j = 0; j < k; ++j) {
      float a = fabsf(xr[r * k + j]);
      if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
      for (int j = 0; j < k; ++j) qx[r * k + j] = 0;
      row_scale[r] = 0.0f;
      continue;
    }
    float inv = 127.0f / amax;
    for (int j = 0; j < k; ++j) {
      float t = xr[r * k + j] * inv;
      float q = nearbyintf(t);
      if (q > 127.0f) q = 127.0f;
      if (q < -127.0f) q = -127.0f;
      qx[r * k + j] = (int8_t)q;
    }
    row_scale[r] = amax / 127.0f;
  }
  free(xr);
  return OR_OK;
}

/* q_w of one fp16 weight: RNE(v * 127 / 3.453125) as an exact rational.
 * v = V * 2^-24 with V an integer, 3.453125 = 1768 * 2^-9, so
 * v * 127 / 3.453125 = V * 127 / (1768 * 2^15). */
int or_quant_weight(uint16_t vbits) {
  double v = or_f16_to_f64(vbits);
  long long V = llround(ldexp(v, 24));          /* exact: fp16 values are multiples of 2^-24 */
  long long num = V * 127LL;
  long long den = 1768LL * 32768LL;
  long long an = num < 0 ? -num : num;
  long long q = an / den, rem = an % den;
  if (2 * rem > den || (2 * rem == den && (q & 1))) q += 1;  /* ties to even */
  return (int)(num < 0 ? -q : q);
}

/* acc [M][n] int64 = qx @ qw; returns OR_ERR_OVERFLOW if any |acc| >= 2^31. */
int or_int8_acc(const int8_t *qx, const int8_t *qw, int M, int k, int n, int64_t *acc) {
  int overflow = 0;
#pragma omp parallel for schedule(static) reduction(| : overflow)
  for (long r = 0; r < M; ++r) {
    int64_t *ar = acc + r * n;
    for (int j = 0; j < n; ++j) ar[j] = 0;
    for (int i = 0; i < k; ++i) {
      int64_t a = qx[r * k + i];
      const int8_t *wr = qw + (long)i * n;
      for (int j = 0; j < n; ++j) ar[j] += a * (int64_t)wr[j];
    }
    for (int j = 0; j < n; ++j)
      if (ar[j] >= 2147483648LL || ar[j] < -2147483648LL) overflow = 1;
  }
  return overflow ? OR_ERR_OVERFLOW : OR_OK;
}

int or_linear_int8(const uint16_t *x, int M, int k, int n, const uint16_t *trellis,
                   const uint16_t *suh, const uint16_t *svh, int K,
                   int8_t *qx, float *row_scale, int8_t *qw, int64_t *acc, double *y) {
  int rc = check_linear(M, k, n, K);
  if (rc) return rc;
  uint16_t *W = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)k * n);
  if (!W) return OR_ERR_SHAPE;
  or_reconstruct(trellis, k, n, K, W);
#pragma omp parallel for schedule(static)
  for (long i = 0; i < (long)k * n; ++i) qw[i] = (int8_t)or_quant_weight(W[i]);
  free(W);
  or_quant_act(x, suh, M, k, qx, row_scale);
  rc = or_int8_acc(qx, qw, M, k, n, acc);
  double sw = 3.453125 / 127.0;
  for (long r = 0; r < M; ++r)
    for (int j = 0; j < n; ++j)
      y[r * n + j] = (double)acc[r * n + j] * (double)row_scale[r] * sw;
  or_rht_out_f64(y, svh, M, n);
  return rc;
}

/* ------------------------------------------------------------------------- */
/* Routed experts ([README-moe], [ARC-2B])                                     */
/* ------------------------------------------------------------------------- */

/* float64 linear with a float64 input row (the down projection's input h is
 * not an fp16 tensor in the definition). */
static void lin_f64_in(const double *xin, int k, int n, const uint16_t *W,
                       const uint16_t *suh, const uint16_t *svh, double *y) {
  double scale = ldexp(1.0, -3) / sqrt(2.0);
  double *xr = (double *)malloc(sizeof(double) * (size_t)k);
  for (int b = 0; b < k; b += 128) {
    double v[128];
    for (int i = 0; i < 128; ++i) v[i] = xin[b + i] * or_f16_to_f64(suh[b + i]);
    or_fwht128_f64(v);
    for (int i = 0; i < 128; ++i) xr[b + i] = v[i] * scale;
  }
  for (int j = 0; j < n; ++j) y[j] = 0.0;
  for (int i = 0; i < k; ++i) {
    const uint16_t *wr = W + (long)i * n;
    for (int j = 0; j < n; ++j) y[j] += xr[i] * or_f16_to_f64(wr[j]);
  }
  or_rht_out_f64(y, svh, 1, n);
  free(xr);
}

/*
 * Per token t and slot s: e = ids[t][s];
 *   g = lin(x_t; gate_e), u = lin(x_t; up_e)   (gate is slot 0, up slot 1 of w13)
 *   h = g / (1 + exp(-g)) * u                  (SiLU(g) * u)
 *   d = lin(h; down_e)                         (the single slot of w2)
 *   y_t = sum_s w[t][s] * d                    (weight on the down output only)
 * Every step in float64; each projection has its own suh/svh and, being a
 * linear of this file, its own input and output transforms.  Experts' weights
 * are dequantised once per expert used.  Only the tokens listed in `tok`
 * (n_tok of them) are evaluated, so callers can sample a large batch.
 *
 * Per-expert widths ("EXL3 checkpoints on the native engine (tracker) #832",
 * comment of Oct 17: the format keeps each expert's own width): expert e of w13 has width
 * K13[e] and of w2 K2[e].  Each arena packs the experts in id order, expert
 * e's slots right after expert e-1's, so expert e starts at the sum of the
 * earlier experts' sizes (nslots * (k/16) * (n/16) * 16 * K words each).
 */
int or_moe_k(const uint16_t *x, int T, int hidden, const int32_t *ids, const float *weights,
             int topk, int E,
             const uint16_t *w13_trellis, const uint16_t *w13_suh, const uint16_t *w13_svh,
             int inter, const int32_t *K13,
             const uint16_t *w2_trellis, const uint16_t *w2_suh, const uint16_t *w2_svh,
             const int32_t *K2,
             const int32_t *tok, int n_tok, double *y /* [n_tok][hidden] */) {
  if (hidden % 128 || inter % 128 || T < 0 || topk < 1 || E < 1) return OR_ERR_SHAPE;
  for (int e = 0; e < E; ++e)
    if (K13[e] < 1 || K13[e] > 8 || K2[e] < 1 || K2[e] > 8) return OR_ERR_BITS;
  /* word offset of each expert in the two arenas */
  long *off13 = (long *)malloc(sizeof(long) * (size_t)E);
  long *off2 = (long *)malloc(sizeof(long) * (size_t)E);
  long a13 = 0, a2 = 0;
  for (int e = 0; e < E; ++e) {
    off13[e] = a13;
    off2[e] = a2;
    a13 += 2L * (hidden / 16) * (inter / 16) * 16 * K13[e];
    a2 += (long)(inter / 16) * (hidden / 16) * 16 * K2[e];
  }
  char *need = (char *)calloc((size_t)E, 1);
  for (int i = 0; i < n_tok; ++i) {
    if (tok[i] < 0 || tok[i] >= T) { free(need); free(off13); free(off2); return OR_ERR_SHAPE; }
    for (int s = 0; s < topk; ++s) {
      int e = ids[(long)tok[i] * topk + s];
      if (e < 0 || e >= E) { free(need); free(off13); free(off2); return OR_ERR_SHAPE; }
      need[e] = 1;
    }
  }
  uint16_t **Wg = (uint16_t **)calloc((size_t)E, sizeof(uint16_t *));
  uint16_t **Wu = (uint16_t **)calloc((size_t)E, sizeof(uint16_t *));
  uint16_t **Wd = (uint16_t **)calloc((size_t)E, sizeof(uint16_t *));
  for (int e = 0; e < E; ++e) {
    if (!need[e]) continue;
    long slot13 = (long)(hidden / 16) * (inter / 16) * 16 * K13[e];
    Wg[e] = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)hidden * inter);
    Wu[e] = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)hidden * inter);
    Wd[e] = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)inter * hidden);
    or_reconstruct(w13_trellis + off13[e], hidden, inter, K13[e], Wg[e]);
    or_reconstruct(w13_trellis + off13[e] + slot13, hidden, inter, K13[e], Wu[e]);
    or_reconstruct(w2_trellis + off2[e], inter, hidden, K2[e], Wd[e]);
  }
#pragma omp parallel for schedule(dynamic)
  for (int i = 0; i < n_tok; ++i) {
    long t = tok[i];
    double *g = (double *)malloc(sizeof(double) * (size_t)inter);
    double *u = (double *)malloc(sizeof(double) * (size_t)inter);
    double *h = (double *)malloc(sizeof(double) * (size_t)inter);
    double *d = (double *)malloc(sizeof(double) * (size_t)hidden);
    double *yt = y + (long)i * hidden;
    for (int j = 0; j < hidden; ++j) yt[j] = 0.0;
    for (int s = 0; s < topk; ++s) {
      int e = ids[t * topk + s];
      double w = (double)weights[t * topk + s];
      const uint16_t *xt = x + t * hidden;
      or_linear_w(xt, 1, hidden, inter, Wg[e], w13_suh + (2L * e + 0) * hidden,
                  w13_svh + (2L * e + 0) * inter, g);
      or_linear_w(xt, 1, hidden, inter, Wu[e], w13_suh + (2L * e + 1) * hidden,
                  w13_svh + (2L * e + 1) * inter, u);
      for (int j = 0; j < inter; ++j) h[j] = g[j] / (1.0 + exp(-g[j])) * u[j];
      lin_f64_in(h, inter, hidden, Wd[e], w2_suh + (long)e * inter, w2_svh + (long)e * hidden, d);
      for (int j = 0; j < hidden; ++j) yt[j] += w * d[j];
    }
    free(g); free(u); free(h); free(d);
  }
  for (int e = 0; e < E; ++e) { free(Wg[e]); free(Wu[e]); free(Wd[e]); }
  free(Wg); free(Wu); free(Wd); free(need); free(off13); free(off2);
  return OR_OK;
}

/* One width for all experts of each projection kind: the arenas are
 * [E][nslots][k/16][n/16][16K], the packed layout above with equal sizes. */
int or_moe(const uint16_t *x, int T, int hidden, const int32_t *ids, const float *weights,
           int topk, int E,
           const uint16_t *w13_trellis, const uint16_t *w13_suh, const uint16_t *w13_svh,
           int inter, int K13,
           const uint16_t *w2_trellis, const uint16_t *w2_suh, const uint16_t *w2_svh, int K2,
           const int32_t *tok, int n_tok, double *y /* [n_tok][hidden] */) {
  if (K13 < 1 || K13 > 8 || K2 < 1 || K2 > 8) return OR_ERR_BITS;
  if (E < 1) return OR_ERR_SHAPE;
  int32_t *k13 = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
  int32_t *k2 = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
  for (int e = 0; e < E; ++e) { k13[e] = K13; k2[e] = K2; }
  int rc = or_moe_k(x, T, hidden, ids, weights, topk, E, w13_trellis, w13_suh, w13_svh, inter, k13,
                    w2_trellis, w2_suh, w2_svh, k2, tok, n_tok, y);
  free(k13); free(k2);
  return rc;
}
