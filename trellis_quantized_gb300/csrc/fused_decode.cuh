// fused_decode.cuh -- decoding trellis tiles from shared memory straight into
// tcgen05 operands (shared by the small-M linear and the grouped experts).
//
// One 64-deep k step of a 128-column tile covers 4 x 8 trellis tiles.  A
// decoder item is (tile, row group q): G = 8 / gcd(K, 8) rows of 16 weights
// from CPL = K / gcd(K, 8) 16-byte chunks.  Each weight's 16-bit state is
// hashed (IMAD), byte-summed by DP4A seeded with 0x6400 (the fp16 value
// 1024 + B), and either 1534 is subtracted in half2, which leaves the exact
// integer B - 510 as fp16, or 1024 + B is kept and the caller removes
// 1534 * sum x' per token; sigma is applied by the caller's epilogue.  The values go
// to an MN-major, 128-byte-swizzled operand: row k holds 64 n values, 8-row k
// groups are 2 KB apart and 64-wide n atoms 1 KB apart (descriptor LBO =
// 1024, SBO = 2048).
#pragma once

#include "exl3_common.cuh"
#include "tc_ptx.cuh"
#include "trellis_window.cuh"

namespace exl3 {
namespace ftc {

constexpr int BN = 128, BK = 64;             // output columns per CTA, k per step
constexpr int W_BYTES = BK * BN * 2;         // decoded weight operand of one step
constexpr int NGRP = 2;   // decoder groups (alternate k steps)
constexpr int NDEC = 8;   // decoder warps per group
constexpr int NWARPS = 3 + NGRP * NDEC;

template <int K, int NMAX>
struct Shape {
  // Items.  K = 4 and 8: an item is G = 4 rows of a tile (64 weights, so the
  // per-item costs are shared by 64 weights), read as CPL 16-byte chunks;
  // a pair of k steps has 256 of them.  Other widths (RP): an item is one row
  // pair of a tile, the K + 1 stream words starting at word K * rp, 256 per
  // k step.  Either way all decoder threads are busy.
  static constexpr bool RP = (K != 4 && K != 8);
  static constexpr int G = RP ? 2 : 4;               // rows per lane item
  static constexpr int CPL = RP ? 0 : K * G / 8;     // 16-byte chunks per item
  static constexpr int LPT = 16 / G;             // items per tile
  static constexpr int ROWB = (BN / 16) * 32 * K;   // one tile row of the CTA: 8 tiles
  static constexpr int T_BYTES = 4 * ROWB;          // 4 tile rows per 64-deep k step
  static constexpr int X_BYTES = NMAX * BK * 2;     // x' operand of one step (up to NMAX tokens)
  static constexpr int ITEMS = 32 * LPT;         // (tile, group) items per k step
  static_assert(2 * ITEMS % 256 == 0, "a pair of k steps keeps all 256 decoder threads busy");
  static constexpr int NW = RP ? K : 4 * CPL;    // stream words per item (one more is read)
  // Streaming: a trellis stage is TSTEPS k steps (16 tile rows) fetched by one
  // tensor load; an x' stage is XSTEPS k steps, also one tensor load.  Few,
  // large copies keep one producer thread from limiting the feed.
  static constexpr int TSTEPS = 4;
  static constexpr int T_STAGE = TSTEPS * T_BYTES;
  static constexpr int XSTEPS = NMAX <= 32 ? 4 : 2;
  static constexpr int X_STAGE = XSTEPS * X_BYTES;
  // decoded-weight ring depth in k steps: WS / 2 pair slots, a multiple of
  // the decoder groups (2) and of the small-M kernel's MMA issuers (4 or 2),
  // so that each slot has one decoder group and one issuer
  static constexpr int WS = NMAX <= 32 ? 8 : 4;
  static constexpr int XS = 2;                      // x' ring depth (stages)
  static constexpr int TS_FIT = (227 * 1024 - 2048 - WS * W_BYTES - XS * X_STAGE) / T_STAGE;
  static constexpr int TS = TS_FIT > 8 ? 8 : TS_FIT;   // trellis ring depth (stages)
  static constexpr int SMEM_BYTES = WS * W_BYTES + XS * X_STAGE + TS * T_STAGE + 1024 + 1024;
  static_assert(TS >= 2, "trellis ring too shallow");
};

// MN-major 128B-swizzle descriptor: LBO = n-atom stride, SBO = k-group stride.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(const void *base, uint32_t lbo, uint32_t sbo) {
  const uint64_t addr = tc::smem_u32(base);
  uint64_t d = 0;
  d |= (addr >> 4) & 0x3FFFull;
  d |= (uint64_t)(lbo >> 4) << 16;
  d |= (uint64_t)(sbo >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__host__ __device__ constexpr uint32_t idesc_f16_amn(int M, int N) {
  return tc::idesc_f16(M, N) | (1u << 15);   // A is MN-major
}


__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   tc::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
               : "memory");
}

// Two adjacent weights (columns C, C + 1 of row R) as a half2: DP4A seeded
// with 0x6400 gives the fp16 bits of 1024 + B.  OFS = false subtracts 1534
// (exact) for (B0 - 510, B1 - 510); OFS = true keeps (1024 + B0, 1024 + B1)
// and the caller removes 1534 * sum x' per token after the contraction.
template <int K, int R, int C, bool OFS>
__device__ __forceinline__ uint32_t decode_pair(const uint32_t (&w)[Shape<K, 32>::NW + 1]) {
  const uint32_t s0 = window_at<(16 * R + C) * K>(w), s1 = window_at<(16 * R + C + 1) * K>(w);
  const uint32_t h0 = __dp4a(s0 * kMul1, 0x01010101u, 0x6400u);
  const uint32_t h1 = __dp4a(s1 * kMul1, 0x01010101u, 0x6400u);
  const uint32_t pr = __byte_perm(h0, h1, 0x5410);
  if constexpr (OFS) return pr;
  const __half2 d = __hsub2(*reinterpret_cast<const __half2 *>(&pr), __half2half2(__ushort_as_half(0x65FE)));
  return *reinterpret_cast<const uint32_t *>(&d);
}

// Decode rows R.. of one (tile, row group) item into the operand stage.  The
// item's G rows (G = 2 or 4) start at a multiple of G within the 64-deep k
// step, so they share one 8-row k group and row R sits at kr = kr0 + R =
// kr0 ^ R.  With c = ch ^ kr0 (even), the 16-byte slot of row R's even chunk
// is c ^ R and of its odd chunk c ^ R ^ 1: for R = 0, 1 these are c + R and
// c + 1 - R, for R = 2, 3 the same from c ^ 2.  So with pA = row 0 + 16 c and
// pB = row 0 + 16 (c ^ 2), every store address is one of them plus a
// constant.
template <int K, int R, bool OFS>
__device__ __forceinline__ void decode_rows(const uint32_t (&w)[Shape<K, 32>::NW + 1], uint8_t *pA, uint8_t *pB) {
  if constexpr (R < Shape<K, 32>::G) {
    const uint4 lo = make_uint4(decode_pair<K, R, 0, OFS>(w), decode_pair<K, R, 2, OFS>(w),
                                decode_pair<K, R, 4, OFS>(w), decode_pair<K, R, 6, OFS>(w));
    const uint4 hi = make_uint4(decode_pair<K, R, 8, OFS>(w), decode_pair<K, R, 10, OFS>(w),
                                decode_pair<K, R, 12, OFS>(w), decode_pair<K, R, 14, OFS>(w));
    uint8_t *row = (R < 2 ? pA : pB) + R * 128;
    *reinterpret_cast<uint4 *>(row + ((R & 1) ? 16 : 0)) = lo;
    *reinterpret_cast<uint4 *>(row + ((R & 1) ? 0 : 16)) = hi;
    decode_rows<K, R + 1, OFS>(w, pA, pB);
  }
}

// Decode the item of tile (tkl, tnl) of a k step (tkl: tile row 0..3, tnl:
// tile column 0..7) and row group q into the k step's operand stage.
template <int K, bool OFS = false>
__device__ __forceinline__ void decode_item(const uint32_t (&w)[Shape<K, 32>::NW + 1], uint8_t *bstage, int tkl,
                                            int tnl, int q) {
  constexpr int G = Shape<K, 32>::G;
  static_assert(G == 2 || G == 4, "an item stays inside one 8-row k group");
  const int k0 = tkl * 16 + G * q, kr0 = k0 & 7;
  uint8_t *base = bstage + (k0 >> 3) * 2048 + (tnl >> 2) * 1024 + kr0 * 128;
  const int c = ((tnl & 3) * 2) ^ kr0;
  decode_rows<K, 0, OFS>(w, base + 16 * c, base + 16 * (c ^ 2));
}

// The item's stream words w[0..NW] (w[NW] is the first word of the next item
// of the tile, wrapping at the tile end) from the tile at `tile` in shared
// memory.
template <int K>
__device__ __forceinline__ void load_item(const uint8_t *tile, int q, uint32_t (&w)[Shape<K, 32>::NW + 1]) {
  using S = Shape<K, 32>;
  if constexpr (S::RP) {
    const uint32_t *tw = reinterpret_cast<const uint32_t *>(tile);
    if constexpr ((K & 1) == 0) {
#pragma unroll
      for (int j = 0; j < K / 2; ++j) {
        const uint2 v = *reinterpret_cast<const uint2 *>(tw + K * q + 2 * j);
        w[2 * j] = v.x;
        w[2 * j + 1] = v.y;
      }
    } else {
#pragma unroll
      for (int j = 0; j < K; ++j) w[j] = tw[K * q + j];
    }
    w[K] = tw[K * ((q + 1) & 7)];
  } else {
#pragma unroll
    for (int cc = 0; cc < S::CPL; ++cc) {
      const uint4 v4 = *reinterpret_cast<const uint4 *>(tile + q * 16 * S::CPL + 16 * cc);
      w[4 * cc + 0] = v4.x;
      w[4 * cc + 1] = v4.y;
      w[4 * cc + 2] = v4.z;
      w[4 * cc + 3] = v4.w;
    }
    w[S::NW] = *reinterpret_cast<const uint32_t *>(tile + ((q + 1) % S::LPT) * 16 * S::CPL);
  }
}

// Item -> (tile 0..31 of the step, row group q).  32 consecutive items form
// one warp instruction.
template <int K>
__device__ __forceinline__ void item_map(int it, int &ti, int &q) {
  constexpr int LPT = Shape<K, 32>::LPT;
  if constexpr (Shape<K, 32>::RP) {
    // four tiles per warp, lane = 8 tile + row pair: the words K (8 tile + rp)
    // + j of one load fall in 32 distinct banks (odd K) or 16 distinct 8-byte
    // units per half warp (K = 2, 6)
    const int w = it >> 5, l = it & 31;
    ti = 4 * w + (l >> 3);
    q = l & 7;
  } else {
    // G = 4: one tile row of 8 tiles per warp, four row groups per tile
    static_assert(LPT == 4, "item map");
    ti = it >> 2;
    q = it & 3;
  }
}



// The loop-invariant part of a decoder thread's item (the same item every
// pair): the byte offset of its tile from the start of a k step's tile rows
// in a trellis stage, its row group, and the two store bases of its rows in
// an operand slot (see decode_item).
struct ItemPlan {
  int tile_off, q, opA, opB;
};

template <int K>
__device__ __forceinline__ ItemPlan item_plan(int it) {
  constexpr int G = Shape<K, 32>::G;
  int ti, q;
  item_map<K>(it, ti, q);
  const int tkl = ti >> 3, tnl = ti & 7;
  const int k0 = tkl * 16 + G * q, kr0 = k0 & 7;
  const int base = (k0 >> 3) * 2048 + (tnl >> 2) * 1024 + kr0 * 128;
  const int c = ((tnl & 3) * 2) ^ kr0;
  return ItemPlan{tkl * Shape<K, 32>::ROWB + tnl * 32 * K, q, base + 16 * c, base + 16 * (c ^ 2)};
}

// Load and decode the planned item of the k step whose tile rows start at
// `rows` into the operand slot `slot`.
template <int K, bool OFS>
__device__ __forceinline__ void decode_planned(const uint8_t *rows, uint8_t *slot, const ItemPlan &ip) {
  uint32_t w[Shape<K, 32>::NW + 1];
  load_item<K>(rows + ip.tile_off, ip.q, w);
  decode_rows<K, 0, OFS>(w, slot + ip.opA, slot + ip.opB);
}

}  // namespace ftc
}  // namespace exl3
