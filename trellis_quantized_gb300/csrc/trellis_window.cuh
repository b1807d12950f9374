// trellis_window.cuh -- compile-time window extraction from a lane's stream
// words (shared by the CUDA-core GEMV and the fused tensor-core decode).
//
// A lane holds its part of a tile's bitstream as 32-bit words w[0..N) (LSB
// first, words in stream order); the 16-bit trellis state of a weight is the
// window starting at its bit offset O ("Bringing EXL3 Trellis Quantization to
// 35B MoE on Intel Arc 140V", section 1: trellis codebook decoding; the
// window layout is this library's reading).
#pragma once

#include <stdint.h>

namespace exl3 {

// 16-bit window at compile-time bit offset o of the word array w.  Windows on
// byte offsets 0, 1, 2 of a word cost one instruction; other residues reuse a
// word shifted by (o mod 8) bits, shared between windows of the same residue.
template <int O, int N>
__device__ __forceinline__ uint32_t window_at(const uint32_t (&w)[N]) {
  constexpr int a = O & 7, base = O - a, j = base >> 5, b = base & 31;
  if constexpr (b == 24) {
    return __funnelshift_r(w[O >> 5], w[(O >> 5) + 1], O & 31) & 0xFFFFu;
  } else {
    const uint32_t src = a == 0 ? w[j] : __funnelshift_r(w[j], w[j + 1], a);
    if constexpr (b == 0) return src & 0xFFFFu;
    else if constexpr (b == 16) return src >> 16;
    else return __byte_perm(src, 0u, 0x4421);   // bytes 1, 2 then zeros
  }
}


}  // namespace exl3
