// Packed 4-bit dot products on the vector ALUs, shared by the decode kernels
// (fma_pair also serves the decode attention's bf16 q.k dots).
//
// A code q becomes the 16-bit float f = 1 + q/16 exactly (bf16 bits
// 0x3F80 | q << 3, f16 bits 0x3C00 | q << 6), two codes per shift-and-mask,
// and is multiplied with the activation by a mixed-precision FMA (16-bit
// inputs, fp32 accumulate; the product is exact). For a group with scale s
// and bias b, sum_k (s*q_k + b) v_k = 16 s * sum_k f_k v_k + (b - 16 s) * sum_k v_k.
#pragma once

#include "common.cuh"

namespace moe {

// a0 += f_lo * v_lo, a1 += f_hi * v_hi for one pair of 16-bit values.
template <bool BF16>
MOE_DEVINL void fma_pair(float& a0, float& a1, uint32_t f, uint32_t v) {
  if constexpr (BF16)
    asm("{ .reg .b16 fl, fh, vl, vh;\n\t mov.b32 {fl, fh}, %2;\n\t mov.b32 {vl, vh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, fl, vl, %0;\n\t fma.rn.f32.bf16 %1, fh, vh, %1; }"
        : "+f"(a0), "+f"(a1)
        : "r"(f), "r"(v));
  else
    asm("{ .reg .b16 fl, fh, vl, vh;\n\t mov.b32 {fl, fh}, %2;\n\t mov.b32 {vl, vh}, %3;\n\t"
        "fma.rn.f32.f16 %0, fl, vl, %0;\n\t fma.rn.f32.f16 %1, fh, vh, %1; }"
        : "+f"(a0), "+f"(a1)
        : "r"(f), "r"(v));
}

// a0/a1 += sum over the 8 codes of word w of f_k * v_k, v given as the four
// pairs (v_i, v_{i+4}), i = 0..3 (vp.x .. vp.w): shifting w puts codes i
// and i+4 (bits 4i and 16 + 4i) at the two halves' mantissa tops together.
template <bool BF16>
MOE_DEVINL void word_fdot(uint32_t w, const uint4& vp, float& a0, float& a1) {
  if constexpr (BF16) {
    constexpr uint32_t m = 0x00780078u, one = 0x3F803F80u;
    fma_pair<true>(a0, a1, ((w << 3) & m) | one, vp.x);
    fma_pair<true>(a0, a1, ((w >> 1) & m) | one, vp.y);
    fma_pair<true>(a0, a1, ((w >> 5) & m) | one, vp.z);
    fma_pair<true>(a0, a1, ((w >> 9) & m) | one, vp.w);
  } else {
    constexpr uint32_t m = 0x03C003C0u, one = 0x3C003C00u;
    fma_pair<false>(a0, a1, ((w << 6) & m) | one, vp.x);
    fma_pair<false>(a0, a1, ((w << 2) & m) | one, vp.y);
    fma_pair<false>(a0, a1, ((w >> 2) & m) | one, vp.z);
    fma_pair<false>(a0, a1, ((w >> 6) & m) | one, vp.w);
  }
}

// The four pairs (v_i, v_{i+4}) of 8 consecutive 16-bit values held as 4
// words (v0 v1), (v2 v3), (v4 v5), (v6 v7).
MOE_DEVINL uint4 pair_up(uint4 v) {
  return make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                    __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
}

}  // namespace moe
