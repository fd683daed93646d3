// mxfrag.cuh — register-level pieces of the MXFP4 and f16 GEMVs: E2M1 decode
// into m16n8k16 A fragments and the mma.sync contraction (inline PTX).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace dfm {

// 2^s for s in [-126, 127].
__device__ __forceinline__ float pow2i(int s) {
  return __uint_as_float((uint32_t)(127 + s) << 23);
}

// Four bytes = eight E2M1 codes -> four f16x2 (low nibble in the low half).
// With the fragment layout, one word is the whole A fragment of one k-step.
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// d = A * B (+ c): m16n8k16, f16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1,
                                         const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1),
        "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// E8M0 byte `i` of a packed scale word, as the fp32 value 2^(e - 127).
__device__ __forceinline__ float e8m0_byte(uint32_t w, int i) {
  return __uint_as_float(((w >> (8 * i)) & 0xFFu) << 23);
}

}  // namespace dfm
