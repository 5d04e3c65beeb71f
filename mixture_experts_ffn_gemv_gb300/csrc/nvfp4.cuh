// NVFP4 device helpers of the GEMV arm: e2m1 code pairs widened to f16x2 and
// multiplied by their e4m3 block scale.  e2m1 times e4m3 has at most 6
// significant bits and lies in [2^-10, 2688], so the f16 product is exact.
// Weights and tokens are both widened by nvfp4_word, so however the
// conversion orders a pair's halves, they come out in the same order and dot
// products over them are unchanged.  (The grouped GEMM feeds packed codes to
// the tensor core's block-scaled MMA and widens nothing.)
#pragma once

#include <stdint.h>

namespace moe {

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Two e4m3 block-scale codes (block 0 in the low byte) -> each as an f16x2 splat.
__device__ __forceinline__ void nvfp4_scales(uint32_t two_codes, uint32_t& s0, uint32_t& s1) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two_codes));
    s0 = __byte_perm(h2, 0, 0x1010);
    s1 = __byte_perm(h2, 0, 0x3232);
}

// One e4m3 code -> its value as an f16x2 splat.
__device__ __forceinline__ uint32_t nvfp4_scale1(uint32_t code) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(code * 0x101u)));
    return h2;
}

// Four bytes of e2m1 code pairs -> four f16x2 values, each times the scale s.
__device__ __forceinline__ void nvfp4_word(uint32_t w, uint32_t s, uint32_t (&v)[4]) {
    uint32_t d0, d1, d2, d3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
        : "r"(w));
    v[0] = hmul2(d0, s);
    v[1] = hmul2(d1, s);
    v[2] = hmul2(d2, s);
    v[3] = hmul2(d3, s);
}

}  // namespace moe
