// NVFP4 code expansion for the tensor-memory GEMMs (E2M1 elements, an E4M3 scale per 16 inputs, an fp32
// scale per matrix: the block-scaled checkpoint format of the "Qwen-3.6-35B-A3B-SIQ-K6-K4K3" model card).
#pragma once

#include <stdint.h>

namespace qmoe {

// Four bytes of E2M1 code pairs -> four fp16x2 (byte k -> c[k], low nibble in the low half) by the
// hardware conversion.  Exact: every E2M1 value is an fp16.
__device__ __forceinline__ void nv_e2m1x8_f16(uint32_t u, uint32_t (&c)[4])
{
    asm("{\n.reg .b8 b0, b1, b2, b3;\nmov.b32 {b0, b1, b2, b3}, %4;\n"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\ncvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\ncvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(c[0]), "=r"(c[1]), "=r"(c[2]), "=r"(c[3])
        : "r"(u));
}

// Two E4M3 codes (the low 16 bits of v) -> fp16x2, low byte in the low half.  Exact.
__device__ __forceinline__ uint32_t nv_e4m3x2_f16(uint32_t v)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)v));
    return r;
}

// 8 NVFP4 codes of one block (inputs 0..7 of a 32-bit word) times the block scale (fp16x2, both
// halves equal) -> fp16x2 pairs of inputs (0,4) (1,5) (2,6) (3,7).  Exact: e2m1 * e4m3 has at most 6
// significant bits and lies in [2^-10, 2688].
__device__ __forceinline__ uint4 nv_dequant8(uint32_t u, uint32_t s2)
{
    // register-only PTX (no type punning of fp16 pairs through memory)
    uint32_t c[4];
    uint4 o;
    nv_e2m1x8_f16(u, c);
    asm("{\n.reg .b32 p0, p1, p2, p3;\n"
        "prmt.b32 p0, %4, %6, 0x5410;\nprmt.b32 p1, %4, %6, 0x7632;\n"
        "prmt.b32 p2, %5, %7, 0x5410;\nprmt.b32 p3, %5, %7, 0x7632;\n"
        "mul.rn.f16x2 %0, p0, %8;\nmul.rn.f16x2 %1, p1, %8;\n"
        "mul.rn.f16x2 %2, p2, %8;\nmul.rn.f16x2 %3, p3, %8;\n}"
        : "=r"(o.x), "=r"(o.y), "=r"(o.z), "=r"(o.w)
        : "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(s2));
    return o;
}

// The low (hi = false) or high half of an fp16x2, in both halves.
__device__ __forceinline__ uint32_t nv_bcast(uint32_t s2, bool hi)
{
    return hi ? (s2 >> 16) | (s2 & 0xFFFF0000u) : (s2 & 0xFFFFu) | (s2 << 16);
}

}  // namespace qmoe
