// e4m3_umma.cuh -- FP8-E4M3 operands on the sm_103a tensor cores, shared by the
// kernels that consume an E4M3 K/V cache without decoding it.
//
// An E4M3 cache ("[Perf] Ship the qualified SM70 long-context layout ...",
// What: E4M3 K/V with one fp32 scale each) feeds tcgen05.mma kind::f8f6f4
// directly.  Both operands of such an MMA must be 8-bit, so the fp16 / fp32
// operand of each product (Q for Q.K^T, P for P.V) enters as a three-term
// E4M3 expansion x ~= t1 + t2 / XRATIO + t3 / XRATIO^2: t1 is the E4M3
// rounding of x, t2 that of the scaled remainder, t3 that of the next one.
// With |x| <= 256 a remainder is at most half an E4M3 unit of x (<= 8), so
// XRATIO = 32 keeps every scaled remainder inside E4M3's range (448); the
// expansion carries at least 11 significant bits (fp16's precision) and its
// smallest kept value is 2^-19 (E4M3's smallest subnormal, 2^-9, over 32^2).
// The three terms sit side by side along the MMA's N dimension, so one MMA
// yields the three partial products, which the consumer combines.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "sm100.cuh"

namespace gqa {

// Ratio between consecutive terms of a three-term E4M3 expansion.
constexpr float XRATIO = 32.0f;

// A softmax whose P enters such an expansion keeps P <= 256 (a score may
// exceed its row's reference by at most 8 in log2 units before the reference
// moves) and, when the reference moves, sets it this far below the tile's
// max (log2 units): right after a move the largest P is 2^6, and the
// expansion's floor of 2^-19 sits at least 25 binades below the row's max.
constexpr float REF_SHIFT = 6.0f;

// FP8 UMMA: D (+)= A . B with E4M3 operands from shared memory, f32 accumulator
// (the instruction descriptor's A / B format fields 0 select E4M3 here).
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Two floats -> two E4M3 bytes (round to nearest even, saturating), low byte = a.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// Value of an E4M3 byte pair (low byte first) as two floats.
__device__ __forceinline__ void e4m3x2_val(uint32_t v, float& a, float& b) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)v));
    const __half2 hh = *reinterpret_cast<const __half2*>(&h2);
    a = __low2float(hh);
    b = __high2float(hh);
}

// x ~= t1 + t2 / XRATIO + t3 / XRATIO^2 with t1, t2, t3 E4M3, for two values at
// once, |x| <= 256 (each result holds the pair's two bytes in its low 16 bits).
__device__ __forceinline__ void split3_e4m3x2(float x0, float x1, uint32_t& t1, uint32_t& t2,
                                              uint32_t& t3) {
    float a0, a1;
    t1 = e4m3x2(x0, x1);
    e4m3x2_val(t1, a0, a1);
    const float r0 = (x0 - a0) * XRATIO, r1 = (x1 - a1) * XRATIO;
    t2 = e4m3x2(r0, r1);
    e4m3x2_val(t2, a0, a1);
    t3 = e4m3x2((r0 - a0) * XRATIO, (r1 - a1) * XRATIO);
}

// The three partial products of an expansion, combined: p1 + p2 / 32 + p3 / 1024.
__device__ __forceinline__ float combine3(uint32_t p1, uint32_t p2, uint32_t p3) {
    return fmaf(__uint_as_float(p3), 1.0f / (XRATIO * XRATIO),
                fmaf(__uint_as_float(p2), 1.0f / XRATIO, __uint_as_float(p1)));
}

// ---------------------------------------------------------------- TMEM, 4 / 8 columns
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                   "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t* r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}
// N consecutive columns (N a multiple of 4, at most 32) of this thread's TMEM lane.
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t* r) {
    static_assert(N % 4 == 0 && N > 0 && N <= 32, "column count");
    if constexpr (N >= 16) {
        tmem_ld16(taddr, r);
        if constexpr (N > 16) tmem_ldn<N - 16>(taddr + 16, r + 16);
    } else if constexpr (N >= 8) {
        tmem_ld8(taddr, r);
        if constexpr (N > 8) tmem_ldn<N - 8>(taddr + 8, r + 8);
    } else {
        tmem_ld4(taddr, r);
    }
}
template <int N>
__device__ __forceinline__ void tmem_stn(uint32_t taddr, const uint32_t* r) {
    static_assert(N % 4 == 0 && N > 0 && N <= 32, "column count");
    if constexpr (N >= 16) {
        tmem_st16(taddr, r);
        if constexpr (N > 16) tmem_stn<N - 16>(taddr + 16, r + 16);
    } else if constexpr (N >= 8) {
        tmem_st8(taddr, r);
        if constexpr (N > 8) tmem_stn<N - 8>(taddr + 8, r + 8);
    } else {
        tmem_st4(taddr, r);
    }
}

}  // namespace gqa
