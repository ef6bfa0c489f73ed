// Per-token-group E4M3 quantisation arithmetic shared by the stand-alone
// quantiser kernel and the matmul kernels that quantise their activation
// operand on the fly, so that both produce the same codes and scales bit for
// bit.  For one 128-wide group of a token (reading fixed by the quantiser's
// C-ABI declaration): s = amax / 448 in fp32 (1 where that quotient is 0);
// code = E4M3(x / s) with the correctly rounded fp32 quotient, round to
// nearest even, saturating; the sign bit copied from x.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "../../include/w8a8_block_fp8.h"
#include "ptx.cuh"

namespace w8a8 {
namespace quant {

// Element i (0..15) of a lane's raw words, as fp32 (exact).
template <int KIND>
__device__ __forceinline__ float element(const uint32_t *w, int i)
{
    if constexpr (KIND == W8A8_IN_FP32) {
        return __uint_as_float(w[i]);
    } else if constexpr (KIND == W8A8_IN_BF16) {
        return __uint_as_float((i & 1) ? (w[i >> 1] & 0xffff0000u) : (w[i >> 1] << 16));
    } else {
        const __half2 h = *reinterpret_cast<const __half2 *>(&w[i >> 1]);
        return __half2float((i & 1) ? h.y : h.x);
    }
}

// For elements 4c..4c+3: a word whose byte i carries element 4c+i's sign bit
// in its top bit (the input byte that holds the sign, moved into place).
template <int KIND>
__device__ __forceinline__ uint32_t sign_bytes(const uint32_t *w, int c)
{
    if constexpr (KIND == W8A8_IN_FP32)
        return __byte_perm(__byte_perm(w[4 * c], w[4 * c + 1], 0x7373),
                           __byte_perm(w[4 * c + 2], w[4 * c + 3], 0x7373), 0x5410);
    else
        return __byte_perm(w[2 * c], w[2 * c + 1], 0x7531);
}

// x / s rounded to nearest even on two lanes, given y = RN(1/s) and -s.
// Markstein's method (P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): a
// quotient within one ulp of x/s plus the exactly computed residual
// (x - s*q) times the correctly rounded reciprocal rounds to the correctly
// rounded quotient.  The first correction turns RN(x*y) (within about 2 ulp)
// into such a quotient.  Valid while no step under- or overflows: the caller
// keeps s within [2^-64, 2^64] and |x| <= 448 s (1 + 2^-23), and only
// quotients that round to an E4M3 code other than zero need the last bit
// right (|x/s| >= 2^-11, where every residual stays normal).  The sign of a
// zero quotient may come out wrong; the caller sets every code's sign from x.
__device__ __forceinline__ uint64_t div_by_scale2(uint64_t x, uint64_t neg_s, uint64_t y)
{
    constexpr uint64_t kNegZero = 0x8000000080000000ull;       // x * y + (-0) == RN(x * y)
    uint64_t q = fma2_rn(x, y, kNegZero);
    uint64_t r = fma2_rn(neg_s, q, x);
    q = fma2_rn(r, y, q);
    r = fma2_rn(neg_s, q, x);
    return fma2_rn(r, y, q);
}

// Codes of elements 4c..4c+3: byte i = E4M3(x_i / s) with x_i's sign bit.
template <int KIND, bool FAST>
__device__ __forceinline__ uint32_t encode4(const uint32_t *w, int c, float s, uint64_t neg_s,
                                            uint64_t y)
{
    uint32_t two[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const float x0 = element<KIND>(w, 4 * c + 2 * p), x1 = element<KIND>(w, 4 * c + 2 * p + 1);
        float2 q;
        if constexpr (FAST) {
            unpack2f(div_by_scale2(pack2f(x0, x1), neg_s, y), q.x, q.y);
        } else {
            q.x = __fdiv_rn(x0, s);
            q.y = __fdiv_rn(x1, s);
        }
        // |q| <= 448 (1 + 2^-23) except where a subnormal scale lost precision;
        // the saturating conversion is then the clamp to +-448.
        two[p] = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);
    }
    return __byte_perm(two[0], two[1], 0x5410) | (sign_bytes<KIND>(w, c) & 0x80808080u);
}

// The group scale from the group's absolute maximum.
__device__ __forceinline__ float group_scale(float amax)
{
    if (amax == 0.f)             // all-zero group (kept off the divide's special-case path)
        return 1.f;
    const float s = __fdiv_rn(amax, 448.f);
    return s == 0.f ? 1.f : s;   // a max so small that the quotient underflows
}

// Codes of a lane's 16 elements under scale s, as four words (byte order =
// element order).  The division is the fast exact form where s allows it
// (the same for every lane of a group, so the branch does not diverge).
template <int KIND>
__device__ __forceinline__ uint4 encode16(const uint32_t *w, float s)
{
    uint4 out;
    if (s >= 0x1p-64f && s <= 0x1p64f) {
        const float y = __frcp_rn(s);
        const uint64_t y2 = pack2f(y, y), ns2 = pack2f(-s, -s);
        out.x = encode4<KIND, true>(w, 0, s, ns2, y2);
        out.y = encode4<KIND, true>(w, 1, s, ns2, y2);
        out.z = encode4<KIND, true>(w, 2, s, ns2, y2);
        out.w = encode4<KIND, true>(w, 3, s, ns2, y2);
    } else {
        out.x = encode4<KIND, false>(w, 0, s, 0, 0);
        out.y = encode4<KIND, false>(w, 1, s, 0, 0);
        out.z = encode4<KIND, false>(w, 2, s, 0, 0);
        out.w = encode4<KIND, false>(w, 3, s, 0, 0);
    }
    return out;
}

// |x| maximum over a lane's 16 elements.
template <int KIND>
__device__ __forceinline__ float amax16(const uint32_t *w)
{
    if constexpr (KIND == W8A8_IN_BF16) {
        // Two bf16 lanes at a time: |x| by clearing the sign bits, then
        // max.bf16x2, which like fmaxf returns the other operand when one is
        // NaN and keeps subnormals; the maximum of bf16 values is one of them,
        // so it is exact and equals the fp32 maximum below.
        uint32_t m2 = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t a = w[i] & 0x7fff7fffu;
            asm("max.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(m2), "r"(a));
        }
        return fmaxf(0.f, fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xffff0000u)));
    } else {
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            m = fmaxf(m, fabsf(element<KIND>(w, i)));
        return m;
    }
}

}  // namespace quant
}  // namespace w8a8
