// Per-group promotion shared by the tiled kernels (tokens on the MMA M side):
// one thread owns one TMEM lane (one output row) and 2*NP consecutive
// columns of the group partial P_g, and adds s * P_g to its fp32 accumulator
// pairs, where s = a_s[m,g] * b_s[n/128,g] ("feat: optimize w8a8 block fp8
// matmul for Hopper", FlagGems-vllm PR #693, Description: block-wise
// de-quantisation with FP32 accumulation).
#pragma once

#include "ptx.cuh"

namespace w8a8 {

// The partial is read in 32-column chunks with two register buffers: the load
// of chunk c + 1 is in flight while chunk c's 16 paired FMAs run, so a warp's
// TMEM round trips overlap its own arithmetic.  `release()` hands the buffer
// back after the last FMA.  (Measured on GB300 at 16384 x 4096 x 4096: the same
// time as loading 64 columns at a time and waiting for each load; releasing
// the buffer before the last chunk's FMAs made the CTA-pair kernel 10-20 %
// slower; with the FMAs removed, on the other hand, a launch is 20 % shorter:
// the promotion's cost is its instructions, not its TMEM reads.)  Each output
// element receives exactly one fma per group, in group order.
template <int NP, typename Release>
__device__ __forceinline__ void promote_group(uint64_t (&acc)[NP], uint32_t taddr, uint64_t s2,
                                              Release &&release)
{
    static_assert(NP % 16 == 0, "whole 32-column chunks");
    constexpr int kChunks = NP / 16;
    uint32_t va[32], vb[32];
    tmem_ld32_async(taddr, va);
    tmem_wait_ld32(va);
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        uint32_t(&cur)[32] = (c & 1) ? vb : va;
        uint32_t(&nxt)[32] = (c & 1) ? va : vb;
        if (c + 1 < kChunks)
            tmem_ld32_async(taddr + 32u * static_cast<uint32_t>(c + 1), nxt);
#pragma unroll
        for (int j = 0; j < 16; ++j)
            fma2(acc[16 * c + j], s2, pack2(cur[2 * j], cur[2 * j + 1]));
        if (c + 1 < kChunks)
            tmem_wait_ld32(nxt);
    }
    release();
}

}  // namespace w8a8
