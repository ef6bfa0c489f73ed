// Epilogue shared by the tiled kernels (tokens on the MMA M side): a warp's
// 32 rows of fp32 accumulators leave through swizzled shared-memory chunks and
// TMA stores.
#pragma once

#include "kernels.cuh"
#include "ptx.cuh"

namespace w8a8 {

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_out2(uint64_t pair, bool bf)
{
    float lo, hi;
    unpack2f(pair, lo, hi);
    return bf ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

// Epilogue of one warp: its 32 rows (lane = row) x 2*NP accumulator columns
// (NP fp32 pairs) go out in chunks of 64 bytes per row.  Each chunk is written
// to one of the warp's EB buffers of 2 KB in the layout a TMA store with the
// 64-byte swizzle reads (16-byte piece j of row r at r*64 + 16*(j ^ ((r >> 1) & 3)),
// which also spreads a quarter-warp's 16-byte writes over all banks), then one
// lane issues the store of the box {64 bytes of columns, 32 rows} at (x, y).
// A buffer is rewritten only once the store that last used it (EB stores
// earlier, possibly in the previous tile) has finished reading it.
template <int NP, int EB>
__device__ __forceinline__ void store_tile_rows(const uint64_t (&acc)[NP], const CUtensorMap *tmC,
                                                uint32_t buf0, uint32_t lane, int col0, int y,
                                                int N, int out_kind)
{
    const uint32_t sw = (lane >> 1) & 3u;
    const bool fp32 = out_kind == OUT_FP32;
    const bool bf = out_kind == OUT_BF16;
    const int chunks = fp32 ? NP / 8 : NP / 16;
    const int ccols = fp32 ? 16 : 32;
#pragma unroll
    for (int k = 0; k < NP / 8; ++k) {
        const int x = col0 + ccols * k;
        if (k >= chunks || x >= N)
            break;
        const uint32_t buf = buf0 + 2048u * (k % EB);
        if (lane == 0)
            tma_store_wait_read_n<EB - 1>();
        __syncwarp();
        const uint32_t rowa = buf + lane * 64u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (fp32) {
                const uint64_t p0 = acc[8 * k + 2 * j], p1 = acc[8 * k + 2 * j + 1];
                st_shared_v4(rowa + 16u * (j ^ sw), static_cast<uint32_t>(p0),
                             static_cast<uint32_t>(p0 >> 32), static_cast<uint32_t>(p1),
                             static_cast<uint32_t>(p1 >> 32));
            } else if (k < NP / 16) {
                const int b = 16 * k + 4 * j;
                st_shared_v4(rowa + 16u * (j ^ sw), pack_out2(acc[b], bf),
                             pack_out2(acc[b + 1], bf), pack_out2(acc[b + 2], bf),
                             pack_out2(acc[b + 3], bf));
            }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmC, buf, x, y);
            tma_store_commit();
        }
    }
}

}  // namespace w8a8
