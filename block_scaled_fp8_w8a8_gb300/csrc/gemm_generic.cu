// Generic W8A8 block-FP8 matmul on the CUDA cores: the fall-through for every
// problem outside the tensor-core kernels' guards.
//
// Operation ("feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm
// PR #693, Description; the page's dispatcher routes any shape its
// specialised kernels do not take to one generic kernel):
//   C[m,n] = cast( sum_g a_s[m,g] * b_s[n / block_n, g] * sum_{k in g} A[m,k] B[n,k] )
// with groups g of block_k consecutive k (the last one may be shorter), any
// block_n >= 1, any M, N, K (K = 0 gives zeros), any row strides (in
// elements) for A, B, C, a_s and b_s, and any alignment.
//
// One CTA of 256 threads computes a 64 x 64 tile of C, each thread a 4 x 4
// block.  The K loop runs in chunks of at most 32 that never cross a scale
// group: the chunk's A and B bytes are decoded (exactly: E4M3 -> half -> float)
// into shared memory, each thread accumulates its 16 products of the group in
// fp32 (every product of two E4M3 values is exact in fp32), and at the end of
// a group folds them into its accumulators with one FMA by
// a_s[m, g] * b_s[n / block_n, g].  Plain loads with bounds checks: no TMA, no
// alignment requirement.
#include <cuda_fp8.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace w8a8 {

namespace {

constexpr int kTile = 64;      // rows and columns of C per CTA
constexpr int kChunk = 32;     // K elements staged per round (within one group)
constexpr int kPad = kTile + 1;

__device__ __forceinline__ float e4m3_to_float(uint8_t code)
{
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);
    return __half2float(__half(h));
}

__global__ void __launch_bounds__(256) k_generic(const GenericParams p)
{
    __shared__ float As[kChunk][kPad];
    __shared__ float Bs[kChunk][kPad];
    const int tid = static_cast<int>(threadIdx.x);
    const int tx = tid & 15, ty = tid >> 4;
    // one-dimensional grid over the (M tile, N tile) pairs, N tiles fastest
    const int64_t tiles_n = (p.N + kTile - 1) / kTile;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) / tiles_n * kTile;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) % tiles_n * kTile;

    grid_dependency_wait();

    float acc[4][4], part[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            acc[i][j] = 0.f;

    const int64_t G = p.K > 0 ? (p.K + p.block_k - 1) / p.block_k : 0;
    for (int64_t g = 0; g < G; ++g) {
        const int64_t kg0 = g * p.block_k;
        const int64_t kg1 = min(kg0 + p.block_k, p.K);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                part[i][j] = 0.f;
        for (int64_t k0 = kg0; k0 < kg1; k0 += kChunk) {
            const int kc = static_cast<int>(min(static_cast<int64_t>(kChunk), kg1 - k0));
            // Stage: 64 rows x kc bytes of A and of B, decoded; zeros past M / N.
            for (int e = tid; e < kTile * kChunk; e += 256) {
                const int r = e / kChunk, c = e - (e / kChunk) * kChunk;
                float av = 0.f, bv = 0.f;
                if (c < kc) {
                    const int64_t m = m0 + r, n = n0 + r;
                    // (the debug-bounds build re-checks each index against K)
                    if (m < p.M && in_bounds(k0 + c < p.K, p.status, SITE_BOUNDS_A))
                        av = e4m3_to_float(p.A[m * p.lda + k0 + c]);
                    if (n < p.N && in_bounds(k0 + c < p.K, p.status, SITE_BOUNDS_B))
                        bv = e4m3_to_float(p.B[n * p.ldb + k0 + c]);
                }
                As[c][r] = av;
                Bs[c][r] = bv;
            }
            __syncthreads();
            for (int c = 0; c < kc; ++c) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    a[i] = As[c][ty * 4 + i];
                    b[i] = Bs[c][tx * 4 + i];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        part[i][j] = fmaf(a[i], b[j], part[i][j]);
            }
            __syncthreads();
        }
        // Promotion of the group: acc += (a_s[m,g] * b_s[n/block_n,g]) * part.
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t m = m0 + ty * 4 + i;
            const float sa = m < p.M ? p.a_s[m * p.ld_as + g] : 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t n = n0 + tx * 4 + j;
                const float sb = n < p.N ? p.b_s[(n / p.block_n) * p.ld_bs + g] : 0.f;
                acc[i][j] = fmaf(sa * sb, part[i][j], acc[i][j]);
            }
        }
    }

    grid_launch_dependents();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + ty * 4 + i;
        if (m >= p.M)
            continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t n = n0 + tx * 4 + j;
            if (n >= p.N)
                continue;
            const int64_t idx = m * p.ldc + n;
            if (!in_bounds(n < p.ldc, p.status, SITE_BOUNDS_C))   // (debug-bounds build)
                continue;
            if (p.out_kind == OUT_FP32)
                static_cast<float *>(p.C)[idx] = acc[i][j];
            else if (p.out_kind == OUT_BF16)
                static_cast<__nv_bfloat16 *>(p.C)[idx] = __float2bfloat16_rn(acc[i][j]);
            else
                static_cast<__half *>(p.C)[idx] = __float2half_rn(acc[i][j]);
        }
    }
}

}  // namespace

cudaError_t launch_generic(const GenericParams &p, const LaunchCfg &cfg)
{
    const int64_t tiles = ((p.N + kTile - 1) / kTile) * ((p.M + kTile - 1) / kTile);
    if (tiles <= 0)
        return cudaSuccess;
    if (tiles > 0x7fffffff)
        return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(tiles), 1, 1);
    lc.blockDim = dim3(256, 1, 1);
    lc.dynamicSmemBytes = 0;
    lc.stream = cfg.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = cfg.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&lc, k_generic, p);
}

}  // namespace w8a8
