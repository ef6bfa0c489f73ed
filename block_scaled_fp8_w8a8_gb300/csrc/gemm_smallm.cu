// Small-M W8A8 block-FP8 matmul on the CUDA cores, for decode batches of at
// most 16 tokens.
//
// Operation ("feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm
// PR #693, Description):
//   C[m,n] = cast( sum_g a_s[m,g] * b_s[n/128,g] * sum_{k in g} A[m,k] B[n,k] )
//
// With M <= 16 the product is a handful of dot products per weight row: the
// weight stream is the whole cost, and the tensor-core kernels' fixed chain
// (tensor memory, MMA issue, promotion and TMA-store hand-offs between warps)
// is longer than the arithmetic.  Here one CTA owns 32 weight rows, streams
// them into shared memory with TMA (one 32 x 128-byte box per K group, one
// mbarrier per group; with programmatic dependent launch and static weights
// before the dependency wait), converts the tokens' activations to fp32 in
// shared memory, and computes with paired fp32 FMAs: lane = weight row, the 8
// warps split the 16-element K chunks, so every activation read is a broadcast.
// Each chunk's partial sum is scaled by a_s[m,g] * b_s[n/128,g] as it is added
// (the group sum split into chunk sums: the same value up to fp32 rounding).
// The 8 warps' sums are added in warp order through shared memory and stored.
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace w8a8 {

namespace {

constexpr int kRows = 32;           // weight rows per CTA (one per lane)
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr uint32_t kBoxBytes = kRows * 128;   // one K group of the CTA's rows

struct SmallLayout {
    size_t b_off, a_off, s_off, red_off, bar_off, flag_off, total;
};

__host__ __device__ inline SmallLayout small_layout(int mm, int K, int G)
{
    SmallLayout l;
    l.b_off = 0;                                             // 1024-aligned base
    l.a_off = l.b_off + static_cast<size_t>(G) * kBoxBytes;
    l.s_off = l.a_off + static_cast<size_t>(mm) * K * 4;
    l.red_off = l.s_off + static_cast<size_t>(mm) * G * 4;
    l.bar_off = l.red_off + static_cast<size_t>(kWarps) * kRows * mm * 4;
    l.bar_off = (l.bar_off + 7) & ~static_cast<size_t>(7);
    l.flag_off = l.bar_off + static_cast<size_t>(G) * 8;
    l.total = 1024 + l.flag_off + 16;                        // + alignment slack
    return l;
}

// 16 E4M3 codes -> 16 floats (exact: every E4M3 value is an fp16 value).
__device__ __forceinline__ void decode16(const uint4 v, float (&f)[16])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t pair;
            const unsigned short two = static_cast<unsigned short>(w[i] >> (16 * h));
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(pair) : "h"(two));
            const __half2 hv = *reinterpret_cast<const __half2 *>(&pair);
            f[4 * i + 2 * h] = __low2float(hv);
            f[4 * i + 2 * h + 1] = __high2float(hv);
        }
    }
}

__device__ __forceinline__ void store_out(void *C, size_t idx, float v, int out_kind)
{
    if (out_kind == OUT_FP32)
        static_cast<float *>(C)[idx] = v;
    else if (out_kind == OUT_BF16)
        static_cast<__nv_bfloat16 *>(C)[idx] = __float2bfloat16_rn(v);
    else
        static_cast<__half *>(C)[idx] = __float2half_rn(v);
}

template <int MM>
__global__ void __launch_bounds__(kThreads)
    k_smallm(const __grid_constant__ CUtensorMap tmB, const SmallParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const SmallLayout l = small_layout(MM, p.K, p.G);
    const uint32_t sB = smem_addr(smem + l.b_off);
    float *sA = reinterpret_cast<float *>(smem + l.a_off);
    float *sS = reinterpret_cast<float *>(smem + l.s_off);
    float *sRed = reinterpret_cast<float *>(smem + l.red_off);
    const uint32_t bar0 = smem_addr(smem + l.bar_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + l.flag_off);

    const int tid = static_cast<int>(threadIdx.x);
    const int warp = tid >> 5, lane = tid & 31;
    const int n0 = static_cast<int>(blockIdx.x) * kRows;
    const int nb = n0 / 128;                   // the CTA's rows lie in one b_s row block
    const int G = p.G, K = p.K, M = p.M;

    if (tid == 0) {
        for (int g = 0; g < G; ++g)
            mbar_init(bar0 + 8u * g, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmB);
    }
    __syncthreads();
    const WaitGuard guard{abort_flag, p.status, p.wait_limit};

    auto issue_weights = [&]() {
        for (int g = 0; g < G; ++g) {
            // (debug-bounds build: a box outside B is skipped like a skipped load)
            if (g == p.debug_skip_tma || !in_bounds(n0 < p.N && g * 128 < p.K, p.status, SITE_BOUNDS_B))
                continue;
            mbar_arrive_expect_tx(bar0 + 8u * g, kBoxBytes);
            tma_load_2d(sB + g * kBoxBytes, &tmB, bar0 + 8u * g, g * 128, n0);
        }
    };
    if (tid == 0 && p.prefetch_weights)
        issue_weights();                       // the weights do not depend on the previous grid
    grid_launch_dependents();
    grid_dependency_wait();
    if (tid == 0 && !p.prefetch_weights)
        issue_weights();

    // Activations -> fp32 rows of K in shared memory; folded scales s[m][g].
    const int chunks = K / 16;
    for (int c = tid; c < M * chunks; c += kThreads) {
        const int m = c / chunks, k0 = (c - m * chunks) * 16;
        const uint4 v = in_bounds(m < p.M && k0 + 16 <= p.K, p.status, SITE_BOUNDS_A)
                            ? *reinterpret_cast<const uint4 *>(p.A + static_cast<size_t>(m) * p.lda + k0)
                            : make_uint4(0u, 0u, 0u, 0u);
        float f[16];
        decode16(v, f);
        float4 *dst = reinterpret_cast<float4 *>(sA + static_cast<size_t>(m) * K + k0);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            dst[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
    }
    for (int i = tid; i < M * G; i += kThreads) {
        const int m = i / G, g = i - m * G;
        sS[m * G + g] = in_bounds(m < p.M && nb * 128 < p.N, p.status, SITE_BOUNDS_SCALES)
                            ? p.a_s[static_cast<size_t>(m) * G + g] *
                                  p.b_s[static_cast<size_t>(nb) * G + g]
                            : 0.f;
    }
    __syncthreads();

    // Lane = weight row n0 + lane; warp w takes chunks w, w + 8, ...
    float acc[MM];
#pragma unroll
    for (int m = 0; m < MM; ++m)
        acc[m] = 0.f;
    int ready = -1;                            // last group whose weights this thread saw land
    bool ok = true;
    const uint32_t row_base = sB + static_cast<uint32_t>(lane) * 128u;
    for (int c = warp; c < chunks; c += kWarps) {
        const int g = c >> 3;
        if (g != ready) {
            ok = __all_sync(0xffffffffu, wait_bounded(bar0 + 8u * g, 0, guard, SITE_SMALL_WEIGHTS));
            if (!ok)
                break;
            ready = g;
        }
        // 128-byte swizzle of the TMA box: chunk j of row r sits at (j ^ (r & 7)).
        const uint32_t addr = row_base + g * kBoxBytes +
                              static_cast<uint32_t>(((c & 7) ^ (lane & 7)) * 16);
        uint4 bv;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(bv.x), "=r"(bv.y), "=r"(bv.z), "=r"(bv.w)
                     : "r"(addr));
        float bf[16];
        decode16(bv, bf);
        uint64_t b2[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            b2[j] = pack2f(bf[2 * j], bf[2 * j + 1]);
#pragma unroll
        for (int m = 0; m < MM; ++m) {
            if (m < M) {
                const float4 *a4 = reinterpret_cast<const float4 *>(sA + static_cast<size_t>(m) * K + c * 16);
                uint64_t part0 = 0ull, part1 = 0ull;     // two chains: half the latency
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 a = a4[q];
                    fma2(part0, pack2f(a.x, a.y), b2[2 * q]);
                    fma2(part1, pack2f(a.z, a.w), b2[2 * q + 1]);
                }
                float l0, h0, l1, h1;
                unpack2f(part0, l0, h0);
                unpack2f(part1, l1, h1);
                acc[m] = fmaf(sS[m * G + g], (l0 + h0) + (l1 + h1), acc[m]);
            }
        }
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        // A bounded wait ran out (the status word says where): wait, still
        // bounded, for every weight load that was issued, then leave; C is undefined.
        if (tid == 0)
            for (int g = 0; g < G; ++g)
                if (g != p.debug_skip_tma)
                    wait_drain(bar0 + 8u * g, 0, p.status, p.wait_limit, (SITE_DRAIN << 8) | 4u);
        return;
    }

    // Sum the 8 warps' partials in warp order and store C[m][n0 + r]; the
    // partials sit lane-fastest ([warp][m][row]), so that neither the writes
    // nor the reads below meet bank conflicts.
#pragma unroll
    for (int m = 0; m < MM; ++m)
        sRed[(warp * MM + m) * kRows + lane] = acc[m];
    __syncthreads();
    for (int o = tid; o < kRows * M; o += kThreads) {
        const int m = o / kRows, r = o - m * kRows;
        const int n = n0 + r;
        if (n >= p.N)
            continue;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            s += sRed[(w * MM + m) * kRows + r];
        if (in_bounds(m < p.M, p.status, SITE_BOUNDS_C))
            store_out(p.C, static_cast<size_t>(m) * p.ldc + n, s, p.out_kind);
    }
}

template <int MM>
cudaError_t launch_smallm_t(const CUtensorMap &tmB, const SmallParams &p, const LaunchCfg &cfg)
{
    auto kernel = k_smallm<MM>;
    static volatile int smem_set[kMaxDeviceFlags] = {};
    cudaError_t e = ensure_smem_limit(kernel, smem_set);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((p.N + kRows - 1) / kRows, 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = small_layout(MM, p.K, p.G).total;
    lc.stream = cfg.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = cfg.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&lc, kernel, tmB, p);
}

int mm_for(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

}  // namespace

size_t smallm_smem_bytes(int M, int K)
{
    if (M < 1 || M > kSmallMaxM)
        return 0;
    return small_layout(mm_for(M), K, (K + 127) / 128).total;
}

cudaError_t launch_smallm(const CUtensorMap &tmB, const SmallParams &p, const LaunchCfg &cfg)
{
    switch (mm_for(p.M)) {
    case 1: return launch_smallm_t<1>(tmB, p, cfg);
    case 2: return launch_smallm_t<2>(tmB, p, cfg);
    case 4: return launch_smallm_t<4>(tmB, p, cfg);
    case 8: return launch_smallm_t<8>(tmB, p, cfg);
    default: return launch_smallm_t<16>(tmB, p, cfg);
    }
}

}  // namespace w8a8
