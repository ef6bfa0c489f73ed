// Per-token-group FP8 quantiser: the step that produces the matmul's
// activation operand.  The matmul ("feat: optimize w8a8 block fp8 matmul for
// Hopper", FlagGems-vllm PR #693, Description) consumes E4M3 activations that
// carry one fp32 de-quantisation scale per token and 128-wide K group.  The
// pages do not say how that scale is chosen; this takes the plainest reading,
// the group's absolute maximum over 448 (the largest finite E4M3 magnitude),
// the same rule the seeded workloads use.
//
// For each row m and group g (128 columns, the last one possibly shorter):
//   s[m,g]   = amax_k |X[m,k]| / 448 in fp32 (1 where that quotient is 0)
//   A[m,k]   = e4m3fn_RNE(clamp(X[m,k] / s[m,g], -448, 448)), true fp32 division
//
// HBM-bound: eight lanes per (row, group), 16 elements per lane, 16-byte
// loads and stores, amax by shuffles inside the eight lanes.  The division by
// the scale is the correctly rounded one, computed two lanes at a time from
// the scale's reciprocal with two residual corrections.
#include <algorithm>
#include <cstdio>

#include "../../include/w8a8_block_fp8.h"
#include "kernels.cuh"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace w8a8 {
w8a8_status record_error(w8a8_status st, const char *message);

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Elements per lane and unit: 16.  The raw input words a lane holds for them
// (8 for 16-bit input, 16 for fp32), and the (row, group) units a team of
// eight lanes carries per pass (loaded before any is used).
template <int KIND> struct InFormat {
    static constexpr int kWords = KIND == W8A8_IN_FP32 ? 16 : 8;
    static constexpr int kUnroll = KIND == W8A8_IN_FP32 ? 2 : 4;
};

// A team of eight lanes quantises one (row, group) unit: each lane holds 16
// consecutive elements (two 16-byte loads of bf16/fp16, four of fp32), the
// group's amax is a three-step shuffle reduction inside the team, and each
// lane writes its 16 codes with one 16-byte store.  A warp's four teams take
// four consecutive units, so every pass of a warp reads 512 contiguous
// elements (a row's groups are adjacent and rows follow each other); the
// warp's kUnroll passes are loaded before any is used.
template <int KIND>
__global__ void __launch_bounds__(kThreads, 3)
    k_quant_group128(const void *__restrict__ X, uint8_t *__restrict__ A,
                     float *__restrict__ a_s, unsigned M, unsigned K, unsigned G,
                     unsigned *status)
{
    constexpr int kW = InFormat<KIND>::kWords, kU = InFormat<KIND>::kUnroll;
    constexpr int kEsize = KIND == W8A8_IN_FP32 ? 4 : 2;
    grid_launch_dependents();
    grid_dependency_wait();          // X comes from the work before this launch
    const unsigned warp = threadIdx.x >> 5;
    const unsigned team = (threadIdx.x >> 3) & 3;
    const unsigned lane8 = threadIdx.x & 7;
    const unsigned units = M * G;                              // < 2^31, checked by the host
    // The loop bound is per warp (the shuffles need every lane); a team past
    // the last unit carries zeros and stores nothing.
    const unsigned stride = gridDim.x * kWarps * 4 * kU;
    const unsigned stride_m = stride / G, stride_g = stride - stride_m * G;
    unsigned base = (blockIdx.x * kWarps + warp) * 4 * kU;
    unsigned m = base / G, g = base - m * G;                   // (row, group) of unit `base`
    for (; base < units; base += stride) {
        uint32_t w[kU][kW];
        unsigned row[kU], grp[kU];
        bool in[kU], live[kU];
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            unsigned gj = g + 4 * j + team, mj = m;
            while (gj >= G) {                                  // at most 4 kU / G + 1 steps
                gj -= G;
                ++mj;
            }
            live[j] = base + 4 * j + team < units;
            row[j] = mj;
            grp[j] = gj;
            const unsigned k = gj * 128 + 16 * lane8;
            in[j] = live[j] && k < K;                          // K % 16 == 0: whole chunks
            // (debug-bounds build: the row and the 16 columns lie inside X and A)
            if (in[j] && !in_bounds(mj < M && k + 16 <= K, status, SITE_BOUNDS_A))
                in[j] = false;
            if (in[j]) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    static_cast<const uint8_t *>(X) + (static_cast<size_t>(mj) * K + k) * kEsize);
#pragma unroll
                for (int i = 0; i < kW / 4; ++i) {
                    const uint4 t = src[i];
                    w[j][4 * i] = t.x;
                    w[j][4 * i + 1] = t.y;
                    w[j][4 * i + 2] = t.z;
                    w[j][4 * i + 3] = t.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < kW; ++i)
                    w[j][i] = 0u;
            }
        }
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            float amax = quant::amax16<KIND>(w[j]);
#pragma unroll
            for (int off = 4; off > 0; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const float s = quant::group_scale(amax);
            if (in[j]) {
                const size_t idx = static_cast<size_t>(row[j]) * K + grp[j] * 128 + 16 * lane8;
                *reinterpret_cast<uint4 *>(A + idx) = quant::encode16<KIND>(w[j], s);
            }
            if (live[j] && lane8 == 0 &&
                in_bounds(row[j] < M && grp[j] < G, status, SITE_BOUNDS_SCALES))
                a_s[static_cast<size_t>(row[j]) * G + grp[j]] = s;
        }
        m += stride_m;
        g += stride_g;
        if (g >= G) {
            g -= G;
            ++m;
        }
    }
}

}  // namespace
}  // namespace w8a8

extern "C" w8a8_status w8a8_quantize_fp8_per_token_group(const void *X_dev, w8a8_in_dtype x_dtype,
                                                         void *A_dev, float *a_s_dev, int64_t M,
                                                         int64_t K, int group_size,
                                                         w8a8_stream_t stream)
{
    using namespace w8a8;
    if (M < 0 || K < 0)
        return record_error(W8A8_ERR_INVALID_ARG, "negative size");
    if (x_dtype < W8A8_IN_BF16 || x_dtype > W8A8_IN_FP32)
        return record_error(W8A8_ERR_INVALID_ARG, "unknown input dtype");
    if (group_size != 128)
        return record_error(W8A8_ERR_UNSUPPORTED, "only 128-wide groups are supported");
    if (K < 16 || K % 16 != 0)
        return record_error(W8A8_ERR_UNSUPPORTED, "K must be a positive multiple of 16");
    if (K > (1ll << 31) - 1 || M * ((K + 127) / 128) > (1ll << 31) - 1)
        return record_error(W8A8_ERR_UNSUPPORTED, "M * ceil(K/128) and K must be below 2^31");
    if (M == 0)
        return W8A8_OK;
    if (!X_dev || !A_dev || !a_s_dev)
        return record_error(W8A8_ERR_INVALID_ARG, "null pointer argument");
    if ((reinterpret_cast<uintptr_t>(X_dev) | reinterpret_cast<uintptr_t>(A_dev)) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(a_s_dev) % 4 != 0)
        return record_error(W8A8_ERR_UNSUPPORTED, "X and A must be 16-byte aligned, a_s 4-byte");
    const int G = static_cast<int>((K + 127) / 128);
    const long long units = M * static_cast<long long>(G);
    void (*kernel)(const void *, uint8_t *, float *, unsigned, unsigned, unsigned, unsigned *) =
        x_dtype == W8A8_IN_BF16   ? k_quant_group128<W8A8_IN_BF16>
        : x_dtype == W8A8_IN_FP16 ? k_quant_group128<W8A8_IN_FP16>
                                  : k_quant_group128<W8A8_IN_FP32>;
    const int unroll = x_dtype == W8A8_IN_FP32 ? InFormat<W8A8_IN_FP32>::kUnroll
                                               : InFormat<W8A8_IN_BF16>::kUnroll;
    const long long units_per_pass = static_cast<long long>(kWarps) * 4 * unroll;
    // Persistent grid: as many CTAs as are resident on the GPU at once, each
    // striding over the units.
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "device query: %s", cudaGetErrorString(e));
        return record_error(W8A8_ERR_NO_DEVICE, msg);
    }
    long long blocks = (units + units_per_pass - 1) / units_per_pass;
    blocks = std::min<long long>(blocks, static_cast<long long>(sms) * std::max(per_sm, 1));
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    // The debug-bounds build's checks record into the device status word; the
    // release build compiles them away and passes no address.
    unsigned *status = nullptr;
    if (W8A8_DEBUG_BOUNDS && status_word_address(&status) != cudaSuccess)
        status = nullptr;
    e = cudaLaunchKernelEx(&lc, kernel, X_dev, static_cast<uint8_t *>(A_dev), a_s_dev,
                           static_cast<unsigned>(M), static_cast<unsigned>(K),
                           static_cast<unsigned>(G), status);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "kernel launch: %s", cudaGetErrorString(e));
        return record_error(W8A8_ERR_CUDA, msg);
    }
    return W8A8_OK;
}
