// Split-K matmul for callers that cannot allocate device memory.
//
// The split-K variant needs scratch memory for its fp32 partial sums and its
// per-tile arrival counters.  The regular entry points take that scratch from
// the caller or allocate it with cudaMalloc on first use.  Some callers can do
// neither: a serving runtime that reserves all device memory in its own pool at
// start-up and forbids later allocations, a plugin running inside a host
// application that owns the device memory and exposes no allocator to it, or
// latency-sensitive code where a cudaMalloc / cudaFree would implicitly
// synchronise the device and stall other streams.  This entry point serves
// them: its scratch is a fixed array in device memory that is part of the
// library's module (every GPU that loads the library holds it until the
// process exits), so a call allocates nothing.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/w8a8_block_fp8.h"
#include "kernels.cuh"

namespace w8a8 {
w8a8_status record_error(w8a8_status st, const char *message);
}

namespace {

constexpr size_t kScratchBytes = W8A8_NOALLOC_SCRATCH_BYTES;
using w8a8::kCounterBytes;   // the split-K counter block at the start of the scratch
static_assert(kScratchBytes > kCounterBytes, "scratch must hold the counter block");

// The shared scratch.  In host code this name is only a stand-in for the device
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_dev[kMaxDevices] = {};

// Set-up, once per device, with that device current: look up the device
// address of the scratch array.
w8a8_status scratch_address(void **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return w8a8::record_error(W8A8_ERR_NO_DEVICE, "no usable current CUDA device");
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_dev[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(scratch) failed: %s",
                     cudaGetErrorString(e));
            return w8a8::record_error(W8A8_ERR_CUDA, msg);
        }
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return W8A8_OK;
}

}  // namespace

namespace w8a8 {
// Forget the looked-up addresses (w8a8_shutdown): after a cudaDeviceReset the
// module is reloaded, possibly elsewhere, so the next call repeats the set-up.
void noalloc_forget()
{
    std::lock_guard<std::mutex> lock(g_mutex);
    for (void *&p : g_scratch_dev)
        p = nullptr;
}
}  // namespace w8a8

extern "C" w8a8_status w8a8_block_fp8_matmul_splitk_noalloc(
    const void *A_dev, const float *a_s_dev, const void *B_dev, const float *b_s_dev,
    void *C_dev, int64_t M, int64_t N, int64_t K, int block_n, int block_k,
    w8a8_out_dtype out_dtype, int split_k, w8a8_stream_t stream)
{
    if (split_k < 0)
        return w8a8::record_error(W8A8_ERR_INVALID_ARG, "split_k must be >= 0");
    if (block_n != 128 || block_k != 128)
        return w8a8::record_error(W8A8_ERR_UNSUPPORTED, "only [128, 128] scale blocks");
    w8a8_options opts = {};
    opts.variant = W8A8_VARIANT_SPLITK;
    opts.split_k = split_k;
    w8a8_options plan = {};
    // Checks the problem and sizes the scratch this call needs.
    w8a8_status st = w8a8_block_fp8_plan(M, N, K, out_dtype, &opts, &plan);
    if (st != W8A8_OK)
        return st;
    if (M == 0)
        return W8A8_OK;
    if (plan.workspace_bytes > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "problem needs %zu bytes of split-K scratch; the allocation-free entry point "
                 "has %zu (use fewer splits or the regular entry point)",
                 plan.workspace_bytes, kScratchBytes);
        return w8a8::record_error(W8A8_ERR_WORKSPACE, msg);
    }
    void *scratch = nullptr;
    if ((st = scratch_address(&scratch)) != W8A8_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (plan.workspace_bytes > 0) {
        // The array keeps the previous call's contents: zero the arrival
        // counters this call uses (its partial sums are fully overwritten).
        const int64_t m_tile = plan.m_tile > 0 ? plan.m_tile : 1;
        const size_t tiles = static_cast<size_t>((M + m_tile - 1) / m_tile) * ((N + 127) / 128);
        const size_t bytes = tiles * 4 <= kCounterBytes ? tiles * 4 : kCounterBytes;
        cudaError_t e = cudaMemsetAsync(scratch, 0, bytes, s);
        if (e != cudaSuccess) {
            char msg[256];
            snprintf(msg, sizeof(msg), "cudaMemsetAsync(scratch counters) failed: %s",
                     cudaGetErrorString(e));
            return w8a8::record_error(W8A8_ERR_CUDA, msg);
        }
    }
    opts.workspace_dev = scratch;
    opts.workspace_bytes = kScratchBytes;
    return w8a8_block_fp8_matmul_ex(A_dev, a_s_dev, B_dev, b_s_dev, C_dev, M, N, K, block_n,
                                    block_k, out_dtype, stream, &opts);
}
