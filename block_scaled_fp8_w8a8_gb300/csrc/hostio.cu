// Host-to-device staging for the host-buffer entry point: one kernel reads
// every input of a call straight out of page-locked host memory (mapped into
// the device's address space, read over the CPU-GPU link) and writes it to the
// device staging area.  On a Grace-Blackwell node one such gather replaces the
// four copies of a call and their per-copy latency.
#include <cstdint>

#include "kernels.cuh"
#include "ptx.cuh"

namespace w8a8 {
namespace {

// 16-byte loads where source and destination allow them, then the tail (or a
// whole misaligned segment) byte by byte; grid-stride over each segment.  Under
// programmatic dependent launch the copy starts once the previous grid has
// finished and its writes are visible (a no-op without it), and the next grid
// may start its prologue as soon as every block of this one is running.
__global__ void __launch_bounds__(256) k_gather(const GatherSegs g)
{
    grid_dependency_wait();
    grid_launch_dependents();
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (int i = 0; i < g.count; ++i) {
        const uint8_t *src = g.src[i];
        uint8_t *dst = g.dst[i];
        const size_t n = g.bytes[i];
        const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
        const size_t n16 = vec ? n / 16 : 0;
        for (size_t j = tid; j < n16; j += stride)
            reinterpret_cast<uint4 *>(dst)[j] = reinterpret_cast<const uint4 *>(src)[j];
        for (size_t j = n16 * 16 + tid; j < n; j += stride)
            dst[j] = src[j];
    }
}

}  // namespace

cudaError_t launch_gather(const GatherSegs &segs, int grid, cudaStream_t stream, int pdl)
{
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(grid));
    lc.blockDim = dim3(256);
    lc.dynamicSmemBytes = 0;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&lc, k_gather, segs);
}

}  // namespace w8a8
