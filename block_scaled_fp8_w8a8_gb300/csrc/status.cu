// Per-device status word written by kernels whose bounded waits ran out, and
// the empty kernel that measures the launch floor of a dependent chain.
#include "../../include/w8a8_block_fp8.h"
#include "kernels.cuh"

namespace w8a8 {
w8a8_status record_error(w8a8_status st, const char *message);

__device__ unsigned g_device_status_word;

cudaError_t status_word_address(unsigned **out)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(out), g_device_status_word);
}

}  // namespace w8a8

namespace w8a8 {
namespace {

// One CTA that takes part in programmatic dependent launch and does nothing
// else: the shortest possible link of a dependent kernel chain.
__global__ void k_launch_floor()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace
}  // namespace w8a8

extern "C" w8a8_status w8a8_launch_floor_kernel(int pdl, w8a8_stream_t stream)
{
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(1, 1, 1);
    lc.blockDim = dim3(32, 1, 1);
    lc.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&lc, w8a8::k_launch_floor);
    if (e != cudaSuccess)
        return w8a8::record_error(W8A8_ERR_CUDA, cudaGetErrorString(e));
    return W8A8_OK;
}
