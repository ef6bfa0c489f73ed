// Per-device status word written by kernels whose bounded waits ran out.
#include "kernels.cuh"

namespace w8a8 {

__device__ unsigned g_device_status_word;

cudaError_t status_word_address(unsigned **out)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(out), g_device_status_word);
}

}  // namespace w8a8
