// The device error word.  Kernels whose waits are bounded (mbarrier polls) get
// its address as an argument and write a nonzero code there when a wait gives
// up, then leave; nothing traps.  The host reads and clears it after a sync.
#include <cuda_runtime.h>

#include "gdr_internal.h"

namespace gdr {

__device__ unsigned int g_device_error;

cudaError_t device_error_ptr(unsigned int** ptr) {
    return cudaGetSymbolAddress((void**)ptr, g_device_error);
}

cudaError_t read_and_clear_device_error(unsigned int* code) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
}

}  // namespace gdr
