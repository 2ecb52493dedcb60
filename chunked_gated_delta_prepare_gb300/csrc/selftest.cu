// gdr_selftest_bounded_wait: a check of the library's failure detection on the GPU.
//
// Every wait on an mbarrier in the kernels is bounded: when the phase it waits
// for does not complete within its poll limit, the kernel records
// GDR_ERR_DEVICE_TIMEOUT in the device error word and leaves through its normal
// exit, so the context stays usable and gdr_get_device_status reports it.  This
// entry point runs that path on purpose.  One CTA initialises an mbarrier that
// expects one arrival; with `arrive` = 0 nothing arrives and the wait, given
// `polls` polls, runs out; with `arrive` != 0 the thread arrives first and the
// wait succeeds.  Nothing else is in flight (no TMA, no tensor-core work), and
// no thread spins past its limit.
#include <cuda_runtime.h>

#include "blackwell.cuh"
#include "gdr.h"
#include "gdr_internal.h"

namespace gdr {
namespace {

__global__ void bounded_wait_selftest_kernel(uint32_t polls, int arrive, unsigned int* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        bw::mbar_init(&bar, 1);
        bw::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (arrive) bw::mbar_arrive(&bar);
        bw::mbar_wait(&bar, 0, err, kDeviceErrTimeout, polls);
    }
    __syncthreads();
}

}  // namespace
}  // namespace gdr

extern "C" gdr_status gdr_selftest_bounded_wait(int32_t polls, int32_t arrive, void* stream) {
    if (polls < 1 || (uint32_t)polls > gdr::bw::kMaxPolls) return GDR_ERR_ARG;
    unsigned int* err = nullptr;
    if (gdr::device_error_ptr(&err) != cudaSuccess || !err) return GDR_ERR_CUDA;
    gdr::bounded_wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint32_t)polls, arrive, err);
    return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}
