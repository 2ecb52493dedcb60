// gdr_forward_static_scratch: the staged forward with its scratch taken from a
// fixed array compiled into the library instead of a caller workspace.
//
// Who needs it: callers that must not allocate device memory themselves, such
// as a plugin whose host framework owns every byte of device memory and gives
// out no side buffers, or a latency-critical loop where a cudaMalloc (and the
// device-wide synchronisation it can cause) is not acceptable.  They pass only
// inputs and outputs; the scratch lives in g_static_scratch below.
//
// Costs and rules:
//  * g_static_scratch is GDR_STATIC_SCRATCH_BYTES of device memory that every
//    GPU which loads this part of the library keeps until the process exits.
//  * A problem whose staged scratch (gdr_forward_workspace_bytes) is larger is
//    rejected with GDR_ERR_WORKSPACE before anything is launched.
//  * Every call on a device uses the same array.  Two calls whose kernels can
//    overlap on the GPU (different streams, no ordering between them) race on
//    it and give wrong results; order them, e.g. issue them on one stream.
//  * The array keeps whatever the last call left there.  The staged kernels
//    write every scratch byte they read before reading it, so nothing has to
//    be cleared between calls.
//  * The first call on each device looks up the array's device address (with
//    that device current) and caches it.  Make that first call before any
//    stream capture begins on the calling thread.
//  * The cached address lives as long as the device's primary context.  After a
//    cudaDeviceReset (or any other teardown of that context) the array is a new
//    allocation and the cached address is stale: a process that resets a device
//    must not call this entry point on that device again.
//  * Variant AUTO runs what gdr_forward's AUTO runs when the fused path is left
//    out: the tensor-core stages for bf16 and fp16 io, the CUDA-core stages for
//    fp32 io.
#include <cuda_runtime.h>

#include <mutex>

#include "gdr.h"
#include "gdr_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[GDR_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up once per device).
gdr_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return GDR_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return GDR_OK;
}

}  // namespace

extern "C" gdr_status gdr_forward_static_scratch(const gdr_problem* p, const void* q, const void* k, const void* v,
                                                 const float* g, const void* beta, const float* h0, void* o,
                                                 float* h_final, void* stream) {
    if (!p) return GDR_ERR_NULL;
    if (p->variant == GDR_VARIANT_FUSED || p->variant == GDR_VARIANT_FUSED_TC)
        return GDR_ERR_UNSUPPORTED;   // only the staged variants are offered here
    gdr_problem staged = *p;
    if (staged.variant == GDR_VARIANT_AUTO)
        staged.variant = staged.io_dtype == GDR_F32 ? GDR_VARIANT_SIMT : GDR_VARIANT_TENSOR;
    const size_t need = gdr_forward_workspace_bytes(&staged);
    if (need == 0) {
        // the problem itself is invalid: let gdr_forward report why, launching nothing
        return gdr_forward(&staged, q, k, v, g, beta, h0, o, h_final, nullptr, 0, stream);
    }
    if (need > GDR_STATIC_SCRATCH_BYTES) return GDR_ERR_WORKSPACE;
    void* scratch = nullptr;
    gdr_status st = scratch_address(&scratch);
    if (st != GDR_OK) return st;
    return gdr_forward(&staged, q, k, v, g, beta, h0, o, h_final, scratch, GDR_STATIC_SCRATCH_BYTES, stream);
}
