// Packed variable-length sequences.  Sequence s of a packed tensor [total, ...]
// holds the token rows cu[s] .. cu[s + 1] - 1 (cu: cumulative lengths, device
// int32 [n + 1]).  The library runs such a batch as n rows of T tokens each:
// varlen_pack moves sequence s into row s and fills the rest of the row with
// zero tokens; varlen_unpack moves the first len_s tokens of every row back to
// the packed tensor.  A zero token (beta = 0, g = 0, q = k = v = 0) leaves the
// state as it was and its output is dropped, so row s computes exactly sequence
// s: the partial-chunk reading of the recurrence, carried to the end of the row.
//
// One launch moves up to kMaxCopies tensors (blockIdx.y picks the tensor), each
// a run of token rows of row_bytes bytes, in the widest unit (16, 8, 4, 2 or 1
// bytes) that divides the row and both base addresses.  Spans are clamped:
// start to [0, total], length to [0, min(T, total - start)], so even a cu the
// host did not check cannot address memory outside the tensors.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int kThreads = 256;

struct RowCopies {
    RowCopy t[kMaxCopies];
    int lg[kMaxCopies];   // log2 of the copy unit in bytes
};

__device__ __forceinline__ void seq_span(const int* __restrict__ cu, int s, int64_t total, int T, int64_t* start,
                                         int64_t* len) {
    int64_t a = cu[s];
    a = a < 0 ? 0 : (a > total ? total : a);
    int64_t l = (int64_t)cu[s + 1] - a;
    l = l < 0 ? 0 : (l > T ? T : l);
    if (l > total - a) l = total - a;
    *start = a;
    *len = l;
}

template <typename U, bool PACK>
__device__ __forceinline__ void copy_rows(const RowCopy& c, const int* __restrict__ cu, int n, int64_t total, int T) {
    const int64_t units = c.row_bytes / (int64_t)sizeof(U);
    const int64_t all = (int64_t)n * T * units;
    const U* src = reinterpret_cast<const U*>(c.src);
    U* dst = reinterpret_cast<U*>(c.dst);
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < all; i += (int64_t)gridDim.x * kThreads) {
        const int64_t row = i / units, e = i - row * units;   // padded row s T + t, unit e of it
        const int s = (int)(row / T);
        const int64_t t = row - (int64_t)s * T;
        int64_t start, len;
        seq_span(cu, s, total, T, &start, &len);
        if (PACK) {
            dst[i] = t < len ? src[(start + t) * units + e] : U{};
        } else if (t < len) {
            dst[(start + t) * units + e] = src[i];
        }
    }
}

template <bool PACK>
__global__ void __launch_bounds__(kThreads)
varlen_rows_kernel(RowCopies c, const int* __restrict__ cu, int n, int64_t total, int T) {
    const int y = blockIdx.y;
    switch (c.lg[y]) {
        case 4: copy_rows<uint4, PACK>(c.t[y], cu, n, total, T); break;
        case 3: copy_rows<uint2, PACK>(c.t[y], cu, n, total, T); break;
        case 2: copy_rows<uint32_t, PACK>(c.t[y], cu, n, total, T); break;
        case 1: copy_rows<uint16_t, PACK>(c.t[y], cu, n, total, T); break;
        default: copy_rows<uint8_t, PACK>(c.t[y], cu, n, total, T); break;
    }
}

template <bool PACK>
cudaError_t rows(const RowCopy* copies, int count, const int* cu, int n, int64_t total, int T, cudaStream_t s) {
    if (count <= 0 || count > kMaxCopies || n <= 0 || T <= 0 || total < 0) return cudaErrorInvalidValue;
    RowCopies c{};
    int64_t most = 0;
    for (int i = 0; i < count; ++i) {
        c.t[i] = copies[i];
        if (c.t[i].row_bytes <= 0) return cudaErrorInvalidValue;
        const uintptr_t al = reinterpret_cast<uintptr_t>(c.t[i].src) | reinterpret_cast<uintptr_t>(c.t[i].dst) |
                             static_cast<uintptr_t>(c.t[i].row_bytes);
        int lg = 4;
        while (lg > 0 && (al & ((uintptr_t(1) << lg) - 1)) != 0) --lg;
        c.lg[i] = lg;
        const int64_t all = (int64_t)n * T * (c.t[i].row_bytes >> lg);
        if (all > most) most = all;
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int64_t blocks = (most + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    varlen_rows_kernel<PACK><<<dim3((unsigned)blocks, (unsigned)count), kThreads, 0, s>>>(c, cu, n, total, T);
    return cudaGetLastError();
}

}  // namespace

cudaError_t varlen_pack(const RowCopy* copies, int count, const int* cu, int n, int64_t total, int T,
                        cudaStream_t s) {
    return rows<true>(copies, count, cu, n, total, T, s);
}

cudaError_t varlen_unpack(const RowCopy* copies, int count, const int* cu, int n, int64_t total, int T,
                          cudaStream_t s) {
    return rows<false>(copies, count, cu, n, total, T, s);
}

}  // namespace gdr
