// Packed variable-length sequences.  Sequence s of a packed tensor [total, ...]
// holds the token rows cu[s] .. cu[s + 1] - 1 (cu: cumulative lengths, device
// int32 [n + 1]).  The library computes such a batch in one of two working
// layouts, both made of the batched kernels' whole or partial chunks:
//
//   padded        n rows of T tokens; sequence s is row s, its tail zero tokens;
//   chunk-packed  one row of NT whole chunks; sequence s starts at chunk co[s] and
//                 takes ceil(len_s / C) chunks, its last chunk's tail zero tokens.
//
// A zero token (beta = 0, g = 0, q = k = v = 0) leaves the state as it was and
// its output is dropped, so each sequence computes exactly its own recurrence
// (the partial-chunk reading, carried to the end of its row or chunk).  The
// chunk-packed layout adds fewer than C tokens per sequence; the scans walk each
// sequence's own chunks (blockIdx.z = sequence), every other stage is chunk-local.
//
// varlen_pack moves packed rows into the working layout (zero-filling the rest),
// varlen_unpack moves a sequence's first len_s working rows back.  One launch
// moves up to kMaxCopies tensors (blockIdx.y picks the tensor) in the widest unit
// (16, 8, 4, 2 or 1 bytes) that divides the row and both base addresses.  Every
// index read from cu, co or cs is clamped or range-checked, so no value of them
// addresses memory outside the tensors.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int kThreads = 256;
constexpr int kPlanThreads = 1024;

struct RowCopies {
    RowCopy t[kMaxCopies];
    int lg[kMaxCopies];   // log2 of the copy unit in bytes
};

// packed start of sequence s and its length, clamped to [0, total] and [0, maxlen]
__device__ __forceinline__ void seq_span(const int* __restrict__ cu, int s, int64_t total, int64_t maxlen,
                                         int64_t* start, int64_t* len) {
    int64_t a = cu[s];
    a = a < 0 ? 0 : (a > total ? total : a);
    int64_t l = (int64_t)cu[s + 1] - a;
    l = l < 0 ? 0 : (l > maxlen ? maxlen : l);
    if (l > total - a) l = total - a;
    *start = a;
    *len = l;
}

// working row r -> the packed row it holds, or -1 (a zero token)
__device__ __forceinline__ int64_t packed_row(const VarlenMap& m, int64_t r) {
    int s;
    int64_t t, maxlen;
    if (m.co) {
        const int c = (int)(r / m.C);
        s = m.cs[c];
        if (s < 0 || s >= m.n) return -1;
        const int a = m.co[s], b = m.co[s + 1];
        if (c < a || c >= b) return -1;
        t = r - (int64_t)a * m.C;
        maxlen = (int64_t)(b - a) * m.C;
    } else {
        s = (int)(r / m.T);
        t = r - (int64_t)s * m.T;
        maxlen = m.T;
    }
    int64_t start, len;
    seq_span(m.cu, s, m.total, maxlen, &start, &len);
    return t < len ? start + t : -1;
}

template <typename U, bool PACK>
__device__ __forceinline__ void copy_rows(const RowCopy& c, const VarlenMap& m) {
    const int64_t units = c.row_bytes / (int64_t)sizeof(U);
    const int64_t all = m.rows * units;
    const U* src = reinterpret_cast<const U*>(c.src);
    U* dst = reinterpret_cast<U*>(c.dst);
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < all; i += (int64_t)gridDim.x * kThreads) {
        const int64_t r = i / units, e = i - r * units;   // working row r, unit e of it
        const int64_t p = packed_row(m, r);
        if (PACK) {
            dst[i] = p >= 0 ? src[p * units + e] : U{};
        } else if (p >= 0) {
            dst[p * units + e] = src[i];
        }
    }
}

template <bool PACK>
__global__ void __launch_bounds__(kThreads) varlen_rows_kernel(RowCopies c, VarlenMap m) {
    const int y = blockIdx.y;
    switch (c.lg[y]) {
        case 4: copy_rows<uint4, PACK>(c.t[y], m); break;
        case 3: copy_rows<uint2, PACK>(c.t[y], m); break;
        case 2: copy_rows<uint32_t, PACK>(c.t[y], m); break;
        case 1: copy_rows<uint16_t, PACK>(c.t[y], m); break;
        default: copy_rows<uint8_t, PACK>(c.t[y], m); break;
    }
}

// one CTA: an exclusive prefix sum of the sequences' chunk counts over tiles of kPlanThreads, then the
// chunk -> sequence map
__global__ void __launch_bounds__(kPlanThreads)
varlen_plan_kernel(const int* __restrict__ cu, int n, int64_t total, int C, int NT, int* __restrict__ co,
                   int* __restrict__ cs) {
    __shared__ int wsum[kPlanThreads / 32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < n; base += kPlanThreads) {
        const int s = base + tid;
        int nc = 0;
        if (s < n) {
            int64_t start, len;
            seq_span(cu, s, total, total, &start, &len);
            nc = (int)((len + C - 1) / C);
        }
        int x = nc;   // inclusive scan within the warp, then over the warps' totals
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const int incl = x + (warp ? wsum[warp - 1] : 0);
        if (s < n) co[s] = min(carry + incl - nc, NT);
        __syncthreads();
        if (tid == kPlanThreads - 1) carry += incl;
        __syncthreads();
    }
    if (tid == 0) co[n] = min(carry, NT);
    __syncthreads();
    for (int s = tid; s < n; s += kPlanThreads)
        for (int c = co[s]; c < co[s + 1]; ++c) cs[c] = s;
}

template <bool PACK>
cudaError_t rows(const RowCopy* copies, int count, const VarlenMap& m, cudaStream_t s) {
    if (count <= 0 || count > kMaxCopies || m.n <= 0 || m.rows <= 0 || m.total < 0 || !m.cu) return cudaErrorInvalidValue;
    if (m.co ? (!m.cs || m.C <= 0) : m.T <= 0) return cudaErrorInvalidValue;
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
        const int64_t all = m.rows * (c.t[i].row_bytes >> lg);
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
    varlen_rows_kernel<PACK><<<dim3((unsigned)blocks, (unsigned)count), kThreads, 0, s>>>(c, m);
    return cudaGetLastError();
}

}  // namespace

cudaError_t varlen_pack(const RowCopy* copies, int count, const VarlenMap& m, cudaStream_t s) {
    return rows<true>(copies, count, m, s);
}

cudaError_t varlen_unpack(const RowCopy* copies, int count, const VarlenMap& m, cudaStream_t s) {
    return rows<false>(copies, count, m, s);
}

cudaError_t varlen_plan(const int* cu, int n, int64_t total, int C, int NT, int* co, int* cs, cudaStream_t s) {
    if (!cu || !co || !cs || n <= 0 || C <= 0 || NT < 0 || total < 0) return cudaErrorInvalidValue;
    varlen_plan_kernel<<<1, kPlanThreads, 0, s>>>(cu, n, total, C, NT, co, cs);
    return cudaGetLastError();
}

}  // namespace gdr
