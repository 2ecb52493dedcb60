// Warp-level mma.sync products over tiles in padded shared memory, for the
// backward's per-chunk kernels: bf16 tiles stored row-major with a row stride of
// D + 8 elements (so 8 consecutive rows of an ldmatrix land in distinct banks),
// fp32 accumulation.  A warp computes a 16-row block times NCW 16-column blocks.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "warp_mma.cuh"

namespace gdr {
namespace cm {

using bf16 = __nv_bfloat16;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// acc[j] += opA(rows 16 rb .. +15, all kd) opB(all kd, cols 16 (cb0 + j) .. +15) for j < NCW.
// A row-major [M][lda] (AT: stored as [K][lda], i.e. A^T row-major); B stored [K][ldb] (BT: [N][ldb]).
template <int NCW, int KD, bool AT, bool BT>
__device__ __forceinline__ void wgemm(float (&acc)[NCW][2][4], uint32_t A, int lda, uint32_t B, int ldb, int rb,
                                      int cb0, int mi, int mr) {
#pragma unroll
    for (int k0 = 0; k0 < KD; k0 += 16) {
        uint32_t a[4];
        if constexpr (AT) wm::ldsm_x4_t(A + 2u * ((k0 + 8 * (mi >> 1) + mr) * lda + 16 * rb + 8 * (mi & 1)), a);
        else wm::ldsm_x4(A + 2u * ((16 * rb + 8 * (mi & 1) + mr) * lda + k0 + 8 * (mi >> 1)), a);
#pragma unroll
        for (int j = 0; j < NCW; ++j) {
            const int n0 = 16 * (cb0 + j);
            uint32_t bb[4];
            if constexpr (BT) wm::ldsm_x4(B + 2u * ((n0 + 8 * (mi >> 1) + mr) * ldb + k0 + 8 * (mi & 1)), bb);
            else wm::ldsm_x4_t(B + 2u * ((k0 + 8 * (mi & 1) + mr) * ldb + n0 + 8 * (mi >> 1)), bb);
            wm::mma16816(acc[j][0], a, bb[0], bb[1]);
            wm::mma16816(acc[j][1], a, bb[2], bb[3]);
        }
    }
}

template <int NCW>
__device__ __forceinline__ void zero(float (&acc)[NCW][2][4]) {
#pragma unroll
    for (int j = 0; j < NCW; ++j)
#pragma unroll
        for (int n = 0; n < 2; ++n) acc[j][n][0] = acc[j][n][1] = acc[j][n][2] = acc[j][n][3] = 0.f;
}

// Calls f(row, col, value&) for every element of a warp's tiles (rows 16 rb + ..., cols 16 (cb0 + j) + ...).
template <int NCW, typename F>
__device__ __forceinline__ void each(float (&acc)[NCW][2][4], int rb, int cb0, int g4, int q4, F&& f) {
#pragma unroll
    for (int j = 0; j < NCW; ++j)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) f(16 * rb + g4 + 8 * (e >> 1), 16 * (cb0 + j) + 8 * n + 2 * q4 + (e & 1), acc[j][n][e]);
}

// Calls f(row, col, x0&, x1&) for every pair of adjacent columns (col, col + 1) of a warp's tiles: the
// two accumulator elements a thread holds side by side, so a bf16x2 load or store serves both.
template <int NCW, typename F>
__device__ __forceinline__ void each2(float (&acc)[NCW][2][4], int rb, int cb0, int g4, int q4, F&& f) {
#pragma unroll
    for (int j = 0; j < NCW; ++j)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                f(16 * rb + g4 + 8 * h, 16 * (cb0 + j) + 8 * n + 2 * q4, acc[j][n][2 * h], acc[j][n][2 * h + 1]);
}

// Calls f(j, n, e, row, col) for every pair (e, e + 1) of a warp's accumulator elements: (row, col) and
// (row, col + 1), for epilogues over several accumulators with the same tiling.
template <int NCW, typename F>
__device__ __forceinline__ void each2_at(int rb, int cb0, int g4, int q4, F&& f) {
#pragma unroll
    for (int j = 0; j < NCW; ++j)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int h = 0; h < 2; ++h) f(j, n, 2 * h, 16 * rb + g4 + 8 * h, 16 * (cb0 + j) + 8 * n + 2 * q4);
}

__device__ __forceinline__ float2 bf2(const bf16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void st_bf2(bf16* p, float x0, float x1) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(x0, x1);
}

// rows x D bf16 from shared [rows][D + 8] to global rows of stride gs elements, rows < nrows only:
// 16-byte loads and stores, consecutive threads on consecutive 16-byte pieces of a row.
template <int D, int NTHR>
__device__ __forceinline__ void store_tile(bf16* dst, int64_t gs, const bf16* src, int nrows, int tid) {
    constexpr int per = D / 8;
    for (int idx = tid; idx < nrows * per; idx += NTHR) {
        const int r = idx / per, c8 = idx % per;
        *reinterpret_cast<uint4*>(dst + r * gs + 8 * c8) = *reinterpret_cast<const uint4*>(src + r * (D + 8) + 8 * c8);
    }
}

// rows x D bf16 from global rows of stride gs elements into shared [rows][D + 8]; rows >= nrows read as
// zero.  Asynchronous 16-byte copies (cp.async), so every copy of a phase is in flight at once; the
// caller waits with cp_async_wait_all() and a barrier.
template <int D, int NTHR>
__device__ __forceinline__ void load_tile(bf16* dst, const bf16* src, int64_t gs, int rows, int nrows, int tid) {
    constexpr int per = D / 8;
    for (int idx = tid; idx < rows * per; idx += NTHR) {
        const int r = idx / per, c8 = idx % per;
        bf16* d = dst + r * (D + 8) + 8 * c8;
        if (r < nrows)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(d)), "l"(src + r * gs + 8 * c8)
                         : "memory");
        else
            *reinterpret_cast<uint4*>(d) = make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ float bf(const bf16* p) { return __bfloat162float(*p); }

// sum over the four lanes of a quad (the lanes holding one row's columns), then into the row's shared slot
__device__ __forceinline__ void row_add(float* slot, float v, int q4) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    if (q4 == 0) atomicAdd(slot, v);
}

}  // namespace cm
}  // namespace gdr
