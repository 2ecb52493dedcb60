// Device helpers shared by the tensor-core kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "blackwell.cuh"

namespace gdr {
namespace tc {

constexpr int kTile = 64;        // tokens per tile (rows of every M=64 MMA)
constexpr int kLd = kTile + 1;   // row pitch (floats) of the 64 x 64 fp32 scratch matrices

// TMEM address of (lane, column) for this warp's sub-partition.
__device__ __forceinline__ uint32_t tmem_at(uint32_t base, int warp, int col) {
    return base + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)col;
}

// Row of an M=64 accumulator held by this thread (lanes 16..31 hold none: -1).
__device__ __forceinline__ int m64_row(int warp, int lane) { return lane < 16 ? (warp & 3) * 16 + lane : -1; }

// Byte offset of element (r, c) in a [64 rows][D] bf16 tile stored as D/64
// swizzled atoms of [64][64] (8 KB each), the layout TMA writes for a
// 64-column box and the MMA reads as K-major (along D) or MN-major (along rows).
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
    return (uint32_t)((c >> 6) * 8192) + bw::sw128_offset(r, c & 63);
}

// Shared-memory descriptors for the tile layout above.
// K-major operand [64 rows][D] (contraction along D): k-step kk covers columns 16kk..16kk+15.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
    return bw::sdesc_sw128(tile + (uint32_t)((kk >> 2) * 8192 + (kk & 3) * 32), 16, 1024);
}
// MN-major operand stored [rows = contraction][D = M or N]: k-step kk covers rows 16kk..16kk+15.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kk) {
    return bw::sdesc_sw128(tile + (uint32_t)(kk * 2048), 8192, 1024);
}

// The same layouts for a tile of any row count (multiple of 8): atoms are
// [rows][64] and `rows * 128` bytes apart.
__device__ __forceinline__ uint32_t tile_off_r(int r, int c, int rows) {
    return (uint32_t)((c >> 6) * rows * 128) + bw::sw128_offset(r, c & 63);
}
__device__ __forceinline__ uint64_t desc_kmajor_r(uint32_t tile, int kk, int rows) {
    return bw::sdesc_sw128(tile + (uint32_t)((kk >> 2) * rows * 128 + (kk & 3) * 32), 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnmajor_r(uint32_t tile, int kk, int rows) {
    return bw::sdesc_sw128(tile + (uint32_t)(kk * 2048), (uint32_t)(rows * 128), 1024);
}

// (I + A)^{-1} for the block-diagonal, strictly lower A of a 64-row tile made of
// 64/C chunks of C rows (C = 32 or 64).  A and X are fp32 [64][kLd]; X gets the
// inverse inside each chunk's diagonal block and zeros elsewhere.  R is scratch
// of at least 3 * 16 * 17 floats.  Called by all 128 threads of the CTA.
//
// Blocked forward substitution on 16 x 16 blocks: the diagonal blocks are
// inverted column by column (each column a short chain in registers), then
// the off-diagonal blocks follow by distance from the diagonal:
//     X_ij = -X_ii * sum_{m=j}^{i-1} A_im X_mj        (block indices, i > j)
template <int C>
__device__ __forceinline__ void solve_unit_lower(const float* __restrict__ A, float* __restrict__ X,
                                                 float* __restrict__ R, int tid) {
    constexpr int NB = C / 16;
    constexpr int NCH = kTile / C;
    for (int i = tid; i < kTile * kLd; i += 128) X[i] = 0.f;
    __syncthreads();
    if (tid < 64) {
        const int r0 = (tid >> 4) * 16, c = tid & 15;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float s = (i == c) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < i; ++j) s -= A[(r0 + i) * kLd + r0 + j] * x[j];
            x[i] = (i < c) ? 0.f : s;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) X[(r0 + i) * kLd + r0 + c] = x[i];
    }
    __syncthreads();
#pragma unroll
    for (int L = 1; L < NB; ++L) {
        const int per_chunk = NB - L;
        const int n = per_chunk * NCH * 256;
        for (int idx = tid; idx < n; idx += 128) {
            const int p = idx >> 8, e = idx & 255, a = e >> 4, c = e & 15;
            const int ch = p / per_chunk, bi = L + p % per_chunk, bj = bi - L;
            const int ri = ch * C + bi * 16 + a, cj = ch * C + bj * 16 + c;
            const int m0 = ch * C + bj * 16;            // the sum runs over L * 16 rows m0 .. m0 + 16L - 1
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int mm = 0; mm < L * 16; mm += 2) {
                s0 += A[ri * kLd + m0 + mm] * X[(m0 + mm) * kLd + cj];
                s1 += A[ri * kLd + m0 + mm + 1] * X[(m0 + mm + 1) * kLd + cj];
            }
            R[p * 272 + a * 17 + c] = s0 + s1;
        }
        __syncthreads();
        for (int idx = tid; idx < n; idx += 128) {
            const int p = idx >> 8, e = idx & 255, a = e >> 4, c = e & 15;
            const int ch = p / per_chunk, bi = L + p % per_chunk, bj = bi - L;
            const int ri = ch * C + bi * 16 + a, cj = ch * C + bj * 16 + c;
            const int d0 = ch * C + bi * 16;
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) s += X[ri * kLd + d0 + m] * R[p * 272 + m * 17 + c];
            X[ri * kLd + cj] = -s;
        }
        __syncthreads();
    }
}

// Stores n (multiple of 16) fp32 values as bf16 to 16-byte aligned global memory.
__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* dst, const float* v) {
    uint4 a, b;
    a.x = bw::pack_bf16(v[0], v[1]);
    a.y = bw::pack_bf16(v[2], v[3]);
    a.z = bw::pack_bf16(v[4], v[5]);
    a.w = bw::pack_bf16(v[6], v[7]);
    b.x = bw::pack_bf16(v[8], v[9]);
    b.y = bw::pack_bf16(v[10], v[11]);
    b.z = bw::pack_bf16(v[12], v[13]);
    b.w = bw::pack_bf16(v[14], v[15]);
    reinterpret_cast<uint4*>(dst)[0] = a;
    reinterpret_cast<uint4*>(dst)[1] = b;
}

}  // namespace tc
}  // namespace gdr
