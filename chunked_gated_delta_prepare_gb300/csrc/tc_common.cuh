// Device helpers shared by the tensor-core kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "blackwell.cuh"

namespace gdr {
namespace tc {

constexpr int kTile = 64;        // tokens per tile (rows of every M=64 MMA)

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

}  // namespace tc
}  // namespace gdr
