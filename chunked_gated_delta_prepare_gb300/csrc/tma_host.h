// Host helpers that build TMA descriptors for the library's tensor layouts.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gdr {

// Generic 4-D bf16 map with 128-byte swizzle (box[0] * 2 bytes must be <= 128).
bool make_tmap_bf16_4d(CUtensorMap* map, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                       const uint32_t box[4]);

bool make_tmap_bf16_4d_swz(CUtensorMap* map, const void* base, const uint64_t dims[4],
                           const uint64_t strides_bytes[3], const uint32_t box[4], bool swizzle128);

bool make_tmap_bf16_4d_mode(CUtensorMap* map, const void* base, const uint64_t dims[4],
                            const uint64_t strides_bytes[3], const uint32_t box[4], CUtensorMapSwizzle swizzle);

// [B,T,H,D] bf16 token tensor; box = 64 columns (of D) x `rows` tokens of one (b, h).
bool make_tmap_tokens(CUtensorMap* map, const void* base, int B, int T, int H, int D, int rows);

// [B,NT,H,K,V] bf16 checkpoints; box = 64 columns (of V) x all K rows of one (b, c, h).
bool make_tmap_ckpt(CUtensorMap* map, const void* base, int B, int NT, int H, int K, int V);

// Unswizzled boxes of `cols` columns (cols * 2 a multiple of 16 bytes).
bool make_tmap_tokens_plain(CUtensorMap* map, const void* base, int B, int T, int H, int D, int cols, int rows);
bool make_tmap_ckpt_plain(CUtensorMap* map, const void* base, int B, int NT, int H, int K, int V, int cols);

// 32 columns x `rows` tokens with the 64-byte swizzle (16-byte chunk j of row r at j ^ ((r >> 1) & 3)).
bool make_tmap_tokens_sw64(CUtensorMap* map, const void* base, int B, int T, int H, int D, int rows);

// General boxes: `cols` columns x `rows` tokens (or key rows of a checkpoint), any swizzle.
// 32-byte swizzle: 16-byte chunk j of row r of a 32-byte-row box sits at j ^ ((r >> 2) & 1).
bool make_tmap_tokens_box(CUtensorMap* map, const void* base, int B, int T, int H, int D, int cols, int rows,
                          CUtensorMapSwizzle swizzle);
bool make_tmap_ckpt_box(CUtensorMap* map, const void* base, int B, int NT, int H, int K, int V, int cols, int rows,
                        CUtensorMapSwizzle swizzle);

}  // namespace gdr
