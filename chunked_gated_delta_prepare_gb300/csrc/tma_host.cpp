// Host side of TMA: building CUtensorMap descriptors.  The driver's encoder is
// fetched through the runtime (cudaGetDriverEntryPointByVersion), so the
// library does not link libcuda and loads on machines without a GPU driver.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tma_host.h"

namespace gdr {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void fetch_encoder() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
}  // namespace

bool make_tmap_bf16_4d(CUtensorMap* map, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                       const uint32_t box[4]) {
    return make_tmap_bf16_4d_swz(map, base, dims, strides_bytes, box, true);
}

bool make_tmap_bf16_4d_swz(CUtensorMap* map, const void* base, const uint64_t dims[4],
                           const uint64_t strides_bytes[3], const uint32_t box[4], bool swizzle128) {
    return make_tmap_bf16_4d_mode(map, base, dims, strides_bytes, box,
                                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool make_tmap_bf16_4d_mode(CUtensorMap* map, const void* base, const uint64_t dims[4],
                            const uint64_t strides_bytes[3], const uint32_t box[4], CUtensorMapSwizzle swizzle) {
    std::call_once(g_once, fetch_encoder);
    if (!g_encode) return false;
    cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t gs[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
    cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gd, gs, bx, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Token-major [B,T,H,D] bf16 tensor seen as 4-D (D, H, T, B); box = 64 columns x
// `rows` tokens of one head.  Rows past T read as zero.
bool make_tmap_tokens(CUtensorMap* map, const void* base, int B, int T, int H, int D, int rows) {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t st[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)T * H * D * 2};
    const uint32_t box[4] = {64, 1, (uint32_t)rows, 1};
    return make_tmap_bf16_4d(map, base, dims, st, box);
}

// Checkpoints [B,NT,H,K,V] bf16 seen as 4-D (V, K, H, B*NT); box = 64 columns x K rows.
bool make_tmap_ckpt(CUtensorMap* map, const void* base, int B, int NT, int H, int K, int V) {
    const uint64_t dims[4] = {(uint64_t)V, (uint64_t)K, (uint64_t)H, (uint64_t)B * NT};
    const uint64_t st[3] = {(uint64_t)V * 2, (uint64_t)K * V * 2, (uint64_t)H * K * V * 2};
    const uint32_t box[4] = {64, (uint32_t)K, 1, 1};
    return make_tmap_bf16_4d(map, base, dims, st, box);
}

// Unswizzled variants: box = `cols` columns (cols * 2 bytes, a multiple of 16) x `rows`.
bool make_tmap_tokens_plain(CUtensorMap* map, const void* base, int B, int T, int H, int D, int cols, int rows) {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t st[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)T * H * D * 2};
    const uint32_t box[4] = {(uint32_t)cols, 1, (uint32_t)rows, 1};
    return make_tmap_bf16_4d_swz(map, base, dims, st, box, false);
}

bool make_tmap_ckpt_plain(CUtensorMap* map, const void* base, int B, int NT, int H, int K, int V, int cols) {
    const uint64_t dims[4] = {(uint64_t)V, (uint64_t)K, (uint64_t)H, (uint64_t)B * NT};
    const uint64_t st[3] = {(uint64_t)V * 2, (uint64_t)K * V * 2, (uint64_t)H * K * V * 2};
    const uint32_t box[4] = {(uint32_t)cols, (uint32_t)K, 1, 1};
    return make_tmap_bf16_4d_swz(map, base, dims, st, box, false);
}

// 32-column boxes with the 64-byte swizzle: 16-byte chunk j of row r sits at j ^ ((r >> 1) & 3).
bool make_tmap_tokens_sw64(CUtensorMap* map, const void* base, int B, int T, int H, int D, int rows) {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t st[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)T * H * D * 2};
    const uint32_t box[4] = {32, 1, (uint32_t)rows, 1};
    return make_tmap_bf16_4d_mode(map, base, dims, st, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

// Boxes of `cols` columns x `rows` tokens of one (b, h) with the given swizzle.
bool make_tmap_tokens_box(CUtensorMap* map, const void* base, int B, int T, int H, int D, int cols, int rows,
                          CUtensorMapSwizzle swizzle) {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t st[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)T * H * D * 2};
    const uint32_t box[4] = {(uint32_t)cols, 1, (uint32_t)rows, 1};
    return make_tmap_bf16_4d_mode(map, base, dims, st, box, swizzle);
}

// Checkpoint boxes of `cols` columns (of V) x `rows` key rows of one (b, c, h).
bool make_tmap_ckpt_box(CUtensorMap* map, const void* base, int B, int NT, int H, int K, int V, int cols, int rows,
                        CUtensorMapSwizzle swizzle) {
    const uint64_t dims[4] = {(uint64_t)V, (uint64_t)K, (uint64_t)H, (uint64_t)B * NT};
    const uint64_t st[3] = {(uint64_t)V * 2, (uint64_t)K * V * 2, (uint64_t)H * K * V * 2};
    const uint32_t box[4] = {(uint32_t)cols, (uint32_t)rows, 1, 1};
    return make_tmap_bf16_4d_mode(map, base, dims, st, box, swizzle);
}

}  // namespace gdr
