// Warp-level tensor-core building blocks: mma.sync m16n8k16 (bf16 or fp16 in,
// fp32 accumulate) with ldmatrix / stmatrix.  Used where a short serial chain of
// small products must stay in registers: a dependent tcgen05 MMA returns only
// after a round trip of about 300 SM cycles (issue, commit, mbarrier), while
// mma.sync returns in ~22 cycles and issues every ~8 cycles per scheduler.
//
// Fragment layouts (g = lane / 4, c = lane % 4):
//   A 16x16: a0 (g, 2c..2c+1)  a1 (g+8, 2c..)  a2 (g, 2c+8..)  a3 (g+8, 2c+8..)
//   B 16x8 : b0 (k 2c..2c+1, n g)  b1 (k 2c+8.., n g)
//   C 16x8 : c0,c1 (g, 2c..2c+1)  c2,c3 (g+8, 2c..2c+1)
// so the accumulator of n-tiles 2k and 2k+1 is, packed to bf16, the A operand of k-tile k.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gdr {
namespace wm {

__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same product with fp16 A and B.
__device__ __forceinline__ void mma16816_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Operands of the io type: bf16 (F16 = false) or fp16.
template <bool F16>
__device__ __forceinline__ void mma16816_io(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    if constexpr (F16) mma16816_f16(d, a, b0, b1);
    else mma16816(d, a, b0, b1);
}

// Four 8x8 b16 matrices; lane l gives the address of row l % 8 of matrix l / 8.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
// Stores four 8x8 matrices transposed: fragment column j becomes memory row j.
__device__ __forceinline__ void stsm_x4_t(uint32_t addr, const uint32_t* r) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack2_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
template <bool F16>
__device__ __forceinline__ uint32_t pack2_io(float lo, float hi) {
    if constexpr (F16) return pack2_f16(lo, hi);
    else return pack2(lo, hi);
}

}  // namespace wm
}  // namespace gdr
