// Stitches the segments of the segment-parallel state scan.  One chunk of the
// scan ("kernel_fun/kda/_kernels/bwd_scan.py", module docstring: v' = u - w h,
// h = exp(decay) h + kg^T v') is affine in h, so a run of chunks is one map
// h_end = M h_start + Z; the transfer scan (scan_mma.cu, TRANSFER) writes M and Z
// for every segment.  Per (b, h, 8 value columns), in fp32 on the CUDA cores:
//
//   h_start[0] = h0 (zero if NULL);  h_start[s + 1] = M_s h_start[s] + Z_s;
//   h_final = M_{S-1} h_start[S-1] + Z_{S-1}
//
// REVERSE stitches the backward's state gradient the other way: the reverse
// scan maps the gradient at a segment's end to the one at its start by M_s^T
// (the transpose of the forward map) plus Zb_s, so
//
//   end[S-1] = dh_final (zero if NULL);  end[s-1] = M_s^T end[s] + Zb_s;  dh0 = M_0^T end[0] + Zb_0.
//
// The chain is serial in s, so its latency is the cost: narrow column slices
// give many CTAs, and M_{s+1} and Z_{s+1} stream into shared memory (cp.async,
// double-buffered) while step s computes.  A warp owns K/8 rows of the output;
// lane (r, p) sums the columns j = p (mod 4) of row r, so at each step of the
// sum the warp reads 32 distinct words of M from 32 distinct banks (row stride
// K + 4), and the four partial sums meet by shuffles at the end.
#include <cuda_runtime.h>

#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int kThreads = 256;
constexpr int kCB = 8;   // value columns per CTA

__device__ __forceinline__ void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// h0: the forward's h0 or the backward's dh_final; h_start: the segment starts (forward) or ends
// (REVERSE); h_final: h_final (forward) or dh0 (REVERSE)
template <int K, bool REVERSE>
__global__ void __launch_bounds__(kThreads)
segment_combine_kernel(const float* __restrict__ M, const float* __restrict__ Z, const float* __restrict__ h0,
                       float* __restrict__ h_start, float* __restrict__ h_final, int S, int H, int V) {
    constexpr int LM = K + 4;                   // M row stride (16-byte rows for cp.async)
    constexpr int RPW = K / (kThreads / 32);    // output rows per warp (16 for K = 128, 8 for K = 64)
    constexpr int RG = RPW / 8;                 // groups of 8 rows per warp
    extern __shared__ __align__(16) float smem[];
    float* Ms = smem;                           // [2][K][LM]
    float* Zs = Ms + 2 * K * LM;                // [2][K][8]
    float* hs = Zs + 2 * K * kCB;               // [2][K][8]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = lane >> 2, p = lane & 3;
    const int v0 = blockIdx.x * kCB, h = blockIdx.y, b = blockIdx.z;
    const int64_t hb = ((int64_t)b * H + h) * K * V;

    // step i of the chain handles segment s(i): i forward, S - 1 - i in REVERSE; buffers alternate with i
    auto seg_of = [&](int i) { return REVERSE ? S - 1 - i : i; };
    auto prefetch_step = [&](int i) {
        const int s = seg_of(i);
        const int64_t seg = ((int64_t)b * S + s) * H + h;
        const float* Mg = M + seg * K * K;
        const float* Zg = Z + seg * K * V + v0;
        float* md = Ms + (i & 1) * K * LM;
        float* zd = Zs + (i & 1) * K * kCB;
        for (int e = tid; e < K * K / 4; e += kThreads) {
            const int row = e / (K / 4), c4 = e % (K / 4);
            cp16(md + row * LM + 4 * c4, Mg + (int64_t)row * K + 4 * c4);
        }
        for (int e = tid; e < K * 2; e += kThreads)
            cp16(zd + (e >> 1) * kCB + 4 * (e & 1), Zg + (int64_t)(e >> 1) * V + 4 * (e & 1));
        cp_commit();
    };
    prefetch_step(0);
    for (int e = tid; e < K * kCB; e += kThreads)
        hs[e] = h0 ? h0[hb + (int64_t)(e / kCB) * V + v0 + e % kCB] : 0.f;
    for (int i = 0; i < S; ++i) {
        const int s = seg_of(i);
        const float* hcur = hs + (i & 1) * K * kCB;
        float* hnext = hs + ((i + 1) & 1) * K * kCB;
        cp_wait_all();
        __syncthreads();   // M, Z and h of this step in place; every thread is done with the last step's buffers
        if (i + 1 < S) prefetch_step(i + 1);
        // this step's boundary value (a segment's start, or in REVERSE its end): this CTA's [K x 8] slice
        {
            const int64_t sb = (((int64_t)b * S + s) * H + h) * K * V;
            for (int e = tid; e < K * 2; e += kThreads)
                *reinterpret_cast<float4*>(h_start + sb + (int64_t)(e >> 1) * V + v0 + 4 * (e & 1)) =
                    *reinterpret_cast<const float4*>(hcur + (e >> 1) * kCB + 4 * (e & 1));
        }
        const float* Mc = Ms + (i & 1) * K * LM;
        float acc[RG][kCB];
#pragma unroll
        for (int g = 0; g < RG; ++g)
#pragma unroll
            for (int c = 0; c < kCB; ++c) acc[g][c] = 0.f;
#pragma unroll 4
        for (int j = p; j < K; j += 4) {
            const float4 h0v = *reinterpret_cast<const float4*>(hcur + j * kCB);
            const float4 h1v = *reinterpret_cast<const float4*>(hcur + j * kCB + 4);
#pragma unroll
            for (int g = 0; g < RG; ++g) {
                const int row = warp * RPW + 8 * g + r;
                const float m = REVERSE ? Mc[j * LM + row] : Mc[row * LM + j];   // M^T in REVERSE
                acc[g][0] = fmaf(m, h0v.x, acc[g][0]); acc[g][1] = fmaf(m, h0v.y, acc[g][1]);
                acc[g][2] = fmaf(m, h0v.z, acc[g][2]); acc[g][3] = fmaf(m, h0v.w, acc[g][3]);
                acc[g][4] = fmaf(m, h1v.x, acc[g][4]); acc[g][5] = fmaf(m, h1v.y, acc[g][5]);
                acc[g][6] = fmaf(m, h1v.z, acc[g][6]); acc[g][7] = fmaf(m, h1v.w, acc[g][7]);
            }
        }
        // the four partial sums of each row, then + Z_s into the next step's value
        const float* Zc = Zs + (i & 1) * K * kCB;
#pragma unroll
        for (int g = 0; g < RG; ++g) {
#pragma unroll
            for (int c = 0; c < kCB; ++c) {
                acc[g][c] += __shfl_xor_sync(0xffffffffu, acc[g][c], 1);
                acc[g][c] += __shfl_xor_sync(0xffffffffu, acc[g][c], 2);
            }
            const int row = warp * RPW + 8 * g + r;
            if (p < 2) {   // lanes p = 0, 1 write the row's two float4 halves (static register indices)
                const float4 z = *reinterpret_cast<const float4*>(Zc + row * kCB + 4 * p);
                float4 o;
                o.x = (p ? acc[g][4] : acc[g][0]) + z.x;
                o.y = (p ? acc[g][5] : acc[g][1]) + z.y;
                o.z = (p ? acc[g][6] : acc[g][2]) + z.z;
                o.w = (p ? acc[g][7] : acc[g][3]) + z.w;
                *reinterpret_cast<float4*>(hnext + row * kCB + 4 * p) = o;
            }
        }
    }
    __syncthreads();
    if (h_final) {
        const float* hl = hs + (S & 1) * K * kCB;   // written by the last step
        for (int e = tid; e < K * 2; e += kThreads)
            *reinterpret_cast<float4*>(h_final + hb + (int64_t)(e >> 1) * V + v0 + 4 * (e & 1)) =
                *reinterpret_cast<const float4*>(hl + (e >> 1) * kCB + 4 * (e & 1));
    }
}

template <int K, bool REVERSE>
cudaError_t launch(const Dims& d, int S, const float* M, const float* Z, const float* h0, float* h_start,
                   float* h_final, cudaStream_t s) {
    auto kern = segment_combine_kernel<K, REVERSE>;
    const size_t smem = sizeof(float) * (2 * K * (K + 4) + 4 * K * kCB);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(d.V / kCB, d.H, d.B);
    kern<<<grid, kThreads, smem, s>>>(M, Z, h0, h_start, h_final, S, d.H, d.V);
    return cudaGetLastError();
}

}  // namespace

cudaError_t segment_combine(const Dims& d, int S, const float* M, const float* Z, const float* h0, float* h_start,
                            float* h_final, cudaStream_t s, bool reverse) {
    if (S < 1) return cudaErrorInvalidValue;
    if (reverse)
        return d.K == 64 ? launch<64, true>(d, S, M, Z, h0, h_start, h_final, s)
                         : launch<128, true>(d, S, M, Z, h0, h_start, h_final, s);
    return d.K == 64 ? launch<64, false>(d, S, M, Z, h0, h_start, h_final, s)
                     : launch<128, false>(d, S, M, Z, h0, h_start, h_final, s);
}

}  // namespace gdr
