// The backward's local value gradient on the tensor cores, for the problems the
// fused per-chunk backward does not take (a per-key-dim gate, or 32-token chunks):
//
//   dv_loc = scale tril0(Qt)^T do,   Qt_ij = sum_d q_id k_jd exp(G_id - G_jd)   (j <= i)
//
// per chunk, written in bf16 for the reverse scan to add (dv' = dv_loc + kg dh).
// The scan page's backward forms this term from the gated scores of the
// forward's output ("kernel_fun/kda/_kernels/bwd_scan.py", module docstring).
//
// One CTA of four warps per (chunk, head, batch).  q, k and do sit in padded
// bf16 shared memory; S = q k^T (scalar gate, the gate applied to S) or
// S = (q e^(G - G_ref)) (k e^(G_ref - G))^T (per-key-dim gate, G_ref the chunk's
// middle row, so every factor stays bounded) is an mma.sync product, masked to
// the lower triangle with its diagonal, and dv_loc = scale S^T do another.  A
// chunk whose per-key gate moves further than kExpSafe from its middle row
// forms S exactly in fp32 on the CUDA cores instead.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "chunk_mma.cuh"
#include "gdr_internal.h"

namespace gdr {
namespace {

using bf16 = __nv_bfloat16;
using namespace cm;
constexpr int kThreads = 128;
constexpr float kExpSafe = 40.f;

template <int K, int V, int C, bool PER_K>
struct DvlocLayout {
    static constexpr int LK = K + 8, LV = V + 8, LC = C + 8;
    static constexpr int GW = PER_K ? K : 1;
    static constexpr uint32_t rq = 0;
    static constexpr uint32_t rk = rq + C * LK * 2;
    static constexpr uint32_t rdo = rk + C * LK * 2;
    static constexpr uint32_t rp = rdo + C * LV * 2;
    static constexpr uint32_t rg = rp + C * LC * 2;                 // G [C][GW] fp32
    static constexpr uint32_t bytes = rg + C * GW * 4 + 16;
};

template <int K, int V, int C, bool PER_K>
__global__ void __launch_bounds__(kThreads)
bwd_dvloc_mma_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k, const float* __restrict__ g_cum,
                     const bf16* __restrict__ d_o, bf16* __restrict__ dv_loc, int T, int H, int G, float scale) {
    using L = DvlocLayout<K, V, C, PER_K>;
    constexpr int LK = L::LK, LV = L::LV, LC = L::LC, GW = L::GW;
    constexpr int RB = C / 16;                 // 16-row blocks
    constexpr int CG = 4 / RB;                 // warps per row block
    constexpr int NCC = C / 16 / CG;           // column blocks of S per warp
    constexpr int NCV = V / 16 / CG;           // column blocks of dv_loc per warp
    extern __shared__ __align__(128) unsigned char sm[];
    bf16* Qs = reinterpret_cast<bf16*>(sm + L::rq);
    bf16* Ks = reinterpret_cast<bf16*>(sm + L::rk);
    bf16* DOs = reinterpret_cast<bf16*>(sm + L::rdo);
    bf16* Ps = reinterpret_cast<bf16*>(sm + L::rp);
    float* Gs = reinterpret_cast<float*>(sm + L::rg);
    int* sFlag = reinterpret_cast<int*>(Gs + C * GW);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, q4 = lane & 3, mi = lane >> 3, mr = lane & 7;
    const int rb = warp % RB, cg = warp / RB;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int t0 = c * C, nv = min(C, T - t0);
    const int Hk = H / G;
    const int64_t tok0 = ((int64_t)b * T + t0) * H + h;
    const int64_t ktok0 = ((int64_t)b * T + t0) * Hk + h / G;

    load_tile<K, kThreads>(Qs, q + ktok0 * K, (int64_t)Hk * K, C, nv, tid);
    load_tile<K, kThreads>(Ks, k + ktok0 * K, (int64_t)Hk * K, C, nv, tid);
    load_tile<V, kThreads>(DOs, d_o + tok0 * V, (int64_t)H * V, C, nv, tid);
    cp_async_commit();
    // G past T repeats its last value (q, k and do are zero there)
    if constexpr (PER_K) {
        // 16-byte loads, all of a thread's issued before any is used
        constexpr int NV4 = C * GW / 4 / kThreads;
        float4 gv[NV4];
#pragma unroll
        for (int j = 0; j < NV4; ++j) {
            const int e = 4 * (tid + kThreads * j);
            gv[j] = *reinterpret_cast<const float4*>(g_cum + (tok0 + (int64_t)min(e / GW, nv - 1) * H) * GW + e % GW);
        }
#pragma unroll
        for (int j = 0; j < NV4; ++j) *reinterpret_cast<float4*>(Gs + 4 * (tid + kThreads * j)) = gv[j];
    } else {
        for (int i = tid; i < C; i += kThreads) Gs[i] = g_cum[tok0 + (int64_t)min(i, nv - 1) * H];
    }
    if (tid == 0) *sFlag = 0;
    cp_async_wait<0>();
    __syncthreads();

    const uint32_t aQ = smem_addr(Qs), aK = smem_addr(Ks), aDO = smem_addr(DOs), aP = smem_addr(Ps);
    bool exact = false;
    if constexpr (PER_K) {
        // gated copies around the middle row: q e^(G - G_ref) over q, k e^(G_ref - G) over k
        const int ref = min(C / 2, nv - 1);
        bool big = false;
        for (int i = tid; i < C * K; i += kThreads) {
            const int r = i / K, d = i % K;
            big |= fabsf(Gs[r * K + d] - Gs[ref * K + d]) > kExpSafe;
        }
        if (big) *sFlag = 1;
        __syncthreads();
        exact = *sFlag != 0;
        if (exact) {
            // S exactly: fp32 over every key dim with its own gate
            for (int idx = tid; idx < C * C; idx += kThreads) {
                const int i = idx / C, j = idx % C;
                float s = 0.f;
                if (j <= i)
                    for (int d = 0; d < K; ++d)
                        s += bf(Qs + i * LK + d) * bf(Ks + j * LK + d) * __expf(Gs[i * K + d] - Gs[j * K + d]);
                Ps[i * LC + j] = __float2bfloat16_rn(s);
            }
        } else {
            for (int i = tid; i < C * K; i += kThreads) {
                const int r = i / K, d = i % K;
                const float dg = Gs[r * K + d] - Gs[ref * K + d];
                Qs[r * LK + d] = __float2bfloat16_rn(bf(Qs + r * LK + d) * __expf(dg));
                Ks[r * LK + d] = __float2bfloat16_rn(bf(Ks + r * LK + d) * __expf(-dg));
            }
        }
        __syncthreads();
    }
    if (!exact) {
        // S = Qa Kb^T (or q k^T), masked to j <= i, gated (scalar) and rounded into Ps
        float sacc[NCC][2][4];
        zero(sacc);
        wgemm<NCC, K, false, true>(sacc, aQ, LK, aK, LK, rb, cg * NCC, mi, mr);
        each(sacc, rb, cg * NCC, g4, q4, [&](int r, int col, float& x) {
            float y = col <= r ? x : 0.f;
            if constexpr (!PER_K) y *= col <= r ? __expf(Gs[r] - Gs[col]) : 0.f;
            Ps[r * LC + col] = __float2bfloat16_rn(y);
        });
    }
    __syncthreads();
    // dv_loc = scale P^T do
    float acc[NCV][2][4];
    zero(acc);
    wgemm<NCV, C, true, false>(acc, aP, LC, aDO, LV, rb, cg * NCV, mi, mr);
    each(acc, rb, cg * NCV, g4, q4, [&](int r, int col, float& x) {
        if (r < nv) dv_loc[(tok0 + (int64_t)r * H) * V + col] = __float2bfloat16_rn(scale * x);
    });
}

template <int K, int V, int C, bool PER_K>
cudaError_t launch(const Dims& d, const void* q, const void* k, const float* g_cum, const void* d_o, void* dv_loc,
                   cudaStream_t s) {
    using L = DvlocLayout<K, V, C, PER_K>;
    auto kern = bwd_dvloc_mma_kernel<K, V, C, PER_K>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
    if (e != cudaSuccess) return e;
    const dim3 grid(d.NT, d.H, d.B);
    kern<<<grid, kThreads, L::bytes, s>>>((const bf16*)q, (const bf16*)k, g_cum, (const bf16*)d_o, (bf16*)dv_loc,
                                          d.T, d.H, d.G, d.scale);
    return cudaGetLastError();
}

template <int K, int V, int C>
cudaError_t gate(const Dims& d, const void* q, const void* k, const float* g_cum, const void* d_o, void* dv_loc,
                 cudaStream_t s) {
    return d.per_k ? launch<K, V, C, true>(d, q, k, g_cum, d_o, dv_loc, s)
                   : launch<K, V, C, false>(d, q, k, g_cum, d_o, dv_loc, s);
}

template <int K, int V>
cudaError_t chunk(const Dims& d, const void* q, const void* k, const float* g_cum, const void* d_o, void* dv_loc,
                  cudaStream_t s) {
    return d.C == 32 ? gate<K, V, 32>(d, q, k, g_cum, d_o, dv_loc, s) : gate<K, V, 64>(d, q, k, g_cum, d_o, dv_loc, s);
}

}  // namespace

cudaError_t mma_bwd_dv_local(const Dims& d, const void* q, const void* k, const float* g_cum, const void* d_o,
                             void* dv_loc, cudaStream_t s) {
    if (!d.bf16) return cudaErrorInvalidValue;
    if (d.K == 64 && d.V == 64) return chunk<64, 64>(d, q, k, g_cum, d_o, dv_loc, s);
    if (d.K == 64 && d.V == 128) return chunk<64, 128>(d, q, k, g_cum, d_o, dv_loc, s);
    if (d.K == 128 && d.V == 64) return chunk<128, 64>(d, q, k, g_cum, d_o, dv_loc, s);
    return chunk<128, 128>(d, q, k, g_cum, d_o, dv_loc, s);
}

}  // namespace gdr
