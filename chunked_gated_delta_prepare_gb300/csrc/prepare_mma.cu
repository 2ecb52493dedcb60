// WY prepare for bf16 io ("Reuse P as beta tiles in gated deltanet fused
// prepare": the gated A, its inverse, w and u per chunk).
//
// One CTA of 128 threads per 64-token tile of one (batch, head): one chunk when
// C = 64, two when C = 32 (kept apart by the block-diagonal structure).  Warp w
// owns tile rows 16w .. 16w+15 of every product.
//
//   TMA      k [64 x K], v [64 x V]  -> shared memory (128-byte swizzle)
//   SIMT     G = chunk-local cumsum of g (written out as g_cum), beta
//   mma      S = k k^T            (per-key-dim gate: gated copies k*exp(G-G_ref)
//                                  and k*exp(G_ref-G), G_ref the chunk's middle row,
//                                  keep every factor bounded)
//   SIMT     A_ij = beta_i S_ij exp(G_i - G_j) (i > j, same chunk), X = (I+A)^{-1}
//            by blocked forward substitution in fp32
//   mma      w = (X diag(beta)) (k * exp(G)),  u = (X diag(beta)) v
//
// The products are warp-level mma.sync m16n8k16 (bf16 in, fp32 accumulate) fed
// by ldmatrix from the swizzled tiles: at these sizes (64 x 64 x 128 and
// 64 x 128 x 64 per tile) a tcgen05 MMA's fixed ~240-cycle cost per K=16 step
// makes it slower than mma.sync, and without tensor memory more CTAs fit an SM.
// beta is folded into the columns of X, so v feeds the MMA as TMA left it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "blackwell.cuh"
#include "gdr_internal.h"
#include "tc_common.cuh"
#include "tma_host.h"
#include "warp_mma.cuh"

namespace gdr {
namespace {

using bf16 = __nv_bfloat16;
using namespace tc;

template <int K, int V, int C, bool PER_K>
struct PrepLayout {
    static constexpr int GW = PER_K ? K : 1;
    static constexpr uint32_t kK = 0;                               // k tile [64][K]
    static constexpr uint32_t kV = kK + K * 128;                    // v tile [64][V]
    static constexpr uint32_t kKa = kV + V * 128;                   // KDA: gated k copies
    static constexpr uint32_t kKb = kKa + (PER_K ? K * 128 : 0);
    static constexpr uint32_t kF = kKb + (PER_K ? K * 128 : 0);     // fp32 region
    // fp32 arrays (float offsets from kF)
    static constexpr int fG = 0;                         // G [64][GW]
    static constexpr int fGraw = fG + 64 * GW;           // raw g (scalar gate) [64]
    static constexpr int fB = fGraw + 64;                // beta [64]
    static constexpr int fA = fB + 64;                   // A [64][65]
    static constexpr int fX = fA + kTile * kLd;          // X [64][65]
    static constexpr int fR = fX + kTile * kLd;          // solve scratch [3][16][17]
    static constexpr int fFlag = fR + 3 * 272;           // KDA: exact-path flag
    static constexpr int nF = fFlag + 4;
    static constexpr uint32_t bytes = kF + 4 * nF;
};

// Exponents of the gated k copies are clamped here; a chunk whose gate moves
// by more than kExpSafe from its middle row takes the exact fp32 path for A.
constexpr float kExpClamp = 60.f;
constexpr float kExpSafe = 40.f;

template <int K, int V, int C, bool PER_K>
__global__ void __launch_bounds__(128, 3)
prepare_mma_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                  const float* __restrict__ g, const bf16* __restrict__ beta, bf16* __restrict__ w,
                  bf16* __restrict__ u, float* __restrict__ g_cum, int T, int H, unsigned int* err) {
    using L = PrepLayout<K, V, C, PER_K>;
    constexpr int GW = L::GW;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* F = reinterpret_cast<float*>(sm + L::kF);
    float* sG = F + L::fG;
    float* sGraw = F + L::fGraw;
    float* sB = F + L::fB;
    float* sA = F + L::fA;
    float* sX = F + L::fX;
    float* sR = F + L::fR;
    int* sFlag = reinterpret_cast<int*>(F + L::fFlag);
    __shared__ uint64_t bar_tma;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * kTile, h = blockIdx.y, b = blockIdx.z;
    const int nvalid = min(kTile, T - t0);
    auto row = [&](int t) -> int64_t { return ((int64_t)b * T + t0 + t) * H + h; };
    const uint32_t s_base = bw::smem_u32(sm);

    if (tid == 0) {
        bw::mbar_init(&bar_tma, 1);
        bw::fence_mbar_init();
        *sFlag = 0;
    }
    __syncthreads();

    if (tid == 0) {
        bw::mbar_arrive_expect_tx(&bar_tma, (K + V) * 128);
#pragma unroll
        for (int a = 0; a < K / 64; ++a) bw::tma_load_4d(sm + L::kK + a * 8192, &mk, &bar_tma, a * 64, h, t0, b);
#pragma unroll
        for (int a = 0; a < V / 64; ++a) bw::tma_load_4d(sm + L::kV + a * 8192, &mv, &bar_tma, a * 64, h, t0, b);
    }
    // g, beta (rows past T read as zero)
    for (int i = tid; i < kTile * GW; i += 128) {
        const int t = i / GW;
        const float x = t < nvalid ? g[row(t) * GW + i % GW] : 0.f;
        if (PER_K) sG[i] = x; else sGraw[i] = x;
    }
    for (int i = tid; i < kTile; i += 128) sB[i] = i < nvalid ? __bfloat162float(beta[row(i)]) : 0.f;
    __syncthreads();
    // chunk-local inclusive cumsum
    if (PER_K) {
        for (int col = tid; col < (kTile / C) * K; col += 128) {
            const int ch = col / K, d = col % K;
            float run = 0.f;
            for (int t = ch * C; t < ch * C + C; ++t) {
                run += sG[t * K + d];
                sG[t * K + d] = run;
                if (t < nvalid) g_cum[row(t) * K + d] = run;
            }
        }
    } else if (tid < kTile) {
        const int c0 = (tid / C) * C;
        float run = 0.f;
        for (int t = c0; t <= tid; ++t) run += sGraw[t];
        sG[tid] = run;
        if (tid < nvalid) g_cum[row(tid)] = run;
    }
    __syncthreads();

    bool ok = bw::mbar_wait(&bar_tma, 0, err, kDeviceErrTimeout);

    if (PER_K) {
        // gated copies for S: Ka = k exp(G - G_ref), Kb = k exp(G_ref - G), G_ref = middle row of the chunk
        for (int i = tid; i < kTile * (K / 8); i += 128) {
            const int r = i / (K / 8), lc = i % (K / 8);
            const int ref = (r / C) * C + C / 2;
            const uint32_t off = (uint32_t)((lc >> 3) * 8192 + r * 128 + (((lc & 7) ^ (r & 7)) << 4));
            const uint4 raw = *reinterpret_cast<const uint4*>(sm + L::kK + off);
            const bf16* kv = reinterpret_cast<const bf16*>(&raw);
            float fa[8], fb[8];
            bool big = false;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int d = lc * 8 + e;
                const float dg = sG[r * K + d] - sG[ref * K + d];
                big |= fabsf(dg) > kExpSafe;
                const float x = __bfloat162float(kv[e]);
                fa[e] = x * __expf(fminf(fmaxf(dg, -kExpClamp), kExpClamp));
                fb[e] = x * __expf(fminf(fmaxf(-dg, -kExpClamp), kExpClamp));
            }
            if (big) *sFlag = 1;
            uint4 pa, pb;
            pa.x = bw::pack_bf16(fa[0], fa[1]); pa.y = bw::pack_bf16(fa[2], fa[3]);
            pa.z = bw::pack_bf16(fa[4], fa[5]); pa.w = bw::pack_bf16(fa[6], fa[7]);
            pb.x = bw::pack_bf16(fb[0], fb[1]); pb.y = bw::pack_bf16(fb[2], fb[3]);
            pb.z = bw::pack_bf16(fb[4], fb[5]); pb.w = bw::pack_bf16(fb[6], fb[7]);
            *reinterpret_cast<uint4*>(sm + L::kKa + off) = pa;
            *reinterpret_cast<uint4*>(sm + L::kKb + off) = pb;
        }
        bw::fence_async_shared();
    }
    __syncthreads();

    const int g4 = lane >> 2, q4 = lane & 3, mi = lane >> 3, mr = lane & 7;
    const int i0 = warp * 16 + g4, i1 = i0 + 8;       // the two tile rows of this thread's fragments
    // S = k k^T for this warp's 16 rows: [16 x 64]
    {
        const uint32_t a_t = s_base + (PER_K ? L::kKa : L::kK);
        const uint32_t b_t = s_base + (PER_K ? L::kKb : L::kK);
        float S[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) {
            uint32_t a[4];
            wm::ldsm_x4(a_t + tile_off(warp * 16 + 8 * (mi & 1) + mr, 16 * kk + 8 * (mi >> 1)), a);
#pragma unroll
            for (int jp = 0; jp < 8; jp += 2) {
                uint32_t bfr[4];
                wm::ldsm_x4(b_t + tile_off(8 * jp + 8 * (mi >> 1) + mr, 16 * kk + 8 * (mi & 1)), bfr);
                wm::mma16816(S[jp], a, bfr[0], bfr[1]);
                wm::mma16816(S[jp + 1], a, bfr[2], bfr[3]);
            }
        }
        // A from S: element (i, j) of this thread's fragments
        const int c0 = (i0 / C) * C;                 // i0 and i1 share a chunk (16-row blocks never straddle one)
        const float b0 = sB[i0], b1 = sB[i1];
#pragma unroll
        for (int jn = 0; jn < 8; ++jn) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = 8 * jn + 2 * q4 + e;
                const bool in = j >= c0;
                float a0 = 0.f, a1 = 0.f;
                if (in && j < i0) a0 = PER_K ? b0 * S[jn][e] : b0 * S[jn][e] * __expf(sG[i0] - sG[j]);
                if (in && j < i1) a1 = PER_K ? b1 * S[jn][2 + e] : b1 * S[jn][2 + e] * __expf(sG[i1] - sG[j]);
                sA[i0 * kLd + j] = a0;
                sA[i1 * kLd + j] = a1;
            }
        }
    }
    __syncthreads();
    if (PER_K && *sFlag) {
        // exact fp32 A for chunks with extreme gates: A_ij = beta_i sum_d k_id k_jd exp(G_id - G_jd)
        for (int idx = tid; idx < kTile * kTile; idx += 128) {
            const int i = idx / kTile, j = idx % kTile;
            if (j >= (i / C) * C && j < i) {
                float acc = 0.f;
                for (int d = 0; d < K; ++d) {
                    const float ki = __bfloat162float(*reinterpret_cast<const bf16*>(sm + L::kK + tile_off(i, d)));
                    const float kj = __bfloat162float(*reinterpret_cast<const bf16*>(sm + L::kK + tile_off(j, d)));
                    acc += ki * kj * __expf(sG[i * K + d] - sG[j * K + d]);
                }
                sA[i * kLd + j] = sB[i] * acc;
            }
        }
        __syncthreads();
    }

    // B operand of w: k * exp(G), row-scaled in place (scalar gate) or into Ka (per-key-dim gate)
    for (int i = tid; i < kTile * (K / 8); i += 128) {
        const int r = i / (K / 8), lc = i % (K / 8);
        const uint32_t off = (uint32_t)((lc >> 3) * 8192 + r * 128 + (((lc & 7) ^ (r & 7)) << 4));
        const uint4 raw = *reinterpret_cast<const uint4*>(sm + L::kK + off);
        const bf16* kv = reinterpret_cast<const bf16*>(&raw);
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(kv[e]) * __expf(PER_K ? sG[r * K + lc * 8 + e] : sG[r]);
        uint4 p;
        p.x = bw::pack_bf16(f[0], f[1]); p.y = bw::pack_bf16(f[2], f[3]);
        p.z = bw::pack_bf16(f[4], f[5]); p.w = bw::pack_bf16(f[6], f[7]);
        *reinterpret_cast<uint4*>(sm + (PER_K ? L::kKa : L::kK) + off) = p;
    }

    solve_unit_lower<C>(sA, sX, sR, tid);

    // Tb = X diag(beta) as A fragments of this warp's 16 rows (4 k-tiles of 16 tokens)
    uint32_t ta[4][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int j0 = 16 * kk + 2 * q4, j1 = j0 + 8;
        const float bj0 = sB[j0], bj0b = sB[j0 + 1], bj1 = sB[j1], bj1b = sB[j1 + 1];
        ta[kk][0] = wm::pack2(sX[i0 * kLd + j0] * bj0, sX[i0 * kLd + j0 + 1] * bj0b);
        ta[kk][1] = wm::pack2(sX[i1 * kLd + j0] * bj0, sX[i1 * kLd + j0 + 1] * bj0b);
        ta[kk][2] = wm::pack2(sX[i0 * kLd + j1] * bj1, sX[i0 * kLd + j1 + 1] * bj1b);
        ta[kk][3] = wm::pack2(sX[i1 * kLd + j1] * bj1, sX[i1 * kLd + j1 + 1] * bj1b);
    }
    // out[16 x D] = Tb [16 x 64] * B [64 x D], B = k exp(G) or v read token-major by ldmatrix.trans;
    // bf16 rows straight to global (rows past T are not stored)
    auto product_store = [&](uint32_t b_t, bf16* out, int D) {
        const bool st0 = i0 < nvalid, st1 = i1 < nvalid;
        bf16* r0 = out + row(st0 ? i0 : 0) * D;
        bf16* r1 = out + row(st1 ? i1 : 0) * D;
#pragma unroll 1
        for (int n0 = 0; n0 < D; n0 += 64) {
            float acc[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                for (int jp = 0; jp < 8; jp += 2) {
                    uint32_t bfr[4];
                    wm::ldsm_x4_t(b_t + tile_off(16 * kk + 8 * (mi & 1) + mr, n0 + 8 * jp + 8 * (mi >> 1)), bfr);
                    wm::mma16816(acc[jp], ta[kk], bfr[0], bfr[1]);
                    wm::mma16816(acc[jp + 1], ta[kk], bfr[2], bfr[3]);
                }
            }
            if (ok) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int col = n0 + 8 * j + 2 * q4;
                    if (st0) *reinterpret_cast<uint32_t*>(r0 + col) = wm::pack2(acc[j][0], acc[j][1]);
                    if (st1) *reinterpret_cast<uint32_t*>(r1 + col) = wm::pack2(acc[j][2], acc[j][3]);
                }
            }
        }
    };
    product_store(s_base + (PER_K ? L::kKa : L::kK), w, K);
    product_store(s_base + L::kV, u, V);
}

template <int K, int V, int C, bool PER_K>
cudaError_t launch_prepare(const Dims& d, const void* k, const void* v, const float* g, const void* beta, void* w,
                           void* u, float* g_cum, cudaStream_t s, unsigned int* err) {
    using L = PrepLayout<K, V, C, PER_K>;
    CUtensorMap mk, mv;
    if (!make_tmap_tokens(&mk, k, d.B, d.T, d.H, K, kTile) || !make_tmap_tokens(&mv, v, d.B, d.T, d.H, V, kTile))
        return cudaErrorInvalidValue;
    auto kern = prepare_mma_kernel<K, V, C, PER_K>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((d.T + kTile - 1) / kTile, d.H, d.B);
    kern<<<grid, 128, smem, s>>>(mk, mv, g, (const bf16*)beta, (bf16*)w, (bf16*)u, g_cum, d.T, d.H, err);
    return cudaGetLastError();
}

template <int K, int V, int C>
cudaError_t pick_gate(const Dims& d, const void* k, const void* v, const float* g, const void* beta, void* w, void* u,
                      float* g_cum, cudaStream_t s, unsigned int* err) {
    return d.per_k ? launch_prepare<K, V, C, true>(d, k, v, g, beta, w, u, g_cum, s, err)
                   : launch_prepare<K, V, C, false>(d, k, v, g, beta, w, u, g_cum, s, err);
}

template <int K, int V>
cudaError_t pick_chunk(const Dims& d, const void* k, const void* v, const float* g, const void* beta, void* w, void* u,
                       float* g_cum, cudaStream_t s, unsigned int* err) {
    return d.C == 32 ? pick_gate<K, V, 32>(d, k, v, g, beta, w, u, g_cum, s, err)
                     : pick_gate<K, V, 64>(d, k, v, g, beta, w, u, g_cum, s, err);
}

}  // namespace

cudaError_t mma_prepare(const Dims& d, const void* k, const void* v, const float* g, const void* beta, void* w, void* u,
                       float* g_cum, cudaStream_t s, unsigned int* err) {
    if (!d.bf16) return cudaErrorInvalidValue;
    if (d.K == 64 && d.V == 64) return pick_chunk<64, 64>(d, k, v, g, beta, w, u, g_cum, s, err);
    if (d.K == 64 && d.V == 128) return pick_chunk<64, 128>(d, k, v, g, beta, w, u, g_cum, s, err);
    if (d.K == 128 && d.V == 64) return pick_chunk<128, 64>(d, k, v, g, beta, w, u, g_cum, s, err);
    return pick_chunk<128, 128>(d, k, v, g, beta, w, u, g_cum, s, err);
}

}  // namespace gdr
