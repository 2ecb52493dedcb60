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

template <int K, int V, int C, bool PER_K, bool WITH_P>
struct PrepLayout {
    static constexpr int GW = PER_K ? K : 1;
    static constexpr uint32_t kK = 0;                               // k tile [64][K]
    static constexpr uint32_t kV = kK + K * 128;                    // v tile [64][V]
    static constexpr uint32_t kQ = kV + V * 128;                    // q tile [64][K] (with P)
    static constexpr uint32_t kKa = kQ + (WITH_P ? K * 128 : 0);    // KDA: gated k copies
    static constexpr uint32_t kKb = kKa + (PER_K ? K * 128 : 0);
    static constexpr uint32_t kF = kKb + (PER_K ? K * 128 : 0);     // fp32 region
    // fp32 arrays (float offsets from kF)
    static constexpr int fG = 0;                         // G [64][GW]
    static constexpr int fB = fG + 64 * GW;              // beta [64]
    static constexpr int fA = fB + 64;                   // A [64][65]
    static constexpr int fX = fA + kTile * kLd;          // X [64][65]
    static constexpr int fR = fX + kTile * kLd;          // solve scratch [3][16][17]
    static constexpr int fFlag = fR + 3 * 272;           // KDA: exact-path flag
    static constexpr int nF = fFlag + 4;
    static constexpr uint32_t bytes = kF + 4 * nF;
    static constexpr uint32_t kStageBytes = (K + V) * 128;          // w, u staging reuses the fp32 region
    static_assert(4 * nF >= kStageBytes, "fp32 region must hold the w/u staging");
    static_assert(!WITH_P || (C == 64 && !PER_K), "P is produced for 64-token chunks and a scalar gate");
};

// Exponents of the gated k copies are clamped here; a chunk whose gate moves
// by more than kExpSafe from its middle row takes the exact fp32 path for A.
constexpr float kExpClamp = 60.f;
constexpr float kExpSafe = 40.f;

template <int K, int V, int C, bool PER_K, bool WITH_P>
__global__ void __launch_bounds__(128, WITH_P ? 2 : 3)
prepare_mma_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                   const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mu,
                   const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mp,
                   const float* __restrict__ g, const bf16* __restrict__ beta, float* __restrict__ g_cum,
                   int T, int H, unsigned int* err) {
    using L = PrepLayout<K, V, C, PER_K, WITH_P>;
    constexpr int GW = L::GW;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* F = reinterpret_cast<float*>(sm + L::kF);
    float* sG = F + L::fG;
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
        bw::mbar_arrive_expect_tx(&bar_tma, (K + V + (WITH_P ? K : 0)) * 128);
#pragma unroll
        for (int a = 0; a < K / 64; ++a) bw::tma_load_4d(sm + L::kK + a * 8192, &mk, &bar_tma, a * 64, h, t0, b);
#pragma unroll
        for (int a = 0; a < V / 64; ++a) bw::tma_load_4d(sm + L::kV + a * 8192, &mv, &bar_tma, a * 64, h, t0, b);
        if constexpr (WITH_P) {
#pragma unroll
            for (int a = 0; a < K / 64; ++a) bw::tma_load_4d(sm + L::kQ + a * 8192, &mq, &bar_tma, a * 64, h, t0, b);
        }
    }
    // beta; g (rows past T read as zero)
    for (int i = tid; i < kTile; i += 128) sB[i] = i < nvalid ? __bfloat162float(beta[row(i)]) : 0.f;
    if (PER_K) {
        for (int i = tid; i < kTile * GW; i += 128) {
            const int t = i / GW;
            sG[i] = t < nvalid ? g[row(t) * GW + i % GW] : 0.f;
        }
    } else if (warp == 0) {
        // scalar gate: warp shuffle scan, lane l holds rows l and 32 + l
        float x0 = lane < nvalid ? g[row(lane)] : 0.f;
        float x1 = 32 + lane < nvalid ? g[row(32 + lane)] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
            if (lane >= o) { x0 += y0; x1 += y1; }
        }
        if (C == 64) x1 += __shfl_sync(0xffffffffu, x0, 31);   // one chunk spans both halves
        sG[lane] = x0;
        sG[32 + lane] = x1;
        if (lane < nvalid) g_cum[row(lane)] = x0;
        if (32 + lane < nvalid) g_cum[row(32 + lane)] = x1;
    }
    __syncthreads();
    // chunk-local inclusive cumsum (per-key-dim gate: one thread per key column)
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
        __syncthreads();
    }

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
        float S[8][4], Pq[WITH_P ? 8 : 1][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
        if constexpr (WITH_P) {
#pragma unroll
            for (int j = 0; j < 8; ++j) Pq[j][0] = Pq[j][1] = Pq[j][2] = Pq[j][3] = 0.f;
        }
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) {
            uint32_t a[4], aq[4];
            wm::ldsm_x4(a_t + tile_off(warp * 16 + 8 * (mi & 1) + mr, 16 * kk + 8 * (mi >> 1)), a);
            if constexpr (WITH_P)
                wm::ldsm_x4(s_base + L::kQ + tile_off(warp * 16 + 8 * (mi & 1) + mr, 16 * kk + 8 * (mi >> 1)), aq);
#pragma unroll
            for (int jp = 0; jp < 8; jp += 2) {
                uint32_t bfr[4];
                wm::ldsm_x4(b_t + tile_off(8 * jp + 8 * (mi >> 1) + mr, 16 * kk + 8 * (mi & 1)), bfr);
                wm::mma16816(S[jp], a, bfr[0], bfr[1]);
                wm::mma16816(S[jp + 1], a, bfr[2], bfr[3]);
                if constexpr (WITH_P) {
                    wm::mma16816(Pq[jp % (WITH_P ? 8 : 1)], aq, bfr[0], bfr[1]);
                    wm::mma16816(Pq[(jp + 1) % (WITH_P ? 8 : 1)], aq, bfr[2], bfr[3]);
                }
            }
        }
        if constexpr (WITH_P) {
            // P = tril_0(q k^T * exp(G_i - G_j)) -> bf16 into the q tile's place (q is no longer needed),
            // as a [64][64] tile in the 128-byte swizzle; stored with w and u below
#pragma unroll
            for (int jp = 0; jp < 8; jp += 2) {
                float pv[2][4];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int jn = jp + hh, j0 = 8 * jn + 2 * q4;
                    const float* PjR = Pq[jn % (WITH_P ? 8 : 1)];
                    pv[hh][0] = j0 <= i0 ? PjR[0] * __expf(sG[i0] - sG[j0]) : 0.f;
                    pv[hh][1] = j0 + 1 <= i0 ? PjR[1] * __expf(sG[i0] - sG[j0 + 1]) : 0.f;
                    pv[hh][2] = j0 <= i1 ? PjR[2] * __expf(sG[i1] - sG[j0]) : 0.f;
                    pv[hh][3] = j0 + 1 <= i1 ? PjR[3] * __expf(sG[i1] - sG[j0 + 1]) : 0.f;
                }
                const uint32_t r[4] = {wm::pack2(pv[0][0], pv[0][1]), wm::pack2(pv[0][2], pv[0][3]),
                                       wm::pack2(pv[1][0], pv[1][1]), wm::pack2(pv[1][2], pv[1][3])};
                __syncwarp();
                asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(
                                 s_base + L::kQ + tile_off(warp * 16 + 8 * (mi & 1) + mr, 8 * jp + 8 * (mi >> 1))),
                             "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                             : "memory");
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
    // the fp32 scratch is dead from here on: it becomes the bf16 staging of w and u
    __syncthreads();
    unsigned char* stage = sm + L::kF;
    // out[16 x D] = Tb [16 x 64] * B [64 x D], B = k exp(G) or v read token-major by ldmatrix.trans;
    // bf16 results to the staging tile (128-byte swizzle, 64-column atoms) by stmatrix
    auto product_stage = [&](uint32_t b_t, uint32_t st, int D) {
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
#pragma unroll
            for (int jp = 0; jp < 8; jp += 2) {
                const uint32_t r[4] = {wm::pack2(acc[jp][0], acc[jp][1]), wm::pack2(acc[jp][2], acc[jp][3]),
                                       wm::pack2(acc[jp + 1][0], acc[jp + 1][1]),
                                       wm::pack2(acc[jp + 1][2], acc[jp + 1][3])};
                asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(
                                 st + tile_off(warp * 16 + 8 * (mi & 1) + mr, n0 + 8 * jp + 8 * (mi >> 1))),
                             "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                             : "memory");
            }
        }
    };
    const uint32_t st_w = bw::smem_u32(stage), st_u = st_w + K * 128;
    product_stage(s_base + (PER_K ? L::kKa : L::kK), st_w, K);
    product_stage(s_base + L::kV, st_u, V);
    bw::fence_async_shared();
    __syncthreads();
    if (tid == 0 && ok) {
        // rows past T are clipped by the tensor maps
#pragma unroll
        for (int a = 0; a < K / 64; ++a) bw::tma_store_4d(&mw, stage + a * 8192, a * 64, h, t0, b);
#pragma unroll
        for (int a = 0; a < V / 64; ++a) bw::tma_store_4d(&mu, stage + K * 128 + a * 8192, a * 64, h, t0, b);
        if constexpr (WITH_P) bw::tma_store_4d(&mp, sm + L::kQ, 0, 0, h, b * (T / C) + t0 / C);
        bw::bulk_commit();
        bw::bulk_wait_read<0>();
    }
}

template <int K, int V, int C, bool PER_K, bool WITH_P>
cudaError_t launch_prepare(const Dims& d, const void* q, const void* k, const void* v, const float* g,
                           const void* beta, void* w, void* u, float* g_cum, void* P, cudaStream_t s,
                           unsigned int* err) {
    using L = PrepLayout<K, V, C, PER_K, WITH_P>;
    CUtensorMap mk, mv, mw, mu, mq, mp;
    if (!make_tmap_tokens(&mk, k, d.B, d.T, d.H, K, kTile) || !make_tmap_tokens(&mv, v, d.B, d.T, d.H, V, kTile) ||
        !make_tmap_tokens(&mw, w, d.B, d.T, d.H, K, kTile) || !make_tmap_tokens(&mu, u, d.B, d.T, d.H, V, kTile))
        return cudaErrorInvalidValue;
    mq = mk;
    mp = mw;
    if constexpr (WITH_P) {
        // P [B, NT, H, C, C] seen as (C, C, H, B*NT); one 64 x 64 box per chunk
        const uint64_t dims[4] = {(uint64_t)C, (uint64_t)C, (uint64_t)d.H, (uint64_t)d.B * d.NT};
        const uint64_t st[3] = {(uint64_t)C * 2, (uint64_t)C * C * 2, (uint64_t)d.H * C * C * 2};
        const uint32_t box[4] = {64, 64, 1, 1};
        if (!make_tmap_tokens(&mq, q, d.B, d.T, d.H, K, kTile) || !make_tmap_bf16_4d(&mp, P, dims, st, box))
            return cudaErrorInvalidValue;
    }
    auto kern = prepare_mma_kernel<K, V, C, PER_K, WITH_P>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((d.T + kTile - 1) / kTile, d.H, d.B);
    kern<<<grid, 128, smem, s>>>(mk, mv, mw, mu, mq, mp, g, (const bf16*)beta, g_cum, d.T, d.H, err);
    return cudaGetLastError();
}

template <int K, int V, int C>
cudaError_t pick_gate(const Dims& d, const void* q, const void* k, const void* v, const float* g, const void* beta,
                      void* w, void* u, float* g_cum, void* P, cudaStream_t s, unsigned int* err) {
    if (d.per_k) return launch_prepare<K, V, C, true, false>(d, q, k, v, g, beta, w, u, g_cum, P, s, err);
    if constexpr (C == 64) {
        if (P) return launch_prepare<K, V, C, false, true>(d, q, k, v, g, beta, w, u, g_cum, P, s, err);
    }
    return launch_prepare<K, V, C, false, false>(d, q, k, v, g, beta, w, u, g_cum, P, s, err);
}

template <int K, int V>
cudaError_t pick_chunk(const Dims& d, const void* q, const void* k, const void* v, const float* g, const void* beta,
                       void* w, void* u, float* g_cum, void* P, cudaStream_t s, unsigned int* err) {
    return d.C == 32 ? pick_gate<K, V, 32>(d, q, k, v, g, beta, w, u, g_cum, P, s, err)
                     : pick_gate<K, V, 64>(d, q, k, v, g, beta, w, u, g_cum, P, s, err);
}

}  // namespace

cudaError_t mma_prepare(const Dims& d, const void* k, const void* v, const float* g, const void* beta, void* w,
                        void* u, float* g_cum, cudaStream_t s, unsigned int* err, const void* q, void* P) {
    if (!d.bf16) return cudaErrorInvalidValue;
    if (P && (d.per_k || d.C != 64 || !q)) return cudaErrorInvalidValue;
    if (d.K == 64 && d.V == 64) return pick_chunk<64, 64>(d, q, k, v, g, beta, w, u, g_cum, P, s, err);
    if (d.K == 64 && d.V == 128) return pick_chunk<64, 128>(d, q, k, v, g, beta, w, u, g_cum, P, s, err);
    if (d.K == 128 && d.V == 64) return pick_chunk<128, 64>(d, q, k, v, g, beta, w, u, g_cum, P, s, err);
    return pick_chunk<128, 128>(d, q, k, v, g, beta, w, u, g_cum, P, s, err);
}

}  // namespace gdr
