// Fused state scan + chunk output for bf16 io and a scalar (per-head) gate:
// given w, u and the chunk-local cumulative gate G (from the WY prepare),
//
//   scan   ("kernel_fun/kda/_kernels/bwd_scan.py", module docstring):
//          h_c = state before chunk c;  v'_c = u_c - w_c h_c;
//          h_{c+1} = exp(G_last) h_c + (k exp(G_last - G))^T v'_c
//   output (the o assembly the same page gives to the forward's epilogue warps):
//          o_c = scale [ (q exp(G)) h_c + tril_0(q k^T * exp(G_i - G_j)) v'_c ]
//
// so v' and the checkpoints never leave the chip.  One CTA per (batch, head, 32
// value columns); serial over chunks:
//
//   warps 0-1   recurrence: each owns 16 value columns of h^T as fp32 mma.sync
//               accumulators (as in the standalone scan) and, per chunk, stages
//               bf16 h_c and v'_c in shared memory for the output warps
//   warps 2..   output, one per 16 tokens of the chunk: the gated causal P
//               (S = q k^T computed here, or the tile the prepare wrote) and
//               q exp(G) stay in registers; o = (q e^G) h_c + P v' reads h_c
//               and v' from the staging, and leaves by TMA store
//   2 warps     producer of the recurrence ring: TMA w, u; kg = k exp(G_last - G)
//               built from global loads issued a chunk ahead; the decay
//   2 warps     producer of the output ring: TMA q and k (or P); the chunk's G
//
// The two rings are separate so the output warps, which trail the recurrence,
// never hold it back.  Shared tiles read by ldmatrix use 128-byte (k, q, w, kg)
// or 64-byte (u, h_c, v', o) XOR swizzles, so every access is conflict-free.
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

constexpr int kBV = 32;   // value columns per CTA

// byte offset of 16-byte chunk `ch` (0..3) of row r in a [rows][32] bf16 tile, 64-byte swizzle
__device__ __forceinline__ uint32_t sw64(int r, int ch) { return (uint32_t)(r * 64 + ((ch ^ ((r >> 1) & 3)) << 4)); }
// byte offset of 16-byte chunk (col / 8) of row r in a [rows][K] tile of 64-column atoms, 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int r, int col, int rows) {
    return (uint32_t)((col >> 6) * rows * 128 + r * 128 + ((((col & 63) >> 3) ^ (r & 7)) << 4));
}

template <int K, int C, bool HAS_P>
struct FLayout {
    static constexpr int NS = 2;
    static constexpr int NOW = C / 16;                  // output warps
    static constexpr int kThreads = 32 * (2 + NOW + 4);
    static constexpr uint32_t kKC = C * K * 2;          // [C][K] bf16
    static constexpr uint32_t kU = C * kBV * 2;         // [C][32] bf16
    // recurrence ring: w, kg, u, decay
    static constexpr uint32_t W = 0;
    static constexpr uint32_t KG = W + NS * kKC;
    static constexpr uint32_t U = KG + NS * kKC;
    static constexpr uint32_t GLd = U + NS * kU;        // NS x 4 floats (G_last)
    // output ring: q, k, G
    static constexpr uint32_t Q = GLd + 1024;
    static constexpr uint32_t kKR = HAS_P ? C * C * 2 : kKC;   // P [C][C] or raw k [C][K]
    static constexpr uint32_t KR = Q + NS * kKC;
    static constexpr uint32_t G = KR + NS * kKR;        // NS x C floats
    // staging
    static constexpr uint32_t HC = G + 1024;            // 2 x [K][32] bf16 h_c
    static constexpr uint32_t VP = HC + 2 * K * kBV * 2;
    static constexpr uint32_t OS = VP + 2 * kU;         // NOW x 2 x [16][32] bf16
    static constexpr uint32_t bytes = OS + NOW * 2 * 16 * kBV * 2;
    static_assert(bytes + 1024 <= 232448, "fused scan/output shared memory");
    static_assert(!HAS_P || C == 64, "a precomputed P comes in 64 x 64 tiles");
};

template <int K, int C, bool HAS_P>
__global__ void __launch_bounds__(FLayout<K, C, HAS_P>::kThreads, 1)
fused_scan_output_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mu,
                         const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                         const __grid_constant__ CUtensorMap mo, const bf16* __restrict__ k,
                         const float* __restrict__ g_cum, const float* __restrict__ h0, float* __restrict__ h_final,
                         int T, int H, int V, float scale, unsigned int* err) {
    using L = FLayout<K, C, HAS_P>;
    constexpr int NS = L::NS, NOW = L::NOW;
    constexpr int NT8 = C / 8;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = bw::smem_u32(sm);
    float* sGL = reinterpret_cast<float*>(sm + L::GLd);
    float* sG = reinterpret_cast<float*>(sm + L::G);
    __shared__ uint64_t fullA[NS], emptyA[NS], fullB[NS], emptyB[NS], hv_full[2], hv_empty[2];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.x * kBV, h = blockIdx.y, b = blockIdx.z;
    const int NT = T / C;
    const int g = lane >> 2, q4 = lane & 3, mi = lane >> 3, mr = lane & 7;
    auto row = [&](int t) -> int64_t { return ((int64_t)b * T + t) * H + h; };
    constexpr int kRec0 = 0, kOut0 = 2, kProdA0 = 2 + NOW, kProdB0 = 4 + NOW;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            bw::mbar_init(&fullA[s], 64 + 1);
            bw::mbar_init(&emptyA[s], 2);
            bw::mbar_init(&fullB[s], 64 + 1);
            bw::mbar_init(&emptyB[s], NOW);
        }
        for (int i = 0; i < 2; ++i) {
            bw::mbar_init(&hv_full[i], 2);
            bw::mbar_init(&hv_empty[i], NOW);
        }
        bw::fence_mbar_init();
    }
    __syncthreads();

    if (warp >= kProdA0 && warp < kProdB0) {
        // ------------------------------------------------------------ recurrence-ring producer (64 threads)
        const int pt = tid - 32 * kProdA0;
        constexpr int LC = K / 8, RSTEP = 64 / LC, NI = C / RSTEP;
        const int lc = pt % LC, r0 = pt / LC;
        struct Staged {
            uint4 kr[NI];
            float gr[NI], gl;
        };
        Staged sa;
        auto load_chunk = [&](int c, Staged& st) {   // issued one chunk ahead of its use
            const int t0 = c * C;
#pragma unroll
            for (int j = 0; j < NI; ++j) {
                const int t = r0 + j * RSTEP;
                st.kr[j] = *reinterpret_cast<const uint4*>(k + row(t0 + t) * K + lc * 8);
                st.gr[j] = g_cum[row(t0 + t)];
            }
            st.gl = g_cum[row(t0 + C - 1)];
        };
        auto produce = [&](int c, const Staged& st) -> bool {
            const int s = c % NS;
            if (!bw::mbar_wait(&emptyA[s], ((c / NS) & 1) ^ 1, err, kDeviceErrTimeout)) return false;
            const int t0 = c * C;
            if (pt == 0) {
                bw::mbar_arrive_expect_tx(&fullA[s], L::kKC + L::kU);
#pragma unroll
                for (int a = 0; a < K / 64; ++a)
                    bw::tma_load_4d(sm + L::W + s * L::kKC + a * C * 128, &mw, &fullA[s], a * 64, h, t0, b);
                bw::tma_load_4d(sm + L::U + s * L::kU, &mu, &fullA[s], v0, h, t0, b);
                sGL[s * 4] = st.gl;
            }
            unsigned char* kg_t = sm + L::KG + s * L::kKC;
#pragma unroll
            for (int j = 0; j < NI; ++j) {
                const int t = r0 + j * RSTEP;
                const bf16* kv = reinterpret_cast<const bf16*>(&st.kr[j]);
                const float sc = __expf(st.gl - st.gr[j]);
                uint4 p;
                p.x = bw::pack_bf16(__bfloat162float(kv[0]) * sc, __bfloat162float(kv[1]) * sc);
                p.y = bw::pack_bf16(__bfloat162float(kv[2]) * sc, __bfloat162float(kv[3]) * sc);
                p.z = bw::pack_bf16(__bfloat162float(kv[4]) * sc, __bfloat162float(kv[5]) * sc);
                p.w = bw::pack_bf16(__bfloat162float(kv[6]) * sc, __bfloat162float(kv[7]) * sc);
                *reinterpret_cast<uint4*>(kg_t + sw128(t, lc * 8, C)) = p;
            }
            bw::mbar_arrive(&fullA[s]);
            return true;
        };
        if (NT > 0) load_chunk(0, sa);
        for (int c = 0; c < NT; ++c) {
            if (!produce(c, sa)) break;
            if (c + 1 < NT) load_chunk(c + 1, sa);
        }
        return;
    }
    if (warp >= kProdB0) {
        // ------------------------------------------------------------ output-ring producer (64 threads)
        const int pt = tid - 32 * kProdB0;
        for (int c = 0; c < NT; ++c) {
            const int s = c % NS;
            if (!bw::mbar_wait(&emptyB[s], ((c / NS) & 1) ^ 1, err, kDeviceErrTimeout)) break;
            const int t0 = c * C;
            if (pt == 0) {
                bw::mbar_arrive_expect_tx(&fullB[s], L::kKC + L::kKR);
#pragma unroll
                for (int a = 0; a < K / 64; ++a) {
                    bw::tma_load_4d(sm + L::Q + s * L::kKC + a * C * 128, &mq, &fullB[s], a * 64, h, t0, b);
                    if constexpr (!HAS_P)
                        bw::tma_load_4d(sm + L::KR + s * L::kKR + a * C * 128, &mk, &fullB[s], a * 64, h, t0, b);
                }
                if constexpr (HAS_P) bw::tma_load_4d(sm + L::KR + s * L::kKR, &mk, &fullB[s], 0, 0, h, b * NT + c);
            }
            if (pt < C) sG[s * C + pt] = g_cum[row(t0 + pt)];
            bw::mbar_arrive(&fullB[s]);
        }
        return;
    }

    if (warp < kOut0) {
        // ------------------------------------------------------------ recurrence warps
        constexpr int NJ = K / 8;
        const int vr0 = warp * 16;
        const int64_t state = ((int64_t)b * H + h) * K;
        float hT[NJ][4];
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int d = 8 * j + 2 * q4;
            const int va = v0 + vr0 + g, vb = va + 8;
            if (h0) {
                hT[j][0] = h0[(state + d) * V + va];
                hT[j][1] = h0[(state + d + 1) * V + va];
                hT[j][2] = h0[(state + d) * V + vb];
                hT[j][3] = h0[(state + d + 1) * V + vb];
            } else {
                hT[j][0] = hT[j][1] = hT[j][2] = hT[j][3] = 0.f;
            }
        }
        for (int c = 0; c < NT; ++c) {
            const int s = c % NS, hb = c & 1;
            bw::mbar_wait(&fullA[s], (c / NS) & 1, err, kDeviceErrTimeout);
            const uint32_t w_t = s_base + L::W + s * L::kKC;
            const uint32_t kg_t = s_base + L::KG + s * L::kKC;
            const uint32_t u_t = s_base + L::U + s * L::kU;
            // the staging buffer of chunk c-2 must be released by the output warps
            bw::mbar_wait(&hv_empty[hb], ((c >> 1) & 1) ^ 1, err, kDeviceErrTimeout);
            // h_c -> staging [K][32] (bf16), rows = key index
            {
                const uint32_t st = s_base + L::HC + hb * (K * kBV * 2);
#pragma unroll
                for (int j = 0; j < NJ; j += 2) {
                    const uint32_t r[4] = {wm::pack2(hT[j][0], hT[j][1]), wm::pack2(hT[j][2], hT[j][3]),
                                           wm::pack2(hT[j + 1][0], hT[j + 1][1]), wm::pack2(hT[j + 1][2], hT[j + 1][3])};
                    const int d = 8 * j + 8 * (mi >> 1) + mr;
                    wm::stsm_x4_t(st + sw64(d, (vr0 >> 3) + (mi & 1)), r);
                }
            }
            // D = h^T w^T  [16 x C]
            float D[NT8][4];
#pragma unroll
            for (int j = 0; j < NT8; ++j) D[j][0] = D[j][1] = D[j][2] = D[j][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < K / 16; ++kk) {
                const uint32_t a[4] = {wm::pack2(hT[2 * kk][0], hT[2 * kk][1]), wm::pack2(hT[2 * kk][2], hT[2 * kk][3]),
                                       wm::pack2(hT[2 * kk + 1][0], hT[2 * kk + 1][1]),
                                       wm::pack2(hT[2 * kk + 1][2], hT[2 * kk + 1][3])};
#pragma unroll
                for (int jp = 0; jp < NT8; jp += 2) {
                    uint32_t bfr[4];
                    wm::ldsm_x4(w_t + sw128(8 * jp + 8 * (mi >> 1) + mr, 16 * kk + 8 * (mi & 1), C), bfr);
                    wm::mma16816(D[jp], a, bfr[0], bfr[1]);
                    wm::mma16816(D[jp + 1], a, bfr[2], bfr[3]);
                }
            }
            // v'^T = u^T - D; v' -> staging [C][32]
#pragma unroll
            for (int jp = 0; jp < NT8; jp += 2) {
                uint32_t ur[4];
                wm::ldsm_x4_t(u_t + sw64(8 * jp + 8 * (mi >> 1) + mr, (vr0 >> 3) + (mi & 1)), ur);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 uv = *reinterpret_cast<const __nv_bfloat162*>(&ur[e]);
                    float* dd = D[jp + (e >> 1)] + 2 * (e & 1);
                    dd[0] = __bfloat162float(uv.x) - dd[0];
                    dd[1] = __bfloat162float(uv.y) - dd[1];
                }
            }
            {
                const uint32_t st = s_base + L::VP + hb * L::kU;
#pragma unroll
                for (int jp = 0; jp < NT8; jp += 2) {
                    const uint32_t r[4] = {wm::pack2(D[jp][0], D[jp][1]), wm::pack2(D[jp][2], D[jp][3]),
                                           wm::pack2(D[jp + 1][0], D[jp + 1][1]), wm::pack2(D[jp + 1][2], D[jp + 1][3])};
                    wm::stsm_x4_t(st + sw64(8 * jp + 8 * (mi >> 1) + mr, (vr0 >> 3) + (mi & 1)), r);
                }
            }
            __syncwarp();
            if (lane == 0) bw::mbar_arrive(&hv_full[hb]);
            // h^T = exp(G_last) h^T + v'^T kg
            const float e = __expf(sGL[s * 4]);
#pragma unroll
            for (int j = 0; j < NJ; ++j) { hT[j][0] *= e; hT[j][1] *= e; hT[j][2] *= e; hT[j][3] *= e; }
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk) {
                const uint32_t a[4] = {wm::pack2(D[2 * kk][0], D[2 * kk][1]), wm::pack2(D[2 * kk][2], D[2 * kk][3]),
                                       wm::pack2(D[2 * kk + 1][0], D[2 * kk + 1][1]),
                                       wm::pack2(D[2 * kk + 1][2], D[2 * kk + 1][3])};
#pragma unroll
                for (int jp = 0; jp < NJ; jp += 2) {
                    uint32_t bfr[4];
                    wm::ldsm_x4_t(kg_t + sw128(16 * kk + 8 * (mi & 1) + mr, 8 * jp + 8 * (mi >> 1), C), bfr);
                    wm::mma16816(hT[jp], a, bfr[0], bfr[1]);
                    wm::mma16816(hT[jp + 1], a, bfr[2], bfr[3]);
                }
            }
            __syncwarp();
            if (lane == 0) bw::mbar_arrive(&emptyA[s]);
        }
        if (h_final) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int d = 8 * j + 2 * q4;
                const int va = v0 + vr0 + g, vb = va + 8;
                h_final[(state + d) * V + va] = hT[j][0];
                h_final[(state + d + 1) * V + va] = hT[j][1];
                h_final[(state + d) * V + vb] = hT[j][2];
                h_final[(state + d + 1) * V + vb] = hT[j][3];
            }
        }
        return;
    }

    // ---------------------------------------------------------------- output warps
    const int ow = warp - kOut0;
    const int r0 = ow * 16;                       // this warp's 16 tokens of the chunk
    for (int c = 0; c < NT; ++c) {
        const int s = c % NS, hb = c & 1;
        const int t0 = c * C;
        bw::mbar_wait(&fullB[s], (c / NS) & 1, err, kDeviceErrTimeout);
        const uint32_t q_t = s_base + L::Q + s * L::kKC;
        const uint32_t k_t = s_base + L::KR + s * L::kKR;
        const float* G = sG + s * C;
        const int i0 = r0 + g, i1 = i0 + 8;
        const float Gi0 = G[i0], Gi1 = G[i1];
        // q fragments (A operand, 16 rows x K)
        uint32_t qa[K / 16][4];
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) wm::ldsm_x4(q_t + sw128(r0 + 8 * (mi & 1) + mr, 16 * kk + 8 * (mi >> 1), C), qa[kk]);
        uint32_t pa[C / 16][4];
        if constexpr (HAS_P) {
            // P = tril_0(q k^T * exp(G_i - G_j)) precomputed by the prepare: A fragments straight from its tile
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                wm::ldsm_x4(k_t + sw128(r0 + 8 * (mi & 1) + mr, 16 * kk + 8 * (mi >> 1), C), pa[kk]);
        } else {
        // S = q k^T  [16 x C]
        float S[NT8][4];
#pragma unroll
        for (int j = 0; j < NT8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) {
#pragma unroll
            for (int jp = 0; jp < NT8; jp += 2) {
                uint32_t bfr[4];
                wm::ldsm_x4(k_t + sw128(8 * jp + 8 * (mi >> 1) + mr, 16 * kk + 8 * (mi & 1), C), bfr);
                wm::mma16816(S[jp], qa[kk], bfr[0], bfr[1]);
                wm::mma16816(S[jp + 1], qa[kk], bfr[2], bfr[3]);
            }
        }
        // P = tril_0(S * exp(G_i - G_j)) as A fragments
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk) {
            float pv[2][4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int jn = 2 * kk + hh;
                const int j0 = 8 * jn + 2 * q4;
                const float Gj0 = G[j0], Gj1 = G[j0 + 1];
                pv[hh][0] = j0 <= i0 ? S[jn][0] * __expf(Gi0 - Gj0) : 0.f;
                pv[hh][1] = j0 + 1 <= i0 ? S[jn][1] * __expf(Gi0 - Gj1) : 0.f;
                pv[hh][2] = j0 <= i1 ? S[jn][2] * __expf(Gi1 - Gj0) : 0.f;
                pv[hh][3] = j0 + 1 <= i1 ? S[jn][3] * __expf(Gi1 - Gj1) : 0.f;
            }
            pa[kk][0] = wm::pack2(pv[0][0], pv[0][1]);
            pa[kk][1] = wm::pack2(pv[0][2], pv[0][3]);
            pa[kk][2] = wm::pack2(pv[1][0], pv[1][1]);
            pa[kk][3] = wm::pack2(pv[1][2], pv[1][3]);
        }
        }
        // q exp(G_i) in place
        const float e0 = __expf(Gi0), e1 = __expf(Gi1);
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&qa[kk][e]);
                const float sc = (e & 1) ? e1 : e0;   // a1, a3 hold row i1
                qa[kk][e] = wm::pack2(__bfloat162float(x.x) * sc, __bfloat162float(x.y) * sc);
            }
        }
        // o = (q e^G) h_c + P v'   [16 x 32]
        bw::mbar_wait(&hv_full[hb], (c >> 1) & 1, err, kDeviceErrTimeout);
        const uint32_t hc_t = s_base + L::HC + hb * (K * kBV * 2);
        const uint32_t vp_t = s_base + L::VP + hb * L::kU;
        float o[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) {
#pragma unroll
            for (int jp = 0; jp < 4; jp += 2) {
                uint32_t bfr[4];
                wm::ldsm_x4_t(hc_t + sw64(16 * kk + 8 * (mi & 1) + mr, jp + (mi >> 1)), bfr);
                wm::mma16816(o[jp], qa[kk], bfr[0], bfr[1]);
                wm::mma16816(o[jp + 1], qa[kk], bfr[2], bfr[3]);
            }
        }
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk) {
#pragma unroll
            for (int jp = 0; jp < 4; jp += 2) {
                uint32_t bfr[4];
                wm::ldsm_x4_t(vp_t + sw64(16 * kk + 8 * (mi & 1) + mr, jp + (mi >> 1)), bfr);
                wm::mma16816(o[jp], pa[kk], bfr[0], bfr[1]);
                wm::mma16816(o[jp + 1], pa[kk], bfr[2], bfr[3]);
            }
        }
        __syncwarp();
        if (lane == 0) {
            bw::mbar_arrive(&hv_empty[hb]);
            bw::mbar_arrive(&emptyB[s]);
            bw::bulk_wait_read<1>();     // this warp's o staging from two chunks ago has been read
        }
        __syncwarp();
        // o * scale -> bf16 staging [16][32] -> TMA store
        const uint32_t os = s_base + L::OS + (ow * 2 + hb) * (16 * kBV * 2);
#pragma unroll
        for (int jp = 0; jp < 4; jp += 2) {
            const uint32_t r[4] = {wm::pack2(o[jp][0] * scale, o[jp][1] * scale),
                                   wm::pack2(o[jp][2] * scale, o[jp][3] * scale),
                                   wm::pack2(o[jp + 1][0] * scale, o[jp + 1][1] * scale),
                                   wm::pack2(o[jp + 1][2] * scale, o[jp + 1][3] * scale)};
            // non-transposed: matrix (rows 8*(mi&1).., column chunk jp + (mi>>1))
            asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(
                             os + sw64(8 * (mi & 1) + mr, jp + (mi >> 1))),
                         "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                         : "memory");
        }
        bw::fence_async_shared();
        __syncwarp();
        if (lane == 0) {
            bw::tma_store_4d(&mo, sm + L::OS + (ow * 2 + hb) * (16 * kBV * 2), v0, h, t0 + r0, b);
            bw::bulk_commit();
        }
    }
    if (lane == 0) bw::bulk_wait<0>();
}

template <int K, int C, bool HAS_P>
cudaError_t launch(const Dims& d, const void* q, const void* k, const void* w, const void* u, const float* g_cum,
                   const void* P, const float* h0, void* o, float* h_final, cudaStream_t s, unsigned int* err) {
    using L = FLayout<K, C, HAS_P>;
    CUtensorMap mw, mu, mq, mk, mo;
    if (!make_tmap_tokens(&mw, w, d.B, d.T, d.H, K, C) || !make_tmap_tokens_sw64(&mu, u, d.B, d.T, d.H, d.V, C) ||
        !make_tmap_tokens(&mq, q, d.B, d.T, d.H, K, C) || !make_tmap_tokens_sw64(&mo, o, d.B, d.T, d.H, d.V, 16))
        return cudaErrorInvalidValue;
    if constexpr (HAS_P) {
        // P [B, NT, H, C, C] seen as (C, C, H, B*NT); one C x C box per chunk
        const uint64_t dims[4] = {(uint64_t)C, (uint64_t)C, (uint64_t)d.H, (uint64_t)d.B * d.NT};
        const uint64_t st[3] = {(uint64_t)C * 2, (uint64_t)C * C * 2, (uint64_t)d.H * C * C * 2};
        const uint32_t box[4] = {(uint32_t)C, (uint32_t)C, 1, 1};
        if (!make_tmap_bf16_4d(&mk, P, dims, st, box)) return cudaErrorInvalidValue;
    } else {
        if (!make_tmap_tokens(&mk, k, d.B, d.T, d.H, K, C)) return cudaErrorInvalidValue;
    }
    auto kern = fused_scan_output_kernel<K, C, HAS_P>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(d.V / kBV, d.H, d.B);
    kern<<<grid, L::kThreads, smem, s>>>(mw, mu, mq, mk, mo, (const bf16*)k, g_cum, h0, h_final, d.T, d.H, d.V,
                                         d.scale, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t mma_scan_output(const Dims& d, const void* q, const void* k, const void* w, const void* u,
                            const float* g_cum, const void* P, const float* h0, void* o, float* h_final,
                            cudaStream_t s, unsigned int* err) {
    if (!d.bf16 || d.per_k || (P && d.C != 64)) return cudaErrorInvalidValue;
    if (P) {
        return d.K == 64 ? launch<64, 64, true>(d, q, k, w, u, g_cum, P, h0, o, h_final, s, err)
                         : launch<128, 64, true>(d, q, k, w, u, g_cum, P, h0, o, h_final, s, err);
    }
    if (d.K == 64) return d.C == 32 ? launch<64, 32, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, s, err)
                                    : launch<64, 64, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, s, err);
    return d.C == 32 ? launch<128, 32, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, s, err)
                     : launch<128, 64, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, s, err);
}

}  // namespace gdr
