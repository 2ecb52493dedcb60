// State scan for bf16 io with the recurrence in registers (the re-scan of
// "kernel_fun/kda/_kernels/bwd_scan.py", module docstring: hck[c] = h before the
// update, v' = u - w h, h = exp(decay) h + kg^T v').
//
// One CTA per (batch, head, 32 value columns); serial over chunks.  Each of the
// two recurrence warps owns 16 value columns of h^T (16 x K) as fp32 mma.sync
// accumulator fragments for the whole sequence, so per chunk
//
//   D   = h^T w^T                 [16 x C]   A = bf16(h^T) from its own accumulator
//   v'^T = u^T - D                            u^T fragments by ldmatrix.trans
//   h^T = exp(G_last) * h^T + v'^T kg   [16 x K]   A = bf16(v'^T) from D, accumulating in place
//
// runs as two short dependent mma.sync chains with no shared-memory round trip
// and no barrier between the two warps (a tcgen05 MMA costs ~240 SM cycles per
// K=16 step on this part whatever its shape, which is what this chain cannot afford).
// Four producer warps stream w and u by TMA and build kg = k exp(G_last - G) and
// the decay row into a 2-stage ring, their global loads two chunks ahead; v_new
// and the checkpoints leave through stmatrix.trans into per-warp staging and TMA
// stores.
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

constexpr int kBV = 32;        // value columns per CTA
constexpr int kRecWarps = 2;   // recurrence warps (16 columns each)
constexpr int kProdThreads = 128;
constexpr int kThreads = 32 * kRecWarps + kProdThreads;

template <int K, int C, bool PER_K>
struct MScanLayout {
    static constexpr int NS = 2;
    static constexpr int GW = PER_K ? K : 1;
    static constexpr int GWS = GW < 4 ? 4 : GW;
    static constexpr uint32_t kKC = C * K * 2;                    // [C][K] bf16, 128-byte swizzle
    static constexpr uint32_t kU = C * kBV * 2;                   // [C][32] bf16, plain 64-byte rows
    static constexpr uint32_t kSV = C * 16 * 2;                   // v_new staging [C][16] per warp per buffer
    static constexpr uint32_t kSH = K * 16 * 2;                   // checkpoint staging [K][16]
    static constexpr uint32_t W = 0;
    static constexpr uint32_t KG = W + NS * kKC;
    static constexpr uint32_t U = KG + NS * kKC;
    static constexpr uint32_t SV = U + NS * kU;
    static constexpr uint32_t SH = SV + kRecWarps * 2 * kSV;
    static constexpr uint32_t GL = SH + kRecWarps * 2 * kSH;
    static constexpr uint32_t bytes = GL + NS * 4 * GWS;
    static constexpr uint32_t tx = kKC + kU;
    static constexpr uint32_t full_count = kProdThreads + 1;
};

template <int K, int C, bool PER_K>
__global__ void __launch_bounds__(kThreads, 1)
scan_mma_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mu,
                const __grid_constant__ CUtensorMap mvn, const __grid_constant__ CUtensorMap mck,
                const bf16* __restrict__ k, const float* __restrict__ g_cum, const float* __restrict__ h0,
                int has_ckpt, float* __restrict__ h_final, int T, int H, int V, unsigned int* err) {
    using L = MScanLayout<K, C, PER_K>;
    constexpr int GW = L::GW;
    constexpr int NJ = K / 8;      // n-tiles of h^T (over K)
    constexpr int NT8 = C / 8;     // n-tiles of D (over the chunk's tokens)
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* sGL = reinterpret_cast<float*>(sm + L::GL);
    __shared__ uint64_t full[L::NS], empty[L::NS];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.x * kBV, h = blockIdx.y, b = blockIdx.z;
    const int NT = T / C;
    const uint32_t s_base = bw::smem_u32(sm);
    auto row = [&](int t) -> int64_t { return ((int64_t)b * T + t) * H + h; };

    if (tid == 0) {
        for (int s = 0; s < L::NS; ++s) {
            bw::mbar_init(&full[s], L::full_count);
            bw::mbar_init(&empty[s], kRecWarps);
        }
        bw::fence_mbar_init();
    }
    __syncthreads();

    if (warp >= kRecWarps) {
        // ---------------------------------------------------------------- producers
        const int pt = tid - 32 * kRecWarps;
        constexpr int LC = K / 8;
        constexpr int RSTEP = kProdThreads / LC;
        constexpr int NI = C / RSTEP;
        constexpr int GV = PER_K ? 8 : 1;
        const int lc = pt % LC, r0 = pt / LC;
        // Two register sets: the global loads of chunk c+2 are in flight while
        // chunk c+1 is built, so their latency hides behind a whole chunk step.
        struct Staged {
            uint4 kr[NI];
            float gr[NI][GV], gl8[GV];
        };
        Staged sa, sb;
        auto load_chunk = [&](int c, Staged& st) {   // all of a chunk's global loads issued together
            const int t0 = c * C;
            const float* gl = g_cum + row(t0 + C - 1) * GW;
#pragma unroll
            for (int j = 0; j < NI; ++j) {
                const int t = r0 + j * RSTEP;
                st.kr[j] = *reinterpret_cast<const uint4*>(k + row(t0 + t) * K + lc * 8);
                if constexpr (PER_K) {
                    const float4* gt = reinterpret_cast<const float4*>(g_cum + row(t0 + t) * K + lc * 8);
                    *reinterpret_cast<float4*>(&st.gr[j][0]) = gt[0];
                    *reinterpret_cast<float4*>(&st.gr[j][4]) = gt[1];
                } else {
                    st.gr[j][0] = g_cum[row(t0 + t)];
                }
            }
            if constexpr (PER_K) {
                const float4* g8 = reinterpret_cast<const float4*>(gl + lc * 8);
                *reinterpret_cast<float4*>(&st.gl8[0]) = g8[0];
                *reinterpret_cast<float4*>(&st.gl8[4]) = g8[1];
            } else {
                st.gl8[0] = gl[0];
            }
        };
        auto produce = [&](int c, const Staged& st) -> bool {
            const int s = c % L::NS;
            if (!bw::mbar_wait(&empty[s], ((c / L::NS) & 1) ^ 1, err, kDeviceErrTimeout)) return false;
            const int t0 = c * C;
            if (pt == 0) {
                bw::mbar_arrive_expect_tx(&full[s], L::tx);
#pragma unroll
                for (int a = 0; a < K / 64; ++a)
                    bw::tma_load_4d(sm + L::W + s * L::kKC + a * C * 128, &mw, &full[s], a * 64, h, t0, b);
                bw::tma_load_4d(sm + L::U + s * L::kU, &mu, &full[s], v0, h, t0, b);
            }
            if constexpr (PER_K) {
                const float* gl = g_cum + row(t0 + C - 1) * GW;
                for (int d = pt; d < K; d += kProdThreads) sGL[s * L::GWS + d] = gl[d];
            } else {
                if (pt == 0) sGL[s * L::GWS] = st.gl8[0];
            }
            unsigned char* kg_t = sm + L::KG + s * L::kKC;
#pragma unroll
            for (int j = 0; j < NI; ++j) {
                const int t = r0 + j * RSTEP;
                const bf16* kv = reinterpret_cast<const bf16*>(&st.kr[j]);
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float dg = PER_K ? st.gl8[e % GV] - st.gr[j][e % GV] : st.gl8[0] - st.gr[j][0];
                    f[e] = __bfloat162float(kv[e]) * __expf(dg);
                }
                uint4 p;
                p.x = bw::pack_bf16(f[0], f[1]); p.y = bw::pack_bf16(f[2], f[3]);
                p.z = bw::pack_bf16(f[4], f[5]); p.w = bw::pack_bf16(f[6], f[7]);
                *reinterpret_cast<uint4*>(kg_t + (lc >> 3) * C * 128 + t * 128 + (((lc & 7) ^ (t & 7)) << 4)) = p;
            }
            bw::fence_async_shared();
            bw::mbar_arrive(&full[s]);
            return true;
        };
        if (NT > 0) load_chunk(0, sa);
        if (NT > 1) load_chunk(1, sb);
        for (int c = 0; c < NT; c += 2) {
            if (!produce(c, sa)) break;
            if (c + 2 < NT) load_chunk(c + 2, sa);
            if (c + 1 < NT) {
                if (!produce(c + 1, sb)) break;
                if (c + 3 < NT) load_chunk(c + 3, sb);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- recurrence warps
    const int g = lane >> 2, q4 = lane & 3;
    const int vr0 = warp * 16;                         // this warp's columns within the CTA's 32
    const int mi = lane >> 3, mr = lane & 7;           // ldmatrix/stmatrix: matrix and row this lane addresses
    const int64_t state = ((int64_t)b * H + h) * K;
    float hT[NJ][4];                                   // h^T[v][d]: (g | g+8, 8j + 2q4 | +1)
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
    bool ok = true;
    for (int c = 0; c < NT; ++c) {
        const int s = c % L::NS, hb = c & 1;
        const int t0 = c * C;
        ok = ok && bw::mbar_wait(&full[s], (c / L::NS) & 1, err, kDeviceErrTimeout);
        const uint32_t w_t = s_base + L::W + s * L::kKC;
        const uint32_t kg_t = s_base + L::KG + s * L::kKC;
        const uint32_t u_t = s_base + L::U + s * L::kU;

        // checkpoint c (h before this chunk): stmatrix.trans h^T -> [K][16] staging, TMA store
        if (has_ckpt) {
            if (lane == 0) bw::bulk_wait_read<3>();
            __syncwarp();
            const uint32_t st = s_base + L::SH + (warp * 2 + hb) * L::kSH;
#pragma unroll
            for (int j = 0; j < NJ; j += 2) {
                const uint32_t r[4] = {wm::pack2(hT[j][0], hT[j][1]), wm::pack2(hT[j][2], hT[j][3]),
                                       wm::pack2(hT[j + 1][0], hT[j + 1][1]), wm::pack2(hT[j + 1][2], hT[j + 1][3])};
                const int d = 8 * j + 8 * (mi >> 1) + mr;
                wm::stsm_x4_t(st + d * 32 + (mi & 1) * 16, r);
            }
            bw::fence_async_shared();
            __syncwarp();
            if (lane == 0) {
                bw::tma_store_4d(&mck, sm + L::SH + (warp * 2 + hb) * L::kSH, v0 + vr0, 0, h, b * NT + c);
                bw::bulk_commit();
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
                const int t = 8 * jp + 8 * (mi >> 1) + mr, d = 16 * kk + 8 * (mi & 1);
                uint32_t bfr[4];
                wm::ldsm_x4(w_t + (d >> 6) * C * 128 + t * 128 + ((((d & 63) >> 3) ^ (t & 7)) << 4), bfr);
                wm::mma16816(D[jp], a, bfr[0], bfr[1]);
                wm::mma16816(D[jp + 1], a, bfr[2], bfr[3]);
            }
        }
        // v'^T = u^T - D  (u^T in D's fragment layout straight from ldmatrix.trans)
#pragma unroll
        for (int jp = 0; jp < NT8; jp += 2) {
            const int t = 8 * jp + 8 * (mi >> 1) + mr;
            uint32_t ur[4];
            wm::ldsm_x4_t(u_t + t * 64 + (vr0 + 8 * (mi & 1)) * 2, ur);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 uv = *reinterpret_cast<const __nv_bfloat162*>(&ur[e]);
                float* dd = D[jp + (e >> 1)] + 2 * (e & 1);
                dd[0] = __bfloat162float(uv.x) - dd[0];
                dd[1] = __bfloat162float(uv.y) - dd[1];
            }
        }
        // v_new: stmatrix.trans v'^T -> [C][16] staging, TMA store
        {
            if (lane == 0) {
                if (has_ckpt) bw::bulk_wait_read<3>(); else bw::bulk_wait_read<1>();
            }
            __syncwarp();
            const uint32_t st = s_base + L::SV + (warp * 2 + hb) * L::kSV;
#pragma unroll
            for (int jp = 0; jp < NT8; jp += 2) {
                const uint32_t r[4] = {wm::pack2(D[jp][0], D[jp][1]), wm::pack2(D[jp][2], D[jp][3]),
                                       wm::pack2(D[jp + 1][0], D[jp + 1][1]), wm::pack2(D[jp + 1][2], D[jp + 1][3])};
                const int t = 8 * jp + 8 * (mi >> 1) + mr;
                wm::stsm_x4_t(st + t * 32 + (mi & 1) * 16, r);
            }
            bw::fence_async_shared();
            __syncwarp();
            if (lane == 0) {
                bw::tma_store_4d(&mvn, sm + L::SV + (warp * 2 + hb) * L::kSV, v0 + vr0, h, t0, b);
                bw::bulk_commit();
            }
        }
        // h^T = exp(G_last) h^T + v'^T kg
        const float* gl = sGL + s * L::GWS;
        if constexpr (PER_K) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const float e0 = __expf(gl[8 * j + 2 * q4]), e1 = __expf(gl[8 * j + 2 * q4 + 1]);
                hT[j][0] *= e0; hT[j][1] *= e1; hT[j][2] *= e0; hT[j][3] *= e1;
            }
        } else {
            const float e = __expf(gl[0]);
#pragma unroll
            for (int j = 0; j < NJ; ++j) { hT[j][0] *= e; hT[j][1] *= e; hT[j][2] *= e; hT[j][3] *= e; }
        }
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk) {
            const uint32_t a[4] = {wm::pack2(D[2 * kk][0], D[2 * kk][1]), wm::pack2(D[2 * kk][2], D[2 * kk][3]),
                                   wm::pack2(D[2 * kk + 1][0], D[2 * kk + 1][1]),
                                   wm::pack2(D[2 * kk + 1][2], D[2 * kk + 1][3])};
#pragma unroll
            for (int jp = 0; jp < NJ; jp += 2) {
                const int t = 16 * kk + 8 * (mi & 1) + mr, d = 8 * jp + 8 * (mi >> 1);
                uint32_t bfr[4];
                wm::ldsm_x4_t(kg_t + (d >> 6) * C * 128 + t * 128 + ((((d & 63) >> 3) ^ (t & 7)) << 4), bfr);
                wm::mma16816(hT[jp], a, bfr[0], bfr[1]);
                wm::mma16816(hT[jp + 1], a, bfr[2], bfr[3]);
            }
        }
        __syncwarp();
        if (lane == 0) bw::mbar_arrive(&empty[s]);
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
    if (lane == 0) bw::bulk_wait<0>();
    (void)ok;
}

template <int K, int C, bool PER_K>
cudaError_t launch(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum, const float* h0,
                   void* h_ckpt, void* v_new, float* h_final, cudaStream_t s, unsigned int* err) {
    using L = MScanLayout<K, C, PER_K>;
    CUtensorMap mw, mu, mvn, mck;
    if (!make_tmap_tokens(&mw, w, d.B, d.T, d.H, K, C) ||
        !make_tmap_tokens_plain(&mu, u, d.B, d.T, d.H, d.V, kBV, C) ||
        !make_tmap_tokens_plain(&mvn, v_new, d.B, d.T, d.H, d.V, 16, C))
        return cudaErrorInvalidValue;
    // without checkpoints the map is never used; point it at v_new so it still encodes
    if (!(h_ckpt ? make_tmap_ckpt_plain(&mck, h_ckpt, d.B, d.NT, d.H, K, d.V, 16)
                 : make_tmap_tokens_plain(&mck, v_new, d.B, d.T, d.H, d.V, 16, C)))
        return cudaErrorInvalidValue;
    auto kern = scan_mma_kernel<K, C, PER_K>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(d.V / kBV, d.H, d.B);
    kern<<<grid, kThreads, smem, s>>>(mw, mu, mvn, mck, (const bf16*)k, g_cum, h0, h_ckpt != nullptr, h_final, d.T,
                                      d.H, d.V, err);
    return cudaGetLastError();
}

template <int K, int C>
cudaError_t gate(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum, const float* h0,
                 void* h_ckpt, void* v_new, float* h_final, cudaStream_t s, unsigned int* err) {
    return d.per_k ? launch<K, C, true>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err)
                   : launch<K, C, false>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err);
}

}  // namespace

cudaError_t mma_scan(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum, const float* h0,
                     void* h_ckpt, void* v_new, float* h_final, cudaStream_t s, unsigned int* err) {
    if (!d.bf16) return cudaErrorInvalidValue;
    if (d.K == 64) {
        return d.C == 32 ? gate<64, 32>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err)
                         : gate<64, 64>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err);
    }
    return d.C == 32 ? gate<128, 32>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err)
                     : gate<128, 64>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err);
}

}  // namespace gdr
