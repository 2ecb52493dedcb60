// The backward's reverse state scan for bf16 io, a scalar gate and 64-token
// chunks, with the recurrence in registers.  The pages' backward starts from the
// forward re-scan ("kernel_fun/kda/_kernels/bwd_scan.py", module docstring);
// this is the reverse recurrence that carries the state's gradient back
// through the chunks, the derivative of that scan's update:
//
//   dh_ckpt[c] = dh                                   (gradient of the state after chunk c)
//   dv'        = scale P^T do + (k gamma) dh          P = tril_0(q k^T * exp(G_i - G_j)), gamma = exp(G_L - G)
//   dh         = exp(G_L) dh + scale (q exp(G))^T do - w^T dv'
//
// from c = NT-1 down to 0 (dh = dh_final first; dh0 = dh at the end).
//
// One CTA per (batch, head, 32 value columns), as in the forward scan: four
// recurrence warps split dh^T (32 x K) into (value half vh, key half kh)
// quarters held as fp32 mma.sync accumulator fragments; one producer warp feeds
// a two-stage ring by TMA (k, w, q [C x K] with the 128-byte swizzle, do
// [C x 32] with the 64-byte swizzle, P [C x C]) plus the gate rows.  Per chunk
// and warp:
//
//   D   = dh^T[:, my keys] k[:, my keys]^T * gamma         [16 x C], the chain's first product
//   D  += scale do^T[:, my half of i] P[my half of i, :]   (the two halves sum in the exchange)
//   D   = D_0 + D_1                                         partial sums swapped through shared memory
//   E   = (do^T diag(scale exp(G))) q[:, my keys]           off the chain, issued before the exchange wait
//   dh^T[:, my keys] = exp(G_L) dh^T + E - dv'^T w[:, my keys]
//
// dv' (= D) and the bf16 checkpoints leave through stmatrix.trans staging and
// 16-byte global stores, as in the forward scan.
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

constexpr int kBV = 32;
constexpr int kRecWarps = 4;

constexpr uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }

template <int K, int C>
struct RScanLayout {
    static constexpr int NS = 2;
    static constexpr int KH = K / 2;
    static constexpr int NT8 = C / 8;
    static constexpr int kThreads = 32 * (kRecWarps + 1);
    static constexpr uint32_t kKC = C * K * 2;                     // [C][K] bf16, 128-byte swizzle
    static constexpr uint32_t kD = C * kBV * 2;                    // do [C][32] bf16, 64-byte swizzle
    static constexpr uint32_t kP = C * C * 2;                      // P [C][C] bf16, 128-byte swizzle
    static constexpr uint32_t kX = NT8 * 512;
    static constexpr uint32_t kSH = align1k(KH * 32);
    static constexpr uint32_t kSV = align1k(C / 2 * 32);
    static constexpr uint32_t KB = 0;
    static constexpr uint32_t WB = KB + NS * kKC;
    static constexpr uint32_t QB = WB + NS * kKC;
    static constexpr uint32_t DB = QB + NS * kKC;
    static constexpr uint32_t PB = align1k(DB + NS * kD);
    static constexpr uint32_t X = PB + NS * kP;
    static constexpr uint32_t SH = X + 2 * kRecWarps * kX;
    static constexpr uint32_t SV = SH + kRecWarps * kSH;
    static constexpr uint32_t GAM = SV + kRecWarps * kSV;          // gamma [NS][C]
    static constexpr uint32_t EG = GAM + NS * C * 4;               // scale exp(G) [NS][C]
    static constexpr uint32_t DEC = EG + NS * C * 4;               // exp(G_L) [NS]
    static constexpr uint32_t bytes = DEC + 16 * NS;
    static constexpr uint32_t tx = 3 * kKC + kD + kP;
    static constexpr uint32_t full_count = 32 + 1;
    static_assert(C == 64, "P tiles are 64 x 64");
};

template <int K, int C>
__global__ void __launch_bounds__(RScanLayout<K, C>::kThreads, 1)
bwd_scan_mma_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mw,
                    const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mdo,
                    const __grid_constant__ CUtensorMap mp, const float* __restrict__ g_cum,
                    const float* __restrict__ dh_final, bf16* __restrict__ dh_ckpt, bf16* __restrict__ dv_new,
                    float* __restrict__ dh0, int T, int H, int V, int G, float scale, unsigned int* err) {
    using L = RScanLayout<K, C>;
    constexpr int KH = L::KH, NT8 = L::NT8;
    constexpr int NJH = KH / 8;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[L::NS], empty[L::NS];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.x * kBV, h = blockIdx.y, b = blockIdx.z;
    const int NT = (T + C - 1) / C;
    const uint32_t s_base = bw::smem_u32(sm);
    auto rowc = [&](int t) -> int64_t { return ((int64_t)b * T + min(t, T - 1)) * H + h; };   // G past T: its last value

    if (tid == 0) {
        for (int s = 0; s < L::NS; ++s) {
            bw::mbar_init(&full[s], L::full_count);
            bw::mbar_init(&empty[s], kRecWarps);
        }
        bw::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kRecWarps) {
        // ---------------------------------------------------------------- producer
        float* sGam = reinterpret_cast<float*>(sm + L::GAM);
        float* sEG = reinterpret_cast<float*>(sm + L::EG);
        float* sDec = reinterpret_cast<float*>(sm + L::DEC);
        for (int i = 0; i < NT; ++i) {
            const int c = NT - 1 - i, s = i % L::NS, t0 = c * C;
            const float g0 = g_cum[rowc(t0 + lane)], g1 = g_cum[rowc(t0 + 32 + lane)];
            const float gl = g_cum[rowc(t0 + C - 1)];
            if (!bw::mbar_wait(&empty[s], ((i / L::NS) & 1) ^ 1, err, kDeviceErrTimeout)) break;
            if (lane == 0) {
                bw::mbar_arrive_expect_tx(&full[s], L::tx);
#pragma unroll
                for (int a = 0; a < K / 64; ++a) {
                    bw::tma_load_4d(sm + L::KB + s * L::kKC + a * C * 128, &mk, &full[s], a * 64, h / G, t0, b);
                    bw::tma_load_4d(sm + L::WB + s * L::kKC + a * C * 128, &mw, &full[s], a * 64, h, t0, b);
                    bw::tma_load_4d(sm + L::QB + s * L::kKC + a * C * 128, &mq, &full[s], a * 64, h / G, t0, b);
                }
                bw::tma_load_4d(sm + L::DB + s * L::kD, &mdo, &full[s], v0, h, t0, b);
                bw::tma_load_4d(sm + L::PB + s * L::kP, &mp, &full[s], 0, 0, h, b * NT + c);
                sDec[4 * s] = __expf(gl);
            }
            sGam[s * C + lane] = __expf(gl - g0);
            sGam[s * C + 32 + lane] = __expf(gl - g1);
            sEG[s * C + lane] = scale * __expf(g0);
            sEG[s * C + 32 + lane] = scale * __expf(g1);
            bw::mbar_arrive(&full[s]);
        }
        return;
    }

    // -------------------------------------------------------------------- recurrence warps
    const int g = lane >> 2, q4 = lane & 3;
    const int vh = warp & 1, kh = warp >> 1;
    const int vr0 = vh * 16, d0 = kh * KH;
    const int mi = lane >> 3, mr = lane & 7;
    const int64_t state = ((int64_t)b * H + h) * K;
    const float* sGam = reinterpret_cast<const float*>(sm + L::GAM);
    const float* sEG = reinterpret_cast<const float*>(sm + L::EG);
    const float* sDec = reinterpret_cast<const float*>(sm + L::DEC);
    float dhT[NJH][4];                                 // dh^T[v][d]: (g | g+8, d0 + 8j + 2q4 | +1)
#pragma unroll
    for (int j = 0; j < NJH; ++j) {
        const int d = d0 + 8 * j + 2 * q4;
        const int va = v0 + vr0 + g, vb = va + 8;
        if (dh_final) {
            dhT[j][0] = dh_final[(state + d) * V + va];
            dhT[j][1] = dh_final[(state + d + 1) * V + va];
            dhT[j][2] = dh_final[(state + d) * V + vb];
            dhT[j][3] = dh_final[(state + d + 1) * V + vb];
        } else {
            dhT[j][0] = dhT[j][1] = dhT[j][2] = dhT[j][3] = 0.f;
        }
    }
    auto stage_off = [](int r, int half) -> uint32_t { return r * 32 + ((half ^ ((r >> 2) & 1)) << 4); };
    auto kc_off = [](int t, int d) -> uint32_t {      // element (t, d) of a [C][K] tile, 128-byte swizzle
        return (d >> 6) * C * 128 + t * 128 + ((((d & 63) >> 3) ^ (t & 7)) << 4);
    };
    const uint32_t st_h = s_base + L::SH + warp * L::kSH;
    const uint32_t st_v = s_base + L::SV + warp * L::kSV;
    bool ok = true;
    bool ready = NT > 0 && bw::mbar_test_wait(&full[0], 0);
    for (int i = 0; i < NT; ++i) {
        const int c = NT - 1 - i, s = i % L::NS, t0 = c * C;
        if (!ready) ok = ok && bw::mbar_wait(&full[s], (i / L::NS) & 1, err, kDeviceErrTimeout);
        const uint32_t k_t = s_base + L::KB + s * L::kKC;
        const uint32_t w_t = s_base + L::WB + s * L::kKC;
        const uint32_t q_t = s_base + L::QB + s * L::kKC;
        const uint32_t do_t = s_base + L::DB + s * L::kD;
        const uint32_t p_t = s_base + L::PB + s * L::kP;

        // D = dh^T[:, my keys] k[:, my keys]^T  [16 x C]
        float D[NT8][4];
#pragma unroll
        for (int j = 0; j < NT8; ++j) D[j][0] = D[j][1] = D[j][2] = D[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KH / 16; ++kk) {
            const uint32_t a[4] = {wm::pack2(dhT[2 * kk][0], dhT[2 * kk][1]), wm::pack2(dhT[2 * kk][2], dhT[2 * kk][3]),
                                   wm::pack2(dhT[2 * kk + 1][0], dhT[2 * kk + 1][1]),
                                   wm::pack2(dhT[2 * kk + 1][2], dhT[2 * kk + 1][3])};
#pragma unroll
            for (int jp = 0; jp < NT8; jp += 2) {
                uint32_t bfr[4];
                wm::ldsm_x4(k_t + kc_off(8 * jp + 8 * (mi >> 1) + mr, d0 + 16 * kk + 8 * (mi & 1)), bfr);
                wm::mma16816(D[jp], a, bfr[0], bfr[1]);
                wm::mma16816(D[jp + 1], a, bfr[2], bfr[3]);
            }
        }

        // checkpoint c: the gradient of the state after the chunk, my [KH x 16] quarter
#pragma unroll
        for (int j = 0; j < NJH; j += 2) {
            const uint32_t r[4] = {wm::pack2(dhT[j][0], dhT[j][1]), wm::pack2(dhT[j][2], dhT[j][3]),
                                   wm::pack2(dhT[j + 1][0], dhT[j + 1][1]), wm::pack2(dhT[j + 1][2], dhT[j + 1][3])};
            wm::stsm_x4_t(st_h + stage_off(8 * j + 8 * (mi >> 1) + mr, mi & 1), r);
        }
        __syncwarp();
        {
            bf16* dst = dh_ckpt + ((((int64_t)b * NT + c) * H + h) * K + d0) * V + v0 + vr0;
#pragma unroll
            for (int r16 = 0; r16 < KH / 16; ++r16) {
                const int r = 16 * r16 + (lane >> 1), half = lane & 1;
                const uint4 x = wm::lds128(st_h + stage_off(r, half));
                *reinterpret_cast<uint4*>(dst + (int64_t)r * V + 8 * half) = x;
            }
        }

        // do^T as A fragments, k-step kk covering tokens 16kk .. 16kk+15
        uint32_t da[C / 16][4];
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk) {
            const int t = 16 * kk + 8 * (mi >> 1) + mr;
            const int ch = (vr0 >> 3) + (mi & 1);
            wm::ldsm_x4_t(do_t + t * 64 + ((ch ^ ((t >> 1) & 3)) << 4), da[kk]);
        }
        // D *= gamma (columns); + scale do^T P over my half of the query tokens i
        {
            const float* gam = sGam + s * C;
#pragma unroll
            for (int j = 0; j < NT8; ++j) {
                const float2 gg = *reinterpret_cast<const float2*>(gam + 8 * j + 2 * q4);
                D[j][0] *= gg.x; D[j][1] *= gg.y; D[j][2] *= gg.x; D[j][3] *= gg.y;
            }
            float Dl[NT8][4];
#pragma unroll
            for (int j = 0; j < NT8; ++j) Dl[j][0] = Dl[j][1] = Dl[j][2] = Dl[j][3] = 0.f;
#pragma unroll
            for (int kq = 0; kq < C / 32; ++kq) {
                // do^T for query tokens 16 kk .. of my half, loaded again by address (a runtime
                // choice among da's registers would move da to local memory)
                const int kk = kh * (C / 32) + kq;
                uint32_t ah[4];
                {
                    const int t = 16 * kk + 8 * (mi >> 1) + mr;
                    const int ch = (vr0 >> 3) + (mi & 1);
                    wm::ldsm_x4_t(do_t + t * 64 + ((ch ^ ((t >> 1) & 3)) << 4), ah);
                }
#pragma unroll
                for (int jp = 0; jp < NT8; jp += 2) {
                    const int ri = 16 * kk + 8 * (mi & 1) + mr, tc = 8 * jp + 8 * (mi >> 1);
                    uint32_t bfr[4];
                    wm::ldsm_x4_t(p_t + ri * 128 + (((tc >> 3) ^ (ri & 7)) << 4), bfr);
                    wm::mma16816(Dl[jp], ah, bfr[0], bfr[1]);
                    wm::mma16816(Dl[jp + 1], ah, bfr[2], bfr[3]);
                }
            }
#pragma unroll
            for (int j = 0; j < NT8; ++j) {
                D[j][0] += scale * Dl[j][0]; D[j][1] += scale * Dl[j][1];
                D[j][2] += scale * Dl[j][2]; D[j][3] += scale * Dl[j][3];
            }
        }

        // exchange with the other key half; E = (do^T diag(scale exp(G))) q[:, my keys] fills the wait
        unsigned char* xb = sm + L::X + (i & 1) * kRecWarps * L::kX;
        {
            float4* mine = reinterpret_cast<float4*>(xb + warp * L::kX) + lane;
#pragma unroll
            for (int j = 0; j < NT8; ++j) mine[32 * j] = make_float4(D[j][0], D[j][1], D[j][2], D[j][3]);
        }
        float E[NJH][4];
#pragma unroll
        for (int j = 0; j < NJH; ++j) E[j][0] = E[j][1] = E[j][2] = E[j][3] = 0.f;
        {
            const float* eg = sEG + s * C;
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk) {
                const float2 ea = *reinterpret_cast<const float2*>(eg + 16 * kk + 2 * q4);
                const float2 eb = *reinterpret_cast<const float2*>(eg + 16 * kk + 8 + 2 * q4);
                uint32_t a[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    // a bf16 pair to two floats (a bf16 is the top half of an fp32), scaled, repacked
                    const uint32_t x = da[kk][e];
                    const float2 f = e < 2 ? ea : eb;
                    a[e] = wm::pack2(__uint_as_float(x << 16) * f.x, __uint_as_float(x & 0xffff0000u) * f.y);
                }
#pragma unroll
                for (int jp = 0; jp < NJH; jp += 2) {
                    uint32_t bfr[4];
                    wm::ldsm_x4_t(q_t + kc_off(16 * kk + 8 * (mi & 1) + mr, d0 + 8 * jp + 8 * (mi >> 1)), bfr);
                    wm::mma16816(E[jp], a, bfr[0], bfr[1]);
                    wm::mma16816(E[jp + 1], a, bfr[2], bfr[3]);
                }
            }
        }
        bw::named_bar_sync(1 + vh, 64);
        if (i + 1 < NT) ready = bw::mbar_test_wait(&full[(i + 1) % L::NS], ((i + 1) / L::NS) & 1);
        {
            const float4* other = reinterpret_cast<const float4*>(xb + (warp ^ 2) * L::kX) + lane;
#pragma unroll
            for (int j = 0; j < NT8; ++j) {
                const float4 o = other[32 * j];
                D[j][0] += o.x; D[j][1] += o.y; D[j][2] += o.z; D[j][3] += o.w;
            }
        }

        // dh^T[:, my keys] = exp(G_L) dh^T + E - dv'^T w[:, my keys]
        {
            const float e = sDec[4 * s];
#pragma unroll
            for (int j = 0; j < NJH; ++j) {
                dhT[j][0] = e * dhT[j][0] + E[j][0]; dhT[j][1] = e * dhT[j][1] + E[j][1];
                dhT[j][2] = e * dhT[j][2] + E[j][2]; dhT[j][3] = e * dhT[j][3] + E[j][3];
            }
        }
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk) {
            const uint32_t a[4] = {wm::pack2(-D[2 * kk][0], -D[2 * kk][1]), wm::pack2(-D[2 * kk][2], -D[2 * kk][3]),
                                   wm::pack2(-D[2 * kk + 1][0], -D[2 * kk + 1][1]),
                                   wm::pack2(-D[2 * kk + 1][2], -D[2 * kk + 1][3])};
#pragma unroll
            for (int jp = 0; jp < NJH; jp += 2) {
                uint32_t bfr[4];
                wm::ldsm_x4_t(w_t + kc_off(16 * kk + 8 * (mi & 1) + mr, d0 + 8 * jp + 8 * (mi >> 1)), bfr);
                wm::mma16816(dhT[jp], a, bfr[0], bfr[1]);
                wm::mma16816(dhT[jp + 1], a, bfr[2], bfr[3]);
            }
        }
        __syncwarp();
        if (lane == 0) bw::mbar_arrive(&empty[s]);

        // dv': this key half stores tokens kh C/2 .. of dv'^T
        {
#pragma unroll
            for (int jp = 0; jp < NT8; jp += 2) {
                if ((jp >= NT8 / 2) != (kh == 1)) continue;
                const int jq = jp - kh * (NT8 / 2);
                const uint32_t r[4] = {wm::pack2(D[jp][0], D[jp][1]), wm::pack2(D[jp][2], D[jp][3]),
                                       wm::pack2(D[jp + 1][0], D[jp + 1][1]), wm::pack2(D[jp + 1][2], D[jp + 1][3])};
                wm::stsm_x4_t(st_v + stage_off(8 * jq + 8 * (mi >> 1) + mr, mi & 1), r);
            }
            __syncwarp();
            bf16* dst = dv_new + (((int64_t)b * T + t0 + kh * (C / 2)) * H + h) * V + v0 + vr0;
#pragma unroll
            for (int r32 = 0; r32 < C / 32; ++r32) {
                const int r = 16 * r32 + (lane >> 1), half = lane & 1;
                const uint4 x = wm::lds128(st_v + stage_off(r, half));
                if (t0 + kh * (C / 2) + r < T) *reinterpret_cast<uint4*>(dst + (int64_t)r * H * V + 8 * half) = x;
            }
            __syncwarp();
        }
    }
    if (dh0) {
#pragma unroll
        for (int j = 0; j < NJH; ++j) {
            const int d = d0 + 8 * j + 2 * q4;
            const int va = v0 + vr0 + g, vb = va + 8;
            dh0[(state + d) * V + va] = dhT[j][0];
            dh0[(state + d + 1) * V + va] = dhT[j][1];
            dh0[(state + d) * V + vb] = dhT[j][2];
            dh0[(state + d + 1) * V + vb] = dhT[j][3];
        }
    }
    (void)ok;
}

template <int K>
cudaError_t launch(const Dims& d, const void* q, const void* k, const void* w, const float* g_cum, const void* P,
                   const void* d_o, const float* dh_final, void* dh_ckpt, void* dv_new, float* dh0, cudaStream_t s,
                   unsigned int* err) {
    constexpr int C = 64;
    using L = RScanLayout<K, C>;
    CUtensorMap mk, mw, mq, mdo, mp;
    const uint64_t dims[4] = {(uint64_t)C, (uint64_t)C, (uint64_t)d.H, (uint64_t)d.B * d.NT};
    const uint64_t st[3] = {(uint64_t)C * 2, (uint64_t)C * C * 2, (uint64_t)d.H * C * C * 2};
    const uint32_t box[4] = {64, 64, 1, 1};
    if (!make_tmap_tokens(&mk, k, d.B, d.T, d.Hk, K, C) || !make_tmap_tokens(&mw, w, d.B, d.T, d.H, K, C) ||
        !make_tmap_tokens(&mq, q, d.B, d.T, d.Hk, K, C) || !make_tmap_tokens_sw64(&mdo, d_o, d.B, d.T, d.H, d.V, C) ||
        !make_tmap_bf16_4d(&mp, P, dims, st, box))
        return cudaErrorInvalidValue;
    auto kern = bwd_scan_mma_kernel<K, C>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(d.V / kBV, d.H, d.B);
    kern<<<grid, L::kThreads, smem, s>>>(mk, mw, mq, mdo, mp, g_cum, dh_final, (bf16*)dh_ckpt, (bf16*)dv_new, dh0,
                                         d.T, d.H, d.V, d.G, d.scale, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t mma_bwd_scan(const Dims& d, const void* q, const void* k, const void* w, const float* g_cum, const void* P,
                         const void* d_o, const float* dh_final, void* dh_ckpt, void* dv_new, float* dh0,
                         cudaStream_t s, unsigned int* err) {
    if (!d.bf16 || d.per_k || d.C != 64) return cudaErrorInvalidValue;
    return d.K == 64 ? launch<64>(d, q, k, w, g_cum, P, d_o, dh_final, dh_ckpt, dv_new, dh0, s, err)
                     : launch<128>(d, q, k, w, g_cum, P, d_o, dh_final, dh_ckpt, dv_new, dh0, s, err);
}

}  // namespace gdr
