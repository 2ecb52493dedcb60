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
//
// Without P (a per-key-dim gate, or 32-token chunks) the local term scale P^T do
// comes precomputed (dv_loc, bf16, from the tensor-core dv_local kernel), loaded
// by TMA like the forward scan's u and added by key half 0.  For a per-key-dim
// gate the factors cannot move onto do's columns: four producer warps build
// kg = k exp(G_L - G) and qg = scale q exp(G) per element, as the forward scan's
// producers build kg, and the decay exp(G_L) is a K-vector scaling dh's rows.
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

template <int K, int C, bool PER_K, bool FROM_P>
struct RScanLayout {
    static constexpr int NS = 2;
    static constexpr int KH = K / 2;
    static constexpr int NT8 = C / 8;
    static constexpr int GW = PER_K ? K : 1;
    static constexpr int kProdWarps = PER_K ? 4 : 1;
    static constexpr int kThreads = 32 * (kRecWarps + kProdWarps);
    static constexpr uint32_t kKC = C * K * 2;                     // [C][K] bf16, 128-byte swizzle
    static constexpr uint32_t kD = C * kBV * 2;                    // do or dv_loc [C][32] bf16, 64-byte swizzle
    static constexpr uint32_t kP = FROM_P ? C * C * 2 : 0;         // P [C][C] bf16, 128-byte swizzle
    static constexpr uint32_t kL = FROM_P ? 0 : kD;                // dv_loc slice
    static constexpr uint32_t kX = NT8 * 512;
    static constexpr uint32_t kSH = align1k(KH * 32);
    static constexpr uint32_t kSV = align1k(C / 2 * 32);
    static constexpr uint32_t KB = 0;                              // k (scalar gate, TMA) or kg (built)
    static constexpr uint32_t WB = KB + NS * kKC;
    static constexpr uint32_t QB = WB + NS * kKC;                  // q (scalar gate, TMA) or qg (built)
    static constexpr uint32_t DB = QB + NS * kKC;
    static constexpr uint32_t LB = DB + NS * kD;
    static constexpr uint32_t PB = align1k(LB + NS * kL);
    static constexpr uint32_t X = PB + NS * kP;
    static constexpr uint32_t SH = X + 2 * kRecWarps * kX;
    static constexpr uint32_t SV = SH + kRecWarps * kSH;
    static constexpr uint32_t GAM = SV + kRecWarps * kSV;          // gamma [NS][C] (scalar gate)
    static constexpr uint32_t EG = GAM + NS * C * 4;               // scale exp(G) [NS][C] (scalar gate)
    static constexpr uint32_t DEC = EG + NS * C * 4;               // exp(G_L) [NS][4] or [NS][K]
    static constexpr uint32_t bytes = DEC + NS * (PER_K ? K : 4) * 4;
    static constexpr uint32_t tx = (PER_K ? 1 : 3) * kKC + kD + (FROM_P ? kP : kL);
    static constexpr uint32_t full_count = 32 * kProdWarps + 1;
    static_assert(!FROM_P || (C == 64 && !PER_K), "P tiles: scalar gate, 64 x 64");
};

// co (packed variable-length sequences; NULL otherwise): one data row (B = 1) of whole-chunk runs,
// sequence z = blockIdx.z on the chunks co[z] .. co[z+1]-1, from dh_final[z] back to dh0[z].
template <int K, int C, bool PER_K, bool FROM_P>
__global__ void __launch_bounds__(RScanLayout<K, C, PER_K, FROM_P>::kThreads, 1)
bwd_scan_mma_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mw,
                    const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mdo,
                    const __grid_constant__ CUtensorMap mp, const __grid_constant__ CUtensorMap mdl,
                    const bf16* __restrict__ k_raw, const bf16* __restrict__ q_raw, const float* __restrict__ g_cum,
                    const float* __restrict__ dh_final, bf16* __restrict__ dh_ckpt, bf16* __restrict__ dv_new,
                    float* __restrict__ dh0, const int* __restrict__ co, int T, int H, int V, int G, float scale,
                    unsigned int* err) {
    using L = RScanLayout<K, C, PER_K, FROM_P>;
    constexpr int KH = L::KH, NT8 = L::NT8;
    constexpr int NJH = KH / 8;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[L::NS], empty[L::NS];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.x * kBV, h = blockIdx.y, b = blockIdx.z;
    const int NTall = (T + C - 1) / C;
    // this CTA's chunks: c0 .. c0 + NT - 1 of data row bd (clamped, so any co stays inside the tensors)
    const int c0 = co ? min(max(co[b], 0), NTall) : 0;
    const int NT = co ? min(max(co[b + 1], c0), NTall) - c0 : NTall;
    const int bd = co ? 0 : b;
    const uint32_t s_base = bw::smem_u32(sm);
    auto rowc = [&](int t) -> int64_t { return ((int64_t)bd * T + min(t, T - 1)) * H + h; };   // G past T: its last value

    if (tid == 0) {
        for (int s = 0; s < L::NS; ++s) {
            bw::mbar_init(&full[s], L::full_count);
            bw::mbar_init(&empty[s], kRecWarps);
        }
        bw::fence_mbar_init();
    }
    __syncthreads();

    if (warp >= kRecWarps) {
        float* sDec = reinterpret_cast<float*>(sm + L::DEC);
        if constexpr (!PER_K) {
            // ------------------------------------------------------------ producer (scalar gate)
            constexpr int GPL = C / 32;
            float* sGam = reinterpret_cast<float*>(sm + L::GAM);
            float* sEG = reinterpret_cast<float*>(sm + L::EG);
            for (int i = 0; i < NT; ++i) {
                const int c = NT - 1 - i, s = i % L::NS, t0 = (c0 + c) * C;
                float gv[GPL];
#pragma unroll
                for (int ii = 0; ii < GPL; ++ii) gv[ii] = g_cum[rowc(t0 + 32 * ii + lane)];
                const float gl = g_cum[rowc(t0 + C - 1)];
                if (!bw::mbar_wait(&empty[s], ((i / L::NS) & 1) ^ 1, err, kDeviceErrTimeout)) break;
                if (lane == 0) {
                    bw::mbar_arrive_expect_tx(&full[s], L::tx);
#pragma unroll
                    for (int a = 0; a < K / 64; ++a) {
                        bw::tma_load_4d(sm + L::KB + s * L::kKC + a * C * 128, &mk, &full[s], a * 64, h / G, t0, bd);
                        bw::tma_load_4d(sm + L::WB + s * L::kKC + a * C * 128, &mw, &full[s], a * 64, h, t0, bd);
                        bw::tma_load_4d(sm + L::QB + s * L::kKC + a * C * 128, &mq, &full[s], a * 64, h / G, t0, bd);
                    }
                    bw::tma_load_4d(sm + L::DB + s * L::kD, &mdo, &full[s], v0, h, t0, bd);
                    if constexpr (FROM_P) bw::tma_load_4d(sm + L::PB + s * L::kP, &mp, &full[s], 0, 0, h, bd * NTall + c0 + c);
                    else bw::tma_load_4d(sm + L::LB + s * L::kL, &mdl, &full[s], v0, h, t0, bd);
                    sDec[4 * s] = __expf(gl);
                }
#pragma unroll
                for (int ii = 0; ii < GPL; ++ii) {
                    sGam[s * C + 32 * ii + lane] = __expf(gl - gv[ii]);
                    sEG[s * C + 32 * ii + lane] = scale * __expf(gv[ii]);
                }
                bw::mbar_arrive(&full[s]);
            }
        } else {
            // ------------------------------------------------------------ producers (per-key-dim gate)
            // kg = k exp(G_L - G) and qg = scale q exp(G) from global loads one chunk ahead;
            // w, do and dv_loc by TMA
            constexpr int LC = K / 8, RSTEP = 128 / LC, NI = C / RSTEP;
            const int pt = tid - 32 * kRecWarps;
            const int lc = pt % LC, r0 = pt / LC;
            const int hk = h / G, Hk = H / G;
            uint4 kr[NI], qr[NI];
            float gr[NI][8], gl8[8];
            auto load = [&](int c) {
                const int t0 = (c0 + c) * C;
#pragma unroll
                for (int j = 0; j < NI; ++j) {
                    const int t = t0 + r0 + j * RSTEP;
                    const int64_t krow = ((int64_t)bd * T + t) * Hk + hk;
                    kr[j] = t < T ? *reinterpret_cast<const uint4*>(k_raw + krow * K + lc * 8) : make_uint4(0u, 0u, 0u, 0u);
                    qr[j] = t < T ? *reinterpret_cast<const uint4*>(q_raw + krow * K + lc * 8) : make_uint4(0u, 0u, 0u, 0u);
                    const float4* gt = reinterpret_cast<const float4*>(g_cum + rowc(t) * K + lc * 8);
                    *reinterpret_cast<float4*>(&gr[j][0]) = gt[0];
                    *reinterpret_cast<float4*>(&gr[j][4]) = gt[1];
                }
                const float4* g8 = reinterpret_cast<const float4*>(g_cum + rowc(t0 + C - 1) * K + lc * 8);
                *reinterpret_cast<float4*>(&gl8[0]) = g8[0];
                *reinterpret_cast<float4*>(&gl8[4]) = g8[1];
            };
            auto kc_o = [](int t, int d) -> uint32_t {
                return (d >> 6) * C * 128 + t * 128 + ((((d & 63) >> 3) ^ (t & 7)) << 4);
            };
            if (NT > 0) load(NT - 1);
            for (int i = 0; i < NT; ++i) {
                const int c = NT - 1 - i, s = i % L::NS, t0 = (c0 + c) * C;
                if (!bw::mbar_wait(&empty[s], ((i / L::NS) & 1) ^ 1, err, kDeviceErrTimeout)) break;
                if (pt == 0) {
                    bw::mbar_arrive_expect_tx(&full[s], L::tx);
#pragma unroll
                    for (int a = 0; a < K / 64; ++a)
                        bw::tma_load_4d(sm + L::WB + s * L::kKC + a * C * 128, &mw, &full[s], a * 64, h, t0, bd);
                    bw::tma_load_4d(sm + L::DB + s * L::kD, &mdo, &full[s], v0, h, t0, bd);
                    bw::tma_load_4d(sm + L::LB + s * L::kL, &mdl, &full[s], v0, h, t0, bd);
                }
                if (r0 == 0) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) sDec[s * K + lc * 8 + e] = __expf(gl8[e]);
                }
                unsigned char* kg_t = sm + L::KB + s * L::kKC;
                unsigned char* qg_t = sm + L::QB + s * L::kKC;
#pragma unroll
                for (int j = 0; j < NI; ++j) {
                    const int t = r0 + j * RSTEP;
                    const bf16* kv = reinterpret_cast<const bf16*>(&kr[j]);
                    const bf16* qv = reinterpret_cast<const bf16*>(&qr[j]);
                    float fk[8], fq[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        fk[e] = __bfloat162float(kv[e]) * __expf(gl8[e] - gr[j][e]);
                        fq[e] = scale * __bfloat162float(qv[e]) * __expf(gr[j][e]);
                    }
                    uint4 pk, pq;
                    pk.x = bw::pack_bf16(fk[0], fk[1]); pk.y = bw::pack_bf16(fk[2], fk[3]);
                    pk.z = bw::pack_bf16(fk[4], fk[5]); pk.w = bw::pack_bf16(fk[6], fk[7]);
                    pq.x = bw::pack_bf16(fq[0], fq[1]); pq.y = bw::pack_bf16(fq[2], fq[3]);
                    pq.z = bw::pack_bf16(fq[4], fq[5]); pq.w = bw::pack_bf16(fq[6], fq[7]);
                    *reinterpret_cast<uint4*>(kg_t + kc_o(t, lc * 8)) = pk;
                    *reinterpret_cast<uint4*>(qg_t + kc_o(t, lc * 8)) = pq;
                }
                bw::fence_async_shared();
                bw::mbar_arrive(&full[s]);
                if (i + 1 < NT) load(c - 1);
            }
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
        const int c = NT - 1 - i, s = i % L::NS, t0 = (c0 + c) * C;
        if (!ready) ok = ok && bw::mbar_wait(&full[s], (i / L::NS) & 1, err, kDeviceErrTimeout);
        const uint32_t k_t = s_base + L::KB + s * L::kKC;
        const uint32_t w_t = s_base + L::WB + s * L::kKC;
        const uint32_t q_t = s_base + L::QB + s * L::kKC;
        const uint32_t do_t = s_base + L::DB + s * L::kD;
        const uint32_t p_t = s_base + L::PB + s * L::kP;
        const uint32_t l_t = s_base + L::LB + s * L::kL;

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
            bf16* dst = dh_ckpt + ((((int64_t)bd * NTall + c0 + c) * H + h) * K + d0) * V + v0 + vr0;
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
        // D *= gamma (columns; the per-key-dim gate has it in kg already)
        if constexpr (!PER_K) {
            const float* gam = sGam + s * C;
#pragma unroll
            for (int j = 0; j < NT8; ++j) {
                const float2 gg = *reinterpret_cast<const float2*>(gam + 8 * j + 2 * q4);
                D[j][0] *= gg.x; D[j][1] *= gg.y; D[j][2] *= gg.x; D[j][3] *= gg.y;
            }
        }
        if constexpr (!FROM_P) {
            // + dv_loc^T, by key half 0 (the exchange adds the halves), read in D's layout
            if (kh == 0) {
#pragma unroll
                for (int jp = 0; jp < NT8; jp += 2) {
                    const int t = 8 * jp + 8 * (mi >> 1) + mr;
                    const int ch = (vr0 >> 3) + (mi & 1);
                    uint32_t lr[4];
                    wm::ldsm_x4_t(l_t + t * 64 + ((ch ^ ((t >> 1) & 3)) << 4), lr);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float* dd = D[jp + (e >> 1)] + 2 * (e & 1);
                        dd[0] += __uint_as_float(lr[e] << 16);
                        dd[1] += __uint_as_float(lr[e] & 0xffff0000u);
                    }
                }
            }
        } else {
            // + scale do^T P over my half of the query tokens i
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
                uint32_t a[4];
                if constexpr (PER_K) {
                    // qg carries scale exp(G) per element: do^T as loaded
#pragma unroll
                    for (int e = 0; e < 4; ++e) a[e] = da[kk][e];
                } else {
                    const float2 ea = *reinterpret_cast<const float2*>(eg + 16 * kk + 2 * q4);
                    const float2 eb = *reinterpret_cast<const float2*>(eg + 16 * kk + 8 + 2 * q4);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        // a bf16 pair to two floats (a bf16 is the top half of an fp32), scaled, repacked
                        const uint32_t x = da[kk][e];
                        const float2 f = e < 2 ? ea : eb;
                        a[e] = wm::pack2(__uint_as_float(x << 16) * f.x, __uint_as_float(x & 0xffff0000u) * f.y);
                    }
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
        if constexpr (PER_K) {
            const float* dec = sDec + s * K + d0;
#pragma unroll
            for (int j = 0; j < NJH; ++j) {
                const float2 e = *reinterpret_cast<const float2*>(dec + 8 * j + 2 * q4);
                dhT[j][0] = e.x * dhT[j][0] + E[j][0]; dhT[j][1] = e.y * dhT[j][1] + E[j][1];
                dhT[j][2] = e.x * dhT[j][2] + E[j][2]; dhT[j][3] = e.y * dhT[j][3] + E[j][3];
            }
        } else {
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
            bf16* dst = dv_new + (((int64_t)bd * T + t0 + kh * (C / 2)) * H + h) * V + v0 + vr0;
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

// P [B, NT, H, C, C] (FROM_P) or dv_loc [B, T, H, V] bf16 (otherwise) supplies the local term
template <int K, int C, bool PER_K, bool FROM_P>
cudaError_t launch(const Dims& d, const void* q, const void* k, const void* w, const float* g_cum, const void* P,
                   const void* dv_loc, const void* d_o, const float* dh_final, void* dh_ckpt, void* dv_new,
                   float* dh0, const int* co, int nseq, cudaStream_t s, unsigned int* err) {
    using L = RScanLayout<K, C, PER_K, FROM_P>;
    CUtensorMap mk, mw, mq, mdo, mp, mdl;
    if (!make_tmap_tokens(&mk, k, d.B, d.T, d.Hk, K, C) || !make_tmap_tokens(&mw, w, d.B, d.T, d.H, K, C) ||
        !make_tmap_tokens(&mq, q, d.B, d.T, d.Hk, K, C) || !make_tmap_tokens_sw64(&mdo, d_o, d.B, d.T, d.H, d.V, C))
        return cudaErrorInvalidValue;
    if constexpr (FROM_P) {
        const uint64_t dims[4] = {(uint64_t)C, (uint64_t)C, (uint64_t)d.H, (uint64_t)d.B * d.NT};
        const uint64_t st[3] = {(uint64_t)C * 2, (uint64_t)C * C * 2, (uint64_t)d.H * C * C * 2};
        const uint32_t box[4] = {64, 64, 1, 1};
        if (!make_tmap_bf16_4d(&mp, P, dims, st, box)) return cudaErrorInvalidValue;
        mdl = mdo;
    } else {
        if (!make_tmap_tokens_sw64(&mdl, dv_loc, d.B, d.T, d.H, d.V, C)) return cudaErrorInvalidValue;
        mp = mw;
    }
    auto kern = bwd_scan_mma_kernel<K, C, PER_K, FROM_P>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(d.V / kBV, d.H, co ? nseq : d.B);
    kern<<<grid, L::kThreads, smem, s>>>(mk, mw, mq, mdo, mp, mdl, (const bf16*)k, (const bf16*)q, g_cum, dh_final,
                                         (bf16*)dh_ckpt, (bf16*)dv_new, dh0, co, d.T, d.H, d.V, d.G, d.scale, err);
    return cudaGetLastError();
}

template <int K, int C>
cudaError_t from_dvloc(const Dims& d, const void* q, const void* k, const void* w, const float* g_cum,
                       const void* dv_loc, const void* d_o, const float* dh_final, void* dh_ckpt, void* dv_new,
                       float* dh0, const int* co, int nseq, cudaStream_t s, unsigned int* err) {
    return d.per_k ? launch<K, C, true, false>(d, q, k, w, g_cum, nullptr, dv_loc, d_o, dh_final, dh_ckpt, dv_new,
                                               dh0, co, nseq, s, err)
                   : launch<K, C, false, false>(d, q, k, w, g_cum, nullptr, dv_loc, d_o, dh_final, dh_ckpt, dv_new,
                                                dh0, co, nseq, s, err);
}

}  // namespace

cudaError_t mma_bwd_scan(const Dims& d, const void* q, const void* k, const void* w, const float* g_cum, const void* P,
                         const void* d_o, const float* dh_final, void* dh_ckpt, void* dv_new, float* dh0,
                         cudaStream_t s, unsigned int* err, const int* co, int nseq) {
    if (!d.bf16 || d.per_k || d.C != 64 || (co && (d.B != 1 || nseq < 1))) return cudaErrorInvalidValue;
    return d.K == 64 ? launch<64, 64, false, true>(d, q, k, w, g_cum, P, nullptr, d_o, dh_final, dh_ckpt, dv_new, dh0,
                                                   co, nseq, s, err)
                     : launch<128, 64, false, true>(d, q, k, w, g_cum, P, nullptr, d_o, dh_final, dh_ckpt, dv_new, dh0,
                                                    co, nseq, s, err);
}

cudaError_t mma_bwd_scan_dl(const Dims& d, const void* q, const void* k, const void* w, const float* g_cum,
                            const void* dv_loc, const void* d_o, const float* dh_final, void* dh_ckpt, void* dv_new,
                            float* dh0, cudaStream_t s, unsigned int* err, const int* co, int nseq) {
    if (!d.bf16 || (co && (d.B != 1 || nseq < 1))) return cudaErrorInvalidValue;
    if (d.K == 64)
        return d.C == 32 ? from_dvloc<64, 32>(d, q, k, w, g_cum, dv_loc, d_o, dh_final, dh_ckpt, dv_new, dh0, co, nseq, s, err)
                         : from_dvloc<64, 64>(d, q, k, w, g_cum, dv_loc, d_o, dh_final, dh_ckpt, dv_new, dh0, co, nseq, s, err);
    return d.C == 32 ? from_dvloc<128, 32>(d, q, k, w, g_cum, dv_loc, d_o, dh_final, dh_ckpt, dv_new, dh0, co, nseq, s, err)
                     : from_dvloc<128, 64>(d, q, k, w, g_cum, dv_loc, d_o, dh_final, dh_ckpt, dv_new, dh0, co, nseq, s, err);
}

}  // namespace gdr
