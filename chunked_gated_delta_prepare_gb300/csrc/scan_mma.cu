// State scan for bf16 and fp16 io with the recurrence in registers (the re-scan of
// "kernel_fun/kda/_kernels/bwd_scan.py", module docstring: hck[c] = h before the
// update, v' = u - w h, h = exp(decay) h + kg^T v').
//
// One CTA per (batch, head, 32 value columns); serial over chunks.  Four
// recurrence warps, one per SM sub-partition, split h^T (32 x K) into quarters:
// warp (vh, kh) owns value columns 16vh..16vh+15 and key rows kh K/2 .. of it as
// fp32 mma.sync accumulator fragments for the whole sequence.  Per chunk:
//
//   D_kh  = h^T[:, keys kh] w[:, keys kh]^T     [16 x C]  A = bf16(h^T) from the accumulator
//   D     = D_0 + D_1                           the two key halves swap partial sums through
//                                               shared memory behind a 64-thread named barrier
//   v'^T  = u^T - D                             u^T by ldmatrix.trans
//   h^T[:, keys kh] = exp(G_last) h^T + (v'^T diag(gamma)) k[:, keys kh]      (scalar gate)
//                   = exp(G_last) h^T + v'^T kg[:, keys kh]                    (per-key-dim gate)
//
// with gamma_t = exp(G_last - G_t).  For the scalar gate the factor moves from
// k's rows onto v''s columns (kg^T v' = k^T diag(gamma) v'), so k feeds the MMA
// exactly as TMA loads it and one producer warp (TMA issue plus a C-float gamma
// row) feeds a 3-stage ring.  The per-key-dim gate cannot be moved that way;
// there four producer warps build kg = k exp(G_last - G) from global loads
// issued two chunks ahead.  v_new and the bf16 checkpoints are transposed by
// stmatrix.trans into a per-warp staging tile and leave as 16-byte global
// stores (a TMA store costs the issuing warp ~300 cycles of fence, bulk-group
// wait and issue, too much on this chain); the u tile is 64-byte swizzled, w
// and k 128-byte swizzled, the staging XOR-swizzled, so every ldmatrix and
// stmatrix is free of bank conflicts.  The ring's full barrier for chunk c+1 is
// tested (non-blocking) in the middle of chunk c, so its latency stays off the chain.
// With fp16 io (F16) every operand, checkpoint and v' is fp16 in the same places; the
// state stays fp32.
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
constexpr int kRecWarps = 4;   // (value half, key half)

constexpr uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }

// TRANSFER (the segment maps) writes no checkpoint and no v', so it needs no staging.  At K = 128,
// C = 64 it also runs a 2-stage ring: 106 KB instead of 157 KB, so two CTAs share an SM (scalar
// gate; measured 0.088 ms against 0.107 ms for 256 CTAs, though 10% slower per chunk at one CTA
// per SM).  The smaller tiles fit two CTAs with three stages.
template <int K, int C, bool PER_K, bool TRANSFER = false>
struct MScanLayout {
    static constexpr int NS = TRANSFER && K == 128 && C == 64 ? 2 : 3;   // ring stages
    static constexpr int KH = K / 2;                               // keys per recurrence warp
    static constexpr int NT8 = C / 8;
    static constexpr int GW = PER_K ? K : 1;
    static constexpr int kProdWarps = PER_K ? 4 : 1;
    static constexpr int kThreads = 32 * (kRecWarps + kProdWarps);
    static constexpr uint32_t kKC = C * K * 2;                     // [C][K] bf16, 128-byte swizzle
    static constexpr uint32_t kU = C * kBV * 2;                    // [C][32] bf16, 64-byte swizzle
    static constexpr uint32_t kX = NT8 * 512;                      // one warp's partial D, float4 per (n-tile, lane)
    static constexpr uint32_t kSH = align1k(KH * 32);              // checkpoint staging [KH][16]
    static constexpr uint32_t kSV = align1k(C / 2 * 32);           // v_new staging [C/2][16]
    static constexpr uint32_t W = 0;
    static constexpr uint32_t KB = W + NS * kKC;                   // k (scalar gate) or kg (per-key-dim gate)
    static constexpr uint32_t U = KB + NS * kKC;
    static constexpr uint32_t X = U + NS * kU;
    static constexpr uint32_t SH = X + 2 * kRecWarps * kX;
    static constexpr uint32_t SV = SH + (TRANSFER ? 0 : kRecWarps * kSH);
    static constexpr uint32_t GAM = SV + (TRANSFER ? 0 : kRecWarps * kSV);   // gamma rows [NS][C] (scalar gate)
    static constexpr uint32_t DEC = GAM + NS * C * 4;              // exp(G_last) [NS][GW]
    static constexpr uint32_t bytes = DEC + NS * GW * 4;
    static constexpr uint32_t tx = (PER_K ? 1 : 2) * kKC + kU;
    static constexpr uint32_t full_count = 32 * kProdWarps + 1;
};

// GENERAL: a partial last chunk or grouped value heads.  Whole chunks of ungrouped heads take
// the variant without those guards (the per-key-dim producers' guarded loads measured 60%
// slower on whole chunks).
// TRANSFER: the affine map of every segment of the segment-parallel scan, h_end = M h_start + Z.
// The columns of h evolve independently, so the grid gets K/32 more column slices: slices below
// V/32 run u's columns from a zero state (their final state is Z, written to h_final), the others
// run the columns of the identity with u = 0 (their final state is M, written to m_out [.., K, K]).
// No checkpoint and no v' is written.
// co (packed variable-length sequences; NULL otherwise): the tensors hold one row (B = 1) of whole-chunk
// runs, sequence z on the chunks co[z] .. co[z+1]-1; blockIdx.z is the sequence, whose state starts from
// h0[z] and ends in h_final[z].  Checkpoints and v' land at the chunks' places in the row.
template <int K, int C, bool PER_K, bool GENERAL, bool TRANSFER, bool F16>
__global__ void __launch_bounds__(MScanLayout<K, C, PER_K, TRANSFER>::kThreads, TRANSFER && !PER_K ? 2 : 1)
scan_mma_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mk,
                const __grid_constant__ CUtensorMap mu, const bf16* __restrict__ k, const float* __restrict__ g_cum,
                const float* __restrict__ h0, bf16* __restrict__ h_ckpt, bf16* __restrict__ v_new,
                float* __restrict__ h_final, float* __restrict__ m_out, const int* __restrict__ co, int T, int H,
                int V, int G, unsigned int* err) {
    using L = MScanLayout<K, C, PER_K, TRANSFER>;
    constexpr int GW = L::GW, KH = L::KH, NT8 = L::NT8;
    constexpr int NJH = KH / 8;    // n-tiles of this warp's part of h^T
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[L::NS], empty[L::NS];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool mcols = TRANSFER && (int)blockIdx.x >= V / kBV;   // a slice of the identity's columns
    const int v0 = (mcols ? (int)blockIdx.x - V / kBV : (int)blockIdx.x) * kBV, h = blockIdx.y, b = blockIdx.z;
    const uint32_t tx = mcols ? L::tx - L::kU : L::tx;           // u = 0 there: no u tile
    const int NTall = GENERAL ? (T + C - 1) / C : T / C;   // a last, partial chunk runs as zero tokens past T
    // this CTA's chunks: c0 .. c0 + NT - 1 of data row bd (clamped, so any co stays inside the tensors)
    const int c0 = co ? min(max(co[b], 0), NTall) : 0;
    const int NT = co ? min(max(co[b + 1], c0), NTall) - c0 : NTall;
    const int bd = co ? 0 : b;
    const uint32_t s_base = bw::smem_u32(sm);
    auto row = [&](int t) -> int64_t { return ((int64_t)bd * T + t) * H + h; };
    auto rowc = [&](int t) -> int64_t { return row(GENERAL ? min(t, T - 1) : t); };   // G past T: its last value
    auto krow = [&](int t) -> int64_t {                                                 // k: q/k head h / G
        return GENERAL ? ((int64_t)bd * T + t) * (H / G) + h / G : row(t);
    };
    const int hk = GENERAL ? h / G : h;

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
        float* sDec = reinterpret_cast<float*>(sm + L::DEC);
        if constexpr (!PER_K) {
            // one warp: TMA w, k, u; gamma_t = exp(G_last - G_t) and exp(G_last) from G
            float* sGam = reinterpret_cast<float*>(sm + L::GAM);
            constexpr int GPL = C / 32;                // G values per lane
            float gn[GPL], gln;                        // next chunk's G, loaded a chunk ahead
            auto load_g = [&](int c) {
#pragma unroll
                for (int i = 0; i < GPL; ++i) gn[i] = g_cum[rowc((c0 + c) * C + lane + 32 * i)];
                gln = g_cum[rowc((c0 + c) * C + C - 1)];
            };
            if (NT > 0) load_g(0);
            for (int c = 0; c < NT; ++c) {
                const int s = c % L::NS;
                float gc[GPL], glc = gln;
#pragma unroll
                for (int i = 0; i < GPL; ++i) gc[i] = gn[i];
                if (c + 1 < NT) load_g(c + 1);
                if (!bw::mbar_wait(&empty[s], ((c / L::NS) & 1) ^ 1, err, kDeviceErrTimeout)) break;
                const int t0 = (c0 + c) * C;
                if (lane == 0) {
                    bw::mbar_arrive_expect_tx(&full[s], tx);
#pragma unroll
                    for (int a = 0; a < K / 64; ++a) {
                        bw::tma_load_4d(sm + L::W + s * L::kKC + a * C * 128, &mw, &full[s], a * 64, h, t0, bd);
                        bw::tma_load_4d(sm + L::KB + s * L::kKC + a * C * 128, &mk, &full[s], a * 64, hk, t0, bd);
                    }
                    if (!mcols) bw::tma_load_4d(sm + L::U + s * L::kU, &mu, &full[s], v0, h, t0, bd);
                    sDec[s] = __expf(glc);
                }
#pragma unroll
                for (int i = 0; i < GPL; ++i) sGam[s * C + lane + 32 * i] = __expf(glc - gc[i]);
                bw::mbar_arrive(&full[s]);
            }
        } else {
            // four warps: TMA w, u; kg = k exp(G_last - G) built from global loads two chunks ahead
            constexpr int kProdThreads = 32 * L::kProdWarps;
            constexpr int LC = K / 8;
            constexpr int RSTEP = kProdThreads / LC;
            constexpr int NI = C / RSTEP;
            const int lc = pt % LC, r0 = pt / LC;
            struct Staged {
                uint4 kr[NI];
                float gr[NI][8], gl8[8];
            };
            Staged sa, sb;
            auto load_chunk = [&](int c, Staged& st) {
                const int t0 = (c0 + c) * C;
#pragma unroll
                for (int j = 0; j < NI; ++j) {
                    const int t = r0 + j * RSTEP;
                    st.kr[j] = !GENERAL || t0 + t < T ? *reinterpret_cast<const uint4*>(k + krow(t0 + t) * K + lc * 8)
                                          : make_uint4(0u, 0u, 0u, 0u);
                    const float4* gt = reinterpret_cast<const float4*>(g_cum + rowc(t0 + t) * K + lc * 8);
                    *reinterpret_cast<float4*>(&st.gr[j][0]) = gt[0];
                    *reinterpret_cast<float4*>(&st.gr[j][4]) = gt[1];
                }
                const float4* g8 = reinterpret_cast<const float4*>(g_cum + rowc(t0 + C - 1) * K + lc * 8);
                *reinterpret_cast<float4*>(&st.gl8[0]) = g8[0];
                *reinterpret_cast<float4*>(&st.gl8[4]) = g8[1];
            };
            auto produce = [&](int c, const Staged& st) -> bool {
                const int s = c % L::NS;
                if (!bw::mbar_wait(&empty[s], ((c / L::NS) & 1) ^ 1, err, kDeviceErrTimeout)) return false;
                const int t0 = (c0 + c) * C;
                if (pt == 0) {
                    bw::mbar_arrive_expect_tx(&full[s], tx);
#pragma unroll
                    for (int a = 0; a < K / 64; ++a)
                        bw::tma_load_4d(sm + L::W + s * L::kKC + a * C * 128, &mw, &full[s], a * 64, h, t0, bd);
                    if (!mcols) bw::tma_load_4d(sm + L::U + s * L::kU, &mu, &full[s], v0, h, t0, bd);
                }
                if (r0 == 0) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) sDec[s * GW + lc * 8 + e] = __expf(st.gl8[e]);
                }
                unsigned char* kg_t = sm + L::KB + s * L::kKC;
#pragma unroll
                for (int j = 0; j < NI; ++j) {
                    const int t = r0 + j * RSTEP;
                    float f[8];
                    bw::unpack8_io<F16>(st.kr[j], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] *= __expf(st.gl8[e] - st.gr[j][e]);
                    *reinterpret_cast<uint4*>(kg_t + (lc >> 3) * C * 128 + t * 128 + (((lc & 7) ^ (t & 7)) << 4)) =
                        bw::pack8_io<F16>(f);
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
        }
        return;
    }

    // -------------------------------------------------------------------- recurrence warps
    const int g = lane >> 2, q4 = lane & 3;
    const int vh = warp & 1, kh = warp >> 1;
    const int vr0 = vh * 16;                           // this warp's columns within the CTA's 32
    const int d0 = kh * KH;                            // this warp's first key row
    const int mi = lane >> 3, mr = lane & 7;           // ldmatrix/stmatrix: matrix and row this lane addresses
    const int64_t state = ((int64_t)b * H + h) * K;
    const float* sGam = reinterpret_cast<const float*>(sm + L::GAM);
    const float* sDec = reinterpret_cast<const float*>(sm + L::DEC);
    float hT[NJH][4];                                  // h^T[v][d]: (g | g+8, d0 + 8j + 2q4 | +1)
#pragma unroll
    for (int j = 0; j < NJH; ++j) {
        const int d = d0 + 8 * j + 2 * q4;
        const int va = v0 + vr0 + g, vb = va + 8;
        if (TRANSFER) {   // Z from a zero state; M from the identity (column va of I has its 1 in row va)
            hT[j][0] = mcols && d == va ? 1.f : 0.f;
            hT[j][1] = mcols && d + 1 == va ? 1.f : 0.f;
            hT[j][2] = mcols && d == vb ? 1.f : 0.f;
            hT[j][3] = mcols && d + 1 == vb ? 1.f : 0.f;
        } else if (h0) {
            hT[j][0] = h0[(state + d) * V + va];
            hT[j][1] = h0[(state + d + 1) * V + va];
            hT[j][2] = h0[(state + d) * V + vb];
            hT[j][3] = h0[(state + d + 1) * V + vb];
        } else {
            hT[j][0] = hT[j][1] = hT[j][2] = hT[j][3] = 0.f;
        }
    }
    // staging rows: 16 bf16 columns (32 bytes), 16-byte halves swapped on every other group of four rows
    auto stage_off = [](int r, int half) -> uint32_t { return r * 32 + ((half ^ ((r >> 2) & 1)) << 4); };
    const uint32_t st_h = s_base + L::SH + warp * L::kSH;
    const uint32_t st_v = s_base + L::SV + warp * L::kSV;
    bool ok = true;
    bool ready = NT > 0 && bw::mbar_test_wait(&full[0], 0);
    for (int c = 0; c < NT; ++c) {
        const int s = c % L::NS;
        const int t0 = (c0 + c) * C;
        if (!ready) ok = ok && bw::mbar_wait(&full[s], (c / L::NS) & 1, err, kDeviceErrTimeout);
        const uint32_t w_t = s_base + L::W + s * L::kKC;
        const uint32_t k_t = s_base + L::KB + s * L::kKC;
        const uint32_t u_t = s_base + L::U + s * L::kU;

        // partial D = h^T[:, my keys] w[:, my keys]^T  [16 x C]
        float D[NT8][4];
#pragma unroll
        for (int j = 0; j < NT8; ++j) D[j][0] = D[j][1] = D[j][2] = D[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KH / 16; ++kk) {
            const uint32_t a[4] = {wm::pack2_io<F16>(hT[2 * kk][0], hT[2 * kk][1]),
                                   wm::pack2_io<F16>(hT[2 * kk][2], hT[2 * kk][3]),
                                   wm::pack2_io<F16>(hT[2 * kk + 1][0], hT[2 * kk + 1][1]),
                                   wm::pack2_io<F16>(hT[2 * kk + 1][2], hT[2 * kk + 1][3])};
#pragma unroll
            for (int jp = 0; jp < NT8; jp += 2) {
                const int t = 8 * jp + 8 * (mi >> 1) + mr, d = d0 + 16 * kk + 8 * (mi & 1);
                uint32_t bfr[4];
                wm::ldsm_x4(w_t + (d >> 6) * C * 128 + t * 128 + ((((d & 63) >> 3) ^ (t & 7)) << 4), bfr);
                wm::mma16816_io<F16>(D[jp], a, bfr[0], bfr[1]);
                wm::mma16816_io<F16>(D[jp + 1], a, bfr[2], bfr[3]);
            }
        }

        // checkpoint c (h before this chunk), my [KH x 16] quarter: stmatrix.trans -> staging -> global
        if (h_ckpt) {
#pragma unroll
            for (int j = 0; j < NJH; j += 2) {
                const uint32_t r[4] = {wm::pack2_io<F16>(hT[j][0], hT[j][1]), wm::pack2_io<F16>(hT[j][2], hT[j][3]),
                                       wm::pack2_io<F16>(hT[j + 1][0], hT[j + 1][1]),
                                       wm::pack2_io<F16>(hT[j + 1][2], hT[j + 1][3])};
                wm::stsm_x4_t(st_h + stage_off(8 * j + 8 * (mi >> 1) + mr, mi & 1), r);
            }
            __syncwarp();
            bf16* dst = h_ckpt + ((((int64_t)bd * NTall + c0 + c) * H + h) * K + d0) * V + v0 + vr0;
#pragma unroll
            for (int i = 0; i < KH / 16; ++i) {
                const int r = 16 * i + (lane >> 1), half = lane & 1;
                const uint4 x = wm::lds128(st_h + stage_off(r, half));
                *reinterpret_cast<uint4*>(dst + (int64_t)r * V + 8 * half) = x;
            }
        }

        // u^T fragments (D's layout) ahead of the exchange
        uint32_t ur[NT8 / 2][4];
        if (mcols) {
#pragma unroll
            for (int jp = 0; jp < NT8; jp += 2) ur[jp / 2][0] = ur[jp / 2][1] = ur[jp / 2][2] = ur[jp / 2][3] = 0u;
        } else {
#pragma unroll
            for (int jp = 0; jp < NT8; jp += 2) {
                const int t = 8 * jp + 8 * (mi >> 1) + mr;
                const int ch = (vr0 >> 3) + (mi & 1);
                wm::ldsm_x4_t(u_t + t * 64 + ((ch ^ ((t >> 1) & 3)) << 4), ur[jp / 2]);
            }
        }

        // D = D_0 + D_1: swap partial sums with the other key half of the same value columns
        {
            unsigned char* xb = sm + L::X + (c & 1) * kRecWarps * L::kX;
            float4* mine = reinterpret_cast<float4*>(xb + warp * L::kX) + lane;
            const float4* other = reinterpret_cast<const float4*>(xb + (warp ^ 2) * L::kX) + lane;
#pragma unroll
            for (int j = 0; j < NT8; ++j) mine[32 * j] = make_float4(D[j][0], D[j][1], D[j][2], D[j][3]);
            bw::named_bar_sync(1 + vh, 64);
            if (c + 1 < NT) ready = bw::mbar_test_wait(&full[(c + 1) % L::NS], ((c + 1) / L::NS) & 1);
#pragma unroll
            for (int j = 0; j < NT8; ++j) {
                const float4 o = other[32 * j];
                D[j][0] += o.x; D[j][1] += o.y; D[j][2] += o.z; D[j][3] += o.w;
            }
        }
        // v'^T = u^T - D
#pragma unroll
        for (int jp = 0; jp < NT8; jp += 2) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 uv = bw::unpack2_io<F16>(ur[jp / 2][e]);
                float* dd = D[jp + (e >> 1)] + 2 * (e & 1);
                dd[0] = uv.x - dd[0];
                dd[1] = uv.y - dd[1];
            }
        }

        // h^T[:, my keys] = exp(G_last) h^T + (v'^T diag(gamma)) k   |   + v'^T kg
        if constexpr (PER_K) {
            const float* dec = sDec + s * GW + d0;
#pragma unroll
            for (int j = 0; j < NJH; ++j) {
                const float2 e = *reinterpret_cast<const float2*>(dec + 8 * j + 2 * q4);
                hT[j][0] *= e.x; hT[j][1] *= e.y; hT[j][2] *= e.x; hT[j][3] *= e.y;
            }
        } else {
            const float e = sDec[s];
#pragma unroll
            for (int j = 0; j < NJH; ++j) { hT[j][0] *= e; hT[j][1] *= e; hT[j][2] *= e; hT[j][3] *= e; }
        }
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk) {
            float x0 = 1.f, x1 = 1.f, y0 = 1.f, y1 = 1.f;
            if constexpr (!PER_K) {
                const float2 ga = *reinterpret_cast<const float2*>(sGam + s * C + 16 * kk + 2 * q4);
                const float2 gb = *reinterpret_cast<const float2*>(sGam + s * C + 16 * kk + 8 + 2 * q4);
                x0 = ga.x; x1 = ga.y; y0 = gb.x; y1 = gb.y;
            }
            const uint32_t a[4] = {wm::pack2_io<F16>(D[2 * kk][0] * x0, D[2 * kk][1] * x1),
                                   wm::pack2_io<F16>(D[2 * kk][2] * x0, D[2 * kk][3] * x1),
                                   wm::pack2_io<F16>(D[2 * kk + 1][0] * y0, D[2 * kk + 1][1] * y1),
                                   wm::pack2_io<F16>(D[2 * kk + 1][2] * y0, D[2 * kk + 1][3] * y1)};
#pragma unroll
            for (int jp = 0; jp < NJH; jp += 2) {
                const int t = 16 * kk + 8 * (mi & 1) + mr, d = d0 + 8 * jp + 8 * (mi >> 1);
                uint32_t bfr[4];
                wm::ldsm_x4_t(k_t + (d >> 6) * C * 128 + t * 128 + ((((d & 63) >> 3) ^ (t & 7)) << 4), bfr);
                wm::mma16816_io<F16>(hT[jp], a, bfr[0], bfr[1]);
                wm::mma16816_io<F16>(hT[jp + 1], a, bfr[2], bfr[3]);
            }
        }
        __syncwarp();
        if (lane == 0) bw::mbar_arrive(&empty[s]);

        // v_new: this key half stores tokens kh C/2 .. of v'^T; stmatrix.trans -> staging -> global
        if constexpr (!TRANSFER) {
#pragma unroll
            for (int jp = 0; jp < NT8; jp += 2) {
                if ((jp >= NT8 / 2) != (kh == 1)) continue;   // static register indices, runtime half
                const int jq = jp - kh * (NT8 / 2);
                const uint32_t r[4] = {wm::pack2_io<F16>(D[jp][0], D[jp][1]), wm::pack2_io<F16>(D[jp][2], D[jp][3]),
                                       wm::pack2_io<F16>(D[jp + 1][0], D[jp + 1][1]),
                                       wm::pack2_io<F16>(D[jp + 1][2], D[jp + 1][3])};
                wm::stsm_x4_t(st_v + stage_off(8 * jq + 8 * (mi >> 1) + mr, mi & 1), r);
            }
            __syncwarp();
            bf16* dst = v_new + (((int64_t)bd * T + t0 + kh * (C / 2)) * H + h) * V + v0 + vr0;
#pragma unroll
            for (int i = 0; i < C / 32; ++i) {
                const int r = 16 * i + (lane >> 1), half = lane & 1;
                const uint4 x = wm::lds128(st_v + stage_off(r, half));
                if (!GENERAL || t0 + kh * (C / 2) + r < T)
                    *reinterpret_cast<uint4*>(dst + (int64_t)r * H * V + 8 * half) = x;
            }
            __syncwarp();
        }
    }
    if (h_final) {
        float* out = mcols ? m_out : h_final;
        const int ld = mcols ? K : V;
#pragma unroll
        for (int j = 0; j < NJH; ++j) {
            const int d = d0 + 8 * j + 2 * q4;
            const int va = v0 + vr0 + g, vb = va + 8;
            out[(state + d) * ld + va] = hT[j][0];
            out[(state + d + 1) * ld + va] = hT[j][1];
            out[(state + d) * ld + vb] = hT[j][2];
            out[(state + d + 1) * ld + vb] = hT[j][3];
        }
    }
    (void)ok;
}

template <int K, int C, bool PER_K, bool GENERAL, bool TRANSFER, bool F16>
cudaError_t launch_v(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum, const float* h0,
                     void* h_ckpt, void* v_new, float* h_final, float* m_out, const int* co, int nseq, cudaStream_t s,
                     unsigned int* err) {
    using L = MScanLayout<K, C, PER_K, TRANSFER>;
    CUtensorMap mw, mk, mu;
    if (!make_tmap_tokens(&mw, w, d.B, d.T, d.H, K, C) || !make_tmap_tokens(&mk, k, d.B, d.T, d.Hk, K, C) ||
        !make_tmap_tokens_sw64(&mu, u, d.B, d.T, d.H, d.V, C))
        return cudaErrorInvalidValue;
    auto kern = scan_mma_kernel<K, C, PER_K, GENERAL, TRANSFER, F16>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(d.V / kBV + (TRANSFER ? K / kBV : 0), d.H, co ? nseq : d.B);
    kern<<<grid, L::kThreads, smem, s>>>(mw, mk, mu, (const bf16*)k, g_cum, h0, (bf16*)h_ckpt, (bf16*)v_new,
                                         h_final, m_out, co, d.T, d.H, d.V, d.G, err);
    return cudaGetLastError();
}

template <int K, int C, bool PER_K, bool TRANSFER>
cudaError_t launch(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum, const float* h0,
                   void* h_ckpt, void* v_new, float* h_final, float* m_out, const int* co, int nseq, cudaStream_t s,
                   unsigned int* err) {
    if constexpr (!TRANSFER) {   // fp16 io: the scan proper (the segment maps are bf16 only)
        if (d.f16) {
            if (d.T % C != 0 || d.G != 1)
                return launch_v<K, C, PER_K, true, false, true>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, m_out,
                                                                co, nseq, s, err);
            return launch_v<K, C, PER_K, false, false, true>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, m_out, co,
                                                             nseq, s, err);
        }
    }
    if (d.T % C != 0 || d.G != 1)
        return launch_v<K, C, PER_K, true, TRANSFER, false>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, m_out, co,
                                                            nseq, s, err);
    return launch_v<K, C, PER_K, false, TRANSFER, false>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, m_out, co,
                                                         nseq, s, err);
}

template <bool TRANSFER>
cudaError_t dispatch(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum, const float* h0,
                     void* h_ckpt, void* v_new, float* h_final, float* m_out, const int* co, int nseq, cudaStream_t s,
                     unsigned int* err) {
#define GDR_SCAN_ARGS d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, m_out, co, nseq, s, err
    if (d.K == 64) {
        if (d.C == 32)
            return d.per_k ? launch<64, 32, true, TRANSFER>(GDR_SCAN_ARGS) : launch<64, 32, false, TRANSFER>(GDR_SCAN_ARGS);
        return d.per_k ? launch<64, 64, true, TRANSFER>(GDR_SCAN_ARGS) : launch<64, 64, false, TRANSFER>(GDR_SCAN_ARGS);
    }
    if (d.C == 32)
        return d.per_k ? launch<128, 32, true, TRANSFER>(GDR_SCAN_ARGS) : launch<128, 32, false, TRANSFER>(GDR_SCAN_ARGS);
    return d.per_k ? launch<128, 64, true, TRANSFER>(GDR_SCAN_ARGS) : launch<128, 64, false, TRANSFER>(GDR_SCAN_ARGS);
#undef GDR_SCAN_ARGS
}

}  // namespace

cudaError_t mma_scan(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum, const float* h0,
                     void* h_ckpt, void* v_new, float* h_final, cudaStream_t s, unsigned int* err, const int* co,
                     int nseq) {
    if (!(d.bf16 || d.f16) || (co && (d.B != 1 || nseq < 1))) return cudaErrorInvalidValue;
    return dispatch<false>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, nullptr, co, nseq, s, err);
}

cudaError_t mma_scan_transfer(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum,
                              float* m_out, float* z_out, cudaStream_t s, unsigned int* err) {
    if (!d.bf16 || !m_out || !z_out) return cudaErrorInvalidValue;
    return dispatch<true>(d, k, w, u, g_cum, nullptr, nullptr, nullptr, z_out, m_out, nullptr, 0, s, err);
}

}  // namespace gdr
