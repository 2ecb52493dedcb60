// Fused state scan + chunk output for bf16 or fp16 io and a scalar (per-head) gate:
// given w, u and the chunk-local cumulative gate G (from the WY prepare),
//
//   scan   ("kernel_fun/kda/_kernels/bwd_scan.py", module docstring):
//          h_c = state before chunk c;  v'_c = u_c - w_c h_c;
//          h_{c+1} = exp(G_last) h_c + (k exp(G_last - G))^T v'_c
//   output (the o assembly the same page gives to the forward's epilogue warps):
//          o_c = scale [ exp(G) * (q h_c) + tril_0(q k^T * exp(G_i - G_j)) v'_c ]
//
// so v' and the checkpoints never leave the chip.  One CTA per (batch, head, 32
// value columns); serial over chunks:
//
//   warps 0-3   recurrence, as in the standalone scan: warp (vh, kh) owns value
//               columns 16vh.. and key rows kh K/2.. of h^T in mma.sync
//               accumulators; the key halves swap partial sums of h^T w^T behind
//               a named barrier; gamma_t = exp(G_last - G_t) is folded into v'.
//               Per chunk each warp stages its quarter of bf16 h_c and its half
//               of v' for the output warps (double-buffered)
//   warps 4..   output, one per 16 tokens of the chunk: q h_c (rows then scaled
//               by exp(G_i) in fp32) plus P v', P either the tile the prepare
//               wrote or q k^T gated here; only the k-steps at or below the
//               diagonal of P are taken.  o leaves by 16-byte global stores
//   1 warp      producer of the recurrence ring: TMA w, k, u; gamma; exp(G_last)
//   1 warp      producer of the output ring: TMA q and P (or k); the chunk's G
//
// The two rings are separate so the output warps, which trail the recurrence,
// never hold it back.  Tiles read by ldmatrix use 128-byte (w, k, q, P) or
// 64-byte (u, h_c, v', o) XOR swizzles, so every access is conflict-free.
// With fp16 io (F16) every operand and staged tile is fp16 in the same places; the state
// and the accumulators stay fp32.
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

// byte offset of 16-byte chunk `ch` (0..3) of row r in a [rows][32] bf16 tile, 64-byte swizzle
__device__ __forceinline__ uint32_t sw64(int r, int ch) { return (uint32_t)(r * 64 + ((ch ^ ((r >> 1) & 3)) << 4)); }
// byte offset of 16-byte chunk (col / 8) of row r in a [rows][K] tile of 64-column atoms, 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int r, int col, int rows) {
    return (uint32_t)((col >> 6) * rows * 128 + r * 128 + ((((col & 63) >> 3) ^ (r & 7)) << 4));
}

template <int K, int C, bool HAS_P>
struct FLayout {
    static constexpr int KH = K / 2;
    static constexpr int NT8 = C / 8;
    static constexpr int NOW = C / 16;                  // output warps
    static constexpr int kOut0 = kRecWarps, kProdA = kOut0 + NOW, kProdB = kProdA + 1;
    static constexpr int kThreads = 32 * (kProdB + 1);
    static constexpr uint32_t kKC = C * K * 2;          // [C][K] bf16
    static constexpr uint32_t kU = C * kBV * 2;         // [C][32] bf16
    static constexpr uint32_t kPK = HAS_P ? C * C * 2 : kKC;   // P [C][C] or raw k [C][K]
    static constexpr int NSB = 2;                       // output ring stages
    // recurrence ring: three stages when they fit
    static constexpr uint32_t fixed = 2 * kRecWarps * NT8 * 512 + 2 * K * kBV * 2 + 2 * kU + NSB * (kKC + kPK) +
                                      NOW * 16 * kBV * 2 + 4096;
    static constexpr int NSA = (3 * (2 * kKC + kU) + fixed + 1024 <= 232448) ? 3 : 2;
    static constexpr uint32_t W = 0;
    static constexpr uint32_t KB = W + NSA * kKC;
    static constexpr uint32_t U = KB + NSA * kKC;
    static constexpr uint32_t X = U + NSA * kU;                         // partial-sum exchange, 2 x 4 warps
    static constexpr uint32_t kX = NT8 * 512;
    static constexpr uint32_t HC = X + 2 * kRecWarps * kX;              // 2 x [K][32] bf16 h_c
    static constexpr uint32_t VP = HC + 2 * K * kBV * 2;                // 2 x [C][32] bf16 v'
    static constexpr uint32_t Q = (VP + 2 * kU + 1023) & ~1023u;        // output ring: q
    static constexpr uint32_t PK = Q + NSB * kKC;                       //              P or k
    static constexpr uint32_t OS = PK + NSB * kPK;                      // NOW x [16][32] bf16 o staging
    static constexpr uint32_t GAM = OS + NOW * 16 * kBV * 2;            // NSA x C gamma
    static constexpr uint32_t DEC = GAM + NSA * C * 4;                  // NSA x exp(G_last)
    static constexpr uint32_t GO = DEC + 16;                            // NSB x C G for the output
    static constexpr uint32_t bytes = GO + NSB * C * 4;
    static constexpr uint32_t tx_a = 2 * kKC + kU;
    static constexpr uint32_t tx_b = kKC + kPK;
    static_assert(bytes + 1024 <= 232448, "fused scan/output shared memory");
    static_assert(!HAS_P || C == 64, "a precomputed P comes in 64 x 64 tiles");
};

// GENERAL: a partial last chunk or grouped value heads.  Whole chunks of ungrouped
// heads take the variant without those guards: this kernel's schedule is sensitive
// enough that the guards alone measured 4-7% slower where they are not needed.
// co (packed variable-length sequences; NULL otherwise): one data row (B = 1) of whole-chunk runs,
// sequence z = blockIdx.z on the chunks co[z] .. co[z+1]-1, from h0[z] to h_final[z].
// pcu (with co and P; NULL otherwise): q, k and o are the caller's packed tensors [Tin, ...] rather than
// the chunk-packed row; chunk c of sequence z reads q and k from packed row pcu[z] + c C, the rows past
// the sequence's end in k are zeroed once they land (they hold the next sequence's tokens; their v' is
// zero, but 0 * inf is not), and only o's rows inside the sequence are stored.
template <int K, int C, bool HAS_P, bool GENERAL, bool PACKED, bool F16>
__global__ void __launch_bounds__(FLayout<K, C, HAS_P>::kThreads, 1)
fused_scan_output_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mk,
                         const __grid_constant__ CUtensorMap mu, const __grid_constant__ CUtensorMap mq,
                         const __grid_constant__ CUtensorMap mpk, const float* __restrict__ g_cum,
                         const float* __restrict__ h0, bf16* __restrict__ o, float* __restrict__ h_final,
                         const int* __restrict__ co, const int* __restrict__ pcu, int Tin, int T, int H, int V, int G,
                         float scale, unsigned int* err) {
    using L = FLayout<K, C, HAS_P>;
    constexpr int NSA = L::NSA, NSB = L::NSB, NOW = L::NOW, NT8 = L::NT8, KH = L::KH;
    constexpr int NJH = KH / 8;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = bw::smem_u32(sm);
    __shared__ uint64_t fullA[NSA], emptyA[NSA], fullB[NSB], emptyB[NSB], hv_full[2], hv_empty[2];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.x * kBV, h = blockIdx.y, b = blockIdx.z;
    const int NTall = GENERAL ? (T + C - 1) / C : T / C;   // a last, partial chunk runs as zero tokens past T
    // this CTA's chunks: c0 .. c0 + NT - 1 of data row bd (clamped, so any co stays inside the tensors)
    const int c0 = co ? min(max(co[b], 0), NTall) : 0;
    const int NT = co ? min(max(co[b + 1], c0), NTall) - c0 : NTall;
    const int bd = co ? 0 : b;
    // packed q, k, o: the sequence's first packed row and its length (clamped to the tensor and its chunks)
    const bool packed = PACKED && co && pcu;   // compiled out of the batched variant
    const int in0 = packed ? min(max(pcu[b], 0), Tin) : 0;
    const int len = packed ? min(min(max(pcu[b + 1] - in0, 0), Tin - in0), NT * C) : 0;
    auto qk_row = [&](int c) -> int { return packed ? in0 + c * C : (c0 + c) * C; };
    const int hk = GENERAL ? h / G : h;                  // q/k head of value head h
    const int g = lane >> 2, q4 = lane & 3, mi = lane >> 3, mr = lane & 7;
    auto row = [&](int t) -> int64_t {                   // G past T: its last value
        return ((int64_t)bd * T + (GENERAL ? min(t, T - 1) : t)) * H + h;
    };

    if (tid == 0) {
        for (int s = 0; s < NSA; ++s) {
            bw::mbar_init(&fullA[s], 32 + 1);
            bw::mbar_init(&emptyA[s], kRecWarps);
        }
        for (int s = 0; s < NSB; ++s) {
            bw::mbar_init(&fullB[s], 32 + 1);
            bw::mbar_init(&emptyB[s], NOW);
        }
        for (int i = 0; i < 2; ++i) {
            bw::mbar_init(&hv_full[i], kRecWarps);
            bw::mbar_init(&hv_empty[i], NOW);
        }
        bw::fence_mbar_init();
    }
    __syncthreads();

    if (warp == L::kProdA) {
        // ------------------------------------------------------------ recurrence-ring producer
        float* sGam = reinterpret_cast<float*>(sm + L::GAM);
        float* sDec = reinterpret_cast<float*>(sm + L::DEC);
        constexpr int GPL = C / 32;
        float gn[GPL], gln;
        auto load_g = [&](int c) {
#pragma unroll
            for (int i = 0; i < GPL; ++i) gn[i] = g_cum[row((c0 + c) * C + lane + 32 * i)];
            gln = g_cum[row((c0 + c) * C + C - 1)];
        };
        if (NT > 0) load_g(0);
        for (int c = 0; c < NT; ++c) {
            const int s = c % NSA;
            float gc[GPL], glc = gln;
#pragma unroll
            for (int i = 0; i < GPL; ++i) gc[i] = gn[i];
            if (c + 1 < NT) load_g(c + 1);
            if (!bw::mbar_wait(&emptyA[s], ((c / NSA) & 1) ^ 1, err, kDeviceErrTimeout)) break;
            const int t0 = (c0 + c) * C;
            if (lane == 0) {
                bw::mbar_arrive_expect_tx(&fullA[s], L::tx_a);
#pragma unroll
                for (int a = 0; a < K / 64; ++a) {
                    bw::tma_load_4d(sm + L::W + s * L::kKC + a * C * 128, &mw, &fullA[s], a * 64, h, t0, bd);
                    bw::tma_load_4d(sm + L::KB + s * L::kKC + a * C * 128, &mk, &fullA[s], a * 64, hk, qk_row(c), bd);
                }
                bw::tma_load_4d(sm + L::U + s * L::kU, &mu, &fullA[s], v0, h, t0, bd);
                sDec[s] = __expf(glc);
            }
#pragma unroll
            for (int i = 0; i < GPL; ++i) sGam[s * C + lane + 32 * i] = __expf(glc - gc[i]);
            bw::mbar_arrive(&fullA[s]);
        }
        return;
    }
    if (warp == L::kProdB) {
        // ------------------------------------------------------------ output-ring producer
        float* sG = reinterpret_cast<float*>(sm + L::GO);
        for (int c = 0; c < NT; ++c) {
            const int s = c % NSB;
            const int t0 = (c0 + c) * C;
            float gv[C / 32];
#pragma unroll
            for (int i = 0; i < C / 32; ++i) gv[i] = g_cum[row(t0 + lane + 32 * i)];
            if (!bw::mbar_wait(&emptyB[s], ((c / NSB) & 1) ^ 1, err, kDeviceErrTimeout)) break;
            if (lane == 0) {
                bw::mbar_arrive_expect_tx(&fullB[s], L::tx_b);
#pragma unroll
                for (int a = 0; a < K / 64; ++a) {
                    bw::tma_load_4d(sm + L::Q + s * L::kKC + a * C * 128, &mq, &fullB[s], a * 64, hk, qk_row(c), bd);
                    if constexpr (!HAS_P)
                        bw::tma_load_4d(sm + L::PK + s * L::kPK + a * C * 128, &mpk, &fullB[s], a * 64, hk, t0, bd);
                }
                if constexpr (HAS_P) bw::tma_load_4d(sm + L::PK + s * L::kPK, &mpk, &fullB[s], 0, 0, h, bd * NTall + c0 + c);
            }
#pragma unroll
            for (int i = 0; i < C / 32; ++i) sG[s * C + lane + 32 * i] = gv[i];
            bw::mbar_arrive(&fullB[s]);
        }
        return;
    }

    if (warp < kRecWarps) {
        // ------------------------------------------------------------ recurrence warps
        const int vh = warp & 1, kh = warp >> 1;
        const int vr0 = vh * 16, d0 = kh * KH;
        const int64_t state = ((int64_t)b * H + h) * K;
        const float* sGam = reinterpret_cast<const float*>(sm + L::GAM);
        const float* sDec = reinterpret_cast<const float*>(sm + L::DEC);
        float hT[NJH][4];
#pragma unroll
        for (int j = 0; j < NJH; ++j) {
            const int d = d0 + 8 * j + 2 * q4;
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
        bool ready = NT > 0 && bw::mbar_test_wait(&fullA[0], 0);
        bool hv_free = true;                          // the first two staging buffers start free
        for (int c = 0; c < NT; ++c) {
            const int s = c % NSA, hb = c & 1;
            if (!ready) ok = ok && bw::mbar_wait(&fullA[s], (c / NSA) & 1, err, kDeviceErrTimeout);
            const uint32_t w_t = s_base + L::W + s * L::kKC;
            const uint32_t k_t = s_base + L::KB + s * L::kKC;
            const uint32_t u_t = s_base + L::U + s * L::kU;
            if (packed && (c + 1) * C > len) {
                // the sequence's last, partial chunk: every warp zeroes the k rows past its end itself
                // (the same zeros), so each reads only zeros there; fenced before the slot goes back to TMA
                const int first = max(len - c * C, 0);
                unsigned char* kt = sm + L::KB + s * L::kKC;
                for (int i = lane; i < (C - first) * (K / 8); i += 32) {
                    const int r = first + i / (K / 8), u16 = i % (K / 8);
                    *reinterpret_cast<uint4*>(kt + (u16 >> 3) * C * 128 + r * 128 + (u16 & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                bw::fence_async_shared();
                __syncwarp();
            }

            // partial D = h^T[:, my keys] w[:, my keys]^T  [16 x C]
            float D[NT8][4];
#pragma unroll
            for (int j = 0; j < NT8; ++j) D[j][0] = D[j][1] = D[j][2] = D[j][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KH / 16; ++kk) {
                const uint32_t a[4] = {wm::pack2_io<F16>(hT[2 * kk][0], hT[2 * kk][1]), wm::pack2_io<F16>(hT[2 * kk][2], hT[2 * kk][3]),
                                       wm::pack2_io<F16>(hT[2 * kk + 1][0], hT[2 * kk + 1][1]),
                                       wm::pack2_io<F16>(hT[2 * kk + 1][2], hT[2 * kk + 1][3])};
#pragma unroll
                for (int jp = 0; jp < NT8; jp += 2) {
                    uint32_t bfr[4];
                    wm::ldsm_x4(w_t + sw128(8 * jp + 8 * (mi >> 1) + mr, d0 + 16 * kk + 8 * (mi & 1), C), bfr);
                    wm::mma16816_io<F16>(D[jp], a, bfr[0], bfr[1]);
                    wm::mma16816_io<F16>(D[jp + 1], a, bfr[2], bfr[3]);
                }
            }

            // h_c quarter -> staging [K][32] (rows = key), once the output warps released chunk c-2's
            if (!hv_free) ok = ok && bw::mbar_wait(&hv_empty[hb], ((c >> 1) & 1) ^ 1, err, kDeviceErrTimeout);
            {
                const uint32_t st = s_base + L::HC + hb * (K * kBV * 2);
#pragma unroll
                for (int j = 0; j < NJH; j += 2) {
                    const uint32_t r[4] = {wm::pack2_io<F16>(hT[j][0], hT[j][1]), wm::pack2_io<F16>(hT[j][2], hT[j][3]),
                                           wm::pack2_io<F16>(hT[j + 1][0], hT[j + 1][1]), wm::pack2_io<F16>(hT[j + 1][2], hT[j + 1][3])};
                    wm::stsm_x4_t(st + sw64(d0 + 8 * j + 8 * (mi >> 1) + mr, 2 * vh + (mi & 1)), r);
                }
            }

            // u^T fragments
            uint32_t ur[NT8 / 2][4];
#pragma unroll
            for (int jp = 0; jp < NT8; jp += 2)
                wm::ldsm_x4_t(u_t + sw64(8 * jp + 8 * (mi >> 1) + mr, 2 * vh + (mi & 1)), ur[jp / 2]);

            // D = D_0 + D_1 through shared memory
            {
                unsigned char* xb = sm + L::X + (c & 1) * kRecWarps * L::kX;
                float4* mine = reinterpret_cast<float4*>(xb + warp * L::kX) + lane;
                const float4* other = reinterpret_cast<const float4*>(xb + (warp ^ 2) * L::kX) + lane;
#pragma unroll
                for (int j = 0; j < NT8; ++j) mine[32 * j] = make_float4(D[j][0], D[j][1], D[j][2], D[j][3]);
                bw::named_bar_sync(1 + vh, 64);
                if (c + 1 < NT) {
                    ready = bw::mbar_test_wait(&fullA[(c + 1) % NSA], ((c + 1) / NSA) & 1);
                    hv_free = c + 1 < 2 || bw::mbar_test_wait(&hv_empty[(c + 1) & 1], (((c + 1) >> 1) & 1) ^ 1);
                }
#pragma unroll
                for (int j = 0; j < NT8; ++j) {
                    const float4 x = other[32 * j];
                    D[j][0] += x.x; D[j][1] += x.y; D[j][2] += x.z; D[j][3] += x.w;
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
            // h^T[:, my keys] = exp(G_last) h^T + (v'^T diag(gamma)) k[:, my keys]
            {
                const float e = sDec[s];
#pragma unroll
                for (int j = 0; j < NJH; ++j) { hT[j][0] *= e; hT[j][1] *= e; hT[j][2] *= e; hT[j][3] *= e; }
            }
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk) {
                const float2 ga = *reinterpret_cast<const float2*>(sGam + s * C + 16 * kk + 2 * q4);
                const float2 gb = *reinterpret_cast<const float2*>(sGam + s * C + 16 * kk + 8 + 2 * q4);
                const uint32_t a[4] = {wm::pack2_io<F16>(D[2 * kk][0] * ga.x, D[2 * kk][1] * ga.y),
                                       wm::pack2_io<F16>(D[2 * kk][2] * ga.x, D[2 * kk][3] * ga.y),
                                       wm::pack2_io<F16>(D[2 * kk + 1][0] * gb.x, D[2 * kk + 1][1] * gb.y),
                                       wm::pack2_io<F16>(D[2 * kk + 1][2] * gb.x, D[2 * kk + 1][3] * gb.y)};
#pragma unroll
                for (int jp = 0; jp < NJH; jp += 2) {
                    uint32_t bfr[4];
                    wm::ldsm_x4_t(k_t + sw128(16 * kk + 8 * (mi & 1) + mr, d0 + 8 * jp + 8 * (mi >> 1), C), bfr);
                    wm::mma16816_io<F16>(hT[jp], a, bfr[0], bfr[1]);
                    wm::mma16816_io<F16>(hT[jp + 1], a, bfr[2], bfr[3]);
                }
            }
            __syncwarp();
            if (lane == 0) bw::mbar_arrive(&emptyA[s]);
            // this key half's tokens of v' -> staging [C][32] (rows = token)
            {
                const uint32_t st = s_base + L::VP + hb * L::kU;
#pragma unroll
                for (int jp = 0; jp < NT8; jp += 2) {
                    if ((jp >= NT8 / 2) != (kh == 1)) continue;   // static register indices, runtime half
                    const uint32_t r[4] = {wm::pack2_io<F16>(D[jp][0], D[jp][1]), wm::pack2_io<F16>(D[jp][2], D[jp][3]),
                                           wm::pack2_io<F16>(D[jp + 1][0], D[jp + 1][1]), wm::pack2_io<F16>(D[jp + 1][2], D[jp + 1][3])};
                    wm::stsm_x4_t(st + sw64(8 * jp + 8 * (mi >> 1) + mr, 2 * vh + (mi & 1)), r);
                }
            }
            __syncwarp();
            if (lane == 0) bw::mbar_arrive(&hv_full[hb]);
        }
        if (h_final) {
#pragma unroll
            for (int j = 0; j < NJH; ++j) {
                const int d = d0 + 8 * j + 2 * q4;
                const int va = v0 + vr0 + g, vb = va + 8;
                h_final[(state + d) * V + va] = hT[j][0];
                h_final[(state + d + 1) * V + va] = hT[j][1];
                h_final[(state + d) * V + vb] = hT[j][2];
                h_final[(state + d + 1) * V + vb] = hT[j][3];
            }
        }
        (void)ok;
        return;
    }

    // ---------------------------------------------------------------- output warps
    const int ow = warp - L::kOut0;
    const int r0 = ow * 16;                       // this warp's 16 tokens of the chunk
    const float* sG = reinterpret_cast<const float*>(sm + L::GO);
    const uint32_t os = s_base + L::OS + ow * (16 * kBV * 2);
    bool ok = true;
    for (int c = 0; c < NT; ++c) {
        const int s = c % NSB, hb = c & 1;
        const int t0 = (c0 + c) * C;
        ok = ok && bw::mbar_wait(&fullB[s], (c / NSB) & 1, err, kDeviceErrTimeout);
        const uint32_t q_t = s_base + L::Q + s * L::kKC;
        const uint32_t pk_t = s_base + L::PK + s * L::kPK;
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
            for (int kk = 0; kk < C / 16; ++kk) {
                if (kk > ow) continue;
                wm::ldsm_x4(pk_t + sw128(r0 + 8 * (mi & 1) + mr, 16 * kk + 8 * (mi >> 1), C), pa[kk]);
            }
        } else {
            // S = q k^T  [16 x C], then P = tril_0(S * exp(G_i - G_j)) as A fragments
            float S[NT8][4];
#pragma unroll
            for (int j = 0; j < NT8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < K / 16; ++kk) {
#pragma unroll
                for (int jp = 0; jp < NT8; jp += 2) {
                    if (jp / 2 > ow) continue;           // key blocks above the diagonal are masked anyway
                    uint32_t bfr[4];
                    wm::ldsm_x4(pk_t + sw128(8 * jp + 8 * (mi >> 1) + mr, 16 * kk + 8 * (mi & 1), C), bfr);
                    wm::mma16816_io<F16>(S[jp], qa[kk], bfr[0], bfr[1]);
                    wm::mma16816_io<F16>(S[jp + 1], qa[kk], bfr[2], bfr[3]);
                }
            }
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
                pa[kk][0] = wm::pack2_io<F16>(pv[0][0], pv[0][1]);
                pa[kk][1] = wm::pack2_io<F16>(pv[0][2], pv[0][3]);
                pa[kk][2] = wm::pack2_io<F16>(pv[1][0], pv[1][1]);
                pa[kk][3] = wm::pack2_io<F16>(pv[1][2], pv[1][3]);
            }
        }
        // o = exp(G_i) (q h_c) + P v'   [16 x 32]
        ok = ok && bw::mbar_wait(&hv_full[hb], (c >> 1) & 1, err, kDeviceErrTimeout);
        const uint32_t hc_t = s_base + L::HC + hb * (K * kBV * 2);
        const uint32_t vp_t = s_base + L::VP + hb * L::kU;
        float acc[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) {
#pragma unroll
            for (int jp = 0; jp < 4; jp += 2) {
                uint32_t bfr[4];
                wm::ldsm_x4_t(hc_t + sw64(16 * kk + 8 * (mi & 1) + mr, jp + (mi >> 1)), bfr);
                wm::mma16816_io<F16>(acc[jp], qa[kk], bfr[0], bfr[1]);
                wm::mma16816_io<F16>(acc[jp + 1], qa[kk], bfr[2], bfr[3]);
            }
        }
        {
            const float e0 = __expf(Gi0), e1 = __expf(Gi1);
#pragma unroll
            for (int j = 0; j < 4; ++j) { acc[j][0] *= e0; acc[j][1] *= e0; acc[j][2] *= e1; acc[j][3] *= e1; }
        }
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk) {
            if (kk > ow) continue;                   // P is zero above the diagonal block
#pragma unroll
            for (int jp = 0; jp < 4; jp += 2) {
                uint32_t bfr[4];
                wm::ldsm_x4_t(vp_t + sw64(16 * kk + 8 * (mi & 1) + mr, jp + (mi >> 1)), bfr);
                wm::mma16816_io<F16>(acc[jp], pa[kk], bfr[0], bfr[1]);
                wm::mma16816_io<F16>(acc[jp + 1], pa[kk], bfr[2], bfr[3]);
            }
        }
        __syncwarp();
        if (lane == 0) {
            bw::mbar_arrive(&hv_empty[hb]);
            bw::mbar_arrive(&emptyB[s]);
        }
        // o * scale -> bf16 staging [16][32] -> 16-byte global stores
#pragma unroll
        for (int jp = 0; jp < 4; jp += 2) {
            const uint32_t r[4] = {wm::pack2_io<F16>(acc[jp][0] * scale, acc[jp][1] * scale),
                                   wm::pack2_io<F16>(acc[jp][2] * scale, acc[jp][3] * scale),
                                   wm::pack2_io<F16>(acc[jp + 1][0] * scale, acc[jp + 1][1] * scale),
                                   wm::pack2_io<F16>(acc[jp + 1][2] * scale, acc[jp + 1][3] * scale)};
            asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(
                             os + sw64(8 * (mi & 1) + mr, jp + (mi >> 1))),
                         "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                         : "memory");
        }
        __syncwarp();
        bf16* dst = o + (((int64_t)bd * T + (packed ? in0 + c * C : t0) + r0) * H + h) * V + v0;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int rr = 8 * i + (lane >> 2), ch = lane & 3;
            const uint4 x = wm::lds128(os + sw64(rr, ch));
            const bool in = packed ? c * C + r0 + rr < len : (!GENERAL || t0 + r0 + rr < T);
            if (in) *reinterpret_cast<uint4*>(dst + (int64_t)rr * H * V + 8 * ch) = x;
        }
        __syncwarp();
    }
    (void)ok;
}

template <int K, int C, bool HAS_P, bool GENERAL, bool PACKED, bool F16>
cudaError_t launch_v(const Dims& d, const void* q, const void* k, const void* w, const void* u, const float* g_cum,
                     const void* P, const float* h0, void* o, float* h_final, const int* co, int nseq,
                     const int* pcu, int Tin, cudaStream_t s, unsigned int* err) {
    using L = FLayout<K, C, HAS_P>;
    CUtensorMap mw, mk, mu, mq, mpk;
    const int tq = pcu ? Tin : d.T;   // rows of q and k: the caller's packed tokens, or the data row
    if (!make_tmap_tokens(&mw, w, d.B, d.T, d.H, K, C) || !make_tmap_tokens(&mk, k, d.B, tq, d.Hk, K, C) ||
        !make_tmap_tokens_sw64(&mu, u, d.B, d.T, d.H, d.V, C) || !make_tmap_tokens(&mq, q, d.B, tq, d.Hk, K, C))
        return cudaErrorInvalidValue;
    if constexpr (HAS_P) {
        // P [B, NT, H, C, C] seen as (C, C, H, B*NT); one 64 x 64 box per chunk
        const uint64_t dims[4] = {(uint64_t)C, (uint64_t)C, (uint64_t)d.H, (uint64_t)d.B * d.NT};
        const uint64_t st[3] = {(uint64_t)C * 2, (uint64_t)C * C * 2, (uint64_t)d.H * C * C * 2};
        const uint32_t box[4] = {64, 64, 1, 1};
        if (!make_tmap_bf16_4d(&mpk, P, dims, st, box)) return cudaErrorInvalidValue;
    } else {
        mpk = mk;
    }
    auto kern = fused_scan_output_kernel<K, C, HAS_P, GENERAL, PACKED, F16>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(d.V / kBV, d.H, co ? nseq : d.B);
    kern<<<grid, L::kThreads, smem, s>>>(mw, mk, mu, mq, mpk, g_cum, h0, (bf16*)o, h_final, co, pcu, Tin, d.T, d.H,
                                         d.V, d.G, d.scale, err);
    return cudaGetLastError();
}

template <int K, int C, bool HAS_P>
cudaError_t launch(const Dims& d, const void* q, const void* k, const void* w, const void* u, const float* g_cum,
                   const void* P, const float* h0, void* o, float* h_final, const int* co, int nseq,
                   const int* pcu, int Tin, cudaStream_t s, unsigned int* err) {
    if (d.f16) {   // fp16 io: one unpacked form per shape (the guarded one serves whole chunks too)
        if (pcu) return cudaErrorInvalidValue;
        if (d.T % C != 0 || d.G != 1)
            return launch_v<K, C, HAS_P, true, false, true>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, nullptr,
                                                            0, s, err);
        return launch_v<K, C, HAS_P, false, false, true>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, nullptr, 0,
                                                         s, err);
    }
    if constexpr (HAS_P) {   // packed q, k, o (pcu) only with P
        if (pcu) {
            if (d.T % C != 0 || d.G != 1)
                return launch_v<K, C, true, true, true, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, pcu,
                                                               Tin, s, err);
            return launch_v<K, C, true, false, true, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, pcu,
                                                            Tin, s, err);
        }
    }
    if (d.T % C != 0 || d.G != 1)
        return launch_v<K, C, HAS_P, true, false, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, nullptr, 0,
                                                         s, err);
    return launch_v<K, C, HAS_P, false, false, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, nullptr, 0,
                                                      s, err);
}

}  // namespace

cudaError_t mma_scan_output(const Dims& d, const void* q, const void* k, const void* w, const void* u,
                            const float* g_cum, const void* P, const float* h0, void* o, float* h_final,
                            cudaStream_t s, unsigned int* err, const int* co, int nseq, const int* pcu, int Tin) {
    if (!(d.bf16 || d.f16) || d.per_k || (co && (d.B != 1 || nseq < 1))) return cudaErrorInvalidValue;
    if (pcu && (!co || !P || Tin < 1)) return cudaErrorInvalidValue;
    if (P) {
        if (d.C != 64) return cudaErrorInvalidValue;
        return d.K == 64 ? launch<64, 64, true>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, pcu, Tin, s, err)
                         : launch<128, 64, true>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, pcu, Tin, s, err);
    }
    if (d.K == 64) return d.C == 32 ? launch<64, 32, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, pcu, Tin, s, err)
                                    : launch<64, 64, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, pcu, Tin, s, err);
    return d.C == 32 ? launch<128, 32, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, pcu, Tin, s, err)
                     : launch<128, 64, false>(d, q, k, w, u, g_cum, P, h0, o, h_final, co, nseq, pcu, Tin, s, err);
}

}  // namespace gdr
