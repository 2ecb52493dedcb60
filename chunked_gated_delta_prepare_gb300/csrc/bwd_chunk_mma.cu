// The backward's per-chunk stage for bf16 io and a scalar gate (32- or 64-token
// chunks): every gradient that needs only the chunk's own tiles, in one kernel
// (the pages' backward names this stage wy_dqkg: the WY backward fused with dq,
// dk and the gate gradient; "kernel_fun/kda/_kernels/bwd_scan.py", host wrapper).
//
// Per chunk (rows i, j; G the chunk-local cumsum of g, G_L its last row,
// Gam_ij = exp(G_i - G_j); h = h_ckpt[c], dhn = dh_ckpt[c]; T = (I + A)^{-1}):
//
//   dqg = scale do h^T,  dkg = v' dhn^T,  dw = -dv' h^T
//   Xq  = scale (do v'^T) * Gam, strictly lower;  its diagonal d_i = scale do_i . v'_i
//   dq  = dqg e^G + Xq k + d_i k_i
//   dk  = dkg e^(G_L - G) + Xq^T q + d_i q_i + beta e^G dkb + Y k + Y^T k
//   dkb = T^T dw,  dvb = T^T dv',  dv = beta dvb
//   dA  = strict_lower(-(dkb w^T + dvb u^T))      (w = T kb, u = T vb make T^T dT T^T collapse to this)
//   Y   = beta_i dA_ij Gam_ij
//   dbeta_i = sum_d dkb k e^G + sum_v dvb v + sum_j dA_ij M_ij,  M = Gam * (k k^T)
//   dG_i = sum_d [dqg q e^G + q (Xq k) - k (Xq^T q) - dkg k e^(G_L - G) + dkb kb + k (Y k) - k (Y^T k)]
//          (+ on the chunk's last token: sum of the dkg kg terms of the other rows + e^(G_L) sum h dhn)
//   dg  = reverse cumsum of dG over the chunk
//
// The diagonal of the output scores and the last token's own dkg kg term cancel
// exactly in dG and are left out of it (fp32 rounding of those O(1) pairs would
// otherwise swamp a small dG).  One CTA of eight warps per (chunk, head,
// batch); the tiles sit in shared memory as padded bf16 rows (a row stride of
// D + 8 elements keeps every ldmatrix free of bank conflicts) and every product
// is a warp-level mma.sync m16n8k16 with fp32 accumulation.  Warp w owns the
// 16-row block w % (C/16) and the column group w / (C/16) of every [C x D]
// result, so dq and dk accumulate in registers across all their terms (sixteen
// warps with column quarters measured no faster).  Epilogues work on column
// pairs (one bf16x2 access for two elements), keep the row sums of dG and dbeta
// in registers until the end, and dq and dk leave through shared memory as
// 16-byte row stores: 2.36 -> 1.76 ms on the 32k-token, 32-head problem.  Tile
// loads are cp.async groups issued in the order the products need them, and the
// WY phase's tiles are in flight during the output-score phase.  (A persistent
// CTA prefetching the next chunk's tiles into dead regions measured slower:
// 1.92 ms with cp.async, 2.06 ms with per-row bulk copies.)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "chunk_mma.cuh"
#include "gdr_internal.h"
#include "warp_mma.cuh"

namespace gdr {
namespace {

using bf16 = __nv_bfloat16;
using namespace cm;
constexpr int kThreads = 256;

template <int K, int V, int C>
struct ChunkLayout {
    static constexpr int LK = K + 8, LV = V + 8, LC = C + 8;
    static constexpr uint32_t rq = 0;                              // q
    static constexpr uint32_t rk = rq + C * LK * 2;                // k
    static constexpr uint32_t rdo = rk + C * LK * 2;               // do; later v
    static constexpr uint32_t rvp = rdo + C * LV * 2;              // v'; later u
    static constexpr uint32_t rdv = rvp + C * LV * 2;              // dv'
    static constexpr uint32_t rh = rdv + C * LV * 2;               // h [K][V]; later dkb [C][K] (+ T)
    static constexpr uint32_t rdh = rh + K * LV * 2;               // dhn [K][V]; later dvb [C][V] (+ w)
    static constexpr uint32_t rw = rdh + K * LV * 2;               // dw [C][K]
    static constexpr uint32_t rx = rw + C * LK * 2;                // Xq
    static constexpr uint32_t ry = rx + C * LC * 2;                // Y
    static constexpr uint32_t rf = ry + C * LC * 2;                // fp32 rows
    // the WY phase's T and w, prefetched during phase 2: behind dkb in h's space and behind dvb in
    // dhn's space where those have room, else in space of their own
    static constexpr bool kTinH = K * LV * 2 >= C * LK * 2 + C * LC * 2;
    static constexpr bool kWinDH = K * LV * 2 >= C * LV * 2 + C * LK * 2;
    static constexpr uint32_t rextra = rf + 8 * C * 4;
    static constexpr uint32_t rt = kTinH ? rh + C * LK * 2 : rextra;
    static constexpr uint32_t rw2 = kWinDH ? rdh + C * LV * 2 : rextra + (kTinH ? 0 : C * LC * 2);
    static constexpr uint32_t bytes = rextra + (kTinH ? 0 : C * LC * 2) + (kWinDH ? 0 : C * LK * 2);
    static_assert(C * LK <= K * LV, "dkb fits over h");
    static_assert(bytes <= 227 * 1024, "shared memory");
};

template <int K, int V, int C>
__global__ void __launch_bounds__(kThreads, 1)
bwd_chunk_mma_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v,
                     const bf16* __restrict__ beta, const float* __restrict__ g_cum, const bf16* __restrict__ w,
                     const bf16* __restrict__ u, const bf16* __restrict__ tinv, const bf16* __restrict__ v_new,
                     const bf16* __restrict__ h_ckpt, const bf16* __restrict__ d_o, const bf16* __restrict__ dv_new,
                     const bf16* __restrict__ dh_ckpt, bf16* __restrict__ dq, bf16* __restrict__ dk,
                     bf16* __restrict__ dv, bf16* __restrict__ dbeta, float* __restrict__ dg, int T, int H, int G,
                     float scale) {
    using L = ChunkLayout<K, V, C>;
    constexpr int LK = L::LK, LV = L::LV, LC = L::LC;
    constexpr int RB = C / 16, CG = 8 / RB;             // 16-row blocks; warps sharing each
    constexpr int NK = K / 16 / CG, NV = V / 16 / CG;   // 16-column blocks per warp
    constexpr int NCB = C / 16, NC = NCB >= CG ? NCB / CG : 1;   // C x C results: some warps idle at C = 32
    extern __shared__ __align__(128) unsigned char sm[];
    bf16* Qs = reinterpret_cast<bf16*>(sm + L::rq);
    bf16* Ks = reinterpret_cast<bf16*>(sm + L::rk);
    bf16* DOs = reinterpret_cast<bf16*>(sm + L::rdo);
    bf16* VPs = reinterpret_cast<bf16*>(sm + L::rvp);
    bf16* DVs = reinterpret_cast<bf16*>(sm + L::rdv);
    bf16* Hs = reinterpret_cast<bf16*>(sm + L::rh);
    bf16* DHs = reinterpret_cast<bf16*>(sm + L::rdh);
    bf16* DWs = reinterpret_cast<bf16*>(sm + L::rw);
    bf16* Xs = reinterpret_cast<bf16*>(sm + L::rx);
    bf16* Ys = reinterpret_cast<bf16*>(sm + L::ry);
    float* sG = reinterpret_cast<float*>(sm + L::rf);
    float* sEG = sG + C;      // e^G
    float* sGam = sEG + C;    // e^(G_L - G)
    float* sB = sGam + C;     // beta
    float* sdG = sB + C;      // gate gradient per row
    float* sdB = sdG + C;     // dbeta per row
    float* sDiag = sdB + C;   // scale do_i . v'_i
    float* sS = sDiag + C;    // [0]: sum of dkg kg over the other rows, [1]: sum h dhn

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, q4 = lane & 3, mi = lane >> 3, mr = lane & 7;
    const int rb = warp % RB, cg = warp / RB;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int NT = (T + C - 1) / C;
    const int t0 = c * C, nv = min(C, T - t0);
    const int64_t tok0 = ((int64_t)b * T + t0) * H + h;      // row of token t0, head h
    const int Hk = H / G;
    const int64_t ktok0 = ((int64_t)b * T + t0) * Hk + h / G; // q and k: row of token t0, q/k head h / G
    const int64_t st_off = (((int64_t)b * NT + c) * H + h);  // this chunk's [K][V] / [C][C] block index
    // ---- gate rows and beta
    if (tid < C) {
        const int i = tid;
        const float Gv = g_cum[((int64_t)b * T + t0 + min(i, nv - 1)) * H + h];
        const float GL = g_cum[((int64_t)b * T + t0 + nv - 1) * H + h];
        sG[i] = Gv;
        sEG[i] = __expf(Gv);
        sGam[i] = __expf(GL - Gv);
        sB[i] = i < nv ? __bfloat162float(beta[tok0 + (int64_t)i * H]) : 0.f;
        sdG[i] = 0.f;
        sdB[i] = 0.f;
        if (i < 2) sS[i] = 0.f;
    }
    // ---- phase 1 tiles, in three groups in the order the products need them
    load_tile<V, kThreads>(Hs, h_ckpt + st_off * K * V, V, K, K, tid);
    load_tile<V, kThreads>(DOs, d_o + tok0 * V, (int64_t)H * V, C, nv, tid);
    cp_async_commit();
    load_tile<V, kThreads>(VPs, v_new + tok0 * V, (int64_t)H * V, C, nv, tid);
    load_tile<V, kThreads>(DHs, dh_ckpt + st_off * K * V, V, K, K, tid);
    cp_async_commit();
    load_tile<V, kThreads>(DVs, dv_new + tok0 * V, (int64_t)H * V, C, nv, tid);
    load_tile<K, kThreads>(Qs, q + ktok0 * K, (int64_t)Hk * K, C, nv, tid);
    load_tile<K, kThreads>(Ks, k + ktok0 * K, (int64_t)Hk * K, C, nv, tid);
    cp_async_commit();

    const uint32_t aQ = smem_addr(Qs), aK = smem_addr(Ks), aDO = smem_addr(DOs), aVP = smem_addr(VPs);
    const uint32_t aDV = smem_addr(DVs), aH = smem_addr(Hs), aDH = smem_addr(DHs), aDW = smem_addr(DWs);
    const uint32_t aX = smem_addr(Xs), aY = smem_addr(Ys);
    const int ck = cg * NK, cv = cg * NV, cc = cg * NC;   // this warp's first column block
    const bool cc_active = cc < NCB;                      // a column block of the C x C results

    float accQ[NK][2][4], accK[NK][2][4], tmp[NK][2][4];
    // this thread's partial sums of the gate gradient and of dbeta for rows 16 rb + g4 (index 0) and
    // 16 rb + g4 + 8 (index 1), over its columns of every term; reduced into sdG and sdB once, at the end
    float gr[2] = {0.f, 0.f}, br[2] = {0.f, 0.f};
    // dqg = do h^T (h, do landed)
    cp_async_wait<2>();
    __syncthreads();
    zero(accQ);
    wgemm<NK, V, false, true>(accQ, aDO, LV, aH, LV, rb, ck, mi, mr);
    // dkg = v' dhn^T and the output scores do v'^T (v', dhn landed)
    cp_async_wait<1>();
    __syncthreads();
    zero(accK);
    wgemm<NK, V, false, true>(accK, aVP, LV, aDH, LV, rb, ck, mi, mr);
    // Xq = scale (do v'^T) Gam, strictly lower, with its diagonal apart
    if (cc_active) {
        float xq[NC][2][4];
        zero(xq);
        wgemm<NC, V, false, true>(xq, aDO, LV, aVP, LV, rb, cc, mi, mr);
        each2(xq, rb, cc, g4, q4, [&](int r, int col, float& x0, float& x1) {
            const float y0 = scale * x0, y1 = scale * x1;
            if (col == r) sDiag[r] = y0;
            if (col + 1 == r) sDiag[r] = y1;
            st_bf2(Xs + r * LC + col, col < r ? y0 * __expf(sG[r] - sG[col]) : 0.f,
                   col + 1 < r ? y1 * __expf(sG[r] - sG[col + 1]) : 0.f);
        });
    }
    cp_async_wait<0>();
    __syncthreads();
    // dq's e^G-scaled part and its gate term
    each2(accQ, rb, ck, g4, q4, [&](int r, int col, float& x0, float& x1) {
        const float e = scale * sEG[r];
        const float2 qv = bf2(Qs + r * LK + col);
        x0 *= e;
        x1 *= e;
        gr[(r >> 3) & 1] += x0 * qv.x + x1 * qv.y;
    });
    // dk's e^(G_L - G) part from dkg; the gate terms go to the rows, the last row takes their sum
    {
        float tot = 0.f;
        each2(accK, rb, ck, g4, q4, [&](int r, int col, float& x0, float& x1) {
            const float2 kv = bf2(Ks + r * LK + col);
            const float t = r == nv - 1 ? 0.f : (x0 * kv.x + x1 * kv.y) * sGam[r];
            gr[(r >> 3) & 1] -= t;
            tot += t;
            x0 *= sGam[r];
            x1 *= sGam[r];
        });
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if (lane == 0) atomicAdd(sS, tot);
    }
    // dw = -dv' h^T -> bf16 tile
    zero(tmp);
    wgemm<NK, V, false, true>(tmp, aDV, LV, aH, LV, rb, ck, mi, mr);
    each2(tmp, rb, ck, g4, q4, [&](int r, int col, float& x0, float& x1) { st_bf2(DWs + r * LK + col, -x0, -x1); });
    // sum h dhn, eight elements per step
    {
        float s = 0.f;
        for (int idx = tid; idx < K * V / 8; idx += kThreads) {
            const int d = idx / (V / 8), x = 8 * (idx % (V / 8));
            const uint4 a = *reinterpret_cast<const uint4*>(Hs + d * LV + x);
            const uint4 e = *reinterpret_cast<const uint4*>(DHs + d * LV + x);
            const uint32_t av[4] = {a.x, a.y, a.z, a.w}, ev[4] = {e.x, e.y, e.z, e.w};
    #pragma unroll
            for (int m = 0; m < 4; ++m)
                s += __uint_as_float(av[m] << 16) * __uint_as_float(ev[m] << 16) +
                     __uint_as_float(av[m] & 0xffff0000u) * __uint_as_float(ev[m] & 0xffff0000u);
        }
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) atomicAdd(sS + 1, s);
    }
    __syncthreads();
    // the WY phase's tiles, in flight during phase 2 (h, dhn, do and v' are dead now)
    bf16* Ws = reinterpret_cast<bf16*>(sm + L::rw2);
    bf16* Vs = DOs;
    bf16* Us = VPs;
    bf16* Ts = reinterpret_cast<bf16*>(sm + L::rt);
    load_tile<C, kThreads>(Ts, tinv + st_off * C * C, C, C, C, tid);
    load_tile<K, kThreads>(Ws, w + tok0 * K, (int64_t)H * K, C, nv, tid);
    load_tile<V, kThreads>(Vs, v + tok0 * V, (int64_t)H * V, C, nv, tid);
    load_tile<V, kThreads>(Us, u + tok0 * V, (int64_t)H * V, C, nv, tid);
    cp_async_commit();

    // ---- phase 2: the output scores' other factors
    bf16* DQs = Hs;   // dq staged over the dead h (later dkb's space) for 16-byte row stores
    zero(tmp);
    wgemm<NK, C, false, false>(tmp, aX, LC, aK, LK, rb, ck, mi, mr);      // Xq k
    // dq done: + Xq k + d_i k_i; Xq k's gate term q (Xq k)
    #pragma unroll
    for (int j = 0; j < NK; ++j)
    #pragma unroll
        for (int n = 0; n < 2; ++n)
    #pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int r = 16 * rb + g4 + 8 * h2, col = 16 * (ck + j) + 8 * n + 2 * q4;
                const float x0 = tmp[j][n][2 * h2], x1 = tmp[j][n][2 * h2 + 1];
                const float2 qv = bf2(Qs + r * LK + col), kv = bf2(Ks + r * LK + col);
                gr[h2] += qv.x * x0 + qv.y * x1;
                st_bf2(DQs + r * LK + col, accQ[j][n][2 * h2] + x0 + sDiag[r] * kv.x,
                       accQ[j][n][2 * h2 + 1] + x1 + sDiag[r] * kv.y);
            }
    zero(tmp);
    wgemm<NK, C, true, false>(tmp, aX, LC, aQ, LK, rb, ck, mi, mr);       // Xq^T q
    #pragma unroll
    for (int j = 0; j < NK; ++j)
    #pragma unroll
        for (int n = 0; n < 2; ++n)
    #pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int r = 16 * rb + g4 + 8 * h2, col = 16 * (ck + j) + 8 * n + 2 * q4;
                const float x0 = tmp[j][n][2 * h2], x1 = tmp[j][n][2 * h2 + 1];
                const float2 qv = bf2(Qs + r * LK + col), kv = bf2(Ks + r * LK + col);
                gr[h2] -= kv.x * x0 + kv.y * x1;
                accK[j][n][2 * h2] += x0 + sDiag[r] * qv.x;
                accK[j][n][2 * h2 + 1] += x1 + sDiag[r] * qv.y;
            }
    __syncthreads();
    store_tile<K, kThreads>(dq + tok0 * K, (int64_t)H * K, DQs, nv, tid);

    // ---- phase 3: the WY backward
    bf16* DKBs = Hs;
    bf16* DVBs = DHs;
    cp_async_wait<0>();
    __syncthreads();   // the WY tiles landed; dq's staging has been read
    const uint32_t aT = smem_addr(Ts), aW = smem_addr(Ws), aU = smem_addr(Us);
    // dkb = T^T dw
    zero(tmp);
    wgemm<NK, C, true, false>(tmp, aT, LC, aDW, LK, rb, ck, mi, mr);
    #pragma unroll
    for (int j = 0; j < NK; ++j)
    #pragma unroll
        for (int n = 0; n < 2; ++n)
    #pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int r = 16 * rb + g4 + 8 * h2, col = 16 * (ck + j) + 8 * n + 2 * q4;
                const float x0 = tmp[j][n][2 * h2], x1 = tmp[j][n][2 * h2 + 1];
                const float2 kv = bf2(Ks + r * LK + col);
                const float db = (x0 * kv.x + x1 * kv.y) * sEG[r];   // dkb . k e^G
                br[h2] += db;
                gr[h2] += db * sB[r];                                 // dkb . kb
                st_bf2(DKBs + r * LK + col, x0, x1);
                accK[j][n][2 * h2] += x0 * sB[r] * sEG[r];
                accK[j][n][2 * h2 + 1] += x1 * sB[r] * sEG[r];
            }
    // dvb = T^T dv': dv = beta dvb
    {
        float tv[NV][2][4];
        zero(tv);
        wgemm<NV, C, true, false>(tv, aT, LC, aDV, LV, rb, cv, mi, mr);
        each2(tv, rb, cv, g4, q4, [&](int r, int col, float& x0, float& x1) {
            const float2 vv = bf2(Vs + r * LV + col);
            br[(r >> 3) & 1] += x0 * vv.x + x1 * vv.y;
            st_bf2(DVBs + r * LV + col, x0, x1);
            if (r < nv) st_bf2(dv + (tok0 + (int64_t)r * H) * V + col, sB[r] * x0, sB[r] * x1);
        });
    }
    __syncthreads();
    // dA = strict_lower(-(dkb w^T + dvb u^T)); dbeta's A term against M = Gam (k k^T); Y = beta dA Gam
    if (cc_active) {
        float da[NC][2][4], m[NC][2][4];
        zero(da);
        zero(m);
        wgemm<NC, K, false, true>(da, smem_addr(DKBs), LK, aW, LK, rb, cc, mi, mr);
        wgemm<NC, V, false, true>(da, smem_addr(DVBs), LV, aU, LV, rb, cc, mi, mr);
        wgemm<NC, K, false, true>(m, aK, LK, aK, LK, rb, cc, mi, mr);
    #pragma unroll
        for (int j = 0; j < NC; ++j)
    #pragma unroll
            for (int n = 0; n < 2; ++n)
    #pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int r = 16 * rb + g4 + 8 * h2, col = 16 * (cc + j) + 8 * n + 2 * q4;
                    const float gam0 = col < r ? __expf(sG[r] - sG[col]) : 0.f;
                    const float gam1 = col + 1 < r ? __expf(sG[r] - sG[col + 1]) : 0.f;
                    const float a0 = -da[j][n][2 * h2], a1 = -da[j][n][2 * h2 + 1];
                    br[h2] += a0 * m[j][n][2 * h2] * gam0 + a1 * m[j][n][2 * h2 + 1] * gam1;
                    st_bf2(Ys + r * LC + col, sB[r] * a0 * gam0, sB[r] * a1 * gam1);
                }
    }
    __syncthreads();
    // dk += Y k + Y^T k; their gate terms
    zero(tmp);
    wgemm<NK, C, false, false>(tmp, aY, LC, aK, LK, rb, ck, mi, mr);
    each2(tmp, rb, ck, g4, q4, [&](int r, int col, float& x0, float& x1) {
        const float2 kv = bf2(Ks + r * LK + col);
        gr[(r >> 3) & 1] += kv.x * x0 + kv.y * x1;
    });
    #pragma unroll
    for (int j = 0; j < NK; ++j)
    #pragma unroll
        for (int n = 0; n < 2; ++n)
    #pragma unroll
            for (int e = 0; e < 4; ++e) accK[j][n][e] += tmp[j][n][e];
    zero(tmp);
    wgemm<NK, C, true, false>(tmp, aY, LC, aK, LK, rb, ck, mi, mr);
    bf16* DKS = Hs;   // dk staged over the dead dkb for 16-byte row stores
    #pragma unroll
    for (int j = 0; j < NK; ++j)
    #pragma unroll
        for (int n = 0; n < 2; ++n)
    #pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int r = 16 * rb + g4 + 8 * h2, col = 16 * (ck + j) + 8 * n + 2 * q4;
                const float x0 = tmp[j][n][2 * h2], x1 = tmp[j][n][2 * h2 + 1];
                const float2 kv = bf2(Ks + r * LK + col);
                gr[h2] -= kv.x * x0 + kv.y * x1;
                st_bf2(DKS + r * LK + col, accK[j][n][2 * h2] + x0, accK[j][n][2 * h2 + 1] + x1);
            }
    // the rows' partial sums of dG and dbeta, once
    row_add(sdG + 16 * rb + g4, gr[0], q4);
    row_add(sdG + 16 * rb + g4 + 8, gr[1], q4);
    row_add(sdB + 16 * rb + g4, br[0], q4);
    row_add(sdB + 16 * rb + g4 + 8, br[1], q4);
    __syncthreads();
    store_tile<K, kThreads>(dk + tok0 * K, (int64_t)H * K, DKS, nv, tid);

    // ---- phase 4: the last token's gate terms, the reverse cumsum (a warp's suffix scan), dbeta
    if (warp == 0) {
        const float last = sS[0] + __expf(sG[nv - 1]) * sS[1];
        float lo = sdG[lane] + (lane == nv - 1 ? last : 0.f);                        // rows 0..31
        float hi = C == 64 ? sdG[32 + lane] + (32 + lane == nv - 1 ? last : 0.f) : 0.f;   // rows 32..63
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float a = __shfl_down_sync(0xffffffffu, lo, o), b2 = __shfl_down_sync(0xffffffffu, hi, o);
            if (lane + o < 32) {
                lo += a;
                hi += b2;
            }
        }
        lo += __shfl_sync(0xffffffffu, hi, 0);   // the rows below add the whole upper half
        if (lane < nv) dg[tok0 + (int64_t)lane * H] = lo;
        if (C == 64 && 32 + lane < nv) dg[tok0 + (int64_t)(32 + lane) * H] = hi;
    }
    if (tid < nv) dbeta[tok0 + (int64_t)tid * H] = __float2bfloat16_rn(sdB[tid]);
}

template <int K, int V, int C>
cudaError_t launch(const Dims& d, const void* q, const void* k, const void* v, const void* beta, const float* g_cum,
                   const void* w, const void* u, const void* tinv, const void* v_new, const void* h_ckpt,
                   const void* d_o, const void* dv_new, const void* dh_ckpt, void* dq, void* dk, void* dv,
                   void* dbeta, float* dg, cudaStream_t s) {
    using L = ChunkLayout<K, V, C>;
    auto kern = bwd_chunk_mma_kernel<K, V, C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
    if (e != cudaSuccess) return e;
    const dim3 grid(d.NT, d.H, d.B);
    kern<<<grid, kThreads, L::bytes, s>>>((const bf16*)q, (const bf16*)k, (const bf16*)v, (const bf16*)beta, g_cum,
                                          (const bf16*)w, (const bf16*)u, (const bf16*)tinv, (const bf16*)v_new,
                                          (const bf16*)h_ckpt, (const bf16*)d_o, (const bf16*)dv_new,
                                          (const bf16*)dh_ckpt, (bf16*)dq, (bf16*)dk, (bf16*)dv, (bf16*)dbeta, dg,
                                          d.T, d.H, d.G, d.scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t mma_bwd_chunk(const Dims& d, const void* q, const void* k, const void* v, const void* beta,
                          const float* g_cum, const void* w, const void* u, const void* tinv, const void* v_new,
                          const void* h_ckpt, const void* d_o, const void* dv_new, const void* dh_ckpt, void* dq,
                          void* dk, void* dv, void* dbeta, float* dg, cudaStream_t s) {
    if (!d.bf16 || d.per_k) return cudaErrorInvalidValue;
#define GDR_CHUNK_ARGS d, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new, dh_ckpt, dq, dk, dv, dbeta, dg, s
    if (d.C == 32) {
        if (d.K == 64 && d.V == 64) return launch<64, 64, 32>(GDR_CHUNK_ARGS);
        if (d.K == 64 && d.V == 128) return launch<64, 128, 32>(GDR_CHUNK_ARGS);
        if (d.K == 128 && d.V == 64) return launch<128, 64, 32>(GDR_CHUNK_ARGS);
        return launch<128, 128, 32>(GDR_CHUNK_ARGS);
    }
    if (d.K == 64 && d.V == 64) return launch<64, 64, 64>(GDR_CHUNK_ARGS);
    if (d.K == 64 && d.V == 128) return launch<64, 128, 64>(GDR_CHUNK_ARGS);
    if (d.K == 128 && d.V == 64) return launch<128, 64, 64>(GDR_CHUNK_ARGS);
    return launch<128, 128, 64>(GDR_CHUNK_ARGS);
#undef GDR_CHUNK_ARGS
}

}  // namespace gdr
