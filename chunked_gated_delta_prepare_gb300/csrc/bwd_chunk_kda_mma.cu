// The backward's per-chunk stage for a per-key-dim gate (KDA), bf16 io: the
// wy_dqkg stage of "kernel_fun/kda/_kernels/bwd_scan.py" (host wrapper), the
// per-key-dim counterpart of bwd_chunk_mma.cu.  Per chunk it forms dq, dk, dv,
// dbeta and dg from the chunk's tiles, T = (I + A)^{-1}, the checkpoints h and
// dh_next, v' and dv'.
//
// Every gate factor e^(G_i - G_j) depends on the key dim here, so it cannot be
// folded into a C x C matrix.  Around the chunk's middle row ref, with
// E_id = e^(G_id - G_ref,d):
//
//   Qa = q E,  Kb = k / E,  Ka = k E                 (bf16 tiles)
//   L(X, k)_i = E_i (X Kb)_i,   R(X, q)_j = (X^T Qa)_j / E_j,   M = Ka Kb^T
//   L(Y, k)_i = E_i (Y Kb)_i,   R(Y, k)_j = (Y^T Ka)_j / E_j
//
// and the gate gradient's products need no division: q_i L_i = Qa_i (X Kb)_i,
// k_j R_j = Kb_j (X^T Qa)_j, and so on.  With Xq = scale tril_strict(do v'^T)
// (its diagonal d_i apart), Y = beta_i dA_ij and, per key dim:
//
//   dq = scale (do h^T) e^G + L(Xq, k) + d_i k_i
//   dk = (v' dhn^T) e^(G_L - G) + R(Xq, q) + d_i q_i + beta e^G dkb + L(Y, k) + R(Y, k)
//   dG = scale (do h^T) q e^G + q L(Xq, k) - k R(Xq, q) - (v' dhn^T) kg + dkb kb + k L(Y, k) - k R(Y, k)
//        (+ on the last token, per key: the kg terms of the other rows and e^(G_L) sum_v h dhn)
//   dg = the reverse cumsum of dG over the chunk, per key column
//
// with dkb, dvb, dA and dv as in bwd_chunk_mma.cu.  dG accumulates in registers,
// each warp over its own [C x K] elements, and goes through shared memory once
// for the cumsum.  A chunk whose gate moves further than kExpSafe from its
// middle row sets its flag and writes nothing: the CUDA-core stages then
// recompute that chunk exactly (they skip every chunk whose flag is clear).
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
constexpr float kExpSafe = 40.f;

template <int K, int V, int C>
struct KdaChunkLayout {
    static constexpr int LK = K + 8, LV = V + 8, LC = C + 8;
    static constexpr uint32_t rq = 0;                              // Qa; later k, then Ka
    static constexpr uint32_t rk = rq + C * LK * 2;                // Kb
    static constexpr uint32_t rdo = rk + C * LK * 2;               // do; later v
    static constexpr uint32_t rvp = rdo + C * LV * 2;              // v'; later u
    static constexpr uint32_t rdv = rvp + C * LV * 2;              // dv'
    static constexpr uint32_t rh = rdv + C * LV * 2;               // h [K][V]; later dkb (+ T); then dG fp32
    static constexpr uint32_t rdh = rh + K * LV * 2;               // dhn [K][V]; later dvb (+ w)
    static constexpr uint32_t rw = rdh + K * LV * 2;               // dw [C][K]
    static constexpr uint32_t rx = rw + C * LK * 2;                // Xq
    static constexpr uint32_t ry = rx + C * LC * 2;                // Y
    static constexpr uint32_t re = ry + C * LC * 2;                // E [C][K] bf16
    static constexpr uint32_t rf = re + C * LK * 2;                // fp32 rows and key vectors
    static constexpr uint32_t nf = 4 * C + 5 * K;
    static constexpr bool kTinH = K * LV * 2 >= C * LK * 2 + C * LC * 2;
    static constexpr bool kWinDH = K * LV * 2 >= C * LV * 2 + C * LK * 2;
    static constexpr uint32_t rextra = rf + nf * 4;
    static constexpr uint32_t rt = kTinH ? rh + C * LK * 2 : rextra;
    static constexpr uint32_t rw2 = kWinDH ? rdh + C * LV * 2 : rextra + (kTinH ? 0 : C * LC * 2);
    static constexpr uint32_t bytes = rextra + (kTinH ? 0 : C * LC * 2) + (kWinDH ? 0 : C * LK * 2);
    static_assert(C * LK <= K * LV, "dkb fits over h");
    static_assert(C * K * 4 <= 2 * K * LV * 2, "the dG tile fits over h and dhn");
    static_assert(bytes <= 227 * 1024, "shared memory");
};

template <int K, int V, int C>
__global__ void __launch_bounds__(kThreads, 1)
bwd_chunk_kda_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v,
                     const bf16* __restrict__ beta, const float* __restrict__ g_cum, const bf16* __restrict__ w,
                     const bf16* __restrict__ u, const bf16* __restrict__ tinv, const bf16* __restrict__ v_new,
                     const bf16* __restrict__ h_ckpt, const bf16* __restrict__ d_o, const bf16* __restrict__ dv_new,
                     const bf16* __restrict__ dh_ckpt, bf16* __restrict__ dq, bf16* __restrict__ dk,
                     bf16* __restrict__ dv, bf16* __restrict__ dbeta, float* __restrict__ dg,
                     int* __restrict__ exact_flags, int T, int H, int G, float scale) {
    using L = KdaChunkLayout<K, V, C>;
    constexpr int LK = L::LK, LV = L::LV, LC = L::LC;
    constexpr int RB = C / 16, CG = 8 / RB;
    constexpr int NK = K / 16 / CG, NV = V / 16 / CG;
    constexpr int NCB = C / 16, NC = NCB >= CG ? NCB / CG : 1;
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
    bf16* Es = reinterpret_cast<bf16*>(sm + L::re);
    float* sB = reinterpret_cast<float*>(sm + L::rf);   // beta [C]
    float* sdB = sB + C;                                // dbeta [C]
    float* sDiag = sdB + C;                             // scale do_i . v'_i [C]
    float* sGref = sDiag + C;                           // G_ref [K]
    float* sEref = sGref + K;                           // e^(G_ref) [K]
    float* sEgl = sEref + K;                            // e^(G_L - G_ref) [K]
    float* sHdh = sEgl + K;                             // sum_v h dhn [K]
    float* sTcol = sHdh + K;                            // sum over other rows of dkg kg [K]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, q4 = lane & 3, mi = lane >> 3, mr = lane & 7;
    const int rb = warp % RB, cg = warp / RB;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int NT = (T + C - 1) / C;
    const int t0 = c * C, nv = min(C, T - t0);
    const int64_t tok0 = ((int64_t)b * T + t0) * H + h;
    const int Hk = H / G;
    const int64_t ktok0 = ((int64_t)b * T + t0) * Hk + h / G;
    const int64_t st_off = (((int64_t)b * NT + c) * H + h);
    const int ref = min(C / 2, nv - 1);
    auto Grow = [&](int r) { return g_cum + (tok0 + (int64_t)min(r, nv - 1) * H) * K; };   // G past T: last row

    // ---- the gate around the middle row; a chunk it cannot keep bounded goes to the exact stages
    for (int d = tid; d < K; d += kThreads) {
        const float gref = Grow(ref)[d], gl = Grow(nv - 1)[d];
        sGref[d] = gref;
        sEref[d] = __expf(gref);
        sEgl[d] = __expf(gl - gref);
        sHdh[d] = 0.f;
        sTcol[d] = 0.f;
    }
    for (int i = tid; i < C; i += kThreads) {
        sB[i] = i < nv ? __bfloat162float(beta[tok0 + (int64_t)i * H]) : 0.f;
        sdB[i] = 0.f;
    }
    __syncthreads();
    {
        bool big = false;
        // eight elements per step, the 16-byte loads of all steps issued before any is used
        constexpr int N8 = C * K / 8 / kThreads;
        float4 g8[N8][2];
#pragma unroll
        for (int j = 0; j < N8; ++j) {
            const int e = 8 * (tid + kThreads * j), r = e / K, d = e % K;
            const float4* src = reinterpret_cast<const float4*>(Grow(r) + d);
            g8[j][0] = src[0];
            g8[j][1] = src[1];
        }
#pragma unroll
        for (int j = 0; j < N8; ++j) {
            const int e = 8 * (tid + kThreads * j), r = e / K, d = e % K;
            const float gv[8] = {g8[j][0].x, g8[j][0].y, g8[j][0].z, g8[j][0].w,
                                 g8[j][1].x, g8[j][1].y, g8[j][1].z, g8[j][1].w};
            __nv_bfloat162 ev[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float d0 = gv[2 * m] - sGref[d + 2 * m], d1 = gv[2 * m + 1] - sGref[d + 2 * m + 1];
                big |= fabsf(d0) > kExpSafe || fabsf(d1) > kExpSafe;
                ev[m] = __floats2bfloat162_rn(__expf(d0), __expf(d1));
            }
            *reinterpret_cast<uint4*>(Es + r * LK + d) = *reinterpret_cast<const uint4*>(ev);
        }
        if (__syncthreads_or(big)) {
            if (tid == 0) exact_flags[st_off] = 1;
            return;
        }
        if (tid == 0) exact_flags[st_off] = 0;
    }

    // ---- phase 1 tiles, in the order the products need them
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
    const int ck = cg * NK, cv = cg * NV, cc = cg * NC;
    const bool cc_active = cc < NCB;
    auto E = [&](int r, int d) { return bf(Es + r * LK + d); };

    float accQ[NK][2][4], accK[NK][2][4], accG[NK][2][4], tmp[NK][2][4];
    float br[2] = {0.f, 0.f};   // dbeta's partial sums for rows 16 rb + g4 and + 8, reduced once at the end
    auto f2 = [](const float* p) { return *reinterpret_cast<const float2*>(p); };
    cp_async_wait<2>();
    __syncthreads();
    zero(accQ);
    wgemm<NK, V, false, true>(accQ, aDO, LV, aH, LV, rb, ck, mi, mr);        // do h^T
    cp_async_wait<1>();
    __syncthreads();
    zero(accK);
    wgemm<NK, V, false, true>(accK, aVP, LV, aDH, LV, rb, ck, mi, mr);       // v' dhn^T
    if (cc_active) {
        // Xq = scale (do v'^T), strictly lower, with its diagonal apart (the gates live in Qa, Kb, E)
        float xq[NC][2][4];
        zero(xq);
        wgemm<NC, V, false, true>(xq, aDO, LV, aVP, LV, rb, cc, mi, mr);
        each2(xq, rb, cc, g4, q4, [&](int r, int col, float& x0, float& x1) {
            const float y0 = scale * x0, y1 = scale * x1;
            if (col == r) sDiag[r] = y0;
            if (col + 1 == r) sDiag[r] = y1;
            st_bf2(Xs + r * LC + col, col < r ? y0 : 0.f, col + 1 < r ? y1 : 0.f);
        });
    }
    cp_async_wait<0>();
    __syncthreads();
    // Qa = q E over q, Kb = k / E over k, eight elements at a time
    for (int i = tid; i < C * (K / 8); i += kThreads) {
        const int off = (i / (K / 8)) * LK + 8 * (i % (K / 8));
        uint4 qv = *reinterpret_cast<const uint4*>(Qs + off), kv = *reinterpret_cast<const uint4*>(Ks + off);
        const uint4 ev = *reinterpret_cast<const uint4*>(Es + off);
        __nv_bfloat162* qp = reinterpret_cast<__nv_bfloat162*>(&qv);
        __nv_bfloat162* kp = reinterpret_cast<__nv_bfloat162*>(&kv);
        const __nv_bfloat162* ep = reinterpret_cast<const __nv_bfloat162*>(&ev);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float2 e = __bfloat1622float2(ep[m]), a = __bfloat1622float2(qp[m]), c2 = __bfloat1622float2(kp[m]);
            qp[m] = __floats2bfloat162_rn(a.x * e.x, a.y * e.y);
            kp[m] = __floats2bfloat162_rn(__fdividef(c2.x, e.x), __fdividef(c2.y, e.y));
        }
        *reinterpret_cast<uint4*>(Qs + off) = qv;
        *reinterpret_cast<uint4*>(Ks + off) = kv;
    }
    // sum_v h dhn per key row
    {
        constexpr int TPR = kThreads / K;                       // threads per key row
        const int d = tid / TPR, part = tid % TPR;
        float s = 0.f;
        for (int x = part * (V / TPR); x < (part + 1) * (V / TPR); x += 8) {
            const uint4 a = *reinterpret_cast<const uint4*>(Hs + d * LV + x);
            const uint4 e = *reinterpret_cast<const uint4*>(DHs + d * LV + x);
            const uint32_t av[4] = {a.x, a.y, a.z, a.w}, ev[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
            for (int m = 0; m < 4; ++m)
                s += __uint_as_float(av[m] << 16) * __uint_as_float(ev[m] << 16) +
                     __uint_as_float(av[m] & 0xffff0000u) * __uint_as_float(ev[m] & 0xffff0000u);
        }
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (part == 0) sHdh[d] = s;
    }
    // dw = -dv' h^T -> bf16 tile
    zero(tmp);
    wgemm<NK, V, false, true>(tmp, aDV, LV, aH, LV, rb, ck, mi, mr);
    each2(tmp, rb, ck, g4, q4, [&](int r, int col, float& x0, float& x1) { st_bf2(DWs + r * LK + col, -x0, -x1); });
    __syncthreads();   // Qa, Kb formed
    // accQ = scale dqg e^(G_ref): times E it is dq's e^G part, times Qa its gate term; phase 2 adds
    // Xq Kb, which goes the same two ways
    each2(accQ, rb, ck, g4, q4, [&](int r, int col, float& x0, float& x1) {
        const float2 er = f2(sEref + col);
        x0 *= scale * er.x;
        x1 *= scale * er.y;
    });
    // dk's e^(G_L - G) part from dkg (kg = k e^(G_L - G) = Kb e^(G_L - G_ref)); the last row takes the
    // other rows' kg gate terms, per key column (its own cancels)
#pragma unroll
    for (int j = 0; j < NK; ++j)
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            float cs0 = 0.f, cs1 = 0.f;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int r = 16 * rb + g4 + 8 * h2, col = 16 * (ck + j) + 8 * n + 2 * q4, e = 2 * h2;
                const float x0 = accK[j][n][e], x1 = accK[j][n][e + 1];
                const float2 kb = bf2(Ks + r * LK + col), ev = bf2(Es + r * LK + col), egl = f2(sEgl + col);
                const float t0 = r == nv - 1 ? 0.f : x0 * kb.x * egl.x;
                const float t1 = r == nv - 1 ? 0.f : x1 * kb.y * egl.y;
                accG[j][n][e] = -t0;                                           // dG's first terms
                accG[j][n][e + 1] = -t1;
                cs0 += t0;
                cs1 += t1;
                accK[j][n][e] = __fdividef(x0 * egl.x, ev.x);
                accK[j][n][e + 1] = __fdividef(x1 * egl.y, ev.y);
            }
            // a column's 16 rows sit in the 8 lanes that share q4
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                cs0 += __shfl_xor_sync(0xffffffffu, cs0, o);
                cs1 += __shfl_xor_sync(0xffffffffu, cs1, o);
            }
            if (g4 == 0) {
                const int col = 16 * (ck + j) + 8 * n + 2 * q4;
                atomicAdd(sTcol + col, cs0);
                atomicAdd(sTcol + col + 1, cs1);
            }
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
    wgemm<NK, C, false, false>(accQ, aX, LC, aK, LK, rb, ck, mi, mr);     // + Xq Kb
    each2_at<NK>(rb, ck, g4, q4, [&](int j, int n, int e, int r, int col) {
        const float x0 = accQ[j][n][e], x1 = accQ[j][n][e + 1];
        const float2 qa = bf2(Qs + r * LK + col), kb = bf2(Ks + r * LK + col), ev = bf2(Es + r * LK + col);
        accG[j][n][e] += qa.x * x0;                                           // (dqg e^G + L) q
        accG[j][n][e + 1] += qa.y * x1;
        // dq done: E (scale dqg e^(G_ref) + Xq Kb) + d_i k_i (k = Kb E)
        st_bf2(DQs + r * LK + col, ev.x * (x0 + sDiag[r] * kb.x), ev.y * (x1 + sDiag[r] * kb.y));
    });
    zero(tmp);
    wgemm<NK, C, true, false>(tmp, aX, LC, aQ, LK, rb, ck, mi, mr);       // Xq^T Qa
    each2_at<NK>(rb, ck, g4, q4, [&](int j, int n, int e, int r, int col) {
        const float x0 = tmp[j][n][e], x1 = tmp[j][n][e + 1];
        const float2 qa = bf2(Qs + r * LK + col), kb = bf2(Ks + r * LK + col), ev = bf2(Es + r * LK + col);
        accG[j][n][e] -= kb.x * x0;                                           // k R = Kb (Xq^T Qa)
        accG[j][n][e + 1] -= kb.y * x1;
        accK[j][n][e] += __fdividef(x0 + sDiag[r] * qa.x, ev.x);              // R + d_i q_i (q = Qa / E)
        accK[j][n][e + 1] += __fdividef(x1 + sDiag[r] * qa.y, ev.y);
    });
    __syncthreads();
    store_tile<K, kThreads>(dq + tok0 * K, (int64_t)H * K, DQs, nv, tid);
    // k again, over Qa, for Ka = k E
    load_tile<K, kThreads>(Qs, k + ktok0 * K, (int64_t)Hk * K, C, nv, tid);
    cp_async_commit();

    // ---- phase 3: the WY backward
    bf16* DKBs = Hs;
    bf16* DVBs = DHs;
    cp_async_wait<1>();
    __syncthreads();   // the WY tiles landed; dq's staging has been read
    const uint32_t aT = smem_addr(Ts), aW = smem_addr(Ws), aU = smem_addr(Us);
    // dvb = T^T dv': dv = beta dvb (needs no Ka: it covers the k reload)
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
    zero(tmp);
    wgemm<NK, C, true, false>(tmp, aT, LC, aDW, LK, rb, ck, mi, mr);      // dkb = T^T dw
    cp_async_wait<0>();
    __syncthreads();
    // Ka = k E in place, eight elements at a time
    for (int i = tid; i < C * (K / 8); i += kThreads) {
        const int off = (i / (K / 8)) * LK + 8 * (i % (K / 8));
        uint4 kv = *reinterpret_cast<const uint4*>(Qs + off);
        const uint4 ev = *reinterpret_cast<const uint4*>(Es + off);
        __nv_bfloat162* kp = reinterpret_cast<__nv_bfloat162*>(&kv);
        const __nv_bfloat162* ep = reinterpret_cast<const __nv_bfloat162*>(&ev);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float2 e = __bfloat1622float2(ep[m]), a = __bfloat1622float2(kp[m]);
            kp[m] = __floats2bfloat162_rn(a.x * e.x, a.y * e.y);
        }
        *reinterpret_cast<uint4*>(Qs + off) = kv;
    }
    __syncthreads();
    // dkb's epilogue: dk += beta e^G dkb, dbeta += dkb . k e^G, dG += dkb kb (k e^G = Ka e^(G_ref))
    each2_at<NK>(rb, ck, g4, q4, [&](int j, int n, int e, int r, int col) {
        const float x0 = tmp[j][n][e], x1 = tmp[j][n][e + 1];
        const float2 ka = bf2(Qs + r * LK + col), ev = bf2(Es + r * LK + col), er = f2(sEref + col);
        const float keg0 = ka.x * er.x, keg1 = ka.y * er.y;
        br[(r >> 3) & 1] += x0 * keg0 + x1 * keg1;
        accG[j][n][e] += x0 * sB[r] * keg0;
        accG[j][n][e + 1] += x1 * sB[r] * keg1;
        accK[j][n][e] += sB[r] * ev.x * er.x * x0;
        accK[j][n][e + 1] += sB[r] * ev.y * er.y * x1;
        st_bf2(DKBs + r * LK + col, x0, x1);
    });
    __syncthreads();
    const uint32_t aKa = aQ;
    // dA = strict_lower(-(dkb w^T + dvb u^T)); dbeta's A term against M = Ka Kb^T; Y = beta dA
    if (cc_active) {
        float da[NC][2][4], m[NC][2][4];
        zero(da);
        zero(m);
        wgemm<NC, K, false, true>(da, smem_addr(DKBs), LK, aW, LK, rb, cc, mi, mr);
        wgemm<NC, V, false, true>(da, smem_addr(DVBs), LV, aU, LV, rb, cc, mi, mr);
        wgemm<NC, K, false, true>(m, aKa, LK, aK, LK, rb, cc, mi, mr);
        each2_at<NC>(rb, cc, g4, q4, [&](int j, int n, int e, int r, int col) {
            const float a0 = col < r ? -da[j][n][e] : 0.f, a1 = col + 1 < r ? -da[j][n][e + 1] : 0.f;
            br[(r >> 3) & 1] += a0 * m[j][n][e] + a1 * m[j][n][e + 1];
            st_bf2(Ys + r * LC + col, sB[r] * a0, sB[r] * a1);
        });
    }
    __syncthreads();
    zero(tmp);
    wgemm<NK, C, false, false>(tmp, aY, LC, aK, LK, rb, ck, mi, mr);      // Y Kb
    each2_at<NK>(rb, ck, g4, q4, [&](int j, int n, int e, int r, int col) {
        const float x0 = tmp[j][n][e], x1 = tmp[j][n][e + 1];
        const float2 ka = bf2(Qs + r * LK + col), ev = bf2(Es + r * LK + col);
        accK[j][n][e] += ev.x * x0;                                           // L(Y, k)
        accK[j][n][e + 1] += ev.y * x1;
        accG[j][n][e] += ka.x * x0;                                           // k L(Y, k) = Ka (Y Kb)
        accG[j][n][e + 1] += ka.y * x1;
    });
    zero(tmp);
    wgemm<NK, C, true, false>(tmp, aY, LC, aKa, LK, rb, ck, mi, mr);      // Y^T Ka
    bf16* DKS = Hs;   // dk staged over the dead dkb for 16-byte row stores
    each2_at<NK>(rb, ck, g4, q4, [&](int j, int n, int e, int r, int col) {
        const float x0 = tmp[j][n][e], x1 = tmp[j][n][e + 1];
        const float2 kb = bf2(Ks + r * LK + col), ev = bf2(Es + r * LK + col);
        accG[j][n][e] -= kb.x * x0;                                           // k R(Y, k) = Kb (Y^T Ka)
        accG[j][n][e + 1] -= kb.y * x1;
        st_bf2(DKS + r * LK + col, accK[j][n][e] + __fdividef(x0, ev.x),        // + R(Y, k): dk done
               accK[j][n][e + 1] + __fdividef(x1, ev.y));
    });
    row_add(sdB + 16 * rb + g4, br[0], q4);
    row_add(sdB + 16 * rb + g4 + 8, br[1], q4);
    __syncthreads();
    store_tile<K, kThreads>(dk + tok0 * K, (int64_t)H * K, DKS, nv, tid);
    __syncthreads();   // dk's staging read before dG goes over it

    // ---- phase 4: dG through shared memory, the last row's terms, the reverse cumsum per key column
    float* dGs = reinterpret_cast<float*>(sm + L::rh);                    // [C][K] fp32 over dead h and dhn
    each2(accG, rb, ck, g4, q4, [&](int r, int col, float& x0, float& x1) {
        *reinterpret_cast<float2*>(dGs + r * K + col) = make_float2(x0, x1);
    });
    __syncthreads();
    for (int d = tid; d < K; d += kThreads) {
        dGs[(nv - 1) * K + d] += sTcol[d] + sEgl[d] * sEref[d] * sHdh[d];  // e^(G_L) = e^(G_L - G_ref) e^(G_ref)
        float run = 0.f;
        for (int i = C - 1; i >= 0; --i) {
            run += dGs[i * K + d];
            if (i < nv) dg[(tok0 + (int64_t)i * H) * K + d] = run;
        }
    }
    if (tid < nv) dbeta[tok0 + (int64_t)tid * H] = __float2bfloat16_rn(sdB[tid]);
}

template <int K, int V, int C>
cudaError_t launch(const Dims& d, const void* q, const void* k, const void* v, const void* beta, const float* g_cum,
                   const void* w, const void* u, const void* tinv, const void* v_new, const void* h_ckpt,
                   const void* d_o, const void* dv_new, const void* dh_ckpt, void* dq, void* dk, void* dv,
                   void* dbeta, float* dg, int* flags, cudaStream_t s) {
    using L = KdaChunkLayout<K, V, C>;
    auto kern = bwd_chunk_kda_kernel<K, V, C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
    if (e != cudaSuccess) return e;
    const dim3 grid(d.NT, d.H, d.B);
    kern<<<grid, kThreads, L::bytes, s>>>((const bf16*)q, (const bf16*)k, (const bf16*)v, (const bf16*)beta, g_cum,
                                          (const bf16*)w, (const bf16*)u, (const bf16*)tinv, (const bf16*)v_new,
                                          (const bf16*)h_ckpt, (const bf16*)d_o, (const bf16*)dv_new,
                                          (const bf16*)dh_ckpt, (bf16*)dq, (bf16*)dk, (bf16*)dv, (bf16*)dbeta, dg,
                                          flags, d.T, d.H, d.G, d.scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t mma_bwd_chunk_kda(const Dims& d, const void* q, const void* k, const void* v, const void* beta,
                              const float* g_cum, const void* w, const void* u, const void* tinv, const void* v_new,
                              const void* h_ckpt, const void* d_o, const void* dv_new, const void* dh_ckpt, void* dq,
                              void* dk, void* dv, void* dbeta, float* dg, int* exact_flags, cudaStream_t s) {
    if (!d.bf16 || !d.per_k) return cudaErrorInvalidValue;
#define GDR_KDA_ARGS d, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new, dh_ckpt, dq, dk, dv, dbeta, dg, \
                     exact_flags, s
    if (d.C == 32) {
        if (d.K == 64 && d.V == 64) return launch<64, 64, 32>(GDR_KDA_ARGS);
        if (d.K == 64 && d.V == 128) return launch<64, 128, 32>(GDR_KDA_ARGS);
        if (d.K == 128 && d.V == 64) return launch<128, 64, 32>(GDR_KDA_ARGS);
        return launch<128, 128, 32>(GDR_KDA_ARGS);
    }
    if (d.K == 64 && d.V == 64) return launch<64, 64, 64>(GDR_KDA_ARGS);
    if (d.K == 64 && d.V == 128) return launch<64, 128, 64>(GDR_KDA_ARGS);
    if (d.K == 128 && d.V == 64) return launch<128, 64, 64>(GDR_KDA_ARGS);
    return launch<128, 128, 64>(GDR_KDA_ARGS);
#undef GDR_KDA_ARGS
}

}  // namespace gdr
