// The backward's per-chunk stage for bf16 io, a scalar gate and 64-token chunks,
// fed by TMA: the same arithmetic as bwd_chunk_mma.cu (the pages' wy_dqkg,
// "kernel_fun/kda/_kernels/bwd_scan.py", host wrapper), with every tile in the
// 128-byte swizzle so that a [rows x D] tile is D / 64 TMA boxes instead of
// rows x D / 8 per-thread copies.
//
// A persistent CTA of eight warps per SM walks the (chunk, head, batch) items.
// Each tile load goes into a region that is dead by the time it is issued, so the
// next item's loads overlap this item's work:
//   the next item's q                   once the WY phase starts (q is dead),
//   its do and dv'                      once dvb is formed (v and dv' are dead),
//   its v', dh_next and h               once dA is formed (u, dvb, w and dkb are dead),
//   its k                               at the top of its own iteration,
//   this item's T, w, v, u              after phase 1 (over the dead h and dh_next),
// each group on an mbarrier that thread 0 arms with the group's bytes and then
// fills with TMA boxes.  Phase 1 runs every product that needs no k while k
// lands.  dk is staged over the dead dw.  Tokens past T are the boxes' zero fill.
// The next item's gate rows and beta are read into registers one item ahead too.
//
// The rest follows bwd_chunk_mma.cu: warp w owns the 16-row block w % 4 and the
// column half w / 4 of every [C x D] result; epilogues work on column pairs; the
// row sums of dG and dbeta stay in registers until one reduction; dq and dk leave
// through shared memory as 16-byte row stores; the reverse cumsum is a warp scan.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "blackwell.cuh"
#include "chunk_mma.cuh"
#include "gdr_internal.h"
#include "tma_host.h"
#include "warp_mma.cuh"

namespace gdr {
namespace {

using bf16 = __nv_bfloat16;
using namespace cm;
constexpr int kThreads = 256;
constexpr int C = 64;

// Byte offset of element (r, c) of a tile of R rows stored as 64-column atoms with the 128-byte swizzle
// (the layout a TMA box of 64 columns x R rows writes).
template <int R>
__device__ __forceinline__ uint32_t so(int r, int c) {
    return (uint32_t)((c >> 6) * R * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}

// acc[j] += opA(rows 16 rb .., all kd) opB(all kd, cols 16 (cb0 + j) ..), both operands swizzled tiles.
// A: [M][KD] of RA rows, or (AT) stored as [KD][M] of RA = KD rows.  B: [KD][N] of RB = KD rows, or (BT)
// stored as [N][KD] of RB = N rows.  Eight consecutive rows at one 16-byte column: conflict-free.
template <int NCW, int KD, bool AT, bool BT, int RA, int RB>
__device__ __forceinline__ void sgemm(float (&acc)[NCW][2][4], uint32_t A, uint32_t B, int rb, int cb0, int mi,
                                      int mr) {
#pragma unroll
    for (int k0 = 0; k0 < KD; k0 += 16) {
        uint32_t a[4];
        if constexpr (AT) wm::ldsm_x4_t(A + so<RA>(k0 + 8 * (mi >> 1) + mr, 16 * rb + 8 * (mi & 1)), a);
        else wm::ldsm_x4(A + so<RA>(16 * rb + 8 * (mi & 1) + mr, k0 + 8 * (mi >> 1)), a);
#pragma unroll
        for (int j = 0; j < NCW; ++j) {
            const int n0 = 16 * (cb0 + j);
            uint32_t bb[4];
            if constexpr (BT) wm::ldsm_x4(B + so<RB>(n0 + 8 * (mi >> 1) + mr, k0 + 8 * (mi & 1)), bb);
            else wm::ldsm_x4_t(B + so<RB>(k0 + 8 * (mi & 1) + mr, n0 + 8 * (mi >> 1)), bb);
            wm::mma16816(acc[j][0], a, bb[0], bb[1]);
            wm::mma16816(acc[j][1], a, bb[2], bb[3]);
        }
    }
}

constexpr uint32_t al1k(uint32_t x) { return (x + 1023u) & ~1023u; }

template <int K, int V>
struct TmaChunkLayout {
    static constexpr uint32_t kCK = C * K * 2, kCV = C * V * 2, kKV = K * V * 2, kCC = C * C * 2;
    static constexpr uint32_t rq = 0;                 // q
    static constexpr uint32_t rk = rq + kCK;          // k
    static constexpr uint32_t rdo = rk + kCK;         // do; later v
    static constexpr uint32_t rvp = rdo + kCV;        // v'; later u
    static constexpr uint32_t rdv = rvp + kCV;        // dv'
    static constexpr uint32_t rh = rdv + kCV;         // h [K][V]; later dq's staging, dkb (+ T)
    static constexpr uint32_t rdh = rh + kKV;         // dh_next [K][V]; later dvb (+ w)
    static constexpr uint32_t rw = rdh + kKV;         // dw; later dk's staging
    static constexpr uint32_t rx = rw + kCK;          // Xq
    static constexpr uint32_t ry = rx + kCC;          // Y
    static constexpr uint32_t rf = ry + kCC;          // fp32 rows
    static constexpr bool kTinH = kKV >= kCK + kCC;
    static constexpr bool kWinDH = kKV >= kCV + kCK;
    static constexpr uint32_t rextra = al1k(rf + 8 * C * 4);
    static constexpr uint32_t rt = kTinH ? rh + kCK : rextra;
    static constexpr uint32_t rw2 = kWinDH ? rdh + kCV : rextra + (kTinH ? 0 : kCC);
    static constexpr uint32_t bytes = rextra + (kTinH ? 0 : kCC) + (kWinDH ? 0 : kCK);
    static_assert(kCK <= kKV, "dkb fits over h");
    static_assert(bytes + 1024 <= 227 * 1024, "shared memory");
};

struct Maps {
    CUtensorMap q, k, d_o, v_new, dv_new, h, dh, tinv, w, v, u;
};

template <int K, int V>
__global__ void __launch_bounds__(kThreads, 1)
bwd_chunk_tma_kernel(const __grid_constant__ Maps mp, const bf16* __restrict__ beta, const float* __restrict__ g_cum,
                     bf16* __restrict__ dq, bf16* __restrict__ dk, bf16* __restrict__ dv, bf16* __restrict__ dbeta,
                     float* __restrict__ dg, int B, int T, int H, int G, float scale, unsigned int* err) {
    using L = TmaChunkLayout<K, V>;
    constexpr int RB = C / 16, CG = 8 / RB;             // 16-row blocks; warps sharing each
    constexpr int NK = K / 16 / CG, NV = V / 16 / CG;   // 16-column blocks per warp
    constexpr int NC = C / 16 / CG;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(sm);
    auto tile = [&](uint32_t region) { return reinterpret_cast<bf16*>(sm + region); };
    // element (r, c) of a swizzled tile of R rows
    auto at = [](bf16* t, uint32_t off) { return reinterpret_cast<bf16*>(reinterpret_cast<unsigned char*>(t) + off); };
    bf16 *Qs = tile(L::rq), *Ks = tile(L::rk), *DOs = tile(L::rdo), *VPs = tile(L::rvp), *DVs = tile(L::rdv);
    bf16 *Hs = tile(L::rh), *DHs = tile(L::rdh), *DWs = tile(L::rw), *Xs = tile(L::rx), *Ys = tile(L::ry);
    float* sG = reinterpret_cast<float*>(sm + L::rf);
    float* sEG = sG + C;      // e^G
    float* sGam = sEG + C;    // e^(G_L - G)
    float* sB = sGam + C;     // beta
    float* sdG = sB + C;      // gate gradient per row
    float* sdB = sdG + C;     // dbeta per row
    float* sDiag = sdB + C;   // scale do_i . v'_i
    float* sS = sDiag + C;    // [0]: sum of dkg kg over the other rows, [1]: sum h dhn
    __shared__ uint64_t bars[5];   // q; do, dv'; v', dh_next, h; T, w, v, u; k

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, q4 = lane & 3, mi = lane >> 3, mr = lane & 7;
    const int rb = warp % RB, cg = warp / RB;
    const int NT = (T + C - 1) / C;
    const int n_items = NT * H * B;
    struct Item {
        int c, b, h, t0, nv;
        int64_t tok0;
    };
    auto item = [&](int wi) {   // item wi: chunk wi % NT of head (wi / NT) % H of batch wi / (NT H)
        Item it;
        it.c = wi % NT;
        const int r = wi / NT;
        it.h = r % H;
        it.b = r / H;
        it.t0 = it.c * C;
        it.nv = min(C, T - it.t0);
        it.tok0 = ((int64_t)it.b * T + it.t0) * H + it.h;
        return it;
    };
    // token tiles: D / 64 boxes of 64 columns x C tokens; checkpoint tiles: V / 64 boxes of 64 columns x K rows
    auto tok = [&](uint32_t region, const CUtensorMap* m, int D, int head, const Item& it, uint64_t* bar) {
        for (int a = 0; a < D / 64; ++a) bw::tma_load_4d(sm + region + a * C * 128, m, bar, a * 64, head, it.t0, it.b);
    };
    auto ckpt = [&](uint32_t region, const CUtensorMap* m, int rows, const Item& it, uint64_t* bar) {
        for (int a = 0; a < V / 64; ++a)
            bw::tma_load_4d(sm + region + a * rows * 128, m, bar, a * 64, 0, it.h, it.b * NT + it.c);
    };
    auto load_q = [&](const Item& it) {
        if (tid == 0) {
            bw::fence_async_shared();
            bw::mbar_arrive_expect_tx(&bars[0], L::kCK);
            tok(L::rq, &mp.q, K, it.h / G, it, &bars[0]);
        }
    };
    auto load_p1 = [&](const Item& it) {   // do, dv'
        if (tid == 0) {
            bw::fence_async_shared();
            bw::mbar_arrive_expect_tx(&bars[1], 2 * L::kCV);
            tok(L::rdo, &mp.d_o, V, it.h, it, &bars[1]);
            tok(L::rdv, &mp.dv_new, V, it.h, it, &bars[1]);
        }
    };
    auto load_p2 = [&](const Item& it) {   // v', dh_next, h
        if (tid == 0) {
            bw::fence_async_shared();
            bw::mbar_arrive_expect_tx(&bars[2], L::kCV + 2 * L::kKV);
            tok(L::rvp, &mp.v_new, V, it.h, it, &bars[2]);
            ckpt(L::rdh, &mp.dh, K, it, &bars[2]);
            ckpt(L::rh, &mp.h, K, it, &bars[2]);
        }
    };
    // the next item's gate values, one item ahead (thread i < C holds row i)
    float nG = 0.f, nGL = 0.f, nBeta = 0.f;
    auto load_gate = [&](const Item& it) {
        if (tid < C) {
            const int64_t g0 = (int64_t)it.b * T + it.t0;
            nG = g_cum[(g0 + min(tid, it.nv - 1)) * H + it.h];
            nGL = g_cum[(g0 + it.nv - 1) * H + it.h];
            nBeta = tid < it.nv ? __bfloat162float(beta[it.tok0 + (int64_t)tid * H]) : 0.f;
        }
    };

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) bw::mbar_init(&bars[i], 1);
        bw::fence_mbar_init();
    }
    __syncthreads();
    if ((int)blockIdx.x < n_items) {   // the first item's early loads, as a previous item would have issued them
        const Item it = item(blockIdx.x);
        load_q(it);
        load_p1(it);
        load_p2(it);
        load_gate(it);
    }
    uint32_t par = 0;   // the barriers' phase parity for this CTA's current item
    const uint32_t aQ = sbase + L::rq, aK = sbase + L::rk, aDO = sbase + L::rdo, aVP = sbase + L::rvp;
    const uint32_t aDV = sbase + L::rdv, aH = sbase + L::rh, aDH = sbase + L::rdh, aDW = sbase + L::rw;
    const uint32_t aX = sbase + L::rx, aY = sbase + L::ry;
    const int ck = cg * NK, cv = cg * NV, cc = cg * NC;   // this warp's first column block

    for (int wi = blockIdx.x; wi < n_items; wi += gridDim.x) {
        const Item it = item(wi);
        const int nv = it.nv;
        const int64_t tok0 = it.tok0;
        const bool has_next = wi + (int)gridDim.x < n_items;
        // the previous item is done with every region and row this one writes first; its generic accesses are
        // ordered before the async proxy's writes (each barrier that precedes a TMA issue has this fence)
        bw::fence_async_shared();
        __syncthreads();

        // ---- gate rows and beta (read one item ahead); this item's h and k
        if (tid < C) {
            sG[tid] = nG;
            sEG[tid] = __expf(nG);
            sGam[tid] = __expf(nGL - nG);
            sB[tid] = nBeta;
            sdG[tid] = 0.f;
            sdB[tid] = 0.f;
            if (tid < 2) sS[tid] = 0.f;
        }
        if (tid == 0) {
            bw::fence_async_shared();
            bw::mbar_arrive_expect_tx(&bars[4], L::kCK);
            tok(L::rk, &mp.k, K, it.h / G, it, &bars[4]);
        }

        float accQ[NK][2][4], accK[NK][2][4], tmp[NK][2][4];
        float gr[2] = {0.f, 0.f}, br[2] = {0.f, 0.f};   // row sums of dG and dbeta (rows 16 rb + g4, + 8)
        // every phase-1 product that needs no k: v' dhn^T, do v'^T, do h^T, dv' h^T (the prefetched tiles)
        {
            const bool ok = bw::mbar_wait(&bars[0], par, err, kDeviceErrTimeout) &&
                            bw::mbar_wait(&bars[1], par, err, kDeviceErrTimeout) &&
                            bw::mbar_wait(&bars[2], par, err, kDeviceErrTimeout);
            if (!__syncthreads_and(ok)) return;
        }
        zero(accK);
        sgemm<NK, V, false, true, C, K>(accK, aVP, aDH, rb, ck, mi, mr);    // dkg = v' dhn^T
        {
            // Xq = scale (do v'^T) Gam, strictly lower, with its diagonal apart
            float xq[NC][2][4];
            zero(xq);
            sgemm<NC, V, false, true, C, C>(xq, aDO, aVP, rb, cc, mi, mr);
            each2(xq, rb, cc, g4, q4, [&](int r, int col, float& x0, float& x1) {
                const float y0 = scale * x0, y1 = scale * x1;
                if (col == r) sDiag[r] = y0;
                if (col + 1 == r) sDiag[r] = y1;
                st_bf2(at(Xs, so<C>(r, col)), col < r ? y0 * __expf(sG[r] - sG[col]) : 0.f,
                       col + 1 < r ? y1 * __expf(sG[r] - sG[col + 1]) : 0.f);
            });
        }
        // dw = -dv' h^T -> bf16 tile
        zero(tmp);
        sgemm<NK, V, false, true, C, K>(tmp, aDV, aH, rb, ck, mi, mr);
        each2(tmp, rb, ck, g4, q4, [&](int r, int col, float& x0, float& x1) {
            st_bf2(at(DWs, so<C>(r, col)), -x0, -x1);
        });
        // dqg = do h^T; dq's e^G-scaled part and its gate term
        zero(accQ);
        sgemm<NK, V, false, true, C, K>(accQ, aDO, aH, rb, ck, mi, mr);
        each2(accQ, rb, ck, g4, q4, [&](int r, int col, float& x0, float& x1) {
            const float e = scale * sEG[r];
            const float2 qv = bf2(at(Qs, so<C>(r, col)));
            x0 *= e;
            x1 *= e;
            gr[(r >> 3) & 1] += x0 * qv.x + x1 * qv.y;
        });
        // sum h dhn, eight elements per step
        {
            float s = 0.f;
            for (int idx = tid; idx < K * V / 8; idx += kThreads) {
                const int d = idx / (V / 8), x = 8 * (idx % (V / 8));
                const uint4 a = *reinterpret_cast<const uint4*>(at(Hs, so<K>(d, x)));
                const uint4 e = *reinterpret_cast<const uint4*>(at(DHs, so<K>(d, x)));
                const uint32_t av[4] = {a.x, a.y, a.z, a.w}, ev[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    s += __uint_as_float(av[m] << 16) * __uint_as_float(ev[m] << 16) +
                         __uint_as_float(av[m] & 0xffff0000u) * __uint_as_float(ev[m] & 0xffff0000u);
            }
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) atomicAdd(sS + 1, s);
        }
        // k landed: dk's e^(G_L - G) part from dkg; the gate terms go to the rows, the last row takes their sum
        if (!__syncthreads_and(bw::mbar_wait(&bars[4], par, err, kDeviceErrTimeout))) return;
        {
            float tot = 0.f;
            each2(accK, rb, ck, g4, q4, [&](int r, int col, float& x0, float& x1) {
                const float2 kv = bf2(at(Ks, so<C>(r, col)));
                const float t = r == nv - 1 ? 0.f : (x0 * kv.x + x1 * kv.y) * sGam[r];
                gr[(r >> 3) & 1] -= t;
                tot += t;
                x0 *= sGam[r];
                x1 *= sGam[r];
            });
            for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
            if (lane == 0) atomicAdd(sS, tot);
        }
        bw::fence_async_shared();
        __syncthreads();
        // the WY phase's tiles, in flight during phase 2 (h, dhn, do and v' are dead now)
        bf16* Ws = tile(L::rw2);
        bf16* Vs = DOs;
        bf16* Ts = tile(L::rt);
        if (tid == 0) {
            bw::fence_async_shared();
            bw::mbar_arrive_expect_tx(&bars[3], L::kCC + L::kCK + 2 * L::kCV);
            for (int a = 0; a < C / 64; ++a)
                bw::tma_load_4d(sm + L::rt + a * C * 128, &mp.tinv, &bars[3], a * 64, 0, it.h, it.b * NT + it.c);
            tok(L::rw2, &mp.w, K, it.h, it, &bars[3]);
            tok(L::rdo, &mp.v, V, it.h, it, &bars[3]);
            tok(L::rvp, &mp.u, V, it.h, it, &bars[3]);
        }

        // ---- phase 2: the output scores' other factors
        bf16* DQs = Hs;   // dq staged over the dead h (later dkb's space) for 16-byte row stores
        zero(tmp);
        sgemm<NK, C, false, false, C, C>(tmp, aX, aK, rb, ck, mi, mr);      // Xq k
        each2_at<NK>(rb, ck, g4, q4, [&](int j, int n, int e, int r, int col) {
            const float x0 = tmp[j][n][e], x1 = tmp[j][n][e + 1];
            const float2 qv = bf2(at(Qs, so<C>(r, col))), kv = bf2(at(Ks, so<C>(r, col)));
            gr[(r >> 3) & 1] += qv.x * x0 + qv.y * x1;
            st_bf2(at(DQs, so<C>(r, col)), accQ[j][n][e] + x0 + sDiag[r] * kv.x,
                   accQ[j][n][e + 1] + x1 + sDiag[r] * kv.y);
        });
        zero(tmp);
        sgemm<NK, C, true, false, C, C>(tmp, aX, aQ, rb, ck, mi, mr);       // Xq^T q
        each2_at<NK>(rb, ck, g4, q4, [&](int j, int n, int e, int r, int col) {
            const float x0 = tmp[j][n][e], x1 = tmp[j][n][e + 1];
            const float2 qv = bf2(at(Qs, so<C>(r, col))), kv = bf2(at(Ks, so<C>(r, col)));
            gr[(r >> 3) & 1] -= kv.x * x0 + kv.y * x1;
            accK[j][n][e] += x0 + sDiag[r] * qv.x;
            accK[j][n][e + 1] += x1 + sDiag[r] * qv.y;
        });
        __syncthreads();
        for (int idx = tid; idx < nv * (K / 8); idx += kThreads) {   // dq: 16-byte row stores
            const int r = idx / (K / 8), c8 = 8 * (idx % (K / 8));
            *reinterpret_cast<uint4*>(dq + (tok0 + (int64_t)r * H) * K + c8) =
                *reinterpret_cast<const uint4*>(at(DQs, so<C>(r, c8)));
        }

        // ---- phase 3: the WY backward
        bf16* DKBs = Hs;
        bf16* DVBs = DHs;
        // the WY tiles landed; dq's staging has been read
        bw::fence_async_shared();
        if (!__syncthreads_and(bw::mbar_wait(&bars[3], par, err, kDeviceErrTimeout))) return;
        if (has_next) load_q(item(wi + gridDim.x));   // q is dead from here on
        const uint32_t aT = sbase + L::rt, aW = sbase + L::rw2, aU = sbase + L::rvp;
        // dkb = T^T dw
        zero(tmp);
        sgemm<NK, C, true, false, C, C>(tmp, aT, aDW, rb, ck, mi, mr);
        each2_at<NK>(rb, ck, g4, q4, [&](int j, int n, int e, int r, int col) {
            const float x0 = tmp[j][n][e], x1 = tmp[j][n][e + 1];
            const float2 kv = bf2(at(Ks, so<C>(r, col)));
            const float db = (x0 * kv.x + x1 * kv.y) * sEG[r];   // dkb . k e^G
            br[(r >> 3) & 1] += db;
            gr[(r >> 3) & 1] += db * sB[r];                       // dkb . kb
            st_bf2(at(DKBs, so<C>(r, col)), x0, x1);
            accK[j][n][e] += x0 * sB[r] * sEG[r];
            accK[j][n][e + 1] += x1 * sB[r] * sEG[r];
        });
        // dvb = T^T dv': dv = beta dvb
        {
            float tv[NV][2][4];
            zero(tv);
            sgemm<NV, C, true, false, C, C>(tv, aT, aDV, rb, cv, mi, mr);
            each2(tv, rb, cv, g4, q4, [&](int r, int col, float& x0, float& x1) {
                const float2 vv = bf2(at(Vs, so<C>(r, col)));
                br[(r >> 3) & 1] += x0 * vv.x + x1 * vv.y;
                st_bf2(at(DVBs, so<C>(r, col)), x0, x1);
                if (r < nv) st_bf2(dv + (tok0 + (int64_t)r * H) * V + col, sB[r] * x0, sB[r] * x1);
            });
        }
        bw::fence_async_shared();
        __syncthreads();
        if (has_next) load_p1(item(wi + gridDim.x));   // v and dv' are dead: the next do, dv' over them
        // dA = strict_lower(-(dkb w^T + dvb u^T)); dbeta's A term against M = Gam (k k^T); Y = beta dA Gam
        {
            float da[NC][2][4], m[NC][2][4];
            zero(da);
            zero(m);
            sgemm<NC, K, false, true, C, C>(da, sbase + L::rh, aW, rb, cc, mi, mr);
            sgemm<NC, V, false, true, C, C>(da, sbase + L::rdh, aU, rb, cc, mi, mr);
            sgemm<NC, K, false, true, C, C>(m, aK, aK, rb, cc, mi, mr);
            each2_at<NC>(rb, cc, g4, q4, [&](int j, int n, int e, int r, int col) {
                const float gam0 = col < r ? __expf(sG[r] - sG[col]) : 0.f;
                const float gam1 = col + 1 < r ? __expf(sG[r] - sG[col + 1]) : 0.f;
                const float a0 = -da[j][n][e], a1 = -da[j][n][e + 1];
                br[(r >> 3) & 1] += a0 * m[j][n][e] * gam0 + a1 * m[j][n][e + 1] * gam1;
                st_bf2(at(Ys, so<C>(r, col)), sB[r] * a0 * gam0, sB[r] * a1 * gam1);
            });
        }
        bw::fence_async_shared();
        __syncthreads();
        // v', dh_next, h (and the gate rows) of the next item: u, dvb, w and dkb are dead now
        if (has_next) {
            const Item nx = item(wi + gridDim.x);
            load_p2(nx);
            load_gate(nx);
        }
        // dk += Y k + Y^T k; their gate terms
        zero(tmp);
        sgemm<NK, C, false, false, C, C>(tmp, aY, aK, rb, ck, mi, mr);
        each2(tmp, rb, ck, g4, q4, [&](int r, int col, float& x0, float& x1) {
            const float2 kv = bf2(at(Ks, so<C>(r, col)));
            gr[(r >> 3) & 1] += kv.x * x0 + kv.y * x1;
        });
#pragma unroll
        for (int j = 0; j < NK; ++j)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) accK[j][n][e] += tmp[j][n][e];
        zero(tmp);
        sgemm<NK, C, true, false, C, C>(tmp, aY, aK, rb, ck, mi, mr);
        bf16* DKS = DWs;   // dk staged over the dead dw for 16-byte row stores
        each2_at<NK>(rb, ck, g4, q4, [&](int j, int n, int e, int r, int col) {
            const float x0 = tmp[j][n][e], x1 = tmp[j][n][e + 1];
            const float2 kv = bf2(at(Ks, so<C>(r, col)));
            gr[(r >> 3) & 1] -= kv.x * x0 + kv.y * x1;
            st_bf2(at(DKS, so<C>(r, col)), accK[j][n][e] + x0, accK[j][n][e + 1] + x1);
        });
        // the rows' partial sums of dG and dbeta, once
        row_add(sdG + 16 * rb + g4, gr[0], q4);
        row_add(sdG + 16 * rb + g4 + 8, gr[1], q4);
        row_add(sdB + 16 * rb + g4, br[0], q4);
        row_add(sdB + 16 * rb + g4 + 8, br[1], q4);
        __syncthreads();
        for (int idx = tid; idx < nv * (K / 8); idx += kThreads) {   // dk: 16-byte row stores
            const int r = idx / (K / 8), c8 = 8 * (idx % (K / 8));
            *reinterpret_cast<uint4*>(dk + (tok0 + (int64_t)r * H) * K + c8) =
                *reinterpret_cast<const uint4*>(at(DKS, so<C>(r, c8)));
        }

        // ---- phase 4: the last token's gate terms, the reverse cumsum (a warp's suffix scan), dbeta
        if (warp == 0) {
            const float last = sS[0] + __expf(sG[nv - 1]) * sS[1];
            float lo = sdG[lane] + (lane == nv - 1 ? last : 0.f);            // rows 0..31
            float hi = sdG[32 + lane] + (32 + lane == nv - 1 ? last : 0.f);  // rows 32..63
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
            if (32 + lane < nv) dg[tok0 + (int64_t)(32 + lane) * H] = hi;
        }
        if (tid < nv) dbeta[tok0 + (int64_t)tid * H] = __float2bfloat16_rn(sdB[tid]);
        par ^= 1u;
    }
}

template <int K, int V>
cudaError_t launch(const Dims& d, const void* q, const void* k, const void* v, const void* beta, const float* g_cum,
                   const void* w, const void* u, const void* tinv, const void* v_new, const void* h_ckpt,
                   const void* d_o, const void* dv_new, const void* dh_ckpt, void* dq, void* dk, void* dv,
                   void* dbeta, float* dg, cudaStream_t s, unsigned int* err) {
    using L = TmaChunkLayout<K, V>;
    Maps m;
    if (!make_tmap_tokens(&m.q, q, d.B, d.T, d.Hk, K, C) || !make_tmap_tokens(&m.k, k, d.B, d.T, d.Hk, K, C) ||
        !make_tmap_tokens(&m.d_o, d_o, d.B, d.T, d.H, V, C) || !make_tmap_tokens(&m.v_new, v_new, d.B, d.T, d.H, V, C) ||
        !make_tmap_tokens(&m.dv_new, dv_new, d.B, d.T, d.H, V, C) ||
        !make_tmap_ckpt(&m.h, h_ckpt, d.B, d.NT, d.H, K, V) || !make_tmap_ckpt(&m.dh, dh_ckpt, d.B, d.NT, d.H, K, V) ||
        !make_tmap_ckpt(&m.tinv, tinv, d.B, d.NT, d.H, C, C) || !make_tmap_tokens(&m.w, w, d.B, d.T, d.H, K, C) ||
        !make_tmap_tokens(&m.v, v, d.B, d.T, d.H, V, C) || !make_tmap_tokens(&m.u, u, d.B, d.T, d.H, V, C))
        return cudaErrorInvalidValue;
    auto kern = bwd_chunk_tma_kernel<K, V>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int64_t items = (int64_t)d.NT * d.H * d.B;
    const int grid = (int)(items < sms ? items : sms);
    kern<<<grid, kThreads, smem, s>>>(m, (const bf16*)beta, g_cum, (bf16*)dq, (bf16*)dk, (bf16*)dv, (bf16*)dbeta, dg,
                                      d.B, d.T, d.H, d.G, d.scale, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t mma_bwd_chunk_tma(const Dims& d, const void* q, const void* k, const void* v, const void* beta,
                              const float* g_cum, const void* w, const void* u, const void* tinv, const void* v_new,
                              const void* h_ckpt, const void* d_o, const void* dv_new, const void* dh_ckpt, void* dq,
                              void* dk, void* dv, void* dbeta, float* dg, cudaStream_t s, unsigned int* err) {
    if (!d.bf16 || d.per_k || d.C != C) return cudaErrorInvalidValue;
#define GDR_TMA_ARGS d, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new, dh_ckpt, dq, dk, dv, dbeta, dg, s, err
    if (d.K == 64 && d.V == 64) return launch<64, 64>(GDR_TMA_ARGS);
    if (d.K == 64 && d.V == 128) return launch<64, 128>(GDR_TMA_ARGS);
    if (d.K == 128 && d.V == 64) return launch<128, 64>(GDR_TMA_ARGS);
    return launch<128, 128>(GDR_TMA_ARGS);
#undef GDR_TMA_ARGS
}

}  // namespace gdr
