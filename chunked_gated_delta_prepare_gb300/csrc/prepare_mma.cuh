// WY prepare for bf16 and fp16 io ("Reuse P as beta
// tiles in gated deltanet fused prepare": the gated A, its inverse, w and u per
// chunk).
//
// One CTA of 128 threads per 64-token tile of one (batch, head): one chunk when
// C = 64, two when C = 32 (kept apart by the block-diagonal structure).  Warp I
// owns tile rows 16I .. 16I+15 ("block row I") of every matrix, in registers.
//
//   TMA      k [64 x K], v [64 x V]  -> shared memory (128-byte swizzle)
//   SIMT     G = chunk-local cumsum of g (written out as g_cum), beta
//   mma      S = k k^T            (per-key-dim gate: gated copies k*exp(G-G_ref)
//                                  and k*exp(G_ref-G), G_ref the chunk's middle row,
//                                  keep every factor bounded)
//   regs     A_ij = beta_i S_ij exp(G_i - G_j) (i > j, same chunk), in S's fragments
//   solve    X = (I+A)^{-1} by blocks of 16: each warp inverts its diagonal block
//            in fp32, then level by level (distance from the diagonal)
//                X_IJ = -X_II sum_{M=J}^{I-1} A_IM X_MJ
//            on mma.sync with every operand split into bf16 hi + lo parts
//            (hi*hi + hi*lo + lo*hi: about 16 bits of mantissa, fp32-like), only
//            the 16 x 16 X blocks passing through shared memory
//   mma      w = (X diag(beta exp(G))) k,  u = (X diag(beta)) v   (scalar gate)
//            w = (X diag(beta)) (k * exp(G)), u as above       (per-key-dim gate)
//            each warp skipping the k-steps where its row of X is zero
//
// The products are warp-level mma.sync m16n8k16 (bf16 or fp16 in, fp32 accumulate)
// fed by ldmatrix from the swizzled tiles, or, for S and P, tcgen05 with the
// accumulators in tensor memory (UMMA below).  Measured on the 32k-token,
// 32-head workload (the prepare alone over the whole GPU / the overlapped
// forward): every product on mma.sync 0.386 / 0.799 ms; S and P on tcgen05
// 0.392 / 0.786 ms; S, P, w and u on tcgen05 0.409 / 0.797 ms.  At three CTAs
// per SM a tile is latency-bound: tcgen05 shortens S and P (the warps wait for
// one product instead of issuing up to 64 mma each), but w and u each add a
// round trip and a second pass through the same 128 TMEM columns.
// beta (and, for a scalar gate, exp(G)) is folded into the columns of X, so k
// and v feed the MMA as TMA left them.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

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
    // SPLITG (per-key-dim gate, K = V = 128): G passes through a [64][64] half tile, one half of the keys
    // at a time; k e^G is written over k as the gated copies are made; v lands in Kb's place once S is
    // formed; the solve's scratch takes the dead Ka and G-half tiles.  67 KB: three CTAs per SM.
    static constexpr bool SPLITG = PER_K && K == 128 && V == 128;
    static constexpr uint32_t kK = 0;                               // k tile [64][K] (SPLITG: then k exp(G))
    static constexpr uint32_t kKb0 = kK + K * 128;                  // SPLITG: Kb, then v
    static constexpr uint32_t kV = SPLITG ? kKb0 : kK + K * 128;   // v tile [64][V]
    static constexpr uint32_t kQ = kV + (SPLITG ? K * 128 : V * 128);   // q tile [64][K] (with P)
    static constexpr uint32_t kKa = kQ + (WITH_P ? K * 128 : 0);    // KDA: gated k copies
    static constexpr uint32_t kKb = SPLITG ? kKb0 : kKa + (PER_K ? K * 128 : 0);
    static constexpr uint32_t kGh = kKa + (PER_K ? K * 128 : 0);    // SPLITG: G half [64][64] fp32
    static constexpr uint32_t kF = SPLITG ? kGh + 64 * 64 * 4 : kKb + (PER_K ? K * 128 : 0);   // fp32 / block scratch
    // byte offsets from kF
    static constexpr uint32_t fG = 0;                                // G [64][GW] fp32 (SPLITG: in the half tile)
    static constexpr uint32_t fB = fG + (SPLITG ? 0 : 64 * GW * 4);  // beta [64] fp32
    static constexpr uint32_t fE = fB + 64 * 4;                      // exp(G) [64] fp32 (scalar gate)
    static constexpr uint32_t fFlag = fE + 64 * 4;                   // KDA: exact-path flag
    static constexpr uint32_t fTot = fFlag + 16;                     // SPLITG: the cumsum's block totals
    // The solve's scratch.  With a per-key-dim gate and K = 128 it reuses the 32 KB of G, dead by then
    // (the last reader is the k exp(G) rescale, a barrier before the solve): two CTAs per SM.  SPLITG puts it
    // over the Ka and G-half tiles.
    static constexpr uint32_t kDw = 2 * 16 * 17 * 4;
    static constexpr uint32_t kSolveBytes = ((4 * kDw + 1023) & ~1023u) + 14 * 2 * 512;
    static constexpr bool kAliasG = PER_K && !SPLITG && 64 * GW * 4 >= kSolveBytes;
    static constexpr uint32_t kScr = SPLITG ? kKa : kF;              // the scratch's base
    static constexpr uint32_t fD = (kAliasG || SPLITG) ? 0 : fFlag + 16;   // per warp: A_II, X_II fp32 [16][17] each
    static constexpr uint32_t fXs = (fD + 4 * kDw + 1023) & ~1023u;  // X blocks (M, J), J <= M: hi, lo bf16 [16][16]
    static constexpr uint32_t kXb = 2 * 512;
    static constexpr uint32_t fSs = fXs + 10 * kXb;                  // per warp: S_IJ hi, lo bf16 [16][16]
    static constexpr uint32_t solve_end = fSs + 4 * kXb;
    static constexpr uint32_t scratch = SPLITG ? 2 * K * 128 : (kAliasG ? fFlag + 16 : solve_end);   // from kScr
    static constexpr uint32_t bytes = SPLITG ? kF + fTot + 2048 : kF + scratch;
    static_assert(!kAliasG || solve_end <= 64 * GW * 4, "the solve's scratch fits in G's space");
    static_assert(!SPLITG || solve_end <= scratch, "the solve's scratch fits over Ka and the G half");
    // KDA exact path: A fp32 [64][64] over the Ka and Kb tiles (dead once S = Ka Kb^T is formed; SPLITG: Ka)
    static_assert(!PER_K || 64 * 64 * 4 <= (SPLITG ? 1 : 2) * K * 128, "the exact A fits");
    static_assert(!WITH_P || (C == 64 && !PER_K), "P is produced for 64-token chunks and a scalar gate");
};

// Slot of X block (M, J), J <= M, in the packed lower-triangular store.
__device__ __forceinline__ int xslot(int M, int J) { return M * (M + 1) / 2 + J; }

// 16 x 16 bf16 block with 32-byte rows: the 16-byte halves swap on every other
// group of four rows, so 8-row ldmatrix/stmatrix accesses are conflict-free.
__device__ __forceinline__ uint32_t blk_off(int r, int half) { return r * 32 + ((half ^ ((r >> 2) & 1)) << 4); }

// bf16 hi + lo split of an fp32 pair, packed as mma operands.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = wm::pack2(x0 - hf.x, x1 - hf.y);
}

// A-operand (k-tile) hi/lo parts of a 16 x 16 block held as two C fragments (n-tiles 0, 1).
__device__ __forceinline__ void split_afrag(const float (&c0)[4], const float (&c1)[4], uint32_t (&hi)[4],
                                            uint32_t (&lo)[4]) {
    split2(c0[0], c0[1], hi[0], lo[0]);
    split2(c0[2], c0[3], hi[1], lo[1]);
    split2(c1[0], c1[1], hi[2], lo[2]);
    split2(c1[2], c1[3], hi[3], lo[3]);
}

// Stores a 16 x 16 block held as two C fragments into hi and lo bf16 blocks (stmatrix).
__device__ __forceinline__ void store_block_split(uint32_t hi_addr, uint32_t lo_addr, const float (&c0)[4],
                                                  const float (&c1)[4], int mi, int mr) {
    uint32_t hi[4], lo[4];
    split_afrag(c0, c1, hi, lo);
    const uint32_t off = blk_off(8 * (mi & 1) + mr, mi >> 1);
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(hi_addr + off), "r"(hi[0]),
                 "r"(hi[1]), "r"(hi[2]), "r"(hi[3])
                 : "memory");
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(lo_addr + off), "r"(lo[0]),
                 "r"(lo[1]), "r"(lo[2]), "r"(lo[3])
                 : "memory");
}

// acc[2][4] += A (hi, lo) * B, B the 16 x 16 block stored row-major [k][n] as hi and lo parts.
__device__ __forceinline__ void mma_block_split(float (&acc)[2][4], const uint32_t (&ahi)[4], const uint32_t (&alo)[4],
                                                uint32_t bhi_addr, uint32_t blo_addr, int mi, int mr) {
    const uint32_t off = blk_off(8 * (mi & 1) + mr, mi >> 1);
    uint32_t bh[4], bl[4];
    wm::ldsm_x4_t(bhi_addr + off, bh);
    wm::ldsm_x4_t(blo_addr + off, bl);
    wm::mma16816(acc[0], ahi, bh[0], bh[1]);
    wm::mma16816(acc[1], ahi, bh[2], bh[3]);
    wm::mma16816(acc[0], ahi, bl[0], bl[1]);
    wm::mma16816(acc[1], ahi, bl[2], bl[3]);
    wm::mma16816(acc[0], alo, bh[0], bh[1]);
    wm::mma16816(acc[1], alo, bh[2], bh[3]);
}

// Exponents of the gated k copies are clamped here; a chunk whose gate moves
// by more than kExpSafe from its middle row takes the exact fp32 path for A.
constexpr float kExpClamp = 60.f;
constexpr float kExpSafe = 40.f;

// EXTRA: grouped value heads (q/k head h / G) or the backward's T output.  The plain forward takes
// the variant without either (its schedule measured slower with them compiled in).
// PACKED (C = 64, packed variable-length sequences read in place): the outputs fill one row of whole
// chunks (B = 1, T = NT C) as the chunk-packed layout places them, while q, k, v, g, beta are read from
// the caller's packed tensors [total, ...]: chunk c of the row is chunk c - co[s] of sequence s = cs[c],
// whose tokens start at cu[s].  Rows past the sequence's end are zero tokens: beta and g read as zero,
// the k, q and v rows zeroed after they land (they hold the next sequence's tokens).
struct PackedIn {
    const int* cu;   // device int32 [n + 1]
    const int* co;   // device int32 [n + 1]
    const int* cs;   // device int32 [NT]
    int n;
    int total;
};

// UMMA (K = V = 128, C = 64, scalar gate, with P, tokens read in place): S = k k^T and P = q k^T on
// tcgen05 instead of mma.sync.  Warp 1 issues both (M = N = 64, K = 128) from one elected lane as soon as
// the k and q tiles land; the accumulators take 128 columns of tensor memory (S, then P), which the warps
// read back with 16x256b loads in the mma.sync accumulator layout, so the gating, the solve and the
// products that follow are shared with the mma.sync form.  An M = 64 accumulator keeps rows 16q .. 16q+15
// in lanes 0 .. 15 of sub-partition q: warp q's own block row.
// F16: q, k, v, beta and the outputs w, u, P are fp16 instead of bf16, so the scans that read them
// multiply operands of one type.  The solve's hi/lo split stays bf16, and so do the per-key-dim gate's
// gated copies for S (factors up to e^40 that fp16 cannot hold; S is their own product, both operands
// bf16); k e^G (at most |k|) is fp16.  beta and k arrive through bf16 pointers either way (two bytes
// per element).
template <int K, int V, int C, bool PER_K, bool WITH_P, bool EXTRA, bool PACKED, bool UMMA, bool F16>
__global__ void __launch_bounds__(128, 3)
prepare_mma_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                   const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mu,
                   const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mp,
                   const float* __restrict__ g, const bf16* __restrict__ beta, float* __restrict__ g_cum,
                   bf16* __restrict__ tinv, int T, int H, int G, PackedIn pin, unsigned int* err,
                   const bf16* __restrict__ k_raw) {
    static_assert(!PACKED || (C == kTile && !PER_K), "packed inputs: whole 64-token chunks, scalar gate");
    static_assert(!UMMA || (K == 128 && V == 128 && C == 64 && !PER_K && WITH_P && !PACKED), "tcgen05 S, P: one shape");
    static_assert(!F16 || !PACKED, "fp16 io: not for packed sequences");
    using L = PrepLayout<K, V, C, PER_K, WITH_P>;
    constexpr int GW = L::GW;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr bool SPLITG = L::SPLITG;
    unsigned char* F = sm + L::kF;
    float* sG = reinterpret_cast<float*>(SPLITG ? sm + L::kGh : F + L::fG);   // SPLITG: the half tile
    float* sB = reinterpret_cast<float*>(F + L::fB);
    float* sE = reinterpret_cast<float*>(F + L::fE);
    int* sFlag = reinterpret_cast<int*>(F + L::fFlag);
    __shared__ uint64_t bar_k, bar_q, bar_v;   // one per tile, each waited on just before its first use
    __shared__ uint64_t bar_s, bar_p;   // UMMA: one per product, each completed once
    __shared__ uint32_t tslot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CTAs run chunk-major, the sequence's last tile first, so the first chunks are the last written and
    // still in L2 when the scan that follows reads them first (one grid dimension: tiles x heads)
    const int ntiles = (T + kTile - 1) / kTile;
    const int h = (int)(blockIdx.x % (unsigned)H), t0 = (ntiles - 1 - (int)(blockIdx.x / (unsigned)H)) * kTile;
    const int b = blockIdx.z;
    const int hk = EXTRA ? h / G : h;                 // q/k head of value head h
    const int nout = min(kTile, T - t0);             // rows of the outputs (g_cum) this tile writes
    int nvalid = nout, t_in = t0, b_in = b, T_in = T; // input rows: how many are real tokens, and where
    if constexpr (PACKED) {
        const int c = t0 / C, sq = pin.cs[c];
        nvalid = 0;
        t_in = 0;
        b_in = 0;
        T_in = pin.total;
        if (sq >= 0 && sq < pin.n && pin.co[sq] <= c && c < pin.co[sq + 1]) {
            const int a = min(max(pin.cu[sq], 0), pin.total);
            const int len = min(max(pin.cu[sq + 1] - a, 0), pin.total - a);
            const int j = c - pin.co[sq];
            t_in = a + j * C;
            nvalid = min(max(len - j * C, 0), kTile);
        }
    }
    auto row = [&](int t) -> int64_t { return ((int64_t)b * T + t0 + t) * H + h; };
    auto row_in = [&](int t) -> int64_t { return ((int64_t)b_in * T_in + t_in + t) * H + h; };
    // rows nvalid.. of a [64][D] tile in the 128-byte swizzle (whole 128-byte rows of every atom) to zero
    auto zero_rows = [&](uint32_t tile, int D, int first, int last, int id, int nthr) {
        const int per = (last - first) * (D / 8);
        for (int i = id; i < per; i += nthr) {
            const int r = first + i / (D / 8), u16 = i % (D / 8);
            *reinterpret_cast<uint4*>(sm + tile + (u16 >> 3) * 8192 + r * 128 + (u16 & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
    };
    const uint32_t s_base = bw::smem_u32(sm);
    // a kernel launched as this one's programmatic dependent (the tcgen05 scan after a prepare with P)
    // may start its setup once every CTA of this grid has begun; it waits for this grid's completion
    // before it reads anything written here
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // beta and (scalar gate) g of the tile, loaded first: their latency runs under the barrier setup and
    // the TMA issue (rows past T read as zero)
    float b_pre = 0.f, g_pre0 = 0.f, g_pre1 = 0.f;
    if (tid < kTile && tid < nvalid) b_pre = bw::load_io<F16>(beta + row_in(tid));
    if (!PER_K && warp == 0) {
        if (lane < nvalid) g_pre0 = g[row_in(lane)];
        if (32 + lane < nvalid) g_pre1 = g[row_in(32 + lane)];
    }

    if (tid == 0) {
        bw::mbar_init(&bar_k, 1);
        bw::mbar_init(&bar_q, 1);
        bw::mbar_init(&bar_v, 1);
        if constexpr (UMMA) {
            bw::mbar_init(&bar_s, 1);
            bw::mbar_init(&bar_p, 1);
        }
        bw::fence_mbar_init();
        *sFlag = 0;
    }
    __syncthreads();

    if (tid == 0) {
        // k first (S = k k^T needs it at once), then q (P), then v (u, the last product)
        bw::mbar_arrive_expect_tx(&bar_k, K * 128);
#pragma unroll
        for (int a = 0; a < K / 64; ++a) bw::tma_load_4d(sm + L::kK + a * 8192, &mk, &bar_k, a * 64, hk, t_in, b_in);
        if constexpr (WITH_P) {
            bw::mbar_arrive_expect_tx(&bar_q, K * 128);
#pragma unroll
            for (int a = 0; a < K / 64; ++a) bw::tma_load_4d(sm + L::kQ + a * 8192, &mq, &bar_q, a * 64, hk, t_in, b_in);
        }
        if constexpr (!SPLITG) {   // SPLITG: v lands in Kb's place once S is formed
            bw::mbar_arrive_expect_tx(&bar_v, V * 128);
#pragma unroll
            for (int a = 0; a < V / 64; ++a) bw::tma_load_4d(sm + L::kV + a * 8192, &mv, &bar_v, a * 64, h, t_in, b_in);
        }
    }
    static_assert(kTile <= 128, "one beta row per thread");
    if (tid < kTile) sB[tid] = b_pre;
    // UMMA: warp 1 (idle while warp 0 scans the gate) takes 128 tensor-memory columns (three CTAs per SM
    // take 384 of the 512) and issues S = k k^T (columns 0..63) and P = q k^T (64..127) as k and q land
    if (UMMA && warp == 1) {
        __syncwarp();
        bw::tmem_alloc(&tslot, 128);
        bw::tmem_relinquish();
        bw::tc_fence_before();
        __syncwarp();
        bw::tc_fence_after();
        const uint32_t t = tslot;
        constexpr uint32_t idS = bw::idesc_io(64, 64, 0, 0, F16);
        bw::mbar_wait(&bar_k, 0, err, kDeviceErrTimeout);   // a timeout is recorded; the stores follow thread 0's waits
        __syncwarp();
        bw::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk)
            bw::mma_bf16_warp(t, desc_kmajor(s_base + L::kK, kk), desc_kmajor(s_base + L::kK, kk), idS, kk > 0);
        bw::mma_commit_warp(&bar_s);
        bw::mbar_wait(&bar_q, 0, err, kDeviceErrTimeout);
        __syncwarp();
        bw::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk)
            bw::mma_bf16_warp(t + 64, desc_kmajor(s_base + L::kQ, kk), desc_kmajor(s_base + L::kK, kk), idS, kk > 0);
        bw::mma_commit_warp(&bar_p);
    }
    if constexpr (PER_K) {
        if constexpr (!SPLITG) {   // SPLITG loads G by halves of the keys, below
            // 16-byte loads, all of a thread's issued before any is used (the tile is 32 KB at K = 128)
            constexpr int NV4 = kTile * GW / 4 / 128;
            float4 gv[NV4];
#pragma unroll
            for (int j = 0; j < NV4; ++j) {
                const int e = 4 * (tid + 128 * j), t = e / GW;
                gv[j] = t < nvalid ? *reinterpret_cast<const float4*>(g + row_in(t) * GW + e % GW)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < NV4; ++j) *reinterpret_cast<float4*>(sG + 4 * (tid + 128 * j)) = gv[j];
        }
    } else if (warp == 0) {
        // scalar gate: warp shuffle scan, lane l holds rows l and 32 + l
        float x0 = g_pre0, x1 = g_pre1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
            if (lane >= o) { x0 += y0; x1 += y1; }
        }
        if (C == 64) x1 += __shfl_sync(0xffffffffu, x0, 31);   // one chunk spans both halves
        sG[lane] = x0;
        sG[32 + lane] = x1;
        sE[lane] = __expf(x0);
        sE[32 + lane] = __expf(x1);
        if (lane < nout) g_cum[row(lane)] = x0;
        if (32 + lane < nout) g_cum[row(32 + lane)] = x1;
    }
    __syncthreads();
    // chunk-local inclusive cumsum (per-key-dim gate) in two levels: thread (column quad cq, row block rb)
    // forms the prefix of its RPB rows of four columns, the block totals pass through the still unused Kb
    // tile, and each block adds the totals of the blocks before it in its chunk
    if constexpr (PER_K && !SPLITG) {
        constexpr int NQ = K / 4, NRB = 128 / NQ, RPB = kTile / NRB;   // K = 128: 32 quads x 4 blocks of 16 rows
        static_assert(NQ * NRB == 128 && C % RPB == 0, "blocks tile the threads and the chunks");
        float4* sG4 = reinterpret_cast<float4*>(sG);
        float4* tot = reinterpret_cast<float4*>(sm + L::kKb);        // [NRB][NQ]
        const int cq = tid % NQ, rb = tid / NQ, r0 = rb * RPB;
        float4 pre[RPB];
        float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RPB; ++i) {
            const float4 x = sG4[(r0 + i) * NQ + cq];
            run.x += x.x; run.y += x.y; run.z += x.z; run.w += x.w;
            pre[i] = run;
        }
        tot[rb * NQ + cq] = run;
        __syncthreads();
        float4 off = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int b2 = (r0 / C) * C / RPB; b2 < rb; ++b2) {   // the blocks before this one in its chunk
            const float4 y = tot[b2 * NQ + cq];
            off.x += y.x; off.y += y.y; off.z += y.z; off.w += y.w;
        }
#pragma unroll
        for (int i = 0; i < RPB; ++i) {
            const int t = r0 + i;
            const float4 v4 = make_float4(off.x + pre[i].x, off.y + pre[i].y, off.z + pre[i].z, off.w + pre[i].w);
            sG4[t * NQ + cq] = v4;
            if (t < nout) *reinterpret_cast<float4*>(g_cum + row(t) * K + 4 * cq) = v4;
        }
        __syncthreads();
    }

    bool ok = bw::mbar_wait(&bar_k, 0, err, kDeviceErrTimeout);
    if (PACKED && nvalid < kTile) zero_rows(L::kK, K, nvalid, kTile, tid, 128);   // a barrier follows

    if constexpr (SPLITG) {
        // per-key-dim gate at K = 128, G by halves of the keys through the [64][64] half tile: load, the
        // chunk-local cumsum in two levels (as below), g_cum, then the gated copies Ka, Kb of those keys
        // and k exp(G) over k
        constexpr int HK = 64, NQ = HK / 4, NRB = 128 / NQ, RPB = kTile / NRB;   // 16 quads x 8 blocks of 8 rows
        static_assert(C % RPB == 0, "row blocks tile the chunks");
        float4* sG4 = reinterpret_cast<float4*>(sG);
        float4* tot = reinterpret_cast<float4*>(F + L::fTot);   // [NRB][NQ]
        const int cq = tid % NQ, rb = tid / NQ, r0 = rb * RPB;
        bool big = false;
        for (int hf = 0; hf < K / HK; ++hf) {
            float4 gv[kTile * HK / 4 / 128];
#pragma unroll
            for (int j = 0; j < kTile * HK / 4 / 128; ++j) {
                const int e = 4 * (tid + 128 * j), t = e / HK;
                gv[j] = t < nvalid ? *reinterpret_cast<const float4*>(g + row_in(t) * GW + hf * HK + e % HK)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < kTile * HK / 4 / 128; ++j) sG4[tid + 128 * j] = gv[j];
            __syncthreads();
            float4 pre[RPB];
            float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < RPB; ++i) {
                const float4 x = sG4[(r0 + i) * NQ + cq];
                run.x += x.x; run.y += x.y; run.z += x.z; run.w += x.w;
                pre[i] = run;
            }
            tot[rb * NQ + cq] = run;
            __syncthreads();
            float4 off = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int b2 = (r0 / C) * C / RPB; b2 < rb; ++b2) {
                const float4 y = tot[b2 * NQ + cq];
                off.x += y.x; off.y += y.y; off.z += y.z; off.w += y.w;
            }
#pragma unroll
            for (int i = 0; i < RPB; ++i) {
                const int t = r0 + i;
                const float4 v4 = make_float4(off.x + pre[i].x, off.y + pre[i].y, off.z + pre[i].z, off.w + pre[i].w);
                sG4[t * NQ + cq] = v4;
                if (t < nout) *reinterpret_cast<float4*>(g_cum + row(t) * K + hf * HK + 4 * cq) = v4;
            }
            __syncthreads();
            // this half's 64 x 64 keys as 512 chunks of eight: Ka, Kb, and k exp(G) over k (each thread
            // rewrites the chunk of k it read)
#pragma unroll
            for (int j = 0; j < kTile * (HK / 8) / 128; ++j) {
                const int i = tid + 128 * j, r = i / (HK / 8), lc = i % (HK / 8);
                const int ref = (r / C) * C + C / 2;
                const uint32_t off = (uint32_t)(hf * 8192 + r * 128 + ((lc ^ (r & 7)) << 4));
                const uint4 raw = *reinterpret_cast<const uint4*>(sm + L::kK + off);
                float kv[8], fa[8], fb[8], fw[8];
                bw::unpack8_io<F16>(raw, kv);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float gr = sG[r * HK + lc * 8 + e];
                    const float dg = gr - sG[ref * HK + lc * 8 + e];
                    big |= fabsf(dg) > kExpSafe;
                    const float x = kv[e];
                    fa[e] = x * __expf(fminf(fmaxf(dg, -kExpClamp), kExpClamp));
                    fb[e] = x * __expf(fminf(fmaxf(-dg, -kExpClamp), kExpClamp));
                    fw[e] = x * __expf(gr);
                }
                uint4 pa, pb, pw;
                pa.x = bw::pack_bf16(fa[0], fa[1]); pa.y = bw::pack_bf16(fa[2], fa[3]);
                pa.z = bw::pack_bf16(fa[4], fa[5]); pa.w = bw::pack_bf16(fa[6], fa[7]);
                pb.x = bw::pack_bf16(fb[0], fb[1]); pb.y = bw::pack_bf16(fb[2], fb[3]);
                pb.z = bw::pack_bf16(fb[4], fb[5]); pb.w = bw::pack_bf16(fb[6], fb[7]);
                pw = bw::pack8_io<F16>(fw);   // an operand of w, beside X in the io type
                *reinterpret_cast<uint4*>(sm + L::kKa + off) = pa;
                *reinterpret_cast<uint4*>(sm + L::kKb + off) = pb;
                *reinterpret_cast<uint4*>(sm + L::kK + off) = pw;
            }
            __syncthreads();   // the half tile is rewritten next (or dead)
        }
        if (big) *sFlag = 1;
        bw::fence_async_shared();
    } else if (PER_K) {
        // gated copies for S: Ka = k exp(G - G_ref), Kb = k exp(G_ref - G), G_ref = middle row of the chunk
        for (int i = tid; i < kTile * (K / 8); i += 128) {
            const int r = i / (K / 8), lc = i % (K / 8);
            const int ref = (r / C) * C + C / 2;
            const uint32_t off = (uint32_t)((lc >> 3) * 8192 + r * 128 + (((lc & 7) ^ (r & 7)) << 4));
            const uint4 raw = *reinterpret_cast<const uint4*>(sm + L::kK + off);
            float kv[8], fa[8], fb[8];
            bw::unpack8_io<F16>(raw, kv);
            bool big = false;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int d = lc * 8 + e;
                const float dg = sG[r * K + d] - sG[ref * K + d];
                big |= fabsf(dg) > kExpSafe;
                const float x = kv[e];
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

    // UMMA: the tensor-memory columns warp 1 took (S at 0..63, P at 64..127) in this warp's sub-partition
    uint32_t tmem = 0, tq = 0;
    if constexpr (UMMA) {
        bw::tc_fence_after();
        tmem = tslot;
        tq = tmem + ((uint32_t)(warp * 32) << 16);
    }

    const int g4 = lane >> 2, q4 = lane & 3, mi = lane >> 3, mr = lane & 7;
    const int i0 = warp * 16 + g4, i1 = i0 + 8;       // the two tile rows of this thread's fragments
    float Af[8][4];                                   // A block row of this warp as C fragments
    // S = k k^T for this warp's 16 rows: [16 x 64]
    {
        const uint32_t a_t = s_base + (PER_K ? L::kKa : L::kK);
        const uint32_t b_t = s_base + (PER_K ? L::kKb : L::kK);
        float S[8][4];
        if constexpr (UMMA) {
            ok = bw::mbar_wait(&bar_s, 0, err, kDeviceErrTimeout) && ok;
            __syncwarp();   // the loads below are warp-wide
            bw::tc_fence_after();
            bw::tmem_ld16x256b_x8(tq, &S[0][0]);
            bw::tmem_ld_wait();
        } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) {
            uint32_t a[4];
            wm::ldsm_x4(a_t + tile_off(warp * 16 + 8 * (mi & 1) + mr, 16 * kk + 8 * (mi >> 1)), a);
#pragma unroll
            for (int jp = 0; jp < 8; jp += 2) {
                // key blocks right of the diagonal block: A is zero there (skipping them measured slower with
                // a per-key-dim gate: 0.212 vs 0.195 ms on the 8192-token KDA workload)
                if (!PER_K && jp / 2 > warp) continue;
                uint32_t bfr[4];
                wm::ldsm_x4(b_t + tile_off(8 * jp + 8 * (mi >> 1) + mr, 16 * kk + 8 * (mi & 1)), bfr);
                wm::mma16816_io<F16 && !PER_K>(S[jp], a, bfr[0], bfr[1]);   // per-key-dim gate: bf16 copies
                wm::mma16816_io<F16 && !PER_K>(S[jp + 1], a, bfr[2], bfr[3]);
            }
        }
        }
        // A from S, in place: element (i, j) of this thread's fragments
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
                Af[jn][e] = a0;
                Af[jn][2 + e] = a1;
            }
        }
    }
    if constexpr (WITH_P) {
        ok = bw::mbar_wait(&bar_q, 0, err, kDeviceErrTimeout) && ok;
        if (PACKED && nvalid < warp * 16 + 16) {   // this warp's own rows of q, which only it reads
            zero_rows(L::kQ, K, max(nvalid, warp * 16), warp * 16 + 16, lane, 32);
            __syncwarp();
        }
        // P = tril_0(q k^T * exp(G_i - G_j)) for this warp's rows (key blocks past the diagonal are
        // zero and skipped) -> bf16 into the q tile's place (each warp overwrites only its own rows of
        // q, after reading them), as a [64][64] tile in the 128-byte swizzle; stored with w and u below
        float Pq[8][4];
        if constexpr (UMMA) {   // the product has read every row of q once its barrier completes
            ok = bw::mbar_wait(&bar_p, 0, err, kDeviceErrTimeout) && ok;
            __syncwarp();
            bw::tc_fence_after();
            bw::tmem_ld16x256b_x8(tq + 64, &Pq[0][0]);
            bw::tmem_ld_wait();
        } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) Pq[j][0] = Pq[j][1] = Pq[j][2] = Pq[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) {
            uint32_t aq[4];
            wm::ldsm_x4(s_base + L::kQ + tile_off(warp * 16 + 8 * (mi & 1) + mr, 16 * kk + 8 * (mi >> 1)), aq);
#pragma unroll
            for (int jp = 0; jp < 8; jp += 2) {
                if (jp / 2 > warp) continue;
                uint32_t bfr[4];
                wm::ldsm_x4(s_base + L::kK + tile_off(8 * jp + 8 * (mi >> 1) + mr, 16 * kk + 8 * (mi & 1)), bfr);
                wm::mma16816_io<F16>(Pq[jp], aq, bfr[0], bfr[1]);
                wm::mma16816_io<F16>(Pq[jp + 1], aq, bfr[2], bfr[3]);
            }
        }
        }
#pragma unroll
        for (int jp = 0; jp < 8; jp += 2) {
            float pv[2][4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int jn = jp + hh, j0 = 8 * jn + 2 * q4;
                pv[hh][0] = j0 <= i0 ? Pq[jn][0] * __expf(sG[i0] - sG[j0]) : 0.f;
                pv[hh][1] = j0 + 1 <= i0 ? Pq[jn][1] * __expf(sG[i0] - sG[j0 + 1]) : 0.f;
                pv[hh][2] = j0 <= i1 ? Pq[jn][2] * __expf(sG[i1] - sG[j0]) : 0.f;
                pv[hh][3] = j0 + 1 <= i1 ? Pq[jn][3] * __expf(sG[i1] - sG[j0 + 1]) : 0.f;
            }
            const uint32_t r[4] = {wm::pack2_io<F16>(pv[0][0], pv[0][1]), wm::pack2_io<F16>(pv[0][2], pv[0][3]),
                                   wm::pack2_io<F16>(pv[1][0], pv[1][1]), wm::pack2_io<F16>(pv[1][2], pv[1][3])};
            __syncwarp();
            asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(
                             s_base + L::kQ + tile_off(warp * 16 + 8 * (mi & 1) + mr, 8 * jp + 8 * (mi >> 1))),
                         "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                         : "memory");
        }
    }
    if (PER_K) {
        __syncthreads();
        if (SPLITG && tid == 0) {   // S is formed: v lands in Kb's place under the solve
            bw::mbar_arrive_expect_tx(&bar_v, V * 128);
#pragma unroll
            for (int a = 0; a < V / 64; ++a) bw::tma_load_4d(sm + L::kV + a * 8192, &mv, &bar_v, a * 64, h, t_in, b_in);
        }
        if (*sFlag) {
            // exact fp32 A for chunks with extreme gates: A_ij = beta_i sum_d k_id k_jd exp(G_id - G_jd)
            // (SPLITG: raw k and G come from global memory, k's tile holding k exp(G) and G only its last half)
            float* sA = reinterpret_cast<float*>(sm + L::kKa);   // over the dead Ka (and Kb) tiles
            const int Hk = EXTRA ? H / G : H;
            auto kval = [&](int i, int d) -> float {
                if constexpr (SPLITG)
                    return i < nvalid ? bw::load_io<F16>(k_raw + (((int64_t)b_in * T_in + t_in + i) * Hk + hk) * K + d)
                                      : 0.f;
                else
                    return bw::load_io<F16>(sm + L::kK + tile_off(i, d));
            };
            auto gval = [&](int i, int d) -> float {
                if constexpr (SPLITG) return i < nvalid ? g_cum[row(i) * K + d] : 0.f;
                else return sG[i * K + d];
            };
            for (int idx = tid; idx < kTile * kTile; idx += 128) {
                const int i = idx / kTile, j = idx % kTile;
                float a = 0.f;
                if (j >= (i / C) * C && j < i && i < nvalid) {   // rows past T have k = 0: A is 0 there
                    float acc = 0.f;
                    for (int d = 0; d < K; ++d) acc += kval(i, d) * kval(j, d) * __expf(gval(i, d) - gval(j, d));
                    a = sB[i] * acc;
                }
                sA[i * 64 + j] = a;
            }
            __syncthreads();
#pragma unroll
            for (int jn = 0; jn < 8; ++jn) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int j = 8 * jn + 2 * q4 + e;
                    Af[jn][e] = sA[i0 * 64 + j];
                    Af[jn][2 + e] = sA[i1 * 64 + j];
                }
            }
            __syncthreads();   // every warp has its A before Ka is rewritten below
        }
        // B operand of w: k * exp(G) per element, into Ka (its gated copy is no longer needed); SPLITG made it
        // over k with the gated copies
        for (int i = tid; i < (SPLITG ? 0 : kTile * (K / 8)); i += 128) {
            const int r = i / (K / 8), lc = i % (K / 8);
            const uint32_t off = (uint32_t)((lc >> 3) * 8192 + r * 128 + (((lc & 7) ^ (r & 7)) << 4));
            const uint4 raw = *reinterpret_cast<const uint4*>(sm + L::kK + off);
            float f[8];
            bw::unpack8_io<F16>(raw, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] *= __expf(sG[r * K + lc * 8 + e]);
            *reinterpret_cast<uint4*>(sm + L::kKa + off) = bw::pack8_io<F16>(f);
        }
        __syncthreads();       // G is dead: the solve's scratch reuses its space
    }

    // ---- X = (I + A)^{-1}: this warp's block row I = warp, blocks X_IJ for J0 <= J <= I
    constexpr int NB = C / 16;                        // 16-row blocks per chunk
    const int I = warp, J0 = (I / NB) * NB;           // first block of this warp's chunk
    float Xr[4][2][4];                                // X_IJ as C fragments (n-tiles of block column J)
#pragma unroll
    for (int J = 0; J < 4; ++J)
#pragma unroll
        for (int n = 0; n < 2; ++n) Xr[J][n][0] = Xr[J][n][1] = Xr[J][n][2] = Xr[J][n][3] = 0.f;
    const uint32_t xs_base = s_base + L::kScr + L::fXs;            // block (M, J) at xslot(M, J) * kXb: hi, then lo
    {
        // diagonal block: A_II to shared memory, 16 lanes invert it column by column in fp32
        float* dA = reinterpret_cast<float*>(sm + L::kScr + L::fD + warp * L::kDw);
        float* dX = dA + 16 * 17;
#pragma unroll
        for (int J = 0; J < 4; ++J) {
            if (J != I) continue;
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int cc = 8 * n + 2 * q4;
                dA[g4 * 17 + cc] = Af[2 * J + n][0];
                dA[g4 * 17 + cc + 1] = Af[2 * J + n][1];
                dA[(g4 + 8) * 17 + cc] = Af[2 * J + n][2];
                dA[(g4 + 8) * 17 + cc + 1] = Af[2 * J + n][3];
            }
        }
        __syncwarp();
        if (lane < 16) {
            const int c = lane;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float s = (i == c) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < i; ++j) s -= dA[i * 17 + j] * x[j];
                x[i] = (i < c) ? 0.f : s;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) dX[i * 17 + c] = x[i];
        }
        __syncwarp();
#pragma unroll
        for (int J = 0; J < 4; ++J) {
            if (J != I) continue;
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int cc = 8 * n + 2 * q4;
                Xr[J][n][0] = dX[g4 * 17 + cc];
                Xr[J][n][1] = dX[g4 * 17 + cc + 1];
                Xr[J][n][2] = dX[(g4 + 8) * 17 + cc];
                Xr[J][n][3] = dX[(g4 + 8) * 17 + cc + 1];
            }
            if (NB > 1) store_block_split(xs_base + xslot(I, J) * L::kXb, xs_base + xslot(I, J) * L::kXb + 512,
                                          Xr[J][0], Xr[J][1], mi, mr);
        }
    }
    // X_II as split A operands (left factor of every off-diagonal block of this row)
    uint32_t xdh[4], xdl[4];
#pragma unroll
    for (int J = 0; J < 4; ++J)
        if (J == I) split_afrag(Xr[J][0], Xr[J][1], xdh, xdl);
#pragma unroll
    for (int Lv = 1; Lv < NB; ++Lv) {
        __syncthreads();                              // blocks of distance < Lv are in shared memory
        if (I - J0 >= Lv) {
            const int J = I - Lv;
            // S_IJ = sum_{M=J}^{I-1} A_IM X_MJ
            float Sb[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int M = 0; M < 3; ++M) {
                if (M < J || M >= I) continue;
                uint32_t ah[4], al[4];
                split_afrag(Af[2 * M], Af[2 * M + 1], ah, al);
                const uint32_t xb = xs_base + xslot(M, J) * L::kXb;
                mma_block_split(Sb, ah, al, xb, xb + 512, mi, mr);
            }
            // X_IJ = -X_II S_IJ  (S_IJ back through this warp's block scratch as the B operand)
            const uint32_t sb = s_base + L::kScr + L::fSs + warp * L::kXb;
            store_block_split(sb, sb + 512, Sb[0], Sb[1], mi, mr);
            __syncwarp();
            float Xb[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            mma_block_split(Xb, xdh, xdl, sb, sb + 512, mi, mr);
#pragma unroll
            for (int Jc = 0; Jc < 3; ++Jc) {
                if (Jc != J) continue;
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) Xr[Jc][n][e] = -Xb[n][e];
                if (Lv + 1 < NB)   // a later level reads it
                    store_block_split(xs_base + xslot(I, Jc) * L::kXb, xs_base + xslot(I, Jc) * L::kXb + 512,
                                      Xr[Jc][0], Xr[Jc][1], mi, mr);
            }
        }
    }

    // X itself, for the backward's WY stage: [B, NT, H, C, C] bf16, this warp's 16 rows of its chunk
    if (EXTRA && tinv && t0 + (I / NB) * C < T) {
        const int ci = t0 / C + I / NB;
        bf16* dst = tinv + (((int64_t)b * ((T + C - 1) / C) + ci) * H + h) * C * C;
        const int r0 = 16 * (I - J0) + g4;
#pragma unroll
        for (int J = 0; J < 4; ++J) {
            if (J < J0 || J >= J0 + NB) continue;
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int col = 16 * (J - J0) + 8 * n + 2 * q4;
                *reinterpret_cast<uint32_t*>(dst + (int64_t)r0 * C + col) = wm::pack2(Xr[J][n][0], Xr[J][n][1]);
                *reinterpret_cast<uint32_t*>(dst + (int64_t)(r0 + 8) * C + col) = wm::pack2(Xr[J][n][2], Xr[J][n][3]);
            }
        }
    }

    // Tb fragments: X diag(beta) for u; X diag(beta exp(G)) for w (scalar gate) or X diag(beta) (per-key-dim)
    uint32_t tu[4][4], tw[4][4];
#pragma unroll
    for (int J = 0; J < 4; ++J) {
        const int j0 = 16 * J + 2 * q4, j1 = j0 + 8;
        const float2 ba = *reinterpret_cast<const float2*>(sB + j0), bb = *reinterpret_cast<const float2*>(sB + j1);
        tu[J][0] = wm::pack2_io<F16>(Xr[J][0][0] * ba.x, Xr[J][0][1] * ba.y);
        tu[J][1] = wm::pack2_io<F16>(Xr[J][0][2] * ba.x, Xr[J][0][3] * ba.y);
        tu[J][2] = wm::pack2_io<F16>(Xr[J][1][0] * bb.x, Xr[J][1][1] * bb.y);
        tu[J][3] = wm::pack2_io<F16>(Xr[J][1][2] * bb.x, Xr[J][1][3] * bb.y);
        if constexpr (PER_K) {
#pragma unroll
            for (int e = 0; e < 4; ++e) tw[J][e] = tu[J][e];
        } else {
            const float2 ea = *reinterpret_cast<const float2*>(sE + j0), eb = *reinterpret_cast<const float2*>(sE + j1);
            tw[J][0] = wm::pack2_io<F16>(Xr[J][0][0] * ba.x * ea.x, Xr[J][0][1] * ba.y * ea.y);
            tw[J][1] = wm::pack2_io<F16>(Xr[J][0][2] * ba.x * ea.x, Xr[J][0][3] * ba.y * ea.y);
            tw[J][2] = wm::pack2_io<F16>(Xr[J][1][0] * bb.x * eb.x, Xr[J][1][1] * bb.y * eb.y);
            tw[J][3] = wm::pack2_io<F16>(Xr[J][1][2] * bb.x * eb.x, Xr[J][1][3] * bb.y * eb.y);
        }
    }
    // The products out[64 x D] = T [64 x 64] * B [64 x D], B = k (or k exp(G)) or v read token-major by
    // ldmatrix.trans, balanced over the warps: each warp takes a quarter of the output columns over every
    // row block (row block I needs the k-steps J0(I) .. I, so row-block ownership would leave warp 3 four
    // times warp 0's work).  The T fragments therefore go through shared memory, over the solve's scratch.
    if constexpr (UMMA) bw::tc_fence_before();   // the S and P loads are complete
    __syncthreads();   // every warp is past the solve's scratch
    if (UMMA && warp == 1) {
        bw::tc_fence_after();
        bw::tmem_dealloc(tmem, 128);
    }
    const uint32_t tw_t = s_base + L::kScr + 1024, tu_t = tw_t + 8192;   // T's [64][64] bf16 tiles
    static_assert(L::scratch >= 1024 + 2 * 8192, "the T tiles fit the solve's scratch");
#pragma unroll
    for (int J = 0; J < 4; ++J) {
        const uint32_t off = tile_off(warp * 16 + 8 * (mi & 1) + mr, 16 * J + 8 * (mi >> 1));
        asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(tw_t + off), "r"(tw[J][0]),
                     "r"(tw[J][1]), "r"(tw[J][2]), "r"(tw[J][3])
                     : "memory");
        asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(tu_t + off), "r"(tu[J][0]),
                     "r"(tu[J][1]), "r"(tu[J][2]), "r"(tu[J][3])
                     : "memory");
    }
    __syncthreads();
    // this warp's D / 4 output columns of all four row blocks; k-steps outside J0(I) .. I multiply zeros
    auto product = [&](uint32_t a_t, uint32_t b_t, auto dcols, float (&acc)[4][decltype(dcols)::value / 32][4]) {
        constexpr int D = decltype(dcols)::value, NW = D / 32;
        const int n0 = warp * (D / 4);
#pragma unroll
        for (int I = 0; I < 4; ++I)
#pragma unroll
            for (int j = 0; j < NW; ++j) acc[I][j][0] = acc[I][j][1] = acc[I][j][2] = acc[I][j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t bfr[NW / 2][4];
#pragma unroll
            for (int jp = 0; jp < NW / 2; ++jp)
                wm::ldsm_x4_t(b_t + tile_off(16 * kk + 8 * (mi & 1) + mr, n0 + 16 * jp + 8 * (mi >> 1)), bfr[jp]);
#pragma unroll
            for (int I = 0; I < 4; ++I) {
                if (kk > I || kk < (I / NB) * NB) continue;
                uint32_t a[4];
                wm::ldsm_x4(a_t + tile_off(16 * I + 8 * (mi & 1) + mr, 16 * kk + 8 * (mi >> 1)), a);
#pragma unroll
                for (int jp = 0; jp < NW / 2; ++jp) {
                    wm::mma16816_io<F16>(acc[I][2 * jp], a, bfr[jp][0], bfr[jp][1]);
                    wm::mma16816_io<F16>(acc[I][2 * jp + 1], a, bfr[jp][2], bfr[jp][3]);
                }
            }
        }
    };
    // bf16 results into a tile of the same layout (128-byte swizzle, 64-column atoms) by stmatrix
    auto stage_out = [&](uint32_t st, auto dcols, const float (&acc)[4][decltype(dcols)::value / 32][4]) {
        constexpr int D = decltype(dcols)::value, NW = D / 32;
        const int n0 = warp * (D / 4);
#pragma unroll
        for (int I = 0; I < 4; ++I)
#pragma unroll
            for (int jp = 0; jp < NW / 2; ++jp) {
                const uint32_t r[4] = {wm::pack2_io<F16>(acc[I][2 * jp][0], acc[I][2 * jp][1]),
                                       wm::pack2_io<F16>(acc[I][2 * jp][2], acc[I][2 * jp][3]),
                                       wm::pack2_io<F16>(acc[I][2 * jp + 1][0], acc[I][2 * jp + 1][1]),
                                       wm::pack2_io<F16>(acc[I][2 * jp + 1][2], acc[I][2 * jp + 1][3])};
                asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(
                                 st + tile_off(16 * I + 8 * (mi & 1) + mr, n0 + 16 * jp + 8 * (mi >> 1))),
                             "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                             : "memory");
            }
    };
    // One tile at a time, the result replacing the tile it was computed from: this warp's products into
    // registers, a barrier (every warp is done reading the tile), then the results over it.  This keeps
    // the CTA at three per SM (no separate staging region).
    auto product_in_place = [&](uint32_t a_t, uint32_t tile, auto dcols) {
        constexpr int D = decltype(dcols)::value;
        float acc[4][D / 32][4];
        product(a_t, tile, dcols, acc);
        __syncthreads();
        stage_out(tile, dcols, acc);
    };
    // w over the tile it reads (k, or its scaled copy Ka), then u over v
    const uint32_t w_tile = (PER_K && !SPLITG) ? L::kKa : L::kK;
    product_in_place(tw_t, s_base + w_tile, std::integral_constant<int, K>{});
    // w and P leave while u is formed (rows past T are clipped by the tensor maps)
    bw::fence_async_shared();
    __syncthreads();
    if (tid == 0 && ok) {
#pragma unroll
        for (int a = 0; a < K / 64; ++a) bw::tma_store_4d(&mw, sm + w_tile + a * 8192, a * 64, h, t0, b);
        if constexpr (WITH_P) bw::tma_store_4d(&mp, sm + L::kQ, 0, 0, h, b * ((T + C - 1) / C) + t0 / C);
        bw::bulk_commit();
    }
    ok = bw::mbar_wait(&bar_v, 0, err, kDeviceErrTimeout) && ok;
    if (PACKED && nvalid < kTile) {   // CTA-uniform
        zero_rows(L::kV, V, nvalid, kTile, tid, 128);
        __syncthreads();
    }
    product_in_place(tu_t, s_base + L::kV, std::integral_constant<int, V>{});
    bw::fence_async_shared();
    __syncthreads();
    if (tid == 0) {
        if (ok) {
#pragma unroll
            for (int a = 0; a < V / 64; ++a) bw::tma_store_4d(&mu, sm + L::kV + a * 8192, a * 64, h, t0, b);
            bw::bulk_commit();
        }
        bw::bulk_wait_read<0>();   // no store may still be reading shared memory when the CTA exits
    }
}

// pdl: launched as the programmatic dependent of the kernel before it in the stream (it may start as
// soon as every CTA of that kernel has signalled, and reads nothing that kernel writes).
template <int K, int V, int C, bool PER_K, bool WITH_P, bool EXTRA, bool PACKED = false, bool UMMA = false,
          bool F16 = false>
cudaError_t launch_prepare_v(const Dims& d, const void* q, const void* k, const void* v, const float* g,
                             const void* beta, void* w, void* u, float* g_cum, void* P, void* tinv, cudaStream_t s,
                             unsigned int* err, PackedIn pin = PackedIn{}, bool pdl = false) {
    using L = PrepLayout<K, V, C, PER_K, WITH_P>;
    CUtensorMap mk, mv, mw, mu, mq, mp;
    // q and k have the Hk q/k heads; every other token tensor the H value heads.  Packed inputs: one
    // row of the caller's total tokens.
    const int bi = PACKED ? 1 : d.B, ti = PACKED ? pin.total : d.T;
    if (!make_tmap_tokens(&mk, k, bi, ti, d.Hk, K, kTile) || !make_tmap_tokens(&mv, v, bi, ti, d.H, V, kTile) ||
        !make_tmap_tokens(&mw, w, d.B, d.T, d.H, K, kTile) || !make_tmap_tokens(&mu, u, d.B, d.T, d.H, V, kTile))
        return cudaErrorInvalidValue;
    mq = mk;
    mp = mw;
    if constexpr (WITH_P) {
        // P [B, NT, H, C, C] seen as (C, C, H, B*NT); one 64 x 64 box per chunk
        const uint64_t dims[4] = {(uint64_t)C, (uint64_t)C, (uint64_t)d.H, (uint64_t)d.B * d.NT};
        const uint64_t st[3] = {(uint64_t)C * 2, (uint64_t)C * C * 2, (uint64_t)d.H * C * C * 2};
        const uint32_t box[4] = {64, 64, 1, 1};
        if (!make_tmap_tokens(&mq, q, bi, ti, d.Hk, K, kTile) || !make_tmap_bf16_4d(&mp, P, dims, st, box))
            return cudaErrorInvalidValue;
    }
    auto kern = prepare_mma_kernel<K, V, C, PER_K, WITH_P, EXTRA, PACKED, UMMA, F16>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((d.T + kTile - 1) / kTile) * (unsigned)d.H, 1, d.B);
    if (pdl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, mk, mv, mw, mu, mq, mp, g, (const bf16*)beta, g_cum, (bf16*)tinv, d.T,
                                  d.H, d.G, pin, err, (const bf16*)k);
    }
    kern<<<grid, 128, smem, s>>>(mk, mv, mw, mu, mq, mp, g, (const bf16*)beta, g_cum, (bf16*)tinv, d.T, d.H, d.G,
                                 pin, err, (const bf16*)k);
    return cudaGetLastError();
}

}  // namespace
}  // namespace gdr
