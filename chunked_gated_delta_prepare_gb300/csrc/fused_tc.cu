// State scan + chunk output of one (batch, head) per CTA on the tcgen05 tensor
// cores, for bf16 io (or fp16, scalar gate), K = V = 128 and 64-token chunks
// (any T, grouped value heads):
//
//   scan   ("kernel_fun/kda/_kernels/bwd_scan.py", module docstring):
//          v'_c = u_c - w_c h_c;  h_{c+1} = exp(G_last) h_c + (k exp(G_last - G))^T v'_c
//   output (the o assembly that page gives to the forward's epilogue warps):
//          o_c = scale [ exp(G) * (q h_c) + P_c v'_c ],  P_c = tril_0(q k^T * exp(G_i - G_j))
//
// given w, u, G (g_cum) and P from the WY prepare.  Every product runs transposed, with the
// value dimension as the MMA's M = 128 rows, so the two chain operands that change every
// chunk -- h_c^T and v'_c^T -- are A operands read straight from tensor memory, and the
// per-chunk tiles w, q, k, P are the B operands in shared memory:
//
//   D^T  = h_c^T w^T            M=128 (v) N=64 (t)    K=128 (key)  A: TMEM bf16  B: w [t][key]
//   v'^T = u^T - D^T            CUDA cores (fp32), written back to TMEM as bf16, plain and
//                                scaled by gamma_t = exp(G_last - G_t)
//   dh^T = (v' diag gamma)^T k  M=128 (v) N=128 (key) K=64 (t)     A: TMEM bf16  B: k [t][key]
//   O1^T = h_c^T q^T            M=128     N=64        K=128        A: TMEM bf16  B: q [t][key]
//   O2^T = v'^T P^T             M=128     N=64        K=64         A: TMEM bf16  B: P [i][j]
//   h^T  = exp(G_last) h^T + dh^T   CUDA cores; h stays fp32 in registers for the whole sequence
//   o    = scale (exp(G_t) O1^T + O2^T), stored by the same threads (thread = value column)
//
// Issue order per chunk c: D(c); then O2(c-1), which runs while the CUDA cores form v'(c); dh(c);
// then O1(c), which runs while they update h.  The o epilogue of chunk c-1 runs in the chain warps
// while the tensor cores form dh(c), so neither output product nor the o stores sit between the two
// chain products.  h_c^T and v'^T are double-buffered by chunk parity for the trailing output products.
// The fp32 element work uses the packed two-lane forms (__ffma2_rn, __fmul2_rn), which round each lane
// exactly like the scalar operations.
//
// A per-key-dim gate (GATED) runs the same kernel on the gated operands qg = q exp(G) and
// kg = k exp(G_last - G) that tc_gated_operands writes with P: dh^T = v'^T kg (no gamma, no second copy
// of v'), O2 accumulates onto O1 (o = scale (O1^T + O2^T)), and h decays by exp(G_last) per key.
//
// Warp roles: warp 0 loads each chunk's w, q, k, u, P by TMA into a 3-stage ring and forms
// gamma, exp(G), exp(G_last), reading the next chunk's gate while this one's tiles land; warp 1
// issues the MMAs (one elected lane, fully unrolled, descriptors precomputed); warps 2..17 are
// the chain warps, four per TMEM sub-partition: the warp in sub-partition s, part p owns value
// columns 32s.. (its TMEM lanes), tokens 16p.. of v' and o, and keys 32p.. of h.  Every wait is
// bounded; a wait that gives up records the device error word and the kernel winds down
// through its normal exit.
//
// Where it pays: one CTA carries a whole head, so a problem needs B*H CTAs here against
// B*H*V/32 for the warp-level kernel of fused_mma.cu, but each chunk step costs about 2,700 SM
// cycles here against about 2,400 there (the per-element work of v', h and o on one SM's four
// schedulers, between two dependent MMA round trips; the o stores of a chunk alone cost about 300,
// with lanes v, v^1 trading halves of their token pairs so that each store writes two adjacent
// columns).  Measured on the 2048-token, 64-head workload (256 warp-level CTAs, two waves): 0.056 ms
// here, 0.085 ms there; on the 32k-token, 32-head one (128 CTAs, one wave): 0.670 ms here, 0.601 ms
// there.  Variant AUTO therefore takes this kernel when the warp-level grid would not fit one wave
// of the GPU, and for one long sequence, whose pieces overlap their prepares with it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "blackwell.cuh"
#include "gdr_internal.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace gdr {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kK = 128, kV = 128, kC = 64;
constexpr int kNS = 3;                    // ring stages
constexpr int kChainWarps = 16;           // four per sub-partition
constexpr int kWarp0 = 2;                 // first chain warp
constexpr int kThreads = 32 * (kWarp0 + kChainWarps);

struct TcLayout {
    static constexpr uint32_t kTile = kC * kK * 2;                  // [64][128] bf16, 16 KB
    static constexpr uint32_t W = 0, Q = kTile, KB = 2 * kTile, U = 3 * kTile, P = 4 * kTile;   // in a stage
    static constexpr uint32_t kStage = 4 * kTile + kC * kC * 2;     // 72 KB (a multiple of 1 KB)
    static constexpr uint32_t F = kNS * kStage;                     // per stage: gamma[64], exp(G)[64], exp(G_last)
    static constexpr uint32_t kF = (2 * kC + 4) * 4;
    static constexpr uint32_t bytes = F + kNS * kF;
    static constexpr uint32_t tx = kStage;
    static_assert(bytes + 1024 <= 232448, "tcgen05 scan/output shared memory");
};

// tensor-memory columns (512 allocated)
constexpr uint32_t cHB = 0;      // h_c^T bf16 [128 v][128 key]: two buffers of 64 columns (chunk parity)
constexpr uint32_t cVP = 128;    // v'^T bf16 [128 v][64 t]: two buffers of 32 columns (chunk parity)
constexpr uint32_t cVG = 192;    // (v' diag gamma)^T bf16: 32 columns
constexpr uint32_t cD = 256;     // D^T fp32 (64 columns), then dh^T fp32 (128 columns)
constexpr uint32_t cO1 = 384;    // O1^T fp32, 64 columns
constexpr uint32_t cO2 = 448;    // O2^T fp32, 64 columns

__device__ __forceinline__ void mma_ta(uint32_t d, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* u) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]), "r"(u[8]), "r"(u[9]),
        "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]), "r"(u[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* u) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// GENERAL: a last, partial chunk (T not a multiple of 64) or grouped value heads (G > 1: value head h
// reads q and k of head h / G).  The partial chunk runs as zero tokens past T: the TMA boxes read zeros
// there, the gate repeats its last value (so those tokens neither decay nor move the state) and no o row
// past T is stored.  Whole chunks of ungrouped heads take the variant without those guards.
// GATED (a per-key-dim gate): q and k are the gated operands qg = q exp(G) and kg = k exp(G_last - G)
// (per element, one per value head; see tc_gated_operands), so dh^T = v'^T kg, o = scale (O1^T + O2^T)
// with O2 accumulated onto O1, and the decay exp(G_last) is a vector over the keys.
// F16 (scalar gate): fp16 io.  q, k and the prepare's w, u, P are fp16, and so are the tensor-memory
// operands written here (h_c^T, v'^T), since both operands of one MMA share a type; o is stored as fp16.
template <bool GENERAL, bool GATED, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
tc_scan_output_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mq,
                      const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mu,
                      const __grid_constant__ CUtensorMap mp, const float* __restrict__ g_cum,
                      const float* __restrict__ h0, bf16* __restrict__ o, float* __restrict__ h_final, int T, int H,
                      int NT, int G, float scale, unsigned int* err) {
    using L = TcLayout;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[kNS], empty[kNS], barD, barE, barO, oFree, vpReady, hbReady, drain;
    __shared__ uint32_t tslot;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int hk = GENERAL && !GATED ? h / G : h;         // q/k head of value head h (gated: per value head)

    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            bw::mbar_init(&full[s], 32 + 1);
            bw::mbar_init(&empty[s], 1 + kChainWarps);
        }
        bw::mbar_init(&barD, 1);
        bw::mbar_init(&barE, 1);
        bw::mbar_init(&barO, 1);
        bw::mbar_init(&oFree, kChainWarps);
        bw::mbar_init(&vpReady, kChainWarps);
        bw::mbar_init(&hbReady, kChainWarps);
        bw::mbar_init(&drain, 1);
        bw::fence_mbar_init();
    }
    if (warp == 1) {
        bw::tmem_alloc(&tslot, 512);
        bw::tmem_relinquish();
    }
    __syncthreads();
    bw::tc_fence_after();
    const uint32_t tmem = tslot;
    const uint32_t s_base = bw::smem_u32(sm);
    // every CTA holds its SM now: a kernel launched as this one's programmatic dependent (the next
    // piece's prepare in the overlapped forward) may start on the SMs left free
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // launched as the programmatic dependent of the prepare, the only warp that reads what it wrote
        // waits here for it to complete (a no-op after an ordinary launch)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        constexpr int GW = GATED ? kK : 1;
        const float* gr = g_cum + ((int64_t)b * T * H + h) * GW;
        // G at token t (key d); past T: its last value
        auto gat = [&](int t, int d) { return gr[(int64_t)(GENERAL ? min(t, T - 1) : t) * H * GW + d]; };
        float g0 = 0.f, g1 = 0.f, gl = 0.f, gk[4] = {0.f, 0.f, 0.f, 0.f};
        auto read_gate = [&](int t0) {
            if constexpr (GATED) {
#pragma unroll
                for (int i = 0; i < 4; ++i) gk[i] = gat(t0 + kC - 1, lane + 32 * i);
            } else {
                g0 = gat(t0 + lane, 0);
                g1 = gat(t0 + lane + 32, 0);
                gl = gat(t0 + kC - 1, 0);
            }
        };
        if (NT > 0) read_gate(0);
        int issued = 0;
        for (int c = 0; c < NT; ++c) {
            const int s = c % kNS;
            if (!bw::mbar_wait(&empty[s], ((c / kNS) & 1) ^ 1, err, kDeviceErrTimeout)) break;
            const int t0 = c * kC;
            unsigned char* st = sm + s * L::kStage;
            if (lane == 0) {
                bw::mbar_arrive_expect_tx(&full[s], L::tx);
#pragma unroll
                for (int a = 0; a < kK / 64; ++a) {
                    bw::tma_load_4d(st + L::W + a * 8192, &mw, &full[s], a * 64, h, t0, b);
                    bw::tma_load_4d(st + L::Q + a * 8192, &mq, &full[s], a * 64, hk, t0, b);
                    bw::tma_load_4d(st + L::KB + a * 8192, &mk, &full[s], a * 64, hk, t0, b);
                }
                bw::tma_load_4d(st + L::U, &mu, &full[s], 0, h, t0, b);
                bw::tma_load_4d(st + L::P, &mp, &full[s], 0, 0, h, b * NT + c);
            }
            issued = c + 1;
            // gamma_t = exp(G_last - G_t), exp(G_t), exp(G_last) of the chunk (GATED: exp(G_last) per key);
            // then the next chunk's gate
            float* F = reinterpret_cast<float*>(sm + L::F + s * L::kF);
            if constexpr (GATED) {
#pragma unroll
                for (int i = 0; i < 4; ++i) F[lane + 32 * i] = __expf(gk[i]);
            } else {
                F[lane] = __expf(gl - g0);
                F[lane + 32] = __expf(gl - g1);
                F[kC + lane] = __expf(g0);
                F[kC + lane + 32] = __expf(g1);
                if (lane == 0) F[2 * kC] = __expf(gl);
            }
            bw::mbar_arrive(&full[s]);
            if (c + 1 < NT) read_gate(t0 + kC);
        }
        // no load of this CTA may still be landing when it exits
        for (int c = max(issued - kNS, 0); c < issued; ++c)
            bw::mbar_wait(&full[c % kNS], (c / kNS) & 1, err, kDeviceErrTimeout);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        uint64_t wd[8], kd[4], pd[4];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) wd[kk] = tc::desc_kmajor(s_base + L::W, kk);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            kd[kk] = tc::desc_mnmajor(s_base + L::KB, kk);
            pd[kk] = tc::desc_kmajor(s_base + L::P, kk);
        }
        constexpr uint64_t kQoff = (L::Q - L::W) >> 4;   // the q tile's descriptors: w's plus this start offset
        constexpr uint32_t idT = bw::idesc_io(128, 64, 0, 0, F16);     // N = 64 tokens, B K-major
        constexpr uint32_t idK = bw::idesc_io(128, 128, 0, 1, F16);    // N = 128 keys, B MN-major
        // O2 of a chunk: v'^T P^T, then its output and its stage are complete
        auto issue_o2 = [&](int cc) {
            const uint64_t so = (uint64_t)((cc % kNS) * L::kStage) >> 4;
            const uint32_t vp = cVP + 32 * (cc & 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ta(tmem + (GATED ? cO1 : cO2), tmem + vp + 8 * kk, pd[kk] + so, idT, GATED ? 1u : (uint32_t)(kk > 0));
            bw::mma_commit_warp(&barO);
            bw::mma_commit_warp(&empty[cc % kNS]);
        };
        bool ok = true;
        for (int c = 0; c < NT; ++c) {
            const int s = c % kNS;
            const uint32_t hb = cHB + 64 * (c & 1);                 // h_c^T
            const uint64_t so = (uint64_t)(s * L::kStage) >> 4;     // the stage's start-address offset
            if (!bw::mbar_wait(&full[s], (c / kNS) & 1, err, kDeviceErrTimeout)) { ok = false; break; }
            if (!bw::mbar_wait(&hbReady, c & 1, err, kDeviceErrTimeout)) { ok = false; break; }
            bw::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_ta(tmem + cD, tmem + hb + 8 * kk, wd[kk] + so, idT, kk > 0);
            bw::mma_commit_warp(&barD);
            // the previous chunk's O2 runs while the CUDA cores form this chunk's v'
            if (c >= 1) issue_o2(c - 1);
            if (!bw::mbar_wait(&vpReady, c & 1, err, kDeviceErrTimeout)) { ok = false; break; }
            bw::tc_fence_after();
            const uint32_t va = GATED ? cVP + 32 * (c & 1) : cVG;    // v' (against kg) or (v' diag gamma)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ta(tmem + cD, tmem + va + 8 * kk, kd[kk] + so, idK, kk > 0);
            bw::mma_commit_warp(&barE);
            // O1 runs while the CUDA cores update h; the previous chunk's output must have been read
            if (c >= 1 && !bw::mbar_wait(&oFree, (c - 1) & 1, err, kDeviceErrTimeout)) { ok = false; break; }
            bw::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_ta(tmem + cO1, tmem + hb + 8 * kk, wd[kk] + so + kQoff, idT, kk > 0);
        }
        if (ok && NT > 0) issue_o2(NT - 1);
        // nothing of this CTA's may still be running on the tensor cores when it frees the TMEM
        bw::mma_commit_warp(&drain);
        bw::mbar_wait(&drain, 0, err, kDeviceErrTimeout);
    } else {
        // ------------------------------------------------------------ chain warps
        const int sp = warp & 3, part = (warp - kWarp0) >> 2;
        const int v = sp * 32 + lane;                      // this thread's value column (its TMEM lane)
        const uint32_t lb = tmem + ((uint32_t)(sp * 32) << 16);
        const int key0 = part * 32, tok0 = part * 16;
        const int64_t state = ((int64_t)b * H + h) * kK;
        float hs[32];                                     // h[key0 + j][v], fp32 for the whole sequence
#pragma unroll
        for (int j = 0; j < 32; ++j) hs[j] = h0 ? h0[(state + key0 + j) * kV + v] : 0.f;
        auto store_h = [&](int buf) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[j] = bw::pack_io<F16>(hs[2 * j], hs[2 * j + 1]);
            tmem_st16(lb + cHB + 64 * buf + part * 16, pk);
            tmem_st_wait();
            bw::tc_fence_before();
            __syncwarp();
            if (lane == 0) bw::mbar_arrive(&hbReady);
        };
        // o = scale (exp(G_t) O1^T + O2^T) of chunk cc, tokens tok0 .. tok0 + 15; then its stage is released
        auto epilogue = [&](int cc) -> bool {
            if (!bw::mbar_wait(&barO, cc & 1, err, kDeviceErrTimeout)) return false;
            bw::tc_fence_after();
            float a[16], e[16];
            bw::tmem_ld16(lb + cO1 + tok0, a);
            if constexpr (!GATED) bw::tmem_ld16(lb + cO2 + tok0, e);
            bw::tmem_ld_wait();
            bw::tc_fence_before();
            __syncwarp();
            if (lane == 0) bw::mbar_arrive(&oFree);
            const float* F = reinterpret_cast<const float*>(sm + L::F + (cc % kNS) * L::kF);
            const int tt = cc * kC + tok0;
            const float4* e4 = reinterpret_cast<const float4*>(F + kC + tok0);
            float r[16];
            if constexpr (GATED) {   // o = scale (O1^T + O2^T), one accumulator
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 x = __fmul2_rn(make_float2(scale, scale), make_float2(a[2 * j], a[2 * j + 1]));
                    r[2 * j] = x.x;
                    r[2 * j + 1] = x.y;
                }
            }
#pragma unroll
            for (int j4 = 0; j4 < (GATED ? 0 : 4); ++j4) {
                const float4 eg = e4[j4];
                const float2 r0 = __fmul2_rn(make_float2(scale, scale),
                                             __ffma2_rn(make_float2(eg.x, eg.y), make_float2(a[4 * j4], a[4 * j4 + 1]),
                                                        make_float2(e[4 * j4], e[4 * j4 + 1])));
                const float2 r1 = __fmul2_rn(make_float2(scale, scale),
                                             __ffma2_rn(make_float2(eg.z, eg.w), make_float2(a[4 * j4 + 2], a[4 * j4 + 3]),
                                                        make_float2(e[4 * j4 + 2], e[4 * j4 + 3])));
                r[4 * j4] = r0.x; r[4 * j4 + 1] = r0.y; r[4 * j4 + 2] = r1.x; r[4 * j4 + 3] = r1.y;
            }
            // lanes v, v^1 swap halves of their token pairs: the even lane stores columns v, v+1 of token
            // 2m, the odd lane columns v-1, v of token 2m+1 (one 4-byte store per pair of tokens)
            const int odd = lane & 1;
            bf16* dst = o + (((int64_t)b * T + tt + odd) * H + h) * kV + (v & ~1);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint32_t pk = bw::pack_io<F16>(r[2 * m], r[2 * m + 1]);
                const uint32_t ot = __shfl_xor_sync(0xffffffffu, pk, 1);
                const uint32_t word = odd ? __byte_perm(ot, pk, 0x7632) : __byte_perm(pk, ot, 0x5410);
                if (!GENERAL || tt + 2 * m + odd < T)
                    *reinterpret_cast<uint32_t*>(dst + (int64_t)(2 * m) * H * kV) = word;
            }
            __syncwarp();
            if (lane == 0) bw::mbar_arrive(&empty[cc % kNS]);
            return true;
        };
        store_h(0);
        bool ok = true;
        for (int c = 0; c < NT; ++c) {
            const int s = c % kNS;
            if (!bw::mbar_wait(&full[s], (c / kNS) & 1, err, kDeviceErrTimeout)) { ok = false; break; }
            const unsigned char* us = sm + s * L::kStage + L::U;
            const float* F = reinterpret_cast<const float*>(sm + L::F + s * L::kF);
            float uu[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                uu[j] = bw::load_io<F16>(us + (tok0 + j) * (kV * 2) + v * 2);
            // v'^T = u^T - D^T for tokens tok0 .. tok0 + 15
            if (!bw::mbar_wait(&barD, c & 1, err, kDeviceErrTimeout)) { ok = false; break; }
            bw::tc_fence_after();
            {
                float d[16];
                bw::tmem_ld16(lb + cD + tok0, d);
                bw::tmem_ld_wait();
                uint32_t pv[8], pg[8];
                const float4* g4 = reinterpret_cast<const float4*>(F + tok0);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 x0 = __ffma2_rn(make_float2(d[4 * j], d[4 * j + 1]), make_float2(-1.f, -1.f),
                                                 make_float2(uu[4 * j], uu[4 * j + 1]));
                    const float2 x1 = __ffma2_rn(make_float2(d[4 * j + 2], d[4 * j + 3]), make_float2(-1.f, -1.f),
                                                 make_float2(uu[4 * j + 2], uu[4 * j + 3]));
                    pv[2 * j] = bw::pack_io<F16>(x0.x, x0.y);
                    pv[2 * j + 1] = bw::pack_io<F16>(x1.x, x1.y);
                    if constexpr (!GATED) {
                        const float4 gm = g4[j];
                        const float2 y0 = __fmul2_rn(x0, make_float2(gm.x, gm.y));
                        const float2 y1 = __fmul2_rn(x1, make_float2(gm.z, gm.w));
                        pg[2 * j] = bw::pack_io<F16>(y0.x, y0.y);
                        pg[2 * j + 1] = bw::pack_io<F16>(y1.x, y1.y);
                    }
                }
                tmem_st8(lb + cVP + 32 * (c & 1) + tok0 / 2, pv);
                if constexpr (!GATED) tmem_st8(lb + cVG + tok0 / 2, pg);
                tmem_st_wait();
            }
            bw::tc_fence_before();
            __syncwarp();
            if (lane == 0) bw::mbar_arrive(&vpReady);
            // the previous chunk's output, while the tensor cores form dh
            if (c >= 1 && !epilogue(c - 1)) { ok = false; break; }
            // h^T = exp(G_last) h^T + dh^T for keys key0 .. key0 + 31
            if (!bw::mbar_wait(&barE, c & 1, err, kDeviceErrTimeout)) { ok = false; break; }
            bw::tc_fence_after();
            {
                float d[32];
                bw::tmem_ld32(lb + cD + key0, d);
                bw::tmem_ld_wait();
                if constexpr (GATED) {   // exp(G_last) per key
                    const float2* dk = reinterpret_cast<const float2*>(F + key0);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float2 r = __ffma2_rn(dk[j], make_float2(hs[2 * j], hs[2 * j + 1]),
                                                    make_float2(d[2 * j], d[2 * j + 1]));
                        hs[2 * j] = r.x;
                        hs[2 * j + 1] = r.y;
                    }
                } else {
                    const float dec = F[2 * kC];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float2 r = __ffma2_rn(make_float2(dec, dec), make_float2(hs[2 * j], hs[2 * j + 1]),
                                                    make_float2(d[2 * j], d[2 * j + 1]));
                        hs[2 * j] = r.x;
                        hs[2 * j + 1] = r.y;
                    }
                }
            }
            store_h((c + 1) & 1);
        }
        if (ok && NT > 0) epilogue(NT - 1);
        if (h_final) {
#pragma unroll
            for (int j = 0; j < 32; ++j) h_final[(state + key0 + j) * kV + v] = hs[j];
        }
    }
    bw::tc_fence_before();
    __syncthreads();
    if (warp == 1) bw::tmem_dealloc(tmem, 512);
}

}  // namespace

bool tc_scan_output_supported(const Dims& d) {
    // fp16 io: scalar gate (the prepare's fp16 form)
    const bool io = d.bf16 || (d.f16 && !d.per_k);
    return io && d.K == kK && d.V == kV && d.C == kC && (int64_t)d.B * d.H <= 0x7fffffff;
}

cudaError_t tc_scan_output(const Dims& d, const void* q, const void* k, const void* w, const void* u,
                           const float* g_cum, const void* P, const float* h0, void* o, float* h_final,
                           cudaStream_t s, unsigned int* err, bool pdl) {
    if (!tc_scan_output_supported(d) || !P) return cudaErrorInvalidValue;
    // a per-key-dim gate takes the gated operands qg, kg in place of q, k: one per value head
    const int hq = d.per_k ? d.H : d.Hk;
    CUtensorMap mw, mq, mk, mu, mp;
    if (!make_tmap_tokens(&mw, w, d.B, d.T, d.H, kK, kC) || !make_tmap_tokens(&mq, q, d.B, d.T, hq, kK, kC) ||
        !make_tmap_tokens(&mk, k, d.B, d.T, hq, kK, kC) || !make_tmap_tokens_plain(&mu, u, d.B, d.T, d.H, kV, kV, kC))
        return cudaErrorInvalidValue;
    // P [B, NT, H, C, C] seen as (C, C, H, B*NT); one 64 x 64 box per chunk
    const uint64_t dims[4] = {(uint64_t)kC, (uint64_t)kC, (uint64_t)d.H, (uint64_t)d.B * d.NT};
    const uint64_t st[3] = {(uint64_t)kC * 2, (uint64_t)kC * kC * 2, (uint64_t)d.H * kC * kC * 2};
    const uint32_t box[4] = {64, 64, 1, 1};
    if (!make_tmap_bf16_4d(&mp, P, dims, st, box)) return cudaErrorInvalidValue;
    const size_t smem = TcLayout::bytes + 1024;
    const bool general = d.T % kC != 0 || (!d.per_k && d.G != 1);
    auto kern = d.f16 ? (general ? tc_scan_output_kernel<true, false, true> : tc_scan_output_kernel<false, false, true>)
                : d.per_k ? (general ? tc_scan_output_kernel<true, true, false> : tc_scan_output_kernel<false, true, false>)
                          : (general ? tc_scan_output_kernel<true, false, false>
                                     : tc_scan_output_kernel<false, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (pdl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(d.B * d.H);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, mw, mq, mk, mu, mp, g_cum, h0, (bf16*)o, h_final, d.T, d.H, d.NT, d.G,
                                  d.scale, err);
    }
    kern<<<d.B * d.H, kThreads, smem, s>>>(mw, mq, mk, mu, mp, g_cum, h0, (bf16*)o, h_final, d.T, d.H, d.NT, d.G,
                                          d.scale, err);
    return cudaGetLastError();
}

}  // namespace gdr
