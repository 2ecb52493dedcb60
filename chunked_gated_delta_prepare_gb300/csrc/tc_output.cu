// Tensor-core chunk output for bf16 and fp16 io:
//     o = scale * [ (q * exp(G)) h_c + tril_0(Q~) v' ],   Q~_ij = sum_d q_id k_jd exp(G_id - G_jd)
// (the output assembly that the re-scan page, "kernel_fun/kda/_kernels/bwd_scan.py",
// says the forward's epilogue warps performed).
//
// One CTA of 128 threads per 64-token tile of one (batch, head), all V columns:
//   TMA      q, k [64 x K], v' [64 x V], checkpoint(s) h_c [K x V]
//   MMA 1    S = q k^T                      (M=64, N=64; gated copies for a per-key-dim gate)
//   SIMT     P = tril_0(S * exp(G_i - G_j)) -> bf16;  q <- q * exp(G) in place
//   MMA 2    D = (q exp(G)) h_c             (B = checkpoint, MN-major; with C = 32 the
//                                            tile holds two chunks, each with its own h_c)
//   MMA 3    D += P v'                      (B = v', MN-major)
//   SIMT     o = scale * D -> bf16 -> global
//
// OPS (per-key-dim gate, K = V = 128, C = 64): the gated operands of the tcgen05 scan and output kernel
// instead of o.  The CTA forms P and q exp(G) as above, and kg = k exp(G_last - G) beside the gated copy of
// k (G_last the chunk's last row), and stores the three by TMA: no v', no checkpoints, no MMA 2 or 3.
//
// F16 (fp16 io; not with OPS): q, k, v', the checkpoints, P, q exp(G) and o are fp16, MMA 2 and 3 take
// fp16 operands.  A per-key-dim gate's gated copies for S stay bf16 (their factors reach e^40, past
// fp16's range), so MMA 1 is bf16 there and fp16 for a scalar gate.
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
using namespace tc;

constexpr float kExpClamp = 60.f;
constexpr float kExpSafe = 40.f;

template <int K, int V, int C, bool PER_K, bool OPS = false>
struct OutLayout {
    static constexpr int NCH = kTile / C;                          // chunks per tile
    // With a per-key-dim gate the gate is read from global memory (L2) where needed instead of
    // being staged (32 KB), k's gated copy is written over k, and P over that once S is formed:
    // two CTAs per SM.  OPS keeps no v' and no checkpoints, writes q's gated copy over q and sends qg
    // and kg straight to global memory: two tiles, four CTAs per SM.
    static constexpr uint32_t Q = 0;                               // q, then q exp(G) for chunk 0
    static constexpr uint32_t Kt = Q + K * 128;                    // k (per-key-dim gate: then k exp(Gref - G))
    static constexpr uint32_t VP = Kt + K * 128;                   // v' [64][V] (none with OPS)
    static constexpr uint32_t Hc = VP + (OPS ? 0 : V * 128);       // checkpoints [NCH][K][V] (none with OPS)
    static constexpr uint32_t P = PER_K ? Kt : Hc + NCH * K * V * 2;   // P [64][64]
    static constexpr uint32_t Q1 = PER_K ? Hc + (OPS ? 0 : NCH * K * V * 2) : P + 8192;   // C = 32: q exp(G), chunk 1
    static constexpr uint32_t Qa = OPS ? Q : Q1 + (NCH > 1 ? K * 128 : 0);   // per-key-dim gate: q exp(G - Gref)
    static constexpr uint32_t F = OPS ? Q1 : Qa + (PER_K ? K * 128 : 0);     // fp32: G [64] (scalar gate), flag
    static constexpr uint32_t bytes = F + 4 * ((PER_K ? 0 : kTile) + 4);
    static constexpr uint32_t tmem_cols = OPS ? 64 : 256;          // S at 0 (64 cols), D at 64 (V cols)
};

// OPS: mp is the P store map (otherwise unused), kg_out and qg_out [B, T, H, K] the gated operands'
// outputs (otherwise null).
template <int K, int V, int C, bool PER_K, bool OPS = false, bool F16 = false>
__global__ void __launch_bounds__(128, OPS ? 4 : 1)
tc_output_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mvp, const __grid_constant__ CUtensorMap mh,
                 const __grid_constant__ CUtensorMap mp, const float* __restrict__ g_cum,
                 const bf16* __restrict__ q_raw, const bf16* __restrict__ k_raw, bf16* __restrict__ o, int T, int H,
                 int NT, int G, float scale, unsigned int* err, bf16* __restrict__ kg_out = nullptr,
                 bf16* __restrict__ qg_out = nullptr) {
    static_assert(!OPS || (PER_K && C == 64 && K == V), "gated operands: per-key-dim gate, one chunk per tile");
    static_assert(!(OPS && F16), "gated operands: bf16 io");
    using L = OutLayout<K, V, C, PER_K, OPS>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* sG = reinterpret_cast<float*>(sm + L::F);
    int* sFlag = reinterpret_cast<int*>(sG + (PER_K ? 0 : kTile));
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t tslot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * kTile, h = blockIdx.y, b = blockIdx.z;
    const int nvalid = min(kTile, T - t0);
    auto row = [&](int t) -> int64_t { return ((int64_t)b * T + t0 + t) * H + h; };
    auto krow = [&](int t) -> int64_t { return ((int64_t)b * T + t0 + t) * (H / G) + h / G; };   // q/k head h / G
    // per-key-dim gate: 8 consecutive G values of tile row t from global memory; past T the last
    // row's (q and k are zero there, and a bounded gap keeps the exp range check quiet)
    // per-key-dim gate: a thread's rows of G, eight key columns each, for every step of the loops over the
    // tile's 16-byte groups (its column group lc = tid % (K / 8) is the same at every step), by 16-byte loads
    // issued together before any is used
    constexpr int NIT = kTile * (K / 8) / 128;
    auto load_g_rows = [&](float4 (&ga)[NIT][2]) {
#pragma unroll
        for (int j = 0; j < NIT; ++j) {
            const int i = tid + 128 * j, r = i / (K / 8), lc = i % (K / 8);
            const float4* src = reinterpret_cast<const float4*>(g_cum + row(min(r, nvalid - 1)) * K + lc * 8);
            ga[j][0] = src[0];
            ga[j][1] = src[1];
        }
    };
    auto unpack8 = [](const float4 (&a)[2], float* out) {
        out[0] = a[0].x; out[1] = a[0].y; out[2] = a[0].z; out[3] = a[0].w;
        out[4] = a[1].x; out[5] = a[1].y; out[6] = a[1].z; out[7] = a[1].w;
    };
    const uint32_t s_base = bw::smem_u32(sm);

    if (tid == 0) {
        bw::mbar_init(&bar_tma, 1);
        bw::mbar_init(&bar_mma, 1);
        bw::fence_mbar_init();
        *sFlag = 0;
        // the tiles first: their latency runs under the tensor-memory allocation and the gate loads
        const int nch = OPS ? 0 : (nvalid + C - 1) / C;   // checkpoints that exist for this tile
        bw::mbar_arrive_expect_tx(&bar_tma, 2 * K * 128 + (OPS ? 0 : V * 128) + nch * K * V * 2);
#pragma unroll
        for (int a = 0; a < K / 64; ++a) {
            bw::tma_load_4d(sm + L::Q + a * 8192, &mq, &bar_tma, a * 64, h / G, t0, b);
            bw::tma_load_4d(sm + L::Kt + a * 8192, &mk, &bar_tma, a * 64, h / G, t0, b);
        }
        if constexpr (!OPS) {
#pragma unroll
            for (int a = 0; a < V / 64; ++a) bw::tma_load_4d(sm + L::VP + a * 8192, &mvp, &bar_tma, a * 64, h, t0, b);
        }
        for (int ch = 0; ch < nch; ++ch) {
            const int c = t0 / C + ch;
#pragma unroll
            for (int a = 0; a < V / 64; ++a)
                bw::tma_load_4d(sm + L::Hc + ch * K * V * 2 + a * K * 128, &mh, &bar_tma, a * 64, 0, h, b * NT + c);
        }
    }
    // per-key-dim gate: this thread's rows of G, the middle row of each chunk and (OPS) the chunk's last
    // row.  Without OPS (two CTAs per SM) they are loaded here, in flight together with the tiles; OPS
    // loads them after the tiles' wait, in fewer registers, for four CTAs per SM
    float4 ga[NIT][2], gref[L::NCH][2], glast[2];
    auto load_gates = [&]() {
        load_g_rows(ga);
        if constexpr (OPS) {
            const float4* src = reinterpret_cast<const float4*>(g_cum + row(nvalid - 1) * K + (tid % (K / 8)) * 8);
            glast[0] = src[0];
            glast[1] = src[1];
        }
#pragma unroll
        for (int ch = 0; ch < L::NCH; ++ch) {
            const float4* src = reinterpret_cast<const float4*>(
                g_cum + row(min(ch * C + C / 2, nvalid - 1)) * K + (tid % (K / 8)) * 8);
            gref[ch][0] = src[0];
            gref[ch][1] = src[1];
        }
    };
    if constexpr (PER_K && !OPS) load_gates();
    if (warp == 0) {
        __syncwarp();   // thread 0 issued the loads alone; the allocation is warp-wide
        bw::tmem_alloc(&tslot, L::tmem_cols);
        bw::tmem_relinquish();
    }
    if constexpr (!PER_K)
        for (int i = tid; i < kTile; i += 128) sG[i] = i < nvalid ? g_cum[row(i)] : 0.f;
    if (L::NCH > 1 && nvalid <= C) {
        // a half tile: the second chunk's checkpoint is absent; give its rows a zero state
        for (int i = tid; i < K * V / 8; i += 128)
            *reinterpret_cast<uint4*>(sm + L::Hc + K * V * 2 + i * 16) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    bw::tc_fence_after();
    const uint32_t tmem = tslot;
    bool ok = bw::mbar_wait(&bar_tma, 0, err, kDeviceErrTimeout);

    if constexpr (PER_K) {
        if constexpr (OPS) load_gates();
        // OPS: exp(G_ref) and exp(G_last - G_ref) of this thread's eight key columns (the same at every step),
        // so that qg = (q exp(G - G_ref)) exp(G_ref) and kg = (k exp(G_ref - G)) exp(G_last - G_ref) reuse the
        // gated copies' exponentials where |G - G_ref| <= kExpSafe
        float eref[8], elref[8];
        if constexpr (OPS) {
            float gf0[8], gl0[8];
            unpack8(gref[0], gf0);
            unpack8(glast, gl0);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                eref[e] = __expf(gf0[e]);
                elref[e] = __expf(gl0[e] - gf0[e]);
            }
        }
#pragma unroll
        for (int j = 0; j < NIT; ++j) {
            const int i = tid + 128 * j, r = i / (K / 8), lc = i % (K / 8);
            const uint32_t off = (uint32_t)((lc >> 3) * 8192 + r * 128 + (((lc & 7) ^ (r & 7)) << 4));
            const uint4 rq = *reinterpret_cast<const uint4*>(sm + L::Q + off);
            const uint4 rk = *reinterpret_cast<const uint4*>(sm + L::Kt + off);
            float qv[8], kv[8], fa[8], fb[8], gr[8], gf[8];
            bw::unpack8_io<F16>(rq, qv);
            bw::unpack8_io<F16>(rk, kv);
            unpack8(ga[j], gr);
            unpack8(L::NCH > 1 && r >= C ? gref[L::NCH - 1] : gref[0], gf);
            bool big = false;
            float fq[8], fk[8];   // OPS: qg and kg
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float dg = gr[e] - gf[e];
                const bool far = fabsf(dg) > kExpSafe;
                big |= far;
                const float xq = qv[e], xk = kv[e];
                fa[e] = xq * __expf(fminf(fmaxf(dg, -kExpClamp), kExpClamp));
                fb[e] = xk * __expf(fminf(fmaxf(-dg, -kExpClamp), kExpClamp));
                if constexpr (OPS) {
                    if (!far) {
                        fq[e] = fa[e] * eref[e];
                        fk[e] = fb[e] * elref[e];
                    } else {
                        float gl[8];
                        unpack8(glast, gl);
                        fq[e] = xq * __expf(gr[e]);
                        fk[e] = xk * __expf(gl[e] - gr[e]);
                    }
                }
            }
            if (big) *sFlag = 1;
            if constexpr (OPS) {   // qg and kg straight to global memory: 16 threads write a row's 256 bytes
                uint4 pq, pk;
                pq.x = bw::pack_bf16(fq[0], fq[1]); pq.y = bw::pack_bf16(fq[2], fq[3]);
                pq.z = bw::pack_bf16(fq[4], fq[5]); pq.w = bw::pack_bf16(fq[6], fq[7]);
                pk.x = bw::pack_bf16(fk[0], fk[1]); pk.y = bw::pack_bf16(fk[2], fk[3]);
                pk.z = bw::pack_bf16(fk[4], fk[5]); pk.w = bw::pack_bf16(fk[6], fk[7]);
                if (r < nvalid) {
                    *reinterpret_cast<uint4*>(qg_out + row(r) * K + lc * 8) = pq;
                    *reinterpret_cast<uint4*>(kg_out + row(r) * K + lc * 8) = pk;
                }
            }
            uint4 pa, pb;
            pa.x = bw::pack_bf16(fa[0], fa[1]); pa.y = bw::pack_bf16(fa[2], fa[3]);
            pa.z = bw::pack_bf16(fa[4], fa[5]); pa.w = bw::pack_bf16(fa[6], fa[7]);
            pb.x = bw::pack_bf16(fb[0], fb[1]); pb.y = bw::pack_bf16(fb[2], fb[3]);
            pb.z = bw::pack_bf16(fb[4], fb[5]); pb.w = bw::pack_bf16(fb[6], fb[7]);
            *reinterpret_cast<uint4*>(sm + L::Qa + off) = pa;   // OPS: over q, each thread rewriting what it read
            *reinterpret_cast<uint4*>(sm + L::Kt + off) = pb;   // over k: each thread rewrites what it read
        }
        bw::fence_async_shared();
    }
    __syncthreads();

    // MMA 1: S = q k^T
    if (tid == 0 && ok) {
        bw::tc_fence_after();
        constexpr uint32_t idesc = bw::idesc_io(64, 64, 0, 0, F16 && !PER_K);   // gated copies: bf16
        const uint32_t a_t = s_base + (PER_K ? L::Qa : L::Q);
        const uint32_t b_t = s_base + L::Kt;
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) bw::mma_bf16(tmem, desc_kmajor(a_t, kk), desc_kmajor(b_t, kk), idesc, kk > 0);
        bw::mma_commit(&bar_mma);
    }
    ok = ok && bw::mbar_wait(&bar_mma, 0, err, kDeviceErrTimeout);
    bw::tc_fence_after();

    // P = tril_0(S * gate) -> io type, K-major [64][64]
    {
        const int r = m64_row(warp, lane);
        float s[64];
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) bw::tmem_ld16(tmem_at(tmem, warp, c0), s + c0);
        bw::tmem_ld_wait();
        if (r >= 0) {
            const int ch0 = (r / C) * C;
#pragma unroll
            for (int j = 0; j < 64; j += 8) {
                float pv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int jj = j + e;
                    float x = 0.f;
                    if (jj >= ch0 && jj <= r) {
                        if constexpr (PER_K) x = s[jj];
                        else x = s[jj] * __expf(sG[r] - sG[jj]);
                    }
                    pv[e] = x;
                }
                *reinterpret_cast<uint4*>(sm + L::P + bw::sw128_offset(r, j)) = bw::pack8_io<F16>(pv);
            }
        }
    }
    bw::tc_fence_before();
    __syncthreads();
    if (PER_K && *sFlag) {
        // exact fp32 P for chunks with extreme gates
        for (int idx = tid; idx < kTile * kTile; idx += 128) {
            const int i = idx / kTile, j = idx % kTile;
            if (j >= (i / C) * C && j <= i) {
                float acc = 0.f;
                for (int d = 0; d < K; ++d) {
                    // OPS: q's tile now holds q's gated copy, so raw q comes from global memory too
                    const float qi = OPS ? (i < nvalid ? bw::load_io<F16>(q_raw + krow(i) * K + d) : 0.f)
                                         : bw::load_io<F16>(sm + L::Q + tile_off(i, d));
                    // k's tile now holds its gated copy: raw k and G come from global memory (rare path)
                    const float kj = j < nvalid ? bw::load_io<F16>(k_raw + krow(j) * K + d) : 0.f;
                    const float gi = i < nvalid ? g_cum[row(i) * K + d] : 0.f;
                    const float gj = j < nvalid ? g_cum[row(j) * K + d] : 0.f;
                    acc += qi * kj * __expf(gi - gj);
                }
                bw::store_io<F16>(sm + L::P + bw::sw128_offset(i, j), acc);
            }
        }
        __syncthreads();
    }
    if constexpr (OPS) {
        // P leaves by TMA (rows past T clipped); nothing of the output's second half runs
        bw::fence_async_shared();
        __syncthreads();
        if (tid == 0) {
            if (ok) {
                bw::tma_store_4d(&mp, sm + L::P, 0, 0, h, b * NT + t0 / C);
                bw::bulk_commit();
            }
            bw::bulk_wait_read<0>();
        }
        bw::tc_fence_before();
        __syncthreads();
        if (warp == 0) bw::tmem_dealloc(tmem, L::tmem_cols);
        return;
    }

    // q exp(G) in place (and, for two chunks per tile, split by chunk into Q and Q1)
    float4 gq[PER_K ? NIT : 1][2];
    if constexpr (PER_K) load_g_rows(gq);
#pragma unroll
    for (int j = 0; j < NIT; ++j) {
        const int i = tid + 128 * j, r = i / (K / 8), lc = i % (K / 8);
        const uint32_t off = (uint32_t)((lc >> 3) * 8192 + r * 128 + (((lc & 7) ^ (r & 7)) << 4));
        const uint4 raw = *reinterpret_cast<const uint4*>(sm + L::Q + off);
        float f[8], gr[8];
        bw::unpack8_io<F16>(raw, f);
        if constexpr (PER_K) {
            unpack8(gq[j], gr);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) gr[e] = sG[r];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] *= __expf(gr[e]);
        const uint4 p = bw::pack8_io<F16>(f);
        const uint4 zero = make_uint4(0, 0, 0, 0);
        if (L::NCH > 1) {
            const bool first = r < C;
            *reinterpret_cast<uint4*>(sm + L::Q + off) = first ? p : zero;
            *reinterpret_cast<uint4*>(sm + L::Q1 + off) = first ? zero : p;
        } else {
            *reinterpret_cast<uint4*>(sm + L::Q + off) = p;
        }
    }
    bw::fence_async_shared();
    __syncthreads();

    // MMA 2, 3: D = (q exp(G)) h_c + P v'
    if (tid == 0 && ok) {
        bw::tc_fence_after();
        constexpr uint32_t idesc = bw::idesc_io(64, V, 0, 1, F16);
        const uint32_t d_t = tmem + 64;
#pragma unroll
        for (int ch = 0; ch < L::NCH; ++ch) {
            const uint32_t a_t = s_base + (ch == 0 ? L::Q : L::Q1);
            const uint32_t b_t = s_base + L::Hc + ch * K * V * 2;
#pragma unroll
            for (int kk = 0; kk < K / 16; ++kk)
                bw::mma_bf16(d_t, desc_kmajor(a_t, kk), desc_mnmajor_r(b_t, kk, K), idesc, (ch > 0 || kk > 0));
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            bw::mma_bf16(d_t, desc_kmajor(s_base + L::P, kk), desc_mnmajor(s_base + L::VP, kk), idesc, 1);
        bw::mma_commit(&bar_mma);
    }
    ok = ok && bw::mbar_wait(&bar_mma, 1, err, kDeviceErrTimeout);
    bw::tc_fence_after();
    {
        const int r = m64_row(warp, lane);
        const bool store = r >= 0 && r < nvalid && ok;
        bf16* orow = o + (store ? row(r) * V : 0);
#pragma unroll
        for (int c0 = 0; c0 < V; c0 += 16) {
            float v16[16];
            bw::tmem_ld16(tmem_at(tmem, warp, 64 + c0), v16);
            bw::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) v16[e] *= scale;
            if (store) {
                reinterpret_cast<uint4*>(orow + c0)[0] = bw::pack8_io<F16>(v16);
                reinterpret_cast<uint4*>(orow + c0)[1] = bw::pack8_io<F16>(v16 + 8);
            }
        }
    }
    bw::tc_fence_before();
    __syncthreads();
    if (warp == 0) bw::tmem_dealloc(tmem, L::tmem_cols);
}

template <int K, int V, int C, bool PER_K, bool F16>
cudaError_t launch_output(const Dims& d, const void* q, const void* k, const void* v_new, const void* h_ckpt,
                          const float* g_cum, void* o, cudaStream_t s, unsigned int* err) {
    using L = OutLayout<K, V, C, PER_K>;
    CUtensorMap mq, mk, mvp, mh;
    if (!make_tmap_tokens(&mq, q, d.B, d.T, d.Hk, K, kTile) || !make_tmap_tokens(&mk, k, d.B, d.T, d.Hk, K, kTile) ||
        !make_tmap_tokens(&mvp, v_new, d.B, d.T, d.H, V, kTile) || !make_tmap_ckpt(&mh, h_ckpt, d.B, d.NT, d.H, K, V))
        return cudaErrorInvalidValue;
    auto kern = tc_output_kernel<K, V, C, PER_K, false, F16>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((d.T + kTile - 1) / kTile, d.H, d.B);
    kern<<<grid, 128, smem, s>>>(mq, mk, mvp, mh, mh, g_cum, (const bf16*)q, (const bf16*)k, (bf16*)o, d.T, d.H, d.NT,
                                 d.G, d.scale, err, nullptr, nullptr);
    return cudaGetLastError();
}

template <int K, int V, int C>
cudaError_t out_gate(const Dims& d, const void* q, const void* k, const void* v_new, const void* h_ckpt,
                     const float* g_cum, void* o, cudaStream_t s, unsigned int* err) {
    if (d.f16)
        return d.per_k ? launch_output<K, V, C, true, true>(d, q, k, v_new, h_ckpt, g_cum, o, s, err)
                       : launch_output<K, V, C, false, true>(d, q, k, v_new, h_ckpt, g_cum, o, s, err);
    return d.per_k ? launch_output<K, V, C, true, false>(d, q, k, v_new, h_ckpt, g_cum, o, s, err)
                   : launch_output<K, V, C, false, false>(d, q, k, v_new, h_ckpt, g_cum, o, s, err);
}

template <int K, int V>
cudaError_t out_chunk(const Dims& d, const void* q, const void* k, const void* v_new, const void* h_ckpt,
                      const float* g_cum, void* o, cudaStream_t s, unsigned int* err) {
    return d.C == 32 ? out_gate<K, V, 32>(d, q, k, v_new, h_ckpt, g_cum, o, s, err)
                     : out_gate<K, V, 64>(d, q, k, v_new, h_ckpt, g_cum, o, s, err);
}

}  // namespace

cudaError_t tc_gated_operands(const Dims& d, const void* q, const void* k, const float* g_cum, void* P, void* kg,
                              void* qg, cudaStream_t s, unsigned int* err) {
    constexpr int K = 128, V = 128, C = 64;
    if (!d.bf16 || !d.per_k || d.K != K || d.V != V || d.C != C) return cudaErrorInvalidValue;
    using L = OutLayout<K, V, C, true, true>;
    CUtensorMap mq, mk, mkg, mqg, mp;
    const uint64_t dims[4] = {(uint64_t)C, (uint64_t)C, (uint64_t)d.H, (uint64_t)d.B * d.NT};
    const uint64_t st[3] = {(uint64_t)C * 2, (uint64_t)C * C * 2, (uint64_t)d.H * C * C * 2};
    const uint32_t box[4] = {64, 64, 1, 1};
    if (!make_tmap_tokens(&mq, q, d.B, d.T, d.Hk, K, kTile) || !make_tmap_tokens(&mk, k, d.B, d.T, d.Hk, K, kTile) ||
        !make_tmap_bf16_4d(&mp, P, dims, st, box))
        return cudaErrorInvalidValue;
    mkg = mq;   // unused by the operands form (qg and kg are plain stores)
    mqg = mq;
    auto kern = tc_output_kernel<K, V, C, true, true>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((d.T + kTile - 1) / kTile, d.H, d.B);
    kern<<<grid, 128, smem, s>>>(mq, mk, mkg, mqg, mp, g_cum, (const bf16*)q, (const bf16*)k, nullptr, d.T, d.H, d.NT,
                                 d.G, d.scale, err, (bf16*)kg, (bf16*)qg);
    return cudaGetLastError();
}

cudaError_t tc_output(const Dims& d, const void* q, const void* k, const void* v_new, const void* h_ckpt,
                      const float* g_cum, void* o, cudaStream_t s, unsigned int* err) {
    if (!d.bf16 && !d.f16) return cudaErrorInvalidValue;
    if (d.K == 64 && d.V == 64) return out_chunk<64, 64>(d, q, k, v_new, h_ckpt, g_cum, o, s, err);
    if (d.K == 64) return out_chunk<64, 128>(d, q, k, v_new, h_ckpt, g_cum, o, s, err);
    if (d.V == 64) return out_chunk<128, 64>(d, q, k, v_new, h_ckpt, g_cum, o, s, err);
    return out_chunk<128, 128>(d, q, k, v_new, h_ckpt, g_cum, o, s, err);
}

}  // namespace gdr
