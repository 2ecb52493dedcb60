// Tensor-core state scan for bf16 io (the re-scan of
// "kernel_fun/kda/_kernels/bwd_scan.py", module docstring: hck[c] = h before the
// update, v' = u - w h, h = exp(decay) h + kg^T v').
//
// One CTA per (batch, head, BV value columns), serial over chunks; h [K x BV]
// stays on chip for the whole sequence.  Warps 4-7 produce: TMA for the w and
// u chunk tiles, and kg = k exp(G_last - G) (with the decay row G_last) built
// from global memory straight into a 2-stage ring.  Warps 0-3 run the
// recurrence, one TMEM lane (one accumulator row) per thread:
//
//   MMA a    D_a = h^T w^T   [BV x C]   A = h (bf16, MN-major), B = w (K-major)
//   SIMT     v'^T = u^T - D_a  -> bf16 v'^T (K-major B of MMA b) and v' (TMA-stored as v_new)
//   MMA b    D_b = kg^T v'   [K x BV]   A = kg (MN-major)
//   SIMT     h = exp(G_last) * h + D_b in fp32 registers (the master copy), then
//            bf16 h (double-buffered) for the next MMA a; TMA stores it as the
//            next checkpoint
//
// Every operand is read in the layout TMA or the owning thread produces, so
// nothing is transposed; the recurrence threads touch no global memory inside
// the chunk loop.
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

__device__ __forceinline__ void consumer_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int K, int BV, int C, bool PER_K>
struct ScanLayout {
    static constexpr int NS = 2;                                  // ring stages
    static constexpr int GW = PER_K ? K : 1;
    static constexpr uint32_t kKC = C * K * 2;                    // [C][K] bf16 tile
    static constexpr uint32_t kCB = C * BV * 2;                   // [C][BV] bf16 tile
    static constexpr uint32_t kHB = K * BV * 2;                   // [K][BV] bf16 tile
    static constexpr uint32_t W = 0;                              // ring: w
    static constexpr uint32_t KG = W + NS * kKC;                  // ring: kg
    static constexpr uint32_t U = KG + NS * kKC;                  // ring: u
    static constexpr uint32_t Hs = U + NS * kCB;                  // h, two buffers
    static constexpr uint32_t VP = Hs + 2 * kHB;                  // v'^T [BV][64] (C columns used)
    static constexpr uint32_t VN = VP + BV * 128;                 // v' staging for the v_new store, two buffers
    static constexpr uint32_t GL = VN + 2 * kCB;                  // ring: decay row G_last [GW]
    static constexpr int GWS = GW < 4 ? 4 : GW;                  // ring stride of the decay row
    static constexpr uint32_t bytes = GL + NS * 4 * GWS;
    static constexpr uint32_t tx = kKC + kCB;                     // TMA bytes per ring stage
    static constexpr uint32_t full_count = 128 + 1;               // 128 producer arrivals + the expect_tx
    static constexpr uint32_t tmem_cols = 256;                    // D_a at 0 (C cols), D_b at 64 (BV cols)
    static_assert(bytes + 1024 <= 232448, "scan shared memory");
};

template <int K, int BV, int C, bool PER_K>
__global__ void __launch_bounds__(256, 1)
tc_scan_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mu,
               const __grid_constant__ CUtensorMap mvn, const __grid_constant__ CUtensorMap mck,
               const bf16* __restrict__ k, const float* __restrict__ g_cum, const float* __restrict__ h0,
               int has_ckpt, float* __restrict__ h_final, int T, int H, int V, unsigned int* err) {
    using L = ScanLayout<K, BV, C, PER_K>;
    constexpr int GW = L::GW;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* sGL = reinterpret_cast<float*>(sm + L::GL);
    __shared__ uint64_t full[L::NS], empty[L::NS], bar_a, bar_b;
    __shared__ uint32_t tslot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.x * BV, h = blockIdx.y, b = blockIdx.z;
    const int NT = T / C;
    const uint32_t s_base = bw::smem_u32(sm);
    auto row = [&](int t) -> int64_t { return ((int64_t)b * T + t) * H + h; };

    if (tid == 0) {
        for (int s = 0; s < L::NS; ++s) {
            bw::mbar_init(&full[s], L::full_count);
            bw::mbar_init(&empty[s], 1);
        }
        bw::mbar_init(&bar_a, 1);
        bw::mbar_init(&bar_b, 1);
        bw::fence_mbar_init();
    }
    if (warp == 0) {
        bw::tmem_alloc(&tslot, L::tmem_cols);
        bw::tmem_relinquish();
    }
    __syncthreads();
    bw::tc_fence_after();
    const uint32_t tmem = tslot;

    if (warp >= 4) {
        // ---------------------------------------------------------------- producers (128 threads)
        // Thread pt builds the same 8-column slice lc of kg for NI rows of every chunk;
        // all of a chunk's global loads are issued before any is used.
        const int pt = tid - 128;
        constexpr int LC = K / 8;                  // 16-byte column slices per row
        constexpr int RSTEP = 128 / LC;            // rows between a thread's items
        constexpr int NI = C / RSTEP;              // items per thread per chunk
        const int lc = pt % LC, r0 = pt / LC;
        constexpr int GV = PER_K ? 8 : 1;          // gate values per item
        uint4 kr[NI];
        float gr[NI][GV], gl8[GV];
        // global loads of chunk c's k and cumulative gates, all issued together;
        // called for chunk c+1 before waiting for its ring slot, so their latency
        // overlaps the recurrence of the chunks in flight
        auto load_chunk = [&](int c) {
            const int t0 = c * C;
            const float* gl = g_cum + row(t0 + C - 1) * GW;
#pragma unroll
            for (int j = 0; j < NI; ++j) {
                const int t = r0 + j * RSTEP;
                kr[j] = *reinterpret_cast<const uint4*>(k + row(t0 + t) * K + lc * 8);
                if constexpr (PER_K) {
                    const float4* gt = reinterpret_cast<const float4*>(g_cum + row(t0 + t) * K + lc * 8);
                    *reinterpret_cast<float4*>(&gr[j][0]) = gt[0];
                    *reinterpret_cast<float4*>(&gr[j][4]) = gt[1];
                } else {
                    gr[j][0] = g_cum[row(t0 + t)];
                }
            }
            if constexpr (PER_K) {
                const float4* g8 = reinterpret_cast<const float4*>(gl + lc * 8);
                *reinterpret_cast<float4*>(&gl8[0]) = g8[0];
                *reinterpret_cast<float4*>(&gl8[4]) = g8[1];
            } else {
                gl8[0] = gl[0];
            }
        };
        if (NT > 0) load_chunk(0);
        for (int c = 0; c < NT; ++c) {
            const int s = c % L::NS;
            if (!bw::mbar_wait(&empty[s], ((c / L::NS) & 1) ^ 1, err, kDeviceErrTimeout)) break;
            const int t0 = c * C;
            if (pt == 0) {
                bw::mbar_arrive_expect_tx(&full[s], L::tx);
#pragma unroll
                for (int a = 0; a < K / 64; ++a)
                    bw::tma_load_4d(sm + L::W + s * L::kKC + a * C * 128, &mw, &full[s], a * 64, h, t0, b);
#pragma unroll
                for (int a = 0; a < BV / 64; ++a)
                    bw::tma_load_4d(sm + L::U + s * L::kCB + a * C * 128, &mu, &full[s], v0 + a * 64, h, t0, b);
            }
            if constexpr (PER_K) {
                const float* gl = g_cum + row(t0 + C - 1) * GW;
                for (int d = pt; d < K; d += 128) sGL[s * L::GWS + d] = gl[d];
            } else {
                if (pt == 0) sGL[s * L::GWS] = gl8[0];
            }
            unsigned char* kg_t = sm + L::KG + s * L::kKC;
#pragma unroll
            for (int j = 0; j < NI; ++j) {
                const int t = r0 + j * RSTEP;
                const bf16* kv = reinterpret_cast<const bf16*>(&kr[j]);
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float dg = PER_K ? gl8[e % GV] - gr[j][e % GV] : gl8[0] - gr[j][0];
                    f[e] = __bfloat162float(kv[e]) * __expf(dg);
                }
                uint4 p;
                p.x = bw::pack_bf16(f[0], f[1]); p.y = bw::pack_bf16(f[2], f[3]);
                p.z = bw::pack_bf16(f[4], f[5]); p.w = bw::pack_bf16(f[6], f[7]);
                *reinterpret_cast<uint4*>(kg_t + (lc >> 3) * C * 128 + t * 128 + (((lc & 7) ^ (t & 7)) << 4)) = p;
            }
            bw::fence_async_shared();
            bw::mbar_arrive(&full[s]);
            if (c + 1 < NT) load_chunk(c + 1);
        }
    } else {
        // ---------------------------------------------------------------- recurrence (128 threads)
        const int rd = (K == 128) ? tid : m64_row(warp, lane);    // row of D_b (= row of h) held here
        const int rv = (BV == 128) ? tid : m64_row(warp, lane);   // row of D_a (= a value column) held here
        const int64_t state = ((int64_t)b * H + h) * K;

        float hreg[BV];
#pragma unroll
        for (int j = 0; j < BV; ++j) hreg[j] = 0.f;
        if (rd >= 0 && h0) {
            const float4* src = reinterpret_cast<const float4*>(h0 + (state + rd) * V + v0);
#pragma unroll
            for (int j = 0; j < BV / 4; ++j) {
                const float4 x = src[j];
                hreg[4 * j] = x.x; hreg[4 * j + 1] = x.y; hreg[4 * j + 2] = x.z; hreg[4 * j + 3] = x.w;
            }
        }
        auto put_h_smem = [&](int buf) {
            if (rd < 0) return;
            unsigned char* dst = sm + L::Hs + buf * L::kHB;
#pragma unroll
            for (int j = 0; j < BV; j += 8) {
                uint4 p;
                p.x = bw::pack_bf16(hreg[j], hreg[j + 1]);
                p.y = bw::pack_bf16(hreg[j + 2], hreg[j + 3]);
                p.z = bw::pack_bf16(hreg[j + 4], hreg[j + 5]);
                p.w = bw::pack_bf16(hreg[j + 6], hreg[j + 7]);
                *reinterpret_cast<uint4*>(dst + tile_off_r(rd, j, K)) = p;
            }
        };
        auto store_ckpt = [&](int c, int buf) {   // thread 0: checkpoint c from h buffer `buf`
#pragma unroll
            for (int a = 0; a < BV / 64; ++a)
                bw::tma_store_4d(&mck, sm + L::Hs + buf * L::kHB + a * K * 128, v0 + a * 64, 0, h, b * NT + c);
            bw::bulk_commit();
        };
        put_h_smem(0);
        bw::fence_async_shared();
        consumer_barrier();
        if (tid == 0 && has_ckpt) store_ckpt(0, 0);

        bool ok = true;
        for (int c = 0; c < NT; ++c) {
            const int s = c % L::NS, hb = c & 1;
            const int t0 = c * C;
            ok = ok && bw::mbar_wait(&full[s], (c / L::NS) & 1, err, kDeviceErrTimeout);
            const unsigned char* u_t = sm + L::U + s * L::kCB;

            // MMA a: D_a[BV x C] = h^T w^T
            if (tid == 0 && ok) {
                bw::tc_fence_after();
                constexpr uint32_t idesc = bw::idesc_bf16(BV, C, 1, 0);
                const uint32_t h_t = s_base + L::Hs + hb * L::kHB;
                const uint32_t w_t = s_base + L::W + s * L::kKC;
#pragma unroll
                for (int kk = 0; kk < K / 16; ++kk)
                    bw::mma_bf16(tmem, desc_mnmajor_r(h_t, kk, K), desc_kmajor_r(w_t, kk, C), idesc, kk > 0);
                bw::mma_commit(&bar_a);
            }

            // v'^T = u^T - D_a
            ok = ok && bw::mbar_wait(&bar_a, c & 1, err, kDeviceErrTimeout);
            bw::tc_fence_after();
            float vp[C];
#pragma unroll
            for (int t = 0; t < C; t += 32) bw::tmem_ld32(tmem_at(tmem, warp, t), vp + t);
            bw::tmem_ld_wait();
            if (rv >= 0) {
                unsigned char* vn = sm + L::VN + hb * L::kCB;
                // all u loads of a 16-row block first (no stores in between, so they overlap), then the stores
#pragma unroll
                for (int t0h = 0; t0h < C; t0h += 16) {
                    bf16 uu[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) uu[t] = *reinterpret_cast<const bf16*>(u_t + tile_off_r(t0h + t, rv, C));
#pragma unroll
                    for (int t = 0; t < 16; ++t) vp[t0h + t] = __bfloat162float(uu[t]) - vp[t0h + t];
                }
#pragma unroll
                for (int t = 0; t < C; ++t)
                    *reinterpret_cast<bf16*>(vn + tile_off_r(t, rv, C)) = __float2bfloat16_rn(vp[t]);
#pragma unroll
                for (int t = 0; t < C; t += 8) {
                    uint4 p;
                    p.x = bw::pack_bf16(vp[t], vp[t + 1]);
                    p.y = bw::pack_bf16(vp[t + 2], vp[t + 3]);
                    p.z = bw::pack_bf16(vp[t + 4], vp[t + 5]);
                    p.w = bw::pack_bf16(vp[t + 6], vp[t + 7]);
                    *reinterpret_cast<uint4*>(sm + L::VP + tile_off_r(rv, t, BV)) = p;
                }
            }
            bw::fence_async_shared();
            bw::tc_fence_before();
            // every bulk store but the newest (the last checkpoint) has read its smem
            // source: the h buffer and v' staging reused from here on are free
            if (tid == 0) bw::bulk_wait_read<1>();
            consumer_barrier();

            // MMA b: D_b[K x BV] = kg^T v';  store v_new of this chunk
            if (tid == 0 && ok) {
                bw::tc_fence_after();
                constexpr uint32_t idesc = bw::idesc_bf16(K, BV, 1, 0);
                const uint32_t kg_t = s_base + L::KG + s * L::kKC;
#pragma unroll
                for (int kk = 0; kk < C / 16; ++kk)
                    bw::mma_bf16(tmem + 64, desc_mnmajor_r(kg_t, kk, C), desc_kmajor_r(s_base + L::VP, kk, BV),
                                 idesc, kk > 0);
                bw::mma_commit(&bar_b);
#pragma unroll
                for (int a = 0; a < BV / 64; ++a)
                    bw::tma_store_4d(&mvn, sm + L::VN + hb * L::kCB + a * C * 128, v0 + a * 64, h, t0, b);
                bw::bulk_commit();
            }

            // h = exp(G_last) h + D_b
            ok = ok && bw::mbar_wait(&bar_b, c & 1, err, kDeviceErrTimeout);
            bw::tc_fence_after();
            const float* gl = sGL + s * L::GWS;
            const float decay = __expf(PER_K ? gl[rd < 0 ? 0 : rd] : gl[0]);
#pragma unroll
            for (int j = 0; j < BV; j += 32) {
                float dv[32];
                bw::tmem_ld32(tmem_at(tmem, warp, 64 + j), dv);
                bw::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) hreg[j + e] = decay * hreg[j + e] + dv[e];
            }
            put_h_smem(hb ^ 1);
            bw::fence_async_shared();
            bw::tc_fence_before();
            consumer_barrier();
            if (tid == 0) {
                bw::mbar_arrive(&empty[s]);
                if (has_ckpt && c + 1 < NT) store_ckpt(c + 1, hb ^ 1);
            }
        }
        if (h_final && rd >= 0) {
            float4* dst = reinterpret_cast<float4*>(h_final + (state + rd) * V + v0);
#pragma unroll
            for (int j = 0; j < BV / 4; ++j)
                dst[j] = make_float4(hreg[4 * j], hreg[4 * j + 1], hreg[4 * j + 2], hreg[4 * j + 3]);
        }
        if (tid == 0) bw::bulk_wait<0>();
    }
    bw::tc_fence_before();
    __syncthreads();
    if (warp == 0) bw::tmem_dealloc(tmem, L::tmem_cols);
}

template <int K, int BV, int C, bool PER_K>
cudaError_t launch_scan(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum,
                        const float* h0, void* h_ckpt, void* v_new, float* h_final, cudaStream_t s,
                        unsigned int* err) {
    using L = ScanLayout<K, BV, C, PER_K>;
    CUtensorMap mw, mu, mvn, mck;
    if (!make_tmap_tokens(&mw, w, d.B, d.T, d.H, K, C) || !make_tmap_tokens(&mu, u, d.B, d.T, d.H, d.V, C) ||
        !make_tmap_tokens(&mvn, v_new, d.B, d.T, d.H, d.V, C))
        return cudaErrorInvalidValue;
    // without checkpoints the map is never used; point it at v_new so it still encodes
    if (!(h_ckpt ? make_tmap_ckpt(&mck, h_ckpt, d.B, d.NT, d.H, K, d.V)
                 : make_tmap_tokens(&mck, v_new, d.B, d.T, d.H, d.V, C)))
        return cudaErrorInvalidValue;
    auto kern = tc_scan_kernel<K, BV, C, PER_K>;
    const size_t smem = L::bytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(d.V / BV, d.H, d.B);
    kern<<<grid, 256, smem, s>>>(mw, mu, mvn, mck, (const bf16*)k, g_cum, h0, h_ckpt != nullptr, h_final, d.T,
                                 d.H, d.V, err);
    return cudaGetLastError();
}

template <int K, int BV, int C>
cudaError_t scan_gate(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum,
                      const float* h0, void* h_ckpt, void* v_new, float* h_final, cudaStream_t s, unsigned int* err) {
    return d.per_k ? launch_scan<K, BV, C, true>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err)
                   : launch_scan<K, BV, C, false>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err);
}

template <int K, int BV>
cudaError_t scan_chunk(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum,
                       const float* h0, void* h_ckpt, void* v_new, float* h_final, cudaStream_t s, unsigned int* err) {
    return d.C == 32 ? scan_gate<K, BV, 32>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err)
                     : scan_gate<K, BV, 64>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err);
}

}  // namespace

cudaError_t tc_scan(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum, const float* h0,
                    void* h_ckpt, void* v_new, float* h_final, cudaStream_t s, unsigned int* err) {
    if (!d.bf16) return cudaErrorInvalidValue;
    // one CTA per (batch, head) and 64 or 128 value columns
    if (d.K == 64 && d.V == 64) return scan_chunk<64, 64>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err);
    if (d.K == 64) return scan_chunk<64, 128>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err);
    if (d.V == 64) return scan_chunk<128, 64>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err);
    return scan_chunk<128, 128>(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err);
}

}  // namespace gdr
