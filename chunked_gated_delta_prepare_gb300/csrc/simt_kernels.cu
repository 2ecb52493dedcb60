// fp32 CUDA-core kernels for the three stages of the chunked gated delta rule.
//
// This is the exact-fp32 variant: every product and sum is an fp32 FMA on the
// CUDA cores, so an fp32 problem keeps fp32 accuracy end to end.  It runs every
// supported shape (K, V in {64,128}, C in {32,64}, scalar or per-key-dim gate,
// fp32 or bf16 io).  The tensor-core kernels are the fast path for bf16.
//
// Stage math (per batch b, head h, chunk c; G = chunk-local inclusive cumsum of g):
//   prepare ("Reuse P as beta tiles in gated deltanet fused prepare": A_g, its inverse,
//            w = A_g^{-1} k_beta, u = A_g^{-1} v_beta; here k_beta carries exp(G)):
//       A_ij = beta_i sum_d k_id k_jd exp(G_id - G_jd)  (i > j),  X = (I + A)^{-1}
//       w = X (k * beta * exp(G)),  u = X (v * beta)
//   scan ("kernel_fun/kda/_kernels/bwd_scan.py", module docstring):
//       ckpt[c] = h;  v' = u - w h;  h = exp(G_last) * h + (k * exp(G_last - G))^T v'
//   output: o = scale [ (q * exp(G)) ckpt[c] + tril_0(Q~) v' ],  Q~_ij = sum_d q_id k_jd exp(G_id - G_jd)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxChunk = 64;   // C is 32 or 64

__device__ __forceinline__ float ld(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st(__nv_bfloat16* p, int64_t i, float x) { p[i] = __float2bfloat16_rn(x); }
__device__ __forceinline__ float ld(const __half* p, int64_t i) { return __half2float(p[i]); }
__device__ __forceinline__ void st(__half* p, int64_t i, float x) { p[i] = __float2half_rn(x); }

// ------------------------------------------------------------------ prepare
// One CTA per (chunk, head, batch).  Shared memory (fp32):
//   Gs [C][K] or [C]   chunk-local cumsum of g
//   bs [C]             beta
//   ks [C][K+1]        k
//   As [C][C+1]        gated strictly-lower A
//   Xs [C][C+1]        (I + A)^{-1}
//   ys [C][max(K,V)+1] k*beta*exp(G), then reused for v*beta (its lifetimes do not overlap)
template <typename IO, bool PER_K>
__global__ void __launch_bounds__(kThreads, 1)   // the column solve keeps a 64-entry column in registers
simt_prepare_kernel(Dims d, const IO* __restrict__ k, const IO* __restrict__ v, const float* __restrict__ g,
                    const IO* __restrict__ beta, IO* __restrict__ w, IO* __restrict__ u,
                    float* __restrict__ g_cum) {
    extern __shared__ float smem[];
    const int C = d.C, K = d.K, V = d.V, H = d.H;
    const int KP = K + 1, CP = C + 1, YP = (K > V ? K : V) + 1;
    const int GW = PER_K ? K : 1;
    float* Gs = smem;
    float* bs = Gs + C * GW;
    float* ks = bs + C;
    float* As = ks + C * KP;
    float* Xs = As + C * CP;
    float* ys = Xs + C * CP;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const int64_t tok0 = (int64_t)b * d.T + (int64_t)c * C;   // first token of this chunk
    const int nv = min(C, d.T - c * C);                       // tokens of the chunk before T
    auto row = [&](int t) { return (tok0 + t) * H + h; };                 // (token, value head) row index
    auto krow = [&](int t) { return (tok0 + t) * d.Hk + h / d.G; };   // q, k: q/k head h / G

    // tokens past T (a last, partial chunk) read as g = 0, beta = 0, k = v = 0
        for (int i = tid; i < C * GW; i += kThreads) Gs[i] = i / GW < nv ? g[row(i / GW) * GW + i % GW] : 0.f;
    for (int i = tid; i < C; i += kThreads) bs[i] = i < nv ? ld(beta, row(i)) : 0.f;
        for (int i = tid; i < C * K; i += kThreads) ks[(i / K) * KP + i % K] = i / K < nv ? ld(k, krow(i / K) * K + i % K) : 0.f;
    __syncthreads();
    // chunk-local inclusive cumsum, one thread per gate column
    for (int col = tid; col < GW; col += kThreads) {
        float run = 0.f;
        for (int t = 0; t < C; ++t) {
            run += Gs[t * GW + col];
            Gs[t * GW + col] = run;
            if (t < nv) g_cum[row(t) * GW + col] = run;
        }
    }
    __syncthreads();
    // A_ij = beta_i sum_d k_id k_jd exp(G_id - G_jd), i > j: rows i0 .. i0+3 per thread share each load of
    // k_j (four independent sums, each in the same order as one entry alone)
    for (int idx = tid; idx < (C / 4) * C; idx += kThreads) {
        const int i0 = (idx / C) * 4, j = idx % C;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        if (i0 + 3 > j) {
            for (int e = 0; e < K; ++e) {
                const float kj = ks[j * KP + e];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (PER_K) s[r] += ks[(i0 + r) * KP + e] * kj * expf(Gs[(i0 + r) * K + e] - Gs[j * K + e]);
                    else s[r] += ks[(i0 + r) * KP + e] * kj;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = i0 + r;
            float a = 0.f;
            if (i > j) a = PER_K ? bs[i] * s[r] : bs[i] * expf(Gs[i] - Gs[j]) * s[r];
            As[i * CP + j] = a;
        }
    }
    __syncthreads();
    // X = (I + A)^{-1} by forward substitution, one thread per column col, the column in registers:
    // X[col][col] = 1, X[i][col] = -sum_{j=col}^{i-1} A[i][j] X[j][col] for i > col.  The sum runs from
    // j = 0 over the column's zeros above the diagonal, which adds exact zeros: the same sum.
    static_assert(kMaxChunk <= kThreads, "one thread per column");
    if (tid < C) {
        const int col = tid;
        float x[kMaxChunk];
#pragma unroll
        for (int i = 0; i < kMaxChunk; ++i) {
            x[i] = 0.f;
            if (i < C) {
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < i; ++j) s += As[i * CP + j] * x[j];
                x[i] = i < col ? 0.f : (i == col ? 1.f : -s);
            }
        }
#pragma unroll
        for (int i = 0; i < kMaxChunk; ++i)
            if (i < C) Xs[i * CP + col] = x[i];
    }
    for (int i = tid; i < C * K; i += kThreads) {
        const int t = i / K, e = i % K;
        const float gate = expf(Gs[t * GW + (PER_K ? e : 0)]);
        ys[t * YP + e] = ks[t * KP + e] * bs[t] * gate;
    }
    __syncthreads();
    // w = X (k * beta * exp(G)): rows i0 .. i0+3 per thread share each load of the right factor (each
    // row's sum over j <= i in the same order as alone)
    for (int idx = tid; idx < (C / 4) * K; idx += kThreads) {
        const int i0 = (idx / K) * 4, e = idx % K;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j <= i0 + 3; ++j) {
            const float yj = ys[j * YP + e];
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (j <= i0 + r) s[r] += Xs[(i0 + r) * CP + j] * yj;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            if (i0 + r < nv) st(w, row(i0 + r) * K + e, s[r]);
    }
    __syncthreads();
        for (int i = tid; i < C * V; i += kThreads) {
        const int t = i / V, e = i % V;
        ys[t * YP + e] = t < nv ? ld(v, row(t) * V + e) * bs[t] : 0.f;
    }
    __syncthreads();
    // u = X (v * beta), blocked as w
    for (int idx = tid; idx < (C / 4) * V; idx += kThreads) {
        const int i0 = (idx / V) * 4, e = idx % V;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j <= i0 + 3; ++j) {
            const float yj = ys[j * YP + e];
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (j <= i0 + r) s[r] += Xs[(i0 + r) * CP + j] * yj;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            if (i0 + r < nv) st(u, row(i0 + r) * V + e, s[r]);
    }
}

// ------------------------------------------------------------------ scan
// One CTA per (value tile of BV columns, head, batch); serial over chunks.
// Shared memory (fp32): hs [K][BV] state, ws [C][K+1] w, kgs [C][K+1] k*exp(G_last-G),
// us [C][BV+1] u tile, vps [C][BV+1] v', Gl [K] or [1] last-row cumsum.
constexpr int kScanBV = 32;

template <typename IO, bool PER_K>
__global__ void __launch_bounds__(kThreads)
simt_scan_kernel(Dims d, const IO* __restrict__ k, const IO* __restrict__ w, const IO* __restrict__ u,
                 const float* __restrict__ g_cum, const float* __restrict__ h0, IO* __restrict__ h_ckpt,
                 IO* __restrict__ v_new, float* __restrict__ h_final) {
    extern __shared__ float smem[];
    constexpr int BV = kScanBV, BVP = kScanBV + 1;
    const int C = d.C, K = d.K, V = d.V, H = d.H;
    const int KP = K + 1, GW = PER_K ? K : 1;
    float* hs = smem;
    float* ws = hs + K * BV;
    float* kgs = ws + C * KP;
    float* us = kgs + C * KP;
    float* vps = us + C * BVP;
    float* Gl = vps + C * BVP;
    const int vt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int v0 = vt * BV;
    const int tid = threadIdx.x;
    const int64_t state_off = ((int64_t)b * H + h) * K * V;

        for (int i = tid; i < K * BV; i += kThreads) {
        const int e = i / BV, j = i % BV;
        hs[i] = h0 ? h0[state_off + (int64_t)e * V + v0 + j] : 0.f;
    }
    for (int c = 0; c < d.NT; ++c) {
        const int64_t tok0 = (int64_t)b * d.T + (int64_t)c * C;
        const int nv = min(C, d.T - c * C);   // a last, partial chunk: zero w, k, u past T, G held at its last value
        auto row = [&](int t) { return (tok0 + t) * H + h; };
        auto krow = [&](int t) { return (tok0 + t) * d.Hk + h / d.G; };   // q, k: q/k head h / G
        for (int i = tid; i < GW; i += kThreads) Gl[i] = g_cum[row(nv - 1) * GW + i];
        __syncthreads();
        if (h_ckpt) {
            const int64_t ck = (((int64_t)b * d.NT + c) * H + h) * K * V;
            for (int i = tid; i < K * BV; i += kThreads)
                st(h_ckpt, ck + (int64_t)(i / BV) * V + v0 + i % BV, hs[i]);
        }
                for (int i = tid; i < C * K; i += kThreads) {
            const int t = i / K, e = i % K;
            const int gi = PER_K ? e : 0;
            ws[t * KP + e] = t < nv ? ld(w, row(t) * K + e) : 0.f;
            kgs[t * KP + e] = t < nv ? ld(k, krow(t) * K + e) * expf(Gl[gi] - g_cum[row(t) * GW + gi]) : 0.f;
        }
                for (int i = tid; i < C * BV; i += kThreads)
            us[(i / BV) * BVP + i % BV] = i / BV < nv ? ld(u, row(i / BV) * V + v0 + i % BV) : 0.f;
        __syncthreads();
        // v' = u - w h: four rows t0 .. t0+3 per thread share each load of h (four independent sums,
        // each in the same order as one row alone)
        for (int idx = tid; idx < (C / 4) * BV; idx += kThreads) {
            const int t0 = (idx / BV) * 4, j = idx % BV;
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            for (int e = 0; e < K; ++e) {
                const float he = hs[e * BV + j];
#pragma unroll
                for (int r = 0; r < 4; ++r) s[r] += ws[(t0 + r) * KP + e] * he;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = t0 + r;
                const float vp = us[t * BVP + j] - s[r];
                vps[t * BVP + j] = vp;
                if (t < nv) st(v_new, row(t) * V + v0 + j, vp);
            }
        }
        __syncthreads();
        // h = exp(G_last) * h + kg^T v': four key rows per thread share each load of v'
        for (int idx = tid; idx < (K / 4) * BV; idx += kThreads) {
            const int e0 = (idx / BV) * 4, j = idx % BV;
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            for (int t = 0; t < C; ++t) {
                const float vt = vps[t * BVP + j];
#pragma unroll
                for (int r = 0; r < 4; ++r) s[r] += kgs[t * KP + e0 + r] * vt;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int e = e0 + r;
                hs[e * BV + j] = expf(Gl[PER_K ? e : 0]) * hs[e * BV + j] + s[r];
            }
        }
        __syncthreads();
    }
    if (h_final)
        for (int i = tid; i < K * BV; i += kThreads)
            h_final[state_off + (int64_t)(i / BV) * V + v0 + i % BV] = hs[i];
}

// ------------------------------------------------------------------ output
// One CTA per (chunk, head, batch * value tile of 64 columns).
// Shared memory (fp32): qs/ks [C][K+1], Gs [C][K] or [C], Qt [C][C+1], vps [C][65], hs [K][64].
constexpr int kOutVT = 64;

template <typename IO, bool PER_K>
__global__ void __launch_bounds__(kThreads)
simt_output_kernel(Dims d, const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ v_new,
                   const IO* __restrict__ h_ckpt, const float* __restrict__ g_cum, IO* __restrict__ o) {
    extern __shared__ float smem[];
    constexpr int VT = kOutVT, VTP = kOutVT + 1;
    const int C = d.C, K = d.K, V = d.V, H = d.H;
    const int KP = K + 1, CP = C + 1, GW = PER_K ? K : 1;
    const int nvt = V / VT;
    float* qs = smem;
    float* ks = qs + C * KP;
    float* Gs = ks + C * KP;
    float* Qt = Gs + C * GW;
    float* vps = Qt + C * CP;
    float* hs = vps + C * VTP;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z / nvt, vt = blockIdx.z % nvt;
    const int v0 = vt * VT;
    const int tid = threadIdx.x;
    const int64_t tok0 = (int64_t)b * d.T + (int64_t)c * C;
    auto row = [&](int t) { return (tok0 + t) * H + h; };
    auto krow = [&](int t) { return (tok0 + t) * d.Hk + h / d.G; };   // q, k: q/k head h / G
    const int64_t ck = (((int64_t)b * d.NT + c) * H + h) * K * V;
    const int nv = min(C, d.T - c * C);   // a last, partial chunk: zero q, k, v' past T, G held at its last value

        for (int i = tid; i < C * K; i += kThreads) {
        const bool in = i / K < nv;
        qs[(i / K) * KP + i % K] = in ? ld(q, krow(i / K) * K + i % K) : 0.f;
        ks[(i / K) * KP + i % K] = in ? ld(k, krow(i / K) * K + i % K) : 0.f;
    }
        for (int i = tid; i < C * GW; i += kThreads) Gs[i] = g_cum[row(min(i / GW, nv - 1)) * GW + i % GW];
        for (int i = tid; i < C * VT; i += kThreads)
        vps[(i / VT) * VTP + i % VT] = i / VT < nv ? ld(v_new, row(i / VT) * V + v0 + i % VT) : 0.f;
        for (int i = tid; i < K * VT; i += kThreads) hs[i] = ld(h_ckpt, ck + (int64_t)(i / VT) * V + v0 + i % VT);
    __syncthreads();
    // Q~_ij = sum_d q_id k_jd exp(G_id - G_jd), j <= i
    for (int idx = tid; idx < C * C; idx += kThreads) {
        const int i = idx / C, j = idx % C;
        float a = 0.f;
        if (j <= i) {
            float s = 0.f;
            if (PER_K) {
                for (int e = 0; e < K; ++e)
                    s += qs[i * KP + e] * ks[j * KP + e] * expf(Gs[i * K + e] - Gs[j * K + e]);
                a = s;
            } else {
                for (int e = 0; e < K; ++e) s += qs[i * KP + e] * ks[j * KP + e];
                a = expf(Gs[i] - Gs[j]) * s;
            }
        }
        Qt[i * CP + j] = a;
    }
    __syncthreads();
    for (int i = tid; i < C * K; i += kThreads) {
        const int t = i / K, e = i % K;
        qs[t * KP + e] *= expf(Gs[t * GW + (PER_K ? e : 0)]);
    }
    __syncthreads();
    // four rows i0 .. i0+3 per thread share each load of h and of v' (four independent sums, each in the
    // same order as one row alone: the q h terms, then the causal P v' terms)
    for (int idx = tid; idx < (C / 4) * VT; idx += kThreads) {
        const int i0 = (idx / VT) * 4, j = idx % VT;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int e = 0; e < K; ++e) {
            const float he = hs[e * VT + j];
#pragma unroll
            for (int r = 0; r < 4; ++r) s[r] += qs[(i0 + r) * KP + e] * he;
        }
        for (int t = 0; t <= i0 + 3; ++t) {
            const float vt = vps[t * VTP + j];
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (t <= i0 + r) s[r] += Qt[(i0 + r) * CP + t] * vt;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            if (i0 + r < nv) st(o, row(i0 + r) * V + v0 + j, d.scale * s[r]);
    }
}

template <typename Kern>
cudaError_t allow_smem(Kern kern, size_t smem) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace

cudaError_t simt_prepare(const Dims& d, const void* k, const void* v, const float* g, const void* beta,
                         void* w, void* u, float* g_cum, cudaStream_t s) {
    const int GW = d.per_k ? d.K : 1, YP = (d.K > d.V ? d.K : d.V) + 1;
    const size_t smem = sizeof(float) * ((size_t)d.C * GW + d.C + (size_t)d.C * (d.K + 1) +
                                         2 * (size_t)d.C * (d.C + 1) + (size_t)d.C * YP);
    const dim3 grid(d.NT, d.H, d.B);
#define GDR_LAUNCH_PREP(IO, PK)                                                                     \
    do {                                                                                            \
        auto kern = simt_prepare_kernel<IO, PK>;                                                     \
        cudaError_t e = allow_smem(kern, smem);                                             \
        if (e != cudaSuccess) return e;                                                             \
        kern<<<grid, kThreads, smem, s>>>(d, (const IO*)k, (const IO*)v, g, (const IO*)beta, (IO*)w, \
                                          (IO*)u, g_cum);                                           \
    } while (0)
    if (d.bf16) {
        if (d.per_k) GDR_LAUNCH_PREP(__nv_bfloat16, true); else GDR_LAUNCH_PREP(__nv_bfloat16, false);
    } else if (d.f16) {
        if (d.per_k) GDR_LAUNCH_PREP(__half, true); else GDR_LAUNCH_PREP(__half, false);
    } else {
        if (d.per_k) GDR_LAUNCH_PREP(float, true); else GDR_LAUNCH_PREP(float, false);
    }
#undef GDR_LAUNCH_PREP
    return cudaGetLastError();
}

cudaError_t simt_scan(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum,
                      const float* h0, void* h_ckpt, void* v_new, float* h_final, cudaStream_t s) {
    const int GW = d.per_k ? d.K : 1;
    const size_t smem = sizeof(float) * ((size_t)d.K * kScanBV + 2 * (size_t)d.C * (d.K + 1) +
                                         2 * (size_t)d.C * (kScanBV + 1) + GW);
    const dim3 grid(d.V / kScanBV, d.H, d.B);
#define GDR_LAUNCH_SCAN(IO, PK)                                                                       \
    do {                                                                                              \
        auto kern = simt_scan_kernel<IO, PK>;                                                          \
        cudaError_t e = allow_smem(kern, smem);                                               \
        if (e != cudaSuccess) return e;                                                               \
        kern<<<grid, kThreads, smem, s>>>(d, (const IO*)k, (const IO*)w, (const IO*)u, g_cum, h0,     \
                                          (IO*)h_ckpt, (IO*)v_new, h_final);                          \
    } while (0)
    if (d.bf16) {
        if (d.per_k) GDR_LAUNCH_SCAN(__nv_bfloat16, true); else GDR_LAUNCH_SCAN(__nv_bfloat16, false);
    } else if (d.f16) {
        if (d.per_k) GDR_LAUNCH_SCAN(__half, true); else GDR_LAUNCH_SCAN(__half, false);
    } else {
        if (d.per_k) GDR_LAUNCH_SCAN(float, true); else GDR_LAUNCH_SCAN(float, false);
    }
#undef GDR_LAUNCH_SCAN
    return cudaGetLastError();
}

cudaError_t simt_output(const Dims& d, const void* q, const void* k, const void* v_new, const void* h_ckpt,
                        const float* g_cum, void* o, cudaStream_t s) {
    const int GW = d.per_k ? d.K : 1;
    const size_t smem = sizeof(float) * (2 * (size_t)d.C * (d.K + 1) + (size_t)d.C * GW +
                                         (size_t)d.C * (d.C + 1) + (size_t)d.C * (kOutVT + 1) +
                                         (size_t)d.K * kOutVT);
    const dim3 grid(d.NT, d.H, d.B * (d.V / kOutVT));
#define GDR_LAUNCH_OUT(IO, PK)                                                                          \
    do {                                                                                                \
        auto kern = simt_output_kernel<IO, PK>;                                                          \
        cudaError_t e = allow_smem(kern, smem);                                                 \
        if (e != cudaSuccess) return e;                                                                 \
        kern<<<grid, kThreads, smem, s>>>(d, (const IO*)q, (const IO*)k, (const IO*)v_new,              \
                                          (const IO*)h_ckpt, g_cum, (IO*)o);                            \
    } while (0)
    if (d.bf16) {
        if (d.per_k) GDR_LAUNCH_OUT(__nv_bfloat16, true); else GDR_LAUNCH_OUT(__nv_bfloat16, false);
    } else if (d.f16) {
        if (d.per_k) GDR_LAUNCH_OUT(__half, true); else GDR_LAUNCH_OUT(__half, false);
    } else {
        if (d.per_k) GDR_LAUNCH_OUT(float, true); else GDR_LAUNCH_OUT(float, false);
    }
#undef GDR_LAUNCH_OUT
    return cudaGetLastError();
}

}  // namespace gdr
