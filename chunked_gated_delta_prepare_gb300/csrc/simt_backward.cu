// fp32 CUDA-core kernels for the backward of the chunked gated delta rule.
//
// The backward runs the forward prepare and the forward re-scan first (the
// re-scan of "kernel_fun/kda/_kernels/bwd_scan.py", module docstring: h
// checkpointed before each chunk's update, and v' = u - w h), then these four
// stages, each the derivative of one line of the chunked forward.  Per chunk
// (rows i, j; G the chunk-local cumsum of g; G_L its last row; h the state
// before the chunk; dh_next the gradient of the state after it):
//
//   dv_local  dv_loc = scale tril0(Qt)^T do,  Qt_ij = sum_d q_id k_jd e^(G_id - G_jd)
//   scan_dh   serial from the last chunk:  dh_ckpt[c] = dh_next,
//               dv' = dv_loc + kg dh_next,  kg = k e^(G_L - G)
//               dh  = scale (q e^G)^T do + e^(G_L) dh_next - w^T dv'      (dh0 after chunk 0)
//   dqkwg     dqg = scale do h^T, dQt = scale tril0(do v'^T), dkg = v' dh_next^T:
//               dq = dqg e^G + L(dQt, k),  dk_part = R(dQt, q) + dkg e^(G_L - G),  dw = -dv' h^T
//               dG_part = dqg q e^G + q L(dQt, k) - k R(dQt, q) - dkg kg
//                         (+ sum_i dkg_i kg_i + e^(G_L) sum_v h dh_next on the chunk's last token)
//   wy        Tinv = (I + A)^-1 rebuilt, du = dv':
//               dkb = Tinv^T dw, dvb = Tinv^T du, dA = strict_lower(-Tinv^T (dw kb^T + du vb^T) Tinv^T)
//               Y = beta_i dA_ij,  M = A / beta (row-wise)
//               dk = dk_part + beta e^G dkb + L(Y, k) + R(Y, k),  dv = beta dvb
//               dbeta = sum_d dkb k e^G + sum_v dvb v + sum_j dA_ij M_ij
//               dg = reverse cumsum over the chunk of  dG_part + dkb kb + k L(Y, k) - k R(Y, k)
//
// with L(X, Y)_i = sum_j X_ij Y_j e^(G_i - G_j), R(X, Y)_j = sum_i X_ij Y_i e^(G_i - G_j),
// elementwise over the key dim (a scalar gate sums dG over it).  A last, partial
// chunk runs as zero tokens past T; their G repeats the last real value, so the
// last-token term above goes to token T - 1.
//
// Intermediates between the stages (dv_loc, dv', dh_ckpt, dk_part, dw, dG_part)
// are fp32; q, k, v, beta, do, w, v' and h in the problem's io dtype; gradients
// of the io tensors in the io dtype, dg and dh0 in fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;   // key / value columns per pass in dqkwg and wy

__device__ __forceinline__ float ld(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st(__nv_bfloat16* p, int64_t i, float x) { p[i] = __float2bfloat16_rn(x); }
__device__ __forceinline__ float ld(const __half* p, int64_t i) { return __half2float(p[i]); }
__device__ __forceinline__ void st(__half* p, int64_t i, float x) { p[i] = __float2half_rn(x); }

// ------------------------------------------------------------------ dv_local
// One CTA per (chunk, head, batch * value tile of 64).  Shared (fp32):
// qs/ks [C][K+1], Gs [C][GW], Qt [C][C+1], dos [C][65].
constexpr int kLocVT = 64;

template <typename IO, bool PER_K>
__global__ void __launch_bounds__(kThreads)
bwd_dv_local_kernel(Dims d, const IO* __restrict__ q, const IO* __restrict__ k, const float* __restrict__ g_cum,
                    const IO* __restrict__ d_o, float* __restrict__ dv_loc) {
    extern __shared__ float smem[];
    constexpr int VT = kLocVT, VTP = kLocVT + 1;
    const int C = d.C, K = d.K, V = d.V, H = d.H;
    const int KP = K + 1, CP = C + 1, GW = PER_K ? K : 1;
    const int nvt = V / VT;
    float* qs = smem;
    float* ks = qs + C * KP;
    float* Gs = ks + C * KP;
    float* Qt = Gs + C * GW;
    float* dos = Qt + C * CP;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z / nvt, v0 = (blockIdx.z % nvt) * VT;
    const int tid = threadIdx.x;
    const int64_t tok0 = (int64_t)b * d.T + (int64_t)c * C;
    const int nv = min(C, d.T - c * C);
    auto row = [&](int t) { return (tok0 + t) * H + h; };
    auto krow = [&](int t) { return (tok0 + t) * d.Hk + h / d.G; };   // q, k: q/k head h / G

    for (int i = tid; i < C * K; i += kThreads) {
        const bool in = i / K < nv;
        qs[(i / K) * KP + i % K] = in ? ld(q, krow(i / K) * K + i % K) : 0.f;
        ks[(i / K) * KP + i % K] = in ? ld(k, krow(i / K) * K + i % K) : 0.f;
    }
    for (int i = tid; i < C * GW; i += kThreads) Gs[i] = g_cum[row(min(i / GW, nv - 1)) * GW + i % GW];
    for (int i = tid; i < C * VT; i += kThreads)
        dos[(i / VT) * VTP + i % VT] = i / VT < nv ? ld(d_o, row(i / VT) * V + v0 + i % VT) : 0.f;
    __syncthreads();
    for (int idx = tid; idx < C * C; idx += kThreads) {
        const int i = idx / C, j = idx % C;
        float a = 0.f;
        if (j <= i) {
            float s = 0.f;
            if (PER_K) {
                for (int e = 0; e < K; ++e) s += qs[i * KP + e] * ks[j * KP + e] * expf(Gs[i * K + e] - Gs[j * K + e]);
                a = s;
            } else {
                for (int e = 0; e < K; ++e) s += qs[i * KP + e] * ks[j * KP + e];
                a = expf(Gs[i] - Gs[j]) * s;
            }
        }
        Qt[i * CP + j] = a;
    }
    __syncthreads();
    for (int idx = tid; idx < C * VT; idx += kThreads) {
        const int j = idx / VT, x = idx % VT;
        if (j >= nv) continue;
        float s = 0.f;
        for (int i = j; i < C; ++i) s += Qt[i * CP + j] * dos[i * VTP + x];
        dv_loc[row(j) * V + v0 + x] = d.scale * s;
    }
}

// ------------------------------------------------------------------ scan_dh
// One CTA per (value tile of 32, head, batch); serial over chunks from the last.
// Shared (fp32): dhs [K][BV], qgs/ws/kgs [C][K+1], dos/dvs [C][BV+1], Gl [GW].
constexpr int kScanBV = 32;

template <typename IO, bool PER_K>
__global__ void __launch_bounds__(kThreads)
bwd_scan_dh_kernel(Dims d, const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ w,
                   const float* __restrict__ g_cum, const IO* __restrict__ d_o, const float* __restrict__ dv_loc,
                   const float* __restrict__ dh_final, float* __restrict__ dh_ckpt, float* __restrict__ dv_new,
                   float* __restrict__ dh0) {
    extern __shared__ float smem[];
    constexpr int BV = kScanBV, BVP = kScanBV + 1;
    const int C = d.C, K = d.K, V = d.V, H = d.H;
    const int KP = K + 1, GW = PER_K ? K : 1;
    float* dhs = smem;
    float* qgs = dhs + K * BV;
    float* ws = qgs + C * KP;
    float* kgs = ws + C * KP;
    float* dos = kgs + C * KP;
    float* dvs = dos + C * BVP;
    float* Gl = dvs + C * BVP;
    const int v0 = blockIdx.x * BV, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const int64_t state_off = ((int64_t)b * H + h) * K * V;

    for (int i = tid; i < K * BV; i += kThreads)
        dhs[i] = dh_final ? dh_final[state_off + (int64_t)(i / BV) * V + v0 + i % BV] : 0.f;
    for (int c = d.NT - 1; c >= 0; --c) {
        const int64_t tok0 = (int64_t)b * d.T + (int64_t)c * C;
        const int nv = min(C, d.T - c * C);
        auto row = [&](int t) { return (tok0 + t) * H + h; };
        auto krow = [&](int t) { return (tok0 + t) * d.Hk + h / d.G; };   // q, k: q/k head h / G
        for (int i = tid; i < GW; i += kThreads) Gl[i] = g_cum[row(nv - 1) * GW + i];
        __syncthreads();
        const int64_t ck = (((int64_t)b * d.NT + c) * H + h) * K * V;
        for (int i = tid; i < K * BV; i += kThreads) dh_ckpt[ck + (int64_t)(i / BV) * V + v0 + i % BV] = dhs[i];
        for (int i = tid; i < C * K; i += kThreads) {
            const int t = i / K, e = i % K;
            const int gi = PER_K ? e : 0;
            const bool in = t < nv;
            const float G = in ? g_cum[row(t) * GW + gi] : 0.f;
            qgs[t * KP + e] = in ? ld(q, krow(t) * K + e) * expf(G) : 0.f;
            ws[t * KP + e] = in ? ld(w, row(t) * K + e) : 0.f;
            kgs[t * KP + e] = in ? ld(k, krow(t) * K + e) * expf(Gl[gi] - G) : 0.f;
        }
        for (int i = tid; i < C * BV; i += kThreads) {
            const int t = i / BV, j = i % BV;
            const bool in = t < nv;
            dos[t * BVP + j] = in ? ld(d_o, row(t) * V + v0 + j) : 0.f;
            dvs[t * BVP + j] = in ? dv_loc[row(t) * V + v0 + j] : 0.f;
        }
        __syncthreads();
        // dv' = dv_loc + kg dh_next
        for (int idx = tid; idx < C * BV; idx += kThreads) {
            const int t = idx / BV, j = idx % BV;
            float s = dvs[t * BVP + j];
            for (int e = 0; e < K; ++e) s += kgs[t * KP + e] * dhs[e * BV + j];
            dvs[t * BVP + j] = t < nv ? s : 0.f;
            if (t < nv) dv_new[row(t) * V + v0 + j] = s;
        }
        __syncthreads();
        // dh = e^(G_L) dh_next + scale (q e^G)^T do - w^T dv'
        for (int idx = tid; idx < K * BV; idx += kThreads) {
            const int e = idx / BV, j = idx % BV;
            float s1 = 0.f, s2 = 0.f;
            for (int t = 0; t < C; ++t) {
                s1 += qgs[t * KP + e] * dos[t * BVP + j];
                s2 += ws[t * KP + e] * dvs[t * BVP + j];
            }
            dhs[idx] = expf(Gl[PER_K ? e : 0]) * dhs[idx] + d.scale * s1 - s2;
        }
        __syncthreads();
    }
    if (dh0)
        for (int i = tid; i < K * BV; i += kThreads) dh0[state_off + (int64_t)(i / BV) * V + v0 + i % BV] = dhs[i];
}

// ------------------------------------------------------------------ dqkwg
// One CTA per (chunk, head, batch).  Shared (fp32): dos/vps/dvs [C][V+1], dQt [C][C+1],
// then per pass over 32 key columns: hs/dhs [32][V+1], qt/kt/Gt/dGt/tt [C][33]; dGrow [C].
// IT: the type of the reverse scan's dh checkpoints and dv' (fp32 from the CUDA-core scan, bf16 from
// the tensor-core one)
template <typename IO, bool PER_K, typename IT>
__global__ void __launch_bounds__(kThreads)
bwd_dqkwg_kernel(Dims d, const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ v_new,
                 const float* __restrict__ g_cum, const IO* __restrict__ h_ckpt, const IT* __restrict__ dh_ckpt,
                 const IO* __restrict__ d_o, const IT* __restrict__ dv_new, IO* __restrict__ dq,
                 float* __restrict__ dk_part, float* __restrict__ dw, float* __restrict__ dG_part,
                 const int* __restrict__ only) {
    extern __shared__ float smem[];
    constexpr int KT = kTile, KTP = kTile + 1;
    const int C = d.C, K = d.K, V = d.V, H = d.H;
    const int VP = V + 1, CP = C + 1, GW = PER_K ? K : 1;
    float* dos = smem;
    float* vps = dos + C * VP;
    float* dvs = vps + C * VP;
    float* dQt = dvs + C * VP;
    float* hs = dQt + C * CP;
    float* dhs = hs + KT * VP;
    float* qt = dhs + KT * VP;
    float* kt = qt + C * KTP;
    float* Gt = kt + C * KTP;
    float* dGt = Gt + C * KTP;
    float* tt = dGt + C * KTP;
    float* dGrow = tt + C * KTP;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const int64_t tok0 = (int64_t)b * d.T + (int64_t)c * C;
    const int nv = min(C, d.T - c * C);
    auto row = [&](int t) { return (tok0 + t) * H + h; };
    auto krow = [&](int t) { return (tok0 + t) * d.Hk + h / d.G; };   // q, k: q/k head h / G
    const int64_t ck = (((int64_t)b * d.NT + c) * H + h) * K * V;
    if (only && !only[((int64_t)b * d.NT + c) * H + h]) return;   // a chunk another stage has done

    for (int i = tid; i < C * V; i += kThreads) {
        const int t = i / V, x = i % V;
        const bool in = t < nv;
        dos[t * VP + x] = in ? ld(d_o, row(t) * V + x) : 0.f;
        vps[t * VP + x] = in ? ld(v_new, row(t) * V + x) : 0.f;
        dvs[t * VP + x] = in ? ld(dv_new, row(t) * V + x) : 0.f;
    }
    for (int i = tid; i < C; i += kThreads) dGrow[i] = 0.f;
    __syncthreads();
    for (int idx = tid; idx < C * C; idx += kThreads) {
        const int i = idx / C, j = idx % C;
        float s = 0.f;
        if (j <= i)
            for (int x = 0; x < V; ++x) s += dos[i * VP + x] * vps[j * VP + x];
        dQt[i * CP + j] = d.scale * s;
    }
    for (int e0 = 0; e0 < K; e0 += KT) {
        __syncthreads();   // dQt ready; the previous pass is done with the tiles
        for (int i = tid; i < KT * V; i += kThreads) {
            const int e = i / V, x = i % V;
            hs[e * VP + x] = ld(h_ckpt, ck + (int64_t)(e0 + e) * V + x);
            dhs[e * VP + x] = ld(dh_ckpt, ck + (int64_t)(e0 + e) * V + x);
        }
        for (int i = tid; i < C * KT; i += kThreads) {
            const int t = i / KT, e = i % KT;
            const bool in = t < nv;
            qt[t * KTP + e] = in ? ld(q, krow(t) * K + e0 + e) : 0.f;
            kt[t * KTP + e] = in ? ld(k, krow(t) * K + e0 + e) : 0.f;
            Gt[t * KTP + e] = g_cum[row(min(t, nv - 1)) * GW + (PER_K ? e0 + e : 0)];
        }
        __syncthreads();
        for (int idx = tid; idx < C * KT; idx += kThreads) {
            const int i = idx / KT, e = idx % KT;
            float dqg = 0.f, dkg = 0.f, dwv = 0.f;
            for (int x = 0; x < V; ++x) {
                dqg += dos[i * VP + x] * hs[e * VP + x];
                dkg += vps[i * VP + x] * dhs[e * VP + x];
                dwv += dvs[i * VP + x] * hs[e * VP + x];
            }
            dqg *= d.scale;
            const float gi = Gt[i * KTP + e], gL = Gt[(C - 1) * KTP + e];
            // L and R without their diagonal terms: in the gate gradient q_i dQt_ii k_i - k_i dQt_ii q_i
            // cancels exactly, and leaving both out keeps fp32 rounding of O(1) terms out of a small dG
            float L = 0.f, R = 0.f;
            for (int j = 0; j < i; ++j) L += dQt[i * CP + j] * kt[j * KTP + e] * expf(gi - Gt[j * KTP + e]);
            for (int m = i + 1; m < C; ++m) R += dQt[m * CP + i] * qt[m * KTP + e] * expf(Gt[m * KTP + e] - gi);
            const float qi = qt[i * KTP + e], ki = kt[i * KTP + e], dii = dQt[i * CP + i];
            const float eg = expf(gi), ekg = expf(gL - gi);
            const float kg = ki * ekg;
            // the last token's own dkg kg term cancels against its share of the column sum: both left out
            const float t = i == nv - 1 ? 0.f : dkg * kg;
            tt[i * KTP + e] = t;
            dGt[i * KTP + e] = dqg * qi * eg + qi * L - ki * R - t;
            if (i < nv) {
                st(dq, row(i) * K + e0 + e, dqg * eg + L + dii * ki);
                dk_part[row(i) * K + e0 + e] = R + dii * qi + dkg * ekg;
                dw[row(i) * K + e0 + e] = -dwv;
            }
        }
        __syncthreads();
        // the last token's gate: sum_i dkg_i kg_i + e^(G_L) sum_v h dh_next, per key column
        for (int e = tid; e < KT; e += kThreads) {
            float s = 0.f, hd = 0.f;
            for (int i = 0; i < C; ++i) s += tt[i * KTP + e];
            for (int x = 0; x < V; ++x) hd += hs[e * VP + x] * dhs[e * VP + x];
            dGt[(nv - 1) * KTP + e] += s + expf(Gt[(C - 1) * KTP + e]) * hd;
        }
        __syncthreads();
        if (PER_K) {
            for (int i = tid; i < nv * KT; i += kThreads) dG_part[row(i / KT) * K + e0 + i % KT] = dGt[(i / KT) * KTP + i % KT];
        } else {
            for (int i = tid; i < C; i += kThreads) {
                float s = 0.f;
                for (int e = 0; e < KT; ++e) s += dGt[i * KTP + e];
                dGrow[i] += s;
            }
        }
    }
    __syncthreads();
    if (!PER_K)
        for (int i = tid; i < nv; i += kThreads) dG_part[row(i)] = dGrow[i];
}

// ------------------------------------------------------------------ wy
// One CTA per (chunk, head, batch).  Shared (fp32): ks [C][K+1], Gs [C][GW], bs [C],
// Ms/Xs/Ds/Ps [C][C+1], then per pass over 32 columns: at/bt/ct [C][33]; dbs/dGrow [C].
template <typename IO, bool PER_K, typename IT>
__global__ void __launch_bounds__(kThreads)
bwd_wy_kernel(Dims d, const IO* __restrict__ k, const IO* __restrict__ v, const IO* __restrict__ beta,
              const float* __restrict__ g_cum, const float* __restrict__ dw, const IT* __restrict__ du,
              const float* __restrict__ dk_part, const float* __restrict__ dG_part, IO* __restrict__ dk,
              IO* __restrict__ dv, IO* __restrict__ dbeta, float* __restrict__ dg, const int* __restrict__ only) {
    extern __shared__ float smem[];
    constexpr int KT = kTile, KTP = kTile + 1;
    const int C = d.C, K = d.K, V = d.V, H = d.H;
    const int KP = K + 1, CP = C + 1, GW = PER_K ? K : 1;
    float* ks = smem;
    float* Gs = ks + C * KP;
    float* bs = Gs + C * GW;
    float* Ms = bs + C;
    float* Xs = Ms + C * CP;
    float* Ds = Xs + C * CP;
    float* Ps = Ds + C * CP;
    float* at = Ps + C * CP;
    float* bt = at + C * KTP;
    float* ct = bt + C * KTP;
    float* dbs = ct + C * KTP;
    float* dGrow = dbs + C;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const int64_t tok0 = (int64_t)b * d.T + (int64_t)c * C;
    const int nv = min(C, d.T - c * C);
    auto row = [&](int t) { return (tok0 + t) * H + h; };
    auto krow = [&](int t) { return (tok0 + t) * d.Hk + h / d.G; };   // q, k: q/k head h / G
    if (only && !only[((int64_t)b * d.NT + c) * H + h]) return;   // a chunk another stage has done

    for (int i = tid; i < C * K; i += kThreads) ks[(i / K) * KP + i % K] = i / K < nv ? ld(k, krow(i / K) * K + i % K) : 0.f;
    for (int i = tid; i < C * GW; i += kThreads) Gs[i] = g_cum[row(min(i / GW, nv - 1)) * GW + i % GW];
    for (int i = tid; i < C; i += kThreads) {
        bs[i] = i < nv ? ld(beta, row(i)) : 0.f;
        dbs[i] = 0.f;
        dGrow[i] = (!PER_K && i < nv) ? dG_part[row(i)] : 0.f;
    }
    __syncthreads();
    // M_ij = sum_d k_id k_jd e^(G_id - G_jd) for i > j (A = beta_i M); dT accumulator cleared
    for (int idx = tid; idx < C * C; idx += kThreads) {
        const int i = idx / C, j = idx % C;
        float m = 0.f;
        if (i > j) {
            if (PER_K) {
                for (int e = 0; e < K; ++e) m += ks[i * KP + e] * ks[j * KP + e] * expf(Gs[i * K + e] - Gs[j * K + e]);
            } else {
                for (int e = 0; e < K; ++e) m += ks[i * KP + e] * ks[j * KP + e];
                m *= expf(Gs[i] - Gs[j]);
            }
        }
        Ms[i * CP + j] = m;
        Ds[i * CP + j] = 0.f;
    }
    __syncthreads();
    // X = (I + A)^{-1} by forward substitution, one thread per column
    for (int col = tid; col < C; col += kThreads) {
        for (int i = 0; i < col; ++i) Xs[i * CP + col] = 0.f;
        Xs[col * CP + col] = 1.f;
        for (int i = col + 1; i < C; ++i) {
            float s = 0.f;
            for (int j = col; j < i; ++j) s += bs[i] * Ms[i * CP + j] * Xs[j * CP + col];
            Xs[i * CP + col] = -s;
        }
    }
    // dT = dw kb^T + du vb^T, over passes of 32 key columns then 32 value columns
    for (int p0 = 0; p0 < K + V; p0 += KT) {
        const bool keys = p0 < K;
        __syncthreads();
        for (int i = tid; i < C * KT; i += kThreads) {
            const int t = i / KT, e = i % KT;
            const bool in = t < nv;
            if (keys) {
                at[t * KTP + e] = in ? dw[row(t) * K + p0 + e] : 0.f;
                bt[t * KTP + e] = bs[t] * ks[t * KP + p0 + e] * expf(Gs[t * GW + (PER_K ? p0 + e : 0)]);
            } else {
                at[t * KTP + e] = in ? ld(du, row(t) * V + p0 - K + e) : 0.f;
                bt[t * KTP + e] = in ? bs[t] * ld(v, row(t) * V + p0 - K + e) : 0.f;
            }
        }
        __syncthreads();
        for (int idx = tid; idx < C * C; idx += kThreads) {
            const int i = idx / C, j = idx % C;
            float s = 0.f;
            for (int e = 0; e < KT; ++e) s += at[i * KTP + e] * bt[j * KTP + e];
            Ds[i * CP + j] += s;
        }
    }
    __syncthreads();
    // dA = strict_lower(-X^T dT X^T): P = dT X^T, then dA = -X^T P
    for (int idx = tid; idx < C * C; idx += kThreads) {
        const int i = idx / C, j = idx % C;
        float s = 0.f;
        for (int m = 0; m <= j; ++m) s += Ds[i * CP + m] * Xs[j * CP + m];
        Ps[i * CP + j] = s;
    }
    __syncthreads();
    for (int idx = tid; idx < C * C; idx += kThreads) {
        const int i = idx / C, j = idx % C;
        float s = 0.f;
        if (i > j)
            for (int m = i; m < C; ++m) s += Xs[m * CP + i] * Ps[m * CP + j];
        Ds[i * CP + j] = -s;
    }
    __syncthreads();
    // dbeta through A, and Y = beta_i dA_ij (over P)
    for (int i = tid; i < C; i += kThreads) {
        float s = 0.f;
        for (int j = 0; j < i; ++j) s += Ds[i * CP + j] * Ms[i * CP + j];
        dbs[i] += s;
    }
    for (int idx = tid; idx < C * C; idx += kThreads) {
        const int i = idx / C, j = idx % C;
        Ps[i * CP + j] = bs[i] * Ds[i * CP + j];
    }
    // key columns: dk, the gate gradient and dbeta's kb part
    for (int e0 = 0; e0 < K; e0 += KT) {
        __syncthreads();
        for (int i = tid; i < C * KT; i += kThreads) {
            const int t = i / KT, e = i % KT;
            at[t * KTP + e] = t < nv ? dw[row(t) * K + e0 + e] : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < C * KT; idx += kThreads) {
            const int i = idx / KT, e = idx % KT, ee = e0 + e;
            float dkb = 0.f;
            for (int m = i; m < C; ++m) dkb += Xs[m * CP + i] * at[m * KTP + e];
            auto Gof = [&](int r) { return Gs[r * GW + (PER_K ? ee : 0)]; };
            const float gi = Gof(i), ki = ks[i * KP + ee];
            float L = 0.f, R = 0.f;
            for (int j = 0; j < i; ++j) L += Ps[i * CP + j] * ks[j * KP + ee] * expf(gi - Gof(j));
            for (int m = i + 1; m < C; ++m) R += Ps[m * CP + i] * ks[m * KP + ee] * expf(Gof(m) - gi);
            const float eg = expf(gi);
            const float kb = bs[i] * ki * eg;
            bt[i * KTP + e] = dkb * ki * eg;                                    // dbeta's kb part
            ct[i * KTP + e] = dkb * kb + ki * L - ki * R;                       // gate gradient
            if (i < nv) st(dk, row(i) * K + ee, dk_part[row(i) * K + ee] + bs[i] * eg * dkb + L + R);
        }
        __syncthreads();
        for (int i = tid; i < C; i += kThreads) {
            float s = 0.f, gsum = 0.f;
            for (int e = 0; e < KT; ++e) { s += bt[i * KTP + e]; gsum += ct[i * KTP + e]; }
            dbs[i] += s;
            if (!PER_K) dGrow[i] += gsum;
        }
        if (PER_K) {
            // dg = reverse cumsum over the chunk of dG_part + this pass's terms, one thread per key column
            for (int e = tid; e < KT; e += kThreads) {
                float run = 0.f;
                for (int i = C - 1; i >= 0; --i) {
                    const float x = ct[i * KTP + e] + (i < nv ? dG_part[row(i) * K + e0 + e] : 0.f);
                    run += x;
                    if (i < nv) dg[row(i) * K + e0 + e] = run;
                }
            }
        }
    }
    // value columns: dv and dbeta's vb part
    for (int x0 = 0; x0 < V; x0 += KT) {
        __syncthreads();
        for (int i = tid; i < C * KT; i += kThreads) {
            const int t = i / KT, x = i % KT;
            const bool in = t < nv;
            at[t * KTP + x] = in ? ld(du, row(t) * V + x0 + x) : 0.f;
            ct[t * KTP + x] = in ? ld(v, row(t) * V + x0 + x) : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < C * KT; idx += kThreads) {
            const int i = idx / KT, x = idx % KT;
            float dvb = 0.f;
            for (int m = i; m < C; ++m) dvb += Xs[m * CP + i] * at[m * KTP + x];
            bt[i * KTP + x] = dvb * ct[i * KTP + x];
            if (i < nv) st(dv, row(i) * V + x0 + x, bs[i] * dvb);
        }
        __syncthreads();
        for (int i = tid; i < C; i += kThreads) {
            float s = 0.f;
            for (int x = 0; x < KT; ++x) s += bt[i * KTP + x];
            dbs[i] += s;
        }
    }
    __syncthreads();
    for (int i = tid; i < nv; i += kThreads) st(dbeta, row(i), dbs[i]);
    if (!PER_K && tid == 0) {
        float run = 0.f;
        for (int i = C - 1; i >= 0; --i) {
            run += dGrow[i];
            if (i < nv) dg[row(i)] = run;
        }
    }
}

// ------------------------------------------------------------------ group sum
// Grouped value heads: dq and dk of a q/k head are the sums over its group of the
// per-value-head gradients.  in [B,T,Hk*G,K] -> out [B,T,Hk,K], summed in fp32.
template <typename IO>
__global__ void __launch_bounds__(kThreads)
group_sum_kernel(const IO* __restrict__ in, IO* __restrict__ out, int64_t rows_out, int G, int K) {
    const int64_t n = rows_out * K;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads) {
        const int64_t r = i / K, x = i % K;
        float s = 0.f;
        for (int gi = 0; gi < G; ++gi) s += ld(in, (r * G + gi) * K + x);
        st(out, i, s);
    }
}

template <typename Kern>
cudaError_t allow_smem(Kern kern, size_t smem) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

#define GDR_DISPATCH(LAUNCH)                                                                  \
    do {                                                                                      \
        if (d.bf16) {                                                                         \
            if (d.per_k) LAUNCH(__nv_bfloat16, true); else LAUNCH(__nv_bfloat16, false);      \
        } else if (d.f16) {                                                                   \
            if (d.per_k) LAUNCH(__half, true); else LAUNCH(__half, false);                    \
        } else {                                                                              \
            if (d.per_k) LAUNCH(float, true); else LAUNCH(float, false);                      \
        }                                                                                     \
    } while (0)

}  // namespace

cudaError_t simt_bwd_dv_local(const Dims& d, const void* q, const void* k, const float* g_cum, const void* d_o,
                              float* dv_loc, cudaStream_t s) {
    const int GW = d.per_k ? d.K : 1;
    const size_t smem = sizeof(float) * (2 * (size_t)d.C * (d.K + 1) + (size_t)d.C * GW +
                                         (size_t)d.C * (d.C + 1) + (size_t)d.C * (kLocVT + 1));
    const dim3 grid(d.NT, d.H, d.B * (d.V / kLocVT));
#define LAUNCH(IO, PK)                                                                                      \
    do {                                                                                                       \
        auto kern = bwd_dv_local_kernel<IO, PK>;                                                           \
        cudaError_t e = allow_smem(kern, smem);                                                             \
        if (e != cudaSuccess) return e;                                                                     \
        kern<<<grid, kThreads, smem, s>>>(d, (const IO*)q, (const IO*)k, g_cum, (const IO*)d_o, dv_loc);    \
    } while (0)
    GDR_DISPATCH(LAUNCH);
#undef LAUNCH
    return cudaGetLastError();
}

cudaError_t simt_bwd_scan_dh(const Dims& d, const void* q, const void* k, const void* w, const float* g_cum,
                             const void* d_o, const float* dv_loc, const float* dh_final, float* dh_ckpt,
                             float* dv_new, float* dh0, cudaStream_t s) {
    const int GW = d.per_k ? d.K : 1;
    const size_t smem = sizeof(float) * ((size_t)d.K * kScanBV + 3 * (size_t)d.C * (d.K + 1) +
                                         2 * (size_t)d.C * (kScanBV + 1) + GW);
    const dim3 grid(d.V / kScanBV, d.H, d.B);
#define LAUNCH(IO, PK)                                                                                     \
    do {                                                                                                      \
        auto kern = bwd_scan_dh_kernel<IO, PK>;                                                           \
        cudaError_t e = allow_smem(kern, smem);                                                            \
        if (e != cudaSuccess) return e;                                                                    \
        kern<<<grid, kThreads, smem, s>>>(d, (const IO*)q, (const IO*)k, (const IO*)w, g_cum,              \
                                          (const IO*)d_o, dv_loc, dh_final, dh_ckpt, dv_new, dh0);         \
    } while (0)
    GDR_DISPATCH(LAUNCH);
#undef LAUNCH
    return cudaGetLastError();
}

cudaError_t simt_bwd_dqkwg(const Dims& d, const void* q, const void* k, const void* v_new, const float* g_cum,
                           const void* h_ckpt, const void* dh_ckpt, const void* d_o, const void* dv_new,
                           void* dq, float* dk_part, float* dw, float* dG_part, cudaStream_t s, bool inter16,
                           const int* only) {
    const size_t C = d.C, V = d.V;
    const size_t smem = sizeof(float) * (3 * C * (V + 1) + C * (C + 1) + 2 * (size_t)kTile * (V + 1) +
                                         5 * C * (kTile + 1) + C);
    const dim3 grid(d.NT, d.H, d.B);
#define LAUNCH_IT(IO, PK, IT)                                                                                \
    do {                                                                                                     \
        auto kern = bwd_dqkwg_kernel<IO, PK, IT>;                                                            \
        cudaError_t e = allow_smem(kern, smem);                                                              \
        if (e != cudaSuccess) return e;                                                                      \
        kern<<<grid, kThreads, smem, s>>>(d, (const IO*)q, (const IO*)k, (const IO*)v_new, g_cum,            \
                                          (const IO*)h_ckpt, (const IT*)dh_ckpt, (const IO*)d_o,             \
                                          (const IT*)dv_new, (IO*)dq, dk_part, dw, dG_part, only);           \
    } while (0)
#define LAUNCH(IO, PK)                                                                                       \
    do {                                                                                                     \
        if (inter16) LAUNCH_IT(IO, PK, IO); else LAUNCH_IT(IO, PK, float);                                 \
    } while (0)
    GDR_DISPATCH(LAUNCH);
#undef LAUNCH
#undef LAUNCH_IT
    return cudaGetLastError();
}

cudaError_t simt_bwd_wy(const Dims& d, const void* k, const void* v, const void* beta, const float* g_cum,
                        const float* dw, const void* du, const float* dk_part, const float* dG_part, void* dk,
                        void* dv, void* dbeta, float* dg, cudaStream_t s, bool inter16, const int* only) {
    const size_t C = d.C, K = d.K, GW = d.per_k ? d.K : 1;
    const size_t smem = sizeof(float) * (C * (K + 1) + C * GW + C + 4 * C * (C + 1) + 3 * C * (kTile + 1) + 2 * C);
    const dim3 grid(d.NT, d.H, d.B);
#define LAUNCH_IT(IO, PK, IT)                                                                                \
    do {                                                                                                     \
        auto kern = bwd_wy_kernel<IO, PK, IT>;                                                               \
        cudaError_t e = allow_smem(kern, smem);                                                              \
        if (e != cudaSuccess) return e;                                                                      \
        kern<<<grid, kThreads, smem, s>>>(d, (const IO*)k, (const IO*)v, (const IO*)beta, g_cum, dw,         \
                                          (const IT*)du, dk_part, dG_part, (IO*)dk, (IO*)dv, (IO*)dbeta, dg, \
                                          only);                                                             \
    } while (0)
#define LAUNCH(IO, PK)                                                                                       \
    do {                                                                                                     \
        if (inter16) LAUNCH_IT(IO, PK, IO); else LAUNCH_IT(IO, PK, float);                                 \
    } while (0)
    GDR_DISPATCH(LAUNCH);
#undef LAUNCH
#undef LAUNCH_IT
    return cudaGetLastError();
}

}  // namespace gdr

namespace gdr {

cudaError_t group_sum_heads(const Dims& d, const void* dq_v, const void* dk_v, void* dq, void* dk, cudaStream_t s) {
    const int64_t rows_out = (int64_t)d.B * d.T * d.Hk;
    const int blocks = (int)std::min<int64_t>((rows_out * d.K + kThreads - 1) / kThreads, 152 * 16);
    if (d.bf16) {
        group_sum_kernel<__nv_bfloat16><<<blocks, kThreads, 0, s>>>((const __nv_bfloat16*)dq_v, (__nv_bfloat16*)dq,
                                                                   rows_out, d.G, d.K);
        group_sum_kernel<__nv_bfloat16><<<blocks, kThreads, 0, s>>>((const __nv_bfloat16*)dk_v, (__nv_bfloat16*)dk,
                                                                   rows_out, d.G, d.K);
    } else if (d.f16) {
        group_sum_kernel<__half><<<blocks, kThreads, 0, s>>>((const __half*)dq_v, (__half*)dq, rows_out, d.G, d.K);
        group_sum_kernel<__half><<<blocks, kThreads, 0, s>>>((const __half*)dk_v, (__half*)dk, rows_out, d.G, d.K);
    } else {
        group_sum_kernel<float><<<blocks, kThreads, 0, s>>>((const float*)dq_v, (float*)dq, rows_out, d.G, d.K);
        group_sum_kernel<float><<<blocks, kThreads, 0, s>>>((const float*)dk_v, (float*)dk, rows_out, d.G, d.K);
    }
    return cudaGetLastError();
}

}  // namespace gdr
