// The C ABI of libgdr (include/gdr.h): argument validation, workspace
// planning and kernel dispatch.  No arithmetic of the method happens here;
// every step runs in the kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <string>

#include "gdr.h"
#include "gdr_internal.h"

namespace {

thread_local std::string t_last_variant;

constexpr int64_t kMaxGridYZ = 65535;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks the descriptor and fills Dims.  Does not look at pointers.
gdr_status check_problem(const gdr_problem* p, gdr::Dims* d) {
    if (!p) return GDR_ERR_NULL;
    if (p->io_dtype != GDR_F32 && p->io_dtype != GDR_BF16 && p->io_dtype != GDR_F16) return GDR_ERR_DTYPE;
    if (p->gate != GDR_GATE_SCALAR && p->gate != GDR_GATE_PER_K) return GDR_ERR_DTYPE;
    if (p->B <= 0 || p->T <= 0 || p->H <= 0 || p->K <= 0 || p->V <= 0 || p->chunk <= 0) return GDR_ERR_SHAPE;
    if ((p->K != 64 && p->K != 128) || (p->V != 64 && p->V != 128)) return GDR_ERR_SHAPE;
    if (p->chunk != 32 && p->chunk != 64) return GDR_ERR_SHAPE;
    // grouped value heads: HV value heads share the H q/k heads in groups of HV / H
    const int64_t HV = p->HV > 0 ? p->HV : p->H;
    if (p->HV < 0 || HV % p->H != 0) return GDR_ERR_SHAPE;
    // grid and 32-bit dims limits: T, B*T*HV fit int32; HV and B*(V/32) fit a grid y/z extent
    if (p->T > INT32_MAX || HV > kMaxGridYZ || p->B * (p->V / 32) > kMaxGridYZ) return GDR_ERR_SHAPE;
    if (p->B > INT32_MAX / p->T || p->B * p->T > INT32_MAX / HV) return GDR_ERR_SHAPE;
    if (std::isnan(p->scale) || std::isinf(p->scale)) return GDR_ERR_ARG;
    if (p->variant < GDR_VARIANT_AUTO || p->variant > GDR_VARIANT_FUSED_TC) return GDR_ERR_ARG;
    if (p->segments < 0) return GDR_ERR_ARG;
    d->B = (int)p->B;
    d->T = (int)p->T;
    d->H = (int)HV;
    d->Hk = (int)p->H;
    d->G = (int)(HV / p->H);
    d->K = (int)p->K;
    d->V = (int)p->V;
    d->C = (int)p->chunk;
    d->NT = (d->T + d->C - 1) / d->C;   // a last, partial chunk counts
    d->per_k = p->gate == GDR_GATE_PER_K;
    d->bf16 = p->io_dtype == GDR_BF16;
    d->f16 = p->io_dtype == GDR_F16;
    d->scale = p->scale > 0.f ? p->scale : 1.0f / std::sqrt((float)p->K);
    return GDR_OK;
}

gdr_status check_ptrs(std::initializer_list<const void*> required, std::initializer_list<const void*> optional) {
    for (const void* q : required)
        if (!q) return GDR_ERR_NULL;
    for (const void* q : required)
        if (!aligned16(q)) return GDR_ERR_ALIGN;
    for (const void* q : optional)
        if (q && !aligned16(q)) return GDR_ERR_ALIGN;
    return GDR_OK;
}

gdr_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA; }

// A single stage runs its tensor-core kernel (bf16 or fp16 io) unless SIMT is asked for.
gdr_status pick_stage(const gdr_problem* p, const gdr::Dims& d, bool* tensor) {
    switch (p->variant) {
        case GDR_VARIANT_SIMT: *tensor = false; return GDR_OK;
        case GDR_VARIANT_TENSOR:
        case GDR_VARIANT_FUSED:
        case GDR_VARIANT_FUSED_TC:
            if (!d.bf16 && !d.f16) return GDR_ERR_UNSUPPORTED;
            *tensor = true;
            return GDR_OK;
        case GDR_VARIANT_AUTO: *tensor = d.bf16 || d.f16; return GDR_OK;
        default: return GDR_ERR_UNSUPPORTED;
    }
}

enum class Path { Simt, Tensor, Fused, FusedTc };

constexpr int kSmCount = 152;   // GB300
constexpr int kPieceChunks = 64;   // the overlapped forward's chunks per piece, at least
bool segments_apply(const gdr_problem* p, const gdr::Dims& d);

// The path a whole forward takes: SIMT (fp32 CUDA-core kernels for every stage),
// TENSOR (the three tensor-core stage kernels, bf16 or fp16 io) or FUSED (the
// prepare, then scan and output in one kernel; scalar gate only).
gdr_status pick_forward(const gdr_problem* p, const gdr::Dims& d, Path* path) {
    const bool io16 = d.bf16 || d.f16;
    switch (p->variant) {
        case GDR_VARIANT_SIMT: *path = Path::Simt; return GDR_OK;
        case GDR_VARIANT_TENSOR:
            if (!io16) return GDR_ERR_UNSUPPORTED;
            *path = Path::Tensor;
            return GDR_OK;
        case GDR_VARIANT_FUSED:
            if (!io16 || d.per_k) return GDR_ERR_UNSUPPORTED;
            *path = Path::Fused;
            return GDR_OK;
        case GDR_VARIANT_FUSED_TC:
            if (!gdr::tc_scan_output_supported(d)) return GDR_ERR_UNSUPPORTED;
            *path = Path::FusedTc;
            return GDR_OK;
        case GDR_VARIANT_AUTO:
            // bf16 with a scalar gate and 64-token chunks: FUSED (its prepare also writes the gated
            // scores, so scan and output run as one kernel) measures fastest; other bf16 problems
            // take the staged tensor-core kernels; fp32 the exact CUDA-core path
            // The tcgen05 form of the fused kernel (see fused_tc.cu) when the warp-level one would need
            // more than one wave of the GPU, or for one long sequence scanned whole, which it runs in
            // pieces overlapped with the prepare (see forward_tc_overlapped).
            // A per-key-dim gate at K = V = 128, C = 64 takes the tcgen05 form too (its gated operands from
            // their own kernel) unless the segment-parallel scan applies.
            // fp16 io follows the same rules; its tcgen05 form takes a scalar gate only (see
            // tc_scan_output_supported), so a per-key-dim gate runs the staged kernels.
            if (!io16) *path = Path::Simt;
            else if (!d.per_k && d.C == 64)
                *path = gdr::tc_scan_output_supported(d) &&
                                ((int64_t)d.B * d.H * (d.V / 32) > kSmCount || (d.B == 1 && d.NT >= 2 * kPieceChunks &&
                                                                                 !segments_apply(p, d)))
                            ? Path::FusedTc
                            : Path::Fused;
            else if (d.per_k && gdr::tc_scan_output_supported(d) && !segments_apply(p, d)) *path = Path::FusedTc;
            else *path = Path::Tensor;
            return GDR_OK;
        default: return GDR_ERR_UNSUPPORTED;
    }
}

const char* path_name(Path p) {
    switch (p) {
        case Path::Simt: return "simt";
        case Path::Tensor: return "tensor";
        case Path::Fused: return "fused";
        default: return "fused_tc";
    }
}

unsigned int* device_error_word() {
    unsigned int* p = nullptr;
    return gdr::device_error_ptr(&p) == cudaSuccess ? p : nullptr;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The segment-parallel scan: the sequence of each (b, h) splits into S segments of NT / S chunks.
// Viewed as B S sequences of T / S tokens, every [B, T, ...] and [B, NT, ...] tensor keeps its memory
// layout, so the scan kernels run the segments as a larger batch.
gdr::Dims segment_view(const gdr::Dims& d, int S) {
    gdr::Dims v = d;
    v.B = d.B * S;
    v.T = d.T / S;
    v.NT = d.NT / S;
    return v;
}

// S for gdr_forward.  Explicit (p->segments > 1): it must divide NT, with whole chunks.  Automatic
// (0): when the serial scan's grid, B HV V/32 CTAs, fills less than half the GPU, the largest
// divisor of NT that keeps the segmented grid within one wave of 152 SMs and every segment at least
// kSegMinChunks chunks long.  The CUDA-core path is never segmented.
constexpr int kSegMinChunks = 16;

gdr_status resolve_segments(const gdr_problem* p, const gdr::Dims& d, bool tensor, int* S) {
    *S = 1;
    if (p->segments == 1 || !tensor) return GDR_OK;
    if (d.f16) return p->segments > 1 ? GDR_ERR_UNSUPPORTED : GDR_OK;   // the segment maps are bf16 kernels
    if (p->segments > 1) {
        if (d.T % d.C != 0 || d.NT % p->segments != 0 || p->segments > kMaxGridYZ / d.B) return GDR_ERR_ARG;
        *S = (int)p->segments;
        return GDR_OK;
    }
    const int64_t base = (int64_t)d.B * d.H * (d.V / 32);
    if (d.T % d.C != 0 || 2 * base > kSmCount) return GDR_OK;
    for (int cand = d.NT / kSegMinChunks; cand >= 2; --cand) {
        if (d.NT % cand == 0 && cand * base <= kSmCount && cand <= kMaxGridYZ / d.B) {
            *S = cand;
            break;
        }
    }
    return GDR_OK;
}

// Whether the tensor-core paths would scan this problem in segments (resolve_segments with S > 1).
bool segments_apply(const gdr_problem* p, const gdr::Dims& d) {
    int S = 1;
    return resolve_segments(p, d, true, &S) == GDR_OK && S > 1;
}

// gdr_forward scratch: g_cum, w, u and (staged paths) v_new, h_ckpt, (S > 1) the segment maps and
// starts, each 256-byte aligned.
struct StagedWorkspace {
    size_t g_cum, w, u, v_new, h_ckpt, P, kg, qg, seg_m, seg_z, seg_h, carry, total;
};

// gated: the tcgen05 path with a per-key-dim gate, which also keeps kg and qg [B, T, H, K] (io dtype)
StagedWorkspace plan_staged(const gdr::Dims& d, bool fused, int S, int pieces = 1, bool gated = false) {
    const size_t e = (d.bf16 || d.f16) ? 2 : 4;
    const size_t rows = (size_t)d.B * d.T * d.H;
    StagedWorkspace ws;
    size_t off = 0;
    ws.g_cum = off; off = round_up(off + rows * (d.per_k ? d.K : 1) * 4, 256);
    ws.w = off;     off = round_up(off + rows * d.K * e, 256);
    ws.u = off;     off = round_up(off + rows * d.V * e, 256);
    ws.v_new = off;
    ws.h_ckpt = off;
    ws.P = off;
    if (!fused) {   // the fused scan/output keeps v' and the checkpoints on chip
        off = round_up(off + rows * d.V * e, 256);
        ws.h_ckpt = off;
        off = round_up(off + (size_t)d.B * d.NT * d.H * d.K * d.V * e, 256);
    } else if (d.C == 64) {   // ... and reads the prepare's gated causal scores [B, NT, H, C, C]
        off = round_up(off + (size_t)d.B * d.NT * d.H * d.C * d.C * e, 256);
    }
    ws.kg = ws.qg = off;
    if (gated) {
        ws.qg = round_up(off + rows * d.K * e, 256);
        off = round_up(ws.qg + rows * d.K * e, 256);
    }
    ws.seg_m = ws.seg_z = ws.seg_h = off;
    if (S > 1) {   // M [B S, H, K, K], Z and the segment starts [B S, H, K, V], fp32
        const size_t maps = (size_t)d.B * S * d.H * d.K;
        ws.seg_z = round_up(off + maps * d.K * 4, 256);
        ws.seg_h = round_up(ws.seg_z + maps * d.V * 4, 256);
        off = round_up(ws.seg_h + maps * d.V * 4, 256);
    }
    ws.carry = off;
    if (pieces > 1)   // the state between pieces of the overlapped forward, [pieces - 1][B, H, K, V] fp32
        off = round_up(off + (size_t)(pieces - 1) * d.B * d.H * d.K * d.V * 4, 256);
    ws.total = off;
    return ws;
}

// ---------------------------------------------------------------- the overlapped tcgen05 forward
// One long sequence on the tcgen05 fused path (B = 1, no segments) runs in pieces of whole chunks on
// the caller's stream: prepare(0), scan(0), prepare(1), scan(1), ...  Each prepare after the first is
// launched as the programmatic dependent of the scan before it: once every scan CTA holds its SM (one
// per head) the next piece's prepare starts on the SMs left free and overlaps the scan.  Each scan is
// an ordinary launch, so it starts after its own piece's prepare and the previous scan; the state
// passes between pieces in fp32 through the workspace.
//
// Piece sizes grow geometrically from kFirstPiece chunks by 3/2: only the first prepare runs alone, and
// each later prepare, on the SMs the scan leaves, is shorter than the scan it overlaps (a scan chunk
// costs about 1.5 us on one SM per head, a prepare chunk about 1.3 us of the whole GPU per 32 heads).
// A piece is never shorter than an equal share of what is left among the pieces still allowed, so
// there are at most kMaxPieces.
constexpr int kFirstPiece = 16;
constexpr int kMaxPieces = 32;

// Chunk offsets of the pieces: bounds[0] = 0 < bounds[1] < ... < bounds[n] = NT; returns n (1: no pieces).
int overlap_bounds(const gdr::Dims& d, Path path, int S, int* bounds) {
    bounds[0] = 0;
    if (path != Path::FusedTc || d.per_k || S != 1 || d.B != 1 || d.NT < 2 * kPieceChunks) {
        bounds[1] = d.NT;
        return 1;
    }
    int n = 0, c = 0, len = kFirstPiece;
    while (c < d.NT) {
        const int share = (d.NT - c + (kMaxPieces - n) - 1) / (kMaxPieces - n);
        len = std::max(len, share);
        c = std::min(d.NT, c + len);
        bounds[++n] = c;
        len += len / 2;
    }
    return n;
}

int overlap_pieces(const gdr::Dims& d, Path path, int S) {
    int bounds[kMaxPieces + 1];
    return overlap_bounds(d, path, S, bounds);
}

gdr_status forward_tc_overlapped(const gdr::Dims& d, const int* bounds, int pieces, const StagedWorkspace& ws,
                                 char* base, const void* q, const void* k, const void* v, const float* g,
                                 const void* beta, const float* h0, void* o, float* h_final, cudaStream_t s,
                                 unsigned int* err) {
    const size_t e = 2;                                 // bf16
    float* carry = reinterpret_cast<float*>(base + ws.carry);
    const size_t state = (size_t)d.H * d.K * d.V;
    for (int i = 0; i < pieces; ++i) {
        const int c0 = bounds[i], c1 = bounds[i + 1];
        const int64_t t0 = (int64_t)c0 * d.C, t1 = std::min<int64_t>(d.T, (int64_t)c1 * d.C);
        gdr::Dims dp = d;
        dp.T = (int)(t1 - t0);
        dp.NT = c1 - c0;
        const char* qp = static_cast<const char*>(q) + (size_t)t0 * d.Hk * d.K * e;
        const char* kp = static_cast<const char*>(k) + (size_t)t0 * d.Hk * d.K * e;
        const char* vp = static_cast<const char*>(v) + (size_t)t0 * d.H * d.V * e;
        const char* bp = static_cast<const char*>(beta) + (size_t)t0 * d.H * e;
        const float* gp = g + t0 * d.H;
        float* g_cum = reinterpret_cast<float*>(base + ws.g_cum) + t0 * d.H;
        char* w = base + ws.w + (size_t)t0 * d.H * d.K * e;
        char* u = base + ws.u + (size_t)t0 * d.H * d.V * e;
        char* P = base + ws.P + (size_t)c0 * d.H * d.C * d.C * e;
        char* op = static_cast<char*>(o) + (size_t)t0 * d.H * d.V * e;
        const float* hin = i == 0 ? h0 : carry + (size_t)(i - 1) * state;
        float* hout = i == pieces - 1 ? h_final : carry + (size_t)i * state;
        cudaError_t ce = gdr::mma_prepare(dp, kp, vp, gp, bp, w, u, g_cum, s, err, qp, P, nullptr, i > 0, true);
        if (ce == cudaSuccess) ce = gdr::tc_scan_output(dp, qp, kp, w, u, g_cum, P, hin, op, hout, s, err);
        if (ce != cudaSuccess) return GDR_ERR_CUDA;
    }
    return GDR_OK;
}

// gdr_backward scratch: the forward's g_cum, w, u, v_new, h_ckpt (io dtype), then the
// backward's fp32 intermediates, each 256-byte aligned.
struct BackwardWorkspace {
    size_t g_cum, w, u, v_new, h_ckpt, dv_loc, dv_new, dh_ckpt, dk_part, dw, dG_part, P, tinv, flags, dq_v, dk_v,
        seg_m, seg_z, seg_h, seg_zb, seg_e, total;
};

// The backward's paths: every stage on the CUDA cores (SIMT); every stage on the tensor cores for a
// scalar gate (FAST: bf16); the same for a per-key-dim gate with the CUDA-core per-chunk stages
// finishing the chunks whose gate the split-gate products cannot take (TENSOR: bf16).
enum class BwdPath { Simt, Tensor, Fast };

BackwardWorkspace plan_backward(const gdr::Dims& d, BwdPath path, int S) {
    const size_t e = (d.bf16 || d.f16) ? 2 : 4;
    const size_t rows = (size_t)d.B * d.T * d.H;
    const size_t gw = d.per_k ? d.K : 1;
    const size_t states = (size_t)d.B * d.NT * d.H * d.K * d.V;
    const size_t tiles = (size_t)d.B * d.NT * d.H * d.C * d.C;
    BackwardWorkspace ws{};
    size_t off = 0;
    auto take = [&](size_t* field, size_t bytes) { *field = off; off = round_up(off + bytes, 256); };
    take(&ws.g_cum, rows * gw * 4);
    take(&ws.w, rows * d.K * e);
    take(&ws.u, rows * d.V * e);
    take(&ws.v_new, rows * d.V * e);
    take(&ws.h_ckpt, states * e);
    if (path == BwdPath::Fast) {   // bf16 gradients of v' and of the states; T; P (C = 64) or dv_loc (C = 32)
        take(&ws.dv_new, rows * d.V * 2);
        take(&ws.dh_ckpt, states * 2);
        if (d.C == 64) take(&ws.P, tiles * 2);
        else take(&ws.dv_loc, rows * d.V * 2);
        take(&ws.tinv, tiles * 2);
    } else if (path == BwdPath::Tensor) {
        // bf16 dv_loc, v' and state gradients; T; the per-chunk flags and the fp32 partials of the chunks the
        // CUDA cores finish
        take(&ws.dv_loc, rows * d.V * 2);
        take(&ws.dv_new, rows * d.V * 2);
        take(&ws.dh_ckpt, states * 2);
        take(&ws.tinv, tiles * 2);
        take(&ws.flags, (size_t)d.B * d.NT * d.H * 4);
        take(&ws.dk_part, rows * d.K * 4);
        take(&ws.dw, rows * d.K * 4);
        take(&ws.dG_part, rows * gw * 4);
    } else {
        take(&ws.dv_loc, rows * d.V * 4);
        take(&ws.dv_new, rows * d.V * 4);
        take(&ws.dh_ckpt, states * 4);
        take(&ws.dk_part, rows * d.K * 4);
        take(&ws.dw, rows * d.K * 4);
        take(&ws.dG_part, rows * gw * 4);
    }
    if (d.G > 1) {   // per-value-head dq and dk, summed over each group at the end
        take(&ws.dq_v, rows * d.K * e);
        take(&ws.dk_v, rows * d.K * e);
    }
    if (S > 1) {     // the segment maps, the re-scan's segment starts, the reverse scan's offsets and ends
        const size_t maps = (size_t)d.B * S * d.H * d.K;
        take(&ws.seg_m, maps * d.K * 4);
        take(&ws.seg_z, maps * d.V * 4);
        take(&ws.seg_h, maps * d.V * 4);
        take(&ws.seg_zb, maps * d.V * 4);
        take(&ws.seg_e, maps * d.V * 4);
    }
    ws.total = off;
    return ws;
}

// AUTO and TENSOR take FAST where it applies; FUSED keeps no checkpoints and is not offered.
gdr_status pick_backward(const gdr_problem* p, const gdr::Dims& d, BwdPath* path) {
    const bool fast = d.bf16 && !d.per_k;
    switch (p->variant) {
        case GDR_VARIANT_SIMT: *path = BwdPath::Simt; return GDR_OK;
        case GDR_VARIANT_TENSOR:
            if (!d.bf16) return GDR_ERR_UNSUPPORTED;
            *path = fast ? BwdPath::Fast : BwdPath::Tensor;
            return GDR_OK;
        case GDR_VARIANT_AUTO:
            *path = !d.bf16 ? BwdPath::Simt : (fast ? BwdPath::Fast : BwdPath::Tensor);
            return GDR_OK;
        default: return GDR_ERR_UNSUPPORTED;
    }
}

// The backward's launches on validated dims d, path and S, with the workspace planned as ws at base.
// co, nseq: packed variable-length sequences in the chunk-packed layout (d has B = 1; S = 1; the
// tensor-core paths), else NULL and 0.
gdr_status run_backward(const gdr::Dims& d, BwdPath path, int S, char* base, const BackwardWorkspace& ws,
                        const void* q, const void* k, const void* v, const float* g, const void* beta,
                        const float* h0, const void* d_o, const float* dh_final, void* dq, void* dk, void* dv,
                        float* dg, void* dbeta, float* dh0, cudaStream_t s, const int* co, int nseq) {
    gdr_status st;
    const bool tensor = path != BwdPath::Simt;
    if (co && (S != 1 || !tensor)) return GDR_ERR_ARG;
    float* g_cum = reinterpret_cast<float*>(base + ws.g_cum);
    void* w = base + ws.w;
    void* u = base + ws.u;
    void* v_new = base + ws.v_new;
    void* h_ckpt = base + ws.h_ckpt;
    float* dv_loc = reinterpret_cast<float*>(base + ws.dv_loc);
    float* dv_new = reinterpret_cast<float*>(base + ws.dv_new);
    float* dh_ckpt = reinterpret_cast<float*>(base + ws.dh_ckpt);
    float* dk_part = reinterpret_cast<float*>(base + ws.dk_part);
    float* dw = reinterpret_cast<float*>(base + ws.dw);
    float* dG_part = reinterpret_cast<float*>(base + ws.dG_part);
    // grouped value heads: the stages write per-value-head dq and dk, summed over each group at the end
    void* const dq_out = dq;
    void* const dk_out = dk;
    if (d.G > 1) {
        dq = base + ws.dq_v;
        dk = base + ws.dk_v;
    }
    // The two serial scans, segment-parallel when S > 1.  The re-scan as the forward does it; the reverse
    // scan once from a zero gradient at every segment end (its dh0 per segment are the offsets Zb), the
    // reverse stitch with the forward maps transposed, then again from the stitched segment ends.
    float* seg_m = reinterpret_cast<float*>(base + ws.seg_m);
    float* seg_z = reinterpret_cast<float*>(base + ws.seg_z);
    float* seg_h = reinterpret_cast<float*>(base + ws.seg_h);
    float* seg_zb = reinterpret_cast<float*>(base + ws.seg_zb);
    float* seg_e = reinterpret_cast<float*>(base + ws.seg_e);
    auto rescan = [&](unsigned int* err) -> gdr_status {
        if (S == 1) return from_cuda(gdr::mma_scan(d, k, w, u, g_cum, h0, h_ckpt, v_new, nullptr, s, err, co, nseq));
        const gdr::Dims ds = segment_view(d, S);
        gdr_status r = from_cuda(gdr::mma_scan_transfer(ds, k, w, u, g_cum, seg_m, seg_z, s, err));
        if (r == GDR_OK) r = from_cuda(gdr::segment_combine(d, S, seg_m, seg_z, h0, seg_h, nullptr, s));
        if (r == GDR_OK) r = from_cuda(gdr::mma_scan(ds, k, w, u, g_cum, seg_h, h_ckpt, v_new, nullptr, s, err));
        return r;
    };
    auto reverse_scan = [&](auto run) -> gdr_status {   // run(dims, dh_final, dh0)
        if (S == 1) return run(d, dh_final, dh0);
        const gdr::Dims ds = segment_view(d, S);
        gdr_status r = run(ds, nullptr, seg_zb);
        if (r == GDR_OK) r = from_cuda(gdr::segment_combine(d, S, seg_m, seg_zb, dh_final, seg_e, dh0, s, true));
        if (r == GDR_OK) r = run(ds, seg_e, nullptr);
        return r;
    };
    if (path == BwdPath::Fast) {
        // every step on the tensor cores: prepare (+ P and T), re-scan, reverse scan, per-chunk stage
        unsigned int* err = device_error_word();
        void* tinv = base + ws.tinv;
        if (d.C == 64) {   // the prepare's gated scores P give the reverse scan its local term
            void* P = base + ws.P;
            if ((st = from_cuda(gdr::mma_prepare(d, k, v, g, beta, w, u, g_cum, s, err, q, P, tinv))) != GDR_OK)
                return st;
            if ((st = rescan(err)) != GDR_OK) return st;
            st = reverse_scan([&](const gdr::Dims& dd, const float* dhf, float* dh0o) {
                return from_cuda(gdr::mma_bwd_scan(dd, q, k, w, g_cum, P, d_o, dhf, dh_ckpt, dv_new, dh0o, s, err, co,
                                                   nseq));
            });
            if (st != GDR_OK) return st;
        } else {           // C = 32: the local term from its own kernel
            if ((st = from_cuda(gdr::mma_prepare(d, k, v, g, beta, w, u, g_cum, s, err, nullptr, nullptr, tinv))) !=
                GDR_OK)
                return st;
            if ((st = rescan(err)) != GDR_OK) return st;
            if ((st = from_cuda(gdr::mma_bwd_dv_local(d, q, k, g_cum, d_o, dv_loc, s))) != GDR_OK) return st;
            st = reverse_scan([&](const gdr::Dims& dd, const float* dhf, float* dh0o) {
                return from_cuda(gdr::mma_bwd_scan_dl(dd, q, k, w, g_cum, dv_loc, d_o, dhf, dh_ckpt, dv_new, dh0o, s,
                                                      err, co, nseq));
            });
            if (st != GDR_OK) return st;
        }
        st = from_cuda(d.C == 64 ? gdr::mma_bwd_chunk_tma(d, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o,
                                                          dv_new, dh_ckpt, dq, dk, dv, dbeta, dg, s, err)
                                 : gdr::mma_bwd_chunk(d, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new,
                                                      dh_ckpt, dq, dk, dv, dbeta, dg, s));
        if (st != GDR_OK) return st;
        if (d.G > 1 && (st = from_cuda(gdr::group_sum_heads(d, dq, dk, dq_out, dk_out, s))) != GDR_OK) return st;
        t_last_variant = "tensor";
        return GDR_OK;
    }
    // forward prepare and re-scan: G, w, u, the checkpoints and v'
    if (tensor) {
        // a per-key-dim gate: prepare (+ T), re-scan, local term, reverse scan and the per-chunk stage on the
        // tensor cores; the CUDA-core per-chunk stages finish the chunks that stage flags
        unsigned int* err = device_error_word();
        void* tinv = base + ws.tinv;
        int* flags = reinterpret_cast<int*>(base + ws.flags);
        if ((st = from_cuda(gdr::mma_prepare(d, k, v, g, beta, w, u, g_cum, s, err, nullptr, nullptr, tinv))) !=
            GDR_OK)
            return st;
        if ((st = rescan(err)) != GDR_OK) return st;
        if ((st = from_cuda(gdr::mma_bwd_dv_local(d, q, k, g_cum, d_o, dv_loc, s))) != GDR_OK) return st;
        st = reverse_scan([&](const gdr::Dims& dd, const float* dhf, float* dh0o) {
            return from_cuda(gdr::mma_bwd_scan_dl(dd, q, k, w, g_cum, dv_loc, d_o, dhf, dh_ckpt, dv_new, dh0o, s, err,
                                                  co, nseq));
        });
        if (st != GDR_OK) return st;
        if ((st = from_cuda(gdr::mma_bwd_chunk_kda(d, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new,
                                                   dh_ckpt, dq, dk, dv, dbeta, dg, flags, s))) != GDR_OK)
            return st;
        if ((st = from_cuda(gdr::simt_bwd_dqkwg(d, q, k, v_new, g_cum, h_ckpt, dh_ckpt, d_o, dv_new, dq, dk_part, dw,
                                                dG_part, s, true, flags))) != GDR_OK)
            return st;
        if ((st = from_cuda(gdr::simt_bwd_wy(d, k, v, beta, g_cum, dw, dv_new, dk_part, dG_part, dk, dv, dbeta, dg, s,
                                             true, flags))) != GDR_OK)
            return st;
        if (d.G > 1 && (st = from_cuda(gdr::group_sum_heads(d, dq, dk, dq_out, dk_out, s))) != GDR_OK) return st;
        t_last_variant = "tensor";
        return GDR_OK;
    } else {
        if ((st = from_cuda(gdr::simt_prepare(d, k, v, g, beta, w, u, g_cum, s))) != GDR_OK) return st;
        if ((st = from_cuda(gdr::simt_scan(d, k, w, u, g_cum, h0, h_ckpt, v_new, nullptr, s))) != GDR_OK) return st;
    }
    if ((st = from_cuda(gdr::simt_bwd_dv_local(d, q, k, g_cum, d_o, dv_loc, s))) != GDR_OK) return st;
    if ((st = from_cuda(gdr::simt_bwd_scan_dh(d, q, k, w, g_cum, d_o, dv_loc, dh_final, dh_ckpt, dv_new, dh0, s))) !=
        GDR_OK)
        return st;
    if ((st = from_cuda(gdr::simt_bwd_dqkwg(d, q, k, v_new, g_cum, h_ckpt, dh_ckpt, d_o, dv_new, dq, dk_part, dw,
                                            dG_part, s))) != GDR_OK)
        return st;
    if ((st = from_cuda(gdr::simt_bwd_wy(d, k, v, beta, g_cum, dw, dv_new, dk_part, dG_part, dk, dv, dbeta, dg, s))) !=
        GDR_OK)
        return st;
    if (d.G > 1 && (st = from_cuda(gdr::group_sum_heads(d, dq, dk, dq_out, dk_out, s))) != GDR_OK) return st;
    t_last_variant = tensor ? "tensor" : "simt";
    return GDR_OK;
}

}  // namespace

extern "C" {

gdr_status gdr_prepare_wy(const gdr_problem* p, const void* k, const void* v, const float* g, const void* beta,
                          void* w, void* u, float* g_cum, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({k, v, g, beta, w, u, g_cum}, {})) != GDR_OK) return st;
    bool tensor = false;
    if ((st = pick_stage(p, d, &tensor)) != GDR_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    st = from_cuda(tensor ? gdr::mma_prepare(d, k, v, g, beta, w, u, g_cum, s, device_error_word())
                          : gdr::simt_prepare(d, k, v, g, beta, w, u, g_cum, s));
    if (st == GDR_OK) t_last_variant = tensor ? "tensor" : "simt";
    return st;
}

gdr_status gdr_scan_h(const gdr_problem* p, const void* k, const void* w, const void* u, const float* g_cum,
                      const float* h0, void* h_ckpt, void* v_new, float* h_final, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({k, w, u, g_cum, v_new}, {h0, h_ckpt, h_final})) != GDR_OK) return st;
    bool tensor = false;
    if ((st = pick_stage(p, d, &tensor)) != GDR_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    st = from_cuda(tensor ? gdr::mma_scan(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s, device_error_word())
                          : gdr::simt_scan(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s));
    if (st == GDR_OK) t_last_variant = tensor ? "tensor" : "simt";
    return st;
}

gdr_status gdr_scan_transfer(const gdr_problem* p, const void* k, const void* w, const void* u, const float* g_cum,
                             int32_t segments, float* M, float* Z, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({k, w, u, g_cum, M, Z}, {})) != GDR_OK) return st;
    if (p->variant == GDR_VARIANT_SIMT || !d.bf16) return GDR_ERR_UNSUPPORTED;
    if (segments < 1 || d.T % d.C != 0 || d.NT % segments != 0 || segments > kMaxGridYZ / d.B) return GDR_ERR_ARG;
    st = from_cuda(gdr::mma_scan_transfer(segment_view(d, segments), k, w, u, g_cum, M, Z, (cudaStream_t)stream,
                                          device_error_word()));
    if (st == GDR_OK) t_last_variant = "tensor";
    return st;
}

gdr_status gdr_scan_combine(const gdr_problem* p, int32_t segments, const float* M, const float* Z, const float* h0,
                            float* h_start, float* h_final, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({M, Z, h_start}, {h0, h_final})) != GDR_OK) return st;
    if (segments < 1 || segments > kMaxGridYZ / d.B) return GDR_ERR_ARG;
    st = from_cuda(gdr::segment_combine(d, segments, M, Z, h0, h_start, h_final, (cudaStream_t)stream));
    if (st == GDR_OK) t_last_variant = "simt";
    return st;
}

gdr_status gdr_scan_combine_reverse(const gdr_problem* p, int32_t segments, const float* M, const float* Zb,
                                    const float* dh_final, float* ends, float* dh0, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({M, Zb, ends}, {dh_final, dh0})) != GDR_OK) return st;
    if (segments < 1 || segments > kMaxGridYZ / d.B) return GDR_ERR_ARG;
    st = from_cuda(gdr::segment_combine(d, segments, M, Zb, dh_final, ends, dh0, (cudaStream_t)stream, true));
    if (st == GDR_OK) t_last_variant = "simt";
    return st;
}

gdr_status gdr_chunk_output(const gdr_problem* p, const void* q, const void* k, const void* v_new,
                            const void* h_ckpt, const float* g_cum, void* o, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, v_new, h_ckpt, g_cum, o}, {})) != GDR_OK) return st;
    bool tensor = false;
    if ((st = pick_stage(p, d, &tensor)) != GDR_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    st = from_cuda(tensor ? gdr::tc_output(d, q, k, v_new, h_ckpt, g_cum, o, s, device_error_word())
                          : gdr::simt_output(d, q, k, v_new, h_ckpt, g_cum, o, s));
    if (st == GDR_OK) t_last_variant = tensor ? "tensor" : "simt";
    return st;
}

size_t gdr_forward_workspace_bytes(const gdr_problem* p) {
    gdr::Dims d;
    if (check_problem(p, &d) != GDR_OK) return 0;
    Path path;
    int S = 1;
    if (pick_forward(p, d, &path) != GDR_OK || resolve_segments(p, d, path != Path::Simt, &S) != GDR_OK) return 0;
    return plan_staged(d, path == Path::Fused || path == Path::FusedTc, S, overlap_pieces(d, path, S),
                       path == Path::FusedTc && d.per_k)
        .total;
}

int gdr_forward_segments(const gdr_problem* p) {
    gdr::Dims d;
    if (check_problem(p, &d) != GDR_OK) return 0;
    Path path;
    int S = 1;
    if (pick_forward(p, d, &path) != GDR_OK || resolve_segments(p, d, path != Path::Simt, &S) != GDR_OK) return 0;
    return S;
}

gdr_status gdr_forward(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                       const void* beta, const float* h0, void* o, float* h_final, void* workspace,
                       size_t workspace_bytes, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, v, g, beta, o}, {h0, h_final})) != GDR_OK) return st;
    Path path;
    if ((st = pick_forward(p, d, &path)) != GDR_OK) return st;
    int S = 1;
    if ((st = resolve_segments(p, d, path != Path::Simt, &S)) != GDR_OK) return st;
    int bounds[kMaxPieces + 1];
    const int pieces = overlap_bounds(d, path, S, bounds);
    const bool gated = path == Path::FusedTc && d.per_k;
    const StagedWorkspace ws = plan_staged(d, path == Path::Fused || path == Path::FusedTc, S, pieces, gated);
    if (!workspace || workspace_bytes < ws.total) return GDR_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDR_ERR_ALIGN;
    char* base = static_cast<char*>(workspace);
    float* g_cum = reinterpret_cast<float*>(base + ws.g_cum);
    void* w = base + ws.w;
    void* u = base + ws.u;
    void* v_new = base + ws.v_new;
    void* h_ckpt = base + ws.h_ckpt;
    cudaStream_t s = (cudaStream_t)stream;
    unsigned int* err = path == Path::Simt ? nullptr : device_error_word();
    if (pieces > 1) {
        if ((st = forward_tc_overlapped(d, bounds, pieces, ws, base, q, k, v, g, beta, h0, o, h_final, s, err)) !=
            GDR_OK)
            return st;
    } else if (path == Path::Simt) {
        if ((st = from_cuda(gdr::simt_prepare(d, k, v, g, beta, w, u, g_cum, s))) != GDR_OK) return st;
        if ((st = from_cuda(gdr::simt_scan(d, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, s))) != GDR_OK) return st;
        if ((st = from_cuda(gdr::simt_output(d, q, k, v_new, h_ckpt, g_cum, o, s))) != GDR_OK) return st;
    } else {
        const bool fused = path == Path::Fused || path == Path::FusedTc;
        void* P = (fused && d.C == 64) ? base + ws.P : nullptr;
        void* kg = base + ws.kg;
        void* qg = base + ws.qg;
        if (gated) {   // per-key-dim gate: the prepare, then P, kg and qg from q, k and G
            if ((st = from_cuda(gdr::mma_prepare(d, k, v, g, beta, w, u, g_cum, s, err))) != GDR_OK) return st;
            if ((st = from_cuda(gdr::tc_gated_operands(d, q, k, g_cum, P, kg, qg, s, err))) != GDR_OK) return st;
        } else if ((st = from_cuda(gdr::mma_prepare(d, k, v, g, beta, w, u, g_cum, s, err, q, P))) != GDR_OK) {
            return st;
        }
        // segments: every segment's map from a zero state, the starts stitched serially, then the
        // scan (and output) of all segments at once from their starts
        gdr::Dims ds = d;
        const float* hs = h0;
        float* hf = h_final;
        if (S > 1) {
            ds = segment_view(d, S);
            float* m = reinterpret_cast<float*>(base + ws.seg_m);
            float* z = reinterpret_cast<float*>(base + ws.seg_z);
            float* starts = reinterpret_cast<float*>(base + ws.seg_h);
            if ((st = from_cuda(gdr::mma_scan_transfer(ds, k, w, u, g_cum, m, z, s, err))) != GDR_OK) return st;
            if ((st = from_cuda(gdr::segment_combine(d, S, m, z, h0, starts, h_final, s))) != GDR_OK) return st;
            hs = starts;
            hf = nullptr;
        }
        if (fused) {
            const cudaError_t e =
                path != Path::FusedTc ? gdr::mma_scan_output(ds, q, k, w, u, g_cum, P, hs, o, hf, s, err)
                : gated               ? gdr::tc_scan_output(ds, qg, kg, w, u, g_cum, P, hs, o, hf, s, err)
                                      : gdr::tc_scan_output(ds, q, k, w, u, g_cum, P, hs, o, hf, s, err, S == 1);
            if ((st = from_cuda(e)) != GDR_OK) return st;
        } else {
            if ((st = from_cuda(gdr::mma_scan(ds, k, w, u, g_cum, hs, h_ckpt, v_new, hf, s, err))) != GDR_OK)
                return st;
            if ((st = from_cuda(gdr::tc_output(d, q, k, v_new, h_ckpt, g_cum, o, s, err))) != GDR_OK) return st;
        }
    }
    t_last_variant = path_name(path);
    return GDR_OK;
}

// ---------------------------------------------------------------- the forward over host tensors
namespace {

constexpr int kHostPiecesDefault = 8;
constexpr int kHostPiecesMax = 64;

// Per token, the bytes of each host tensor the forward reads (q, k, v, g, beta) and writes (o).
struct HostRows {
    size_t q, k, v, g, beta, o;
};
HostRows host_rows(const gdr::Dims& d) {
    const size_t e = d.bf16 || d.f16 ? 2 : 4;
    return {(size_t)d.Hk * d.K * e, (size_t)d.Hk * d.K * e, (size_t)d.H * d.V * e,
            (size_t)d.H * (d.per_k ? d.K : 1) * 4, (size_t)d.H * e, (size_t)d.H * d.V * e};
}

// Device scratch of the host forward: two slots of one piece's inputs and output, the two states the
// pieces alternate between, h0, and one piece's gdr_forward workspace.
struct HostScratch {
    int pieces, chunks_per_piece;
    size_t slot[2][6];   // q, k, v, g, beta, o
    size_t state[2], h0, ws, ws_bytes, total;
};

bool plan_host(const gdr_problem* p, const gdr::Dims& d, int pieces_req, HostScratch* hs) {
    int pieces = pieces_req > 0 ? pieces_req : kHostPiecesDefault;
    pieces = std::min(std::min(pieces, kHostPiecesMax), d.NT);
    const int cpp = (d.NT + pieces - 1) / pieces;   // chunks per piece; the last piece may be shorter
    hs->pieces = (d.NT + cpp - 1) / cpp;
    hs->chunks_per_piece = cpp;
    const int64_t Tp = std::min<int64_t>((int64_t)cpp * d.C, d.T);
    const HostRows r = host_rows(d);
    const size_t rows[6] = {r.q, r.k, r.v, r.g, r.beta, r.o};
    size_t off = 0;
    for (int sl = 0; sl < 2; ++sl)
        for (int i = 0; i < 6; ++i) {
            hs->slot[sl][i] = off;
            off = round_up(off + (size_t)d.B * Tp * rows[i], 256);
        }
    const size_t state = (size_t)d.B * d.H * d.K * d.V * 4;
    hs->state[0] = off; off = round_up(off + state, 256);
    hs->state[1] = off; off = round_up(off + state, 256);
    hs->h0 = off;       off = round_up(off + state, 256);
    // the workspace of the longest piece and of the last one (a different T may plan differently)
    gdr_problem pp = *p;
    pp.T = Tp;
    size_t ws = gdr_forward_workspace_bytes(&pp);
    const int64_t last = d.T - (int64_t)(hs->pieces - 1) * cpp * d.C;
    pp.T = last;
    ws = std::max(ws, gdr_forward_workspace_bytes(&pp));
    hs->ws = off;
    hs->ws_bytes = ws;
    hs->total = round_up(off + ws, 256);
    return true;
}

// One tensor's token range [t0, t0 + n) of every sequence: host [B, T, row] <-> device [B, n, row].
cudaError_t copy_rows(void* dst, const void* src, size_t row, int B, int64_t T, int64_t t0, int64_t n, bool to_device,
                      cudaStream_t s) {
    if (to_device)
        return cudaMemcpy2DAsync(dst, (size_t)n * row, static_cast<const char*>(src) + (size_t)t0 * row, (size_t)T * row,
                                 (size_t)n * row, (size_t)B, cudaMemcpyHostToDevice, s);
    return cudaMemcpy2DAsync(static_cast<char*>(dst) + (size_t)t0 * row, (size_t)T * row, src, (size_t)n * row,
                             (size_t)n * row, (size_t)B, cudaMemcpyDeviceToHost, s);
}

}  // namespace

size_t gdr_forward_host_scratch_bytes(const gdr_problem* p, int32_t pieces) {
    gdr::Dims d;
    if (check_problem(p, &d) != GDR_OK || pieces < 0) return 0;
    HostScratch hs;
    plan_host(p, d, pieces, &hs);
    return hs.total;
}

gdr_status gdr_forward_host(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                            const void* beta, const float* h0, void* o, float* h_final, int32_t pieces, void* scratch,
                            size_t scratch_bytes, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if (pieces < 0) return GDR_ERR_ARG;
    if (!q || !k || !v || !g || !beta || !o) return GDR_ERR_NULL;
    HostScratch hs;
    plan_host(p, d, pieces, &hs);
    if (!scratch || scratch_bytes < hs.total) return GDR_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(scratch) & 255u) != 0) return GDR_ERR_ALIGN;
    char* base = static_cast<char*>(scratch);
    cudaStream_t s = (cudaStream_t)stream;
    const HostRows r = host_rows(d);
    const size_t rows[6] = {r.q, r.k, r.v, r.g, r.beta, r.o};
    const void* src[5] = {q, k, v, g, beta};
    const size_t state = (size_t)d.B * d.H * d.K * d.V * 4;

    // the copies run on two streams of this call's own; everything they do is ordered after the work
    // already queued on `stream` (which may still be using the scratch) and before what follows there
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t start = nullptr, ready[2] = {}, done[2] = {}, out_free[2] = {}, fin = nullptr;
    auto cleanup = [&]() {
        for (cudaEvent_t e : {start, ready[0], ready[1], done[0], done[1], out_free[0], out_free[1], fin})
            if (e) cudaEventDestroy(e);
        if (up) cudaStreamDestroy(up);
        if (down) cudaStreamDestroy(down);
    };
    auto fail = [&](cudaError_t e) {
        cleanup();
        return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
    };
    cudaError_t e = cudaStreamCreateWithFlags(&up, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&down, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&start, &ready[0], &ready[1], &done[0], &done[1], &out_free[0], &out_free[1], &fin})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(up, start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(down, start, 0);
    const float* h_prev = nullptr;
    if (h0 && e == cudaSuccess) {
        e = cudaMemcpyAsync(base + hs.h0, h0, state, cudaMemcpyHostToDevice, s);
        h_prev = reinterpret_cast<const float*>(base + hs.h0);
    }
    if (e != cudaSuccess) return fail(e);

    const int64_t per = (int64_t)hs.chunks_per_piece * d.C;
    for (int i = 0; i < hs.pieces; ++i) {
        const int sl = i & 1;
        const int64_t t0 = (int64_t)i * per, n = std::min<int64_t>(per, d.T - t0);
        char* buf[6];
        for (int j = 0; j < 6; ++j) buf[j] = base + hs.slot[sl][j];
        // inputs of piece i, once piece i - 2 has finished reading this slot
        if (i >= 2) e = cudaStreamWaitEvent(up, done[sl], 0);
        for (int j = 0; j < 5 && e == cudaSuccess; ++j) e = copy_rows(buf[j], src[j], rows[j], d.B, d.T, t0, n, true, up);
        if (e == cudaSuccess) e = cudaEventRecord(ready[sl], up);
        // piece i on the caller's stream, from the state piece i - 1 left, once its output slot is free
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ready[sl], 0);
        if (e == cudaSuccess && i >= 2) e = cudaStreamWaitEvent(s, out_free[sl], 0);
        if (e != cudaSuccess) return fail(e);
        gdr_problem pp = *p;
        pp.T = n;
        float* hout = reinterpret_cast<float*>(base + hs.state[sl]);
        st = gdr_forward(&pp, buf[0], buf[1], buf[2], reinterpret_cast<const float*>(buf[3]), buf[4], h_prev, buf[5],
                         hout, base + hs.ws, hs.ws_bytes, s);
        if (st != GDR_OK) {
            fail(cudaSuccess);
            return st;
        }
        h_prev = hout;
        e = cudaEventRecord(done[sl], s);
        // its output back to the host
        if (e == cudaSuccess) e = cudaStreamWaitEvent(down, done[sl], 0);
        if (e == cudaSuccess) e = copy_rows(o, buf[5], rows[5], d.B, d.T, t0, n, false, down);
        if (e == cudaSuccess) e = cudaEventRecord(out_free[sl], down);
        if (e != cudaSuccess) return fail(e);
    }
    if (h_final) e = cudaMemcpyAsync(h_final, h_prev, state, cudaMemcpyDeviceToHost, s);
    // `stream` completes only after the last output copy
    if (e == cudaSuccess) e = cudaEventRecord(fin, down);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, fin, 0);
    return fail(e);
}

gdr_status gdr_scan_output(const gdr_problem* p, const void* q, const void* k, const void* w, const void* u,
                           const float* g_cum, const void* P, const float* h0, void* o, float* h_final,
                           void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, w, u, g_cum, o}, {P, h0, h_final})) != GDR_OK) return st;
    if (p->variant == GDR_VARIANT_SIMT || !(d.bf16 || d.f16) || (P && d.C != 64)) return GDR_ERR_UNSUPPORTED;
    // a per-key-dim gate: the tcgen05 kernel only, on gdr_gated_operands' P, qg and kg
    if (d.per_k && (p->variant != GDR_VARIANT_FUSED_TC || !P)) return GDR_ERR_UNSUPPORTED;
    // the tcgen05 kernel for variant FUSED_TC, and for AUTO where gdr_forward would take it
    Path path;
    if ((st = pick_forward(p, d, &path)) != GDR_OK) return st;
    bool tc = path == Path::FusedTc;
    if (tc && !P) {   // the tcgen05 kernel takes P from the prepare
        if (p->variant == GDR_VARIANT_FUSED_TC) return GDR_ERR_UNSUPPORTED;
        tc = false;
    }
    st = from_cuda(tc ? gdr::tc_scan_output(d, q, k, w, u, g_cum, P, h0, o, h_final, (cudaStream_t)stream,
                                            device_error_word())
                      : gdr::mma_scan_output(d, q, k, w, u, g_cum, P, h0, o, h_final, (cudaStream_t)stream,
                                             device_error_word()));
    if (st == GDR_OK) t_last_variant = tc ? "fused_tc" : "fused";
    return st;
}

gdr_status gdr_gated_operands(const gdr_problem* p, const void* q, const void* k, const float* g_cum, void* P, void* kg,
                              void* qg, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, g_cum, P, kg, qg}, {})) != GDR_OK) return st;
    if (p->variant == GDR_VARIANT_SIMT || !d.bf16 || !d.per_k || d.K != 128 || d.V != 128 || d.C != 64)
        return GDR_ERR_UNSUPPORTED;
    st = from_cuda(gdr::tc_gated_operands(d, q, k, g_cum, P, kg, qg, (cudaStream_t)stream, device_error_word()));
    if (st == GDR_OK) t_last_variant = "fused_tc";
    return st;
}

gdr_status gdr_prepare_wyp(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                           const void* beta, void* w, void* u, float* g_cum, void* P, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, v, g, beta, w, u, g_cum, P}, {})) != GDR_OK) return st;
    if (p->variant == GDR_VARIANT_SIMT || !(d.bf16 || d.f16) || d.per_k || d.C != 64) return GDR_ERR_UNSUPPORTED;
    st = from_cuda(gdr::mma_prepare(d, k, v, g, beta, w, u, g_cum, (cudaStream_t)stream, device_error_word(), q, P));
    if (st == GDR_OK) t_last_variant = "tensor";
    return st;
}

gdr_status gdr_bwd_dv_local(const gdr_problem* p, const void* q, const void* k, const float* g_cum,
                            const void* d_o, float* dv_loc, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, g_cum, d_o, dv_loc}, {})) != GDR_OK) return st;
    st = from_cuda(gdr::simt_bwd_dv_local(d, q, k, g_cum, d_o, dv_loc, (cudaStream_t)stream));
    if (st == GDR_OK) t_last_variant = "simt";
    return st;
}

gdr_status gdr_bwd_scan_dh(const gdr_problem* p, const void* q, const void* k, const void* w, const float* g_cum,
                           const void* d_o, const float* dv_loc, const float* dh_final, float* dh_ckpt,
                           float* dv_new, float* dh0, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, w, g_cum, d_o, dv_loc, dh_ckpt, dv_new}, {dh_final, dh0})) != GDR_OK) return st;
    st = from_cuda(gdr::simt_bwd_scan_dh(d, q, k, w, g_cum, d_o, dv_loc, dh_final, dh_ckpt, dv_new, dh0,
                                         (cudaStream_t)stream));
    if (st == GDR_OK) t_last_variant = "simt";
    return st;
}

gdr_status gdr_bwd_dqkwg(const gdr_problem* p, const void* q, const void* k, const void* v_new, const float* g_cum,
                         const void* h_ckpt, const void* dh_ckpt, const void* d_o, const void* dv_new, void* dq,
                         float* dk_part, float* dw, float* dG_part, const int* only, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, v_new, g_cum, h_ckpt, dh_ckpt, d_o, dv_new, dq, dk_part, dw, dG_part}, {})) != GDR_OK)
        return st;
    // the tensor path's intermediates (bf16 io, variants other than SIMT) are bf16
    const bool inter16 = d.bf16 && p->variant != GDR_VARIANT_SIMT;
    st = from_cuda(gdr::simt_bwd_dqkwg(d, q, k, v_new, g_cum, h_ckpt, dh_ckpt, d_o, dv_new, dq, dk_part, dw,
                                       dG_part, (cudaStream_t)stream, inter16, only));
    if (st == GDR_OK) t_last_variant = "simt";
    return st;
}

gdr_status gdr_bwd_wy(const gdr_problem* p, const void* k, const void* v, const void* beta, const float* g_cum,
                      const float* dw, const void* dv_new, const float* dk_part, const float* dG_part, void* dk,
                      void* dv, void* dbeta, float* dg, const int* only, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({k, v, beta, g_cum, dw, dv_new, dk_part, dG_part, dk, dv, dbeta, dg}, {})) != GDR_OK)
        return st;
    const bool inter16 = d.bf16 && p->variant != GDR_VARIANT_SIMT;
    st = from_cuda(gdr::simt_bwd_wy(d, k, v, beta, g_cum, dw, dv_new, dk_part, dG_part, dk, dv, dbeta, dg,
                                    (cudaStream_t)stream, inter16, only));
    if (st == GDR_OK) t_last_variant = "simt";
    return st;
}

gdr_status gdr_bwd_dv_local_tc(const gdr_problem* p, const void* q, const void* k, const float* g_cum,
                               const void* d_o, void* dv_loc, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, g_cum, d_o, dv_loc}, {})) != GDR_OK) return st;
    if (p->variant == GDR_VARIANT_SIMT || !d.bf16) return GDR_ERR_UNSUPPORTED;
    st = from_cuda(gdr::mma_bwd_dv_local(d, q, k, g_cum, d_o, dv_loc, (cudaStream_t)stream));
    if (st == GDR_OK) t_last_variant = "tensor";
    return st;
}

gdr_status gdr_bwd_scan_dh_tc(const gdr_problem* p, const void* q, const void* k, const void* w, const float* g_cum,
                              const void* dv_loc, const void* d_o, const float* dh_final, void* dh_ckpt,
                              void* dv_new, float* dh0, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, w, g_cum, dv_loc, d_o, dh_ckpt, dv_new}, {dh_final, dh0})) != GDR_OK) return st;
    if (p->variant == GDR_VARIANT_SIMT || !d.bf16) return GDR_ERR_UNSUPPORTED;
    st = from_cuda(gdr::mma_bwd_scan_dl(d, q, k, w, g_cum, dv_loc, d_o, dh_final, dh_ckpt, dv_new, dh0,
                                        (cudaStream_t)stream, device_error_word()));
    if (st == GDR_OK) t_last_variant = "tensor";
    return st;
}

gdr_status gdr_bwd_prepare(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                           const void* beta, void* w, void* u, float* g_cum, void* P, void* tinv, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, v, g, beta, w, u, g_cum, tinv}, {P})) != GDR_OK) return st;
    if (p->variant == GDR_VARIANT_SIMT || !d.bf16 || (P && (d.per_k || d.C != 64))) return GDR_ERR_UNSUPPORTED;
    st = from_cuda(gdr::mma_prepare(d, k, v, g, beta, w, u, g_cum, (cudaStream_t)stream, device_error_word(),
                                    P ? q : nullptr, P, tinv));
    if (st == GDR_OK) t_last_variant = "tensor";
    return st;
}

gdr_status gdr_bwd_scan_dh_p(const gdr_problem* p, const void* q, const void* k, const void* w, const float* g_cum,
                             const void* P, const void* d_o, const float* dh_final, void* dh_ckpt, void* dv_new,
                             float* dh0, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, w, g_cum, P, d_o, dh_ckpt, dv_new}, {dh_final, dh0})) != GDR_OK) return st;
    if (p->variant == GDR_VARIANT_SIMT || !d.bf16 || d.per_k || d.C != 64) return GDR_ERR_UNSUPPORTED;
    st = from_cuda(gdr::mma_bwd_scan(d, q, k, w, g_cum, P, d_o, dh_final, dh_ckpt, dv_new, dh0, (cudaStream_t)stream,
                                     device_error_word()));
    if (st == GDR_OK) t_last_variant = "tensor";
    return st;
}

gdr_status gdr_bwd_wy_dqkg(const gdr_problem* p, const void* q, const void* k, const void* v, const void* beta,
                           const float* g_cum, const void* w, const void* u, const void* tinv, const void* v_new,
                           const void* h_ckpt, const void* d_o, const void* dv_new, const void* dh_ckpt, void* dq,
                           void* dk, void* dv, void* dbeta, float* dg, int* exact_flags, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new, dh_ckpt, dq, dk, dv, dbeta,
                          dg}, {})) != GDR_OK)
        return st;
    if (p->variant == GDR_VARIANT_SIMT || !d.bf16) return GDR_ERR_UNSUPPORTED;
    if (d.per_k) {
        if (!exact_flags) return GDR_ERR_NULL;
        if ((reinterpret_cast<uintptr_t>(exact_flags) & 3u) != 0) return GDR_ERR_ALIGN;
        st = from_cuda(gdr::mma_bwd_chunk_kda(d, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new,
                                              dh_ckpt, dq, dk, dv, dbeta, dg, exact_flags, (cudaStream_t)stream));
    } else {
        st = from_cuda(d.C == 64 ? gdr::mma_bwd_chunk_tma(d, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o,
                                                          dv_new, dh_ckpt, dq, dk, dv, dbeta, dg, (cudaStream_t)stream,
                                                          device_error_word())
                                 : gdr::mma_bwd_chunk(d, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new,
                                                      dh_ckpt, dq, dk, dv, dbeta, dg, (cudaStream_t)stream));
    }
    if (st == GDR_OK) t_last_variant = "tensor";
    return st;
}

gdr_status gdr_bwd_group_sum(const gdr_problem* p, const void* dq_v, const void* dk_v, void* dq, void* dk,
                             void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({dq_v, dk_v, dq, dk}, {})) != GDR_OK) return st;
    st = from_cuda(gdr::group_sum_heads(d, dq_v, dk_v, dq, dk, (cudaStream_t)stream));
    if (st == GDR_OK) t_last_variant = "simt";
    return st;
}

size_t gdr_backward_workspace_bytes(const gdr_problem* p) {
    gdr::Dims d;
    if (check_problem(p, &d) != GDR_OK) return 0;
    BwdPath path;
    int S = 1;
    if (pick_backward(p, d, &path) != GDR_OK || resolve_segments(p, d, path != BwdPath::Simt, &S) != GDR_OK) return 0;
    return plan_backward(d, path, S).total;
}

gdr_status gdr_backward(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                        const void* beta, const float* h0, const void* d_o, const float* dh_final, void* dq,
                        void* dk, void* dv, float* dg, void* dbeta, float* dh0, void* workspace,
                        size_t workspace_bytes, void* stream) {
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if ((st = check_ptrs({q, k, v, g, beta, d_o, dq, dk, dv, dg, dbeta}, {h0, dh_final, dh0})) != GDR_OK) return st;
    BwdPath path;
    if ((st = pick_backward(p, d, &path)) != GDR_OK) return st;
    const bool tensor = path != BwdPath::Simt;
    int S = 1;
    if ((st = resolve_segments(p, d, tensor, &S)) != GDR_OK) return st;
    const BackwardWorkspace ws = plan_backward(d, path, S);
    if (!workspace || workspace_bytes < ws.total) return GDR_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDR_ERR_ALIGN;
    return run_backward(d, path, S, static_cast<char*>(workspace), ws, q, k, v, g, beta, h0, d_o, dh_final, dq, dk, dv,
                        dg, dbeta, dh0, (cudaStream_t)stream, nullptr, 0);
}

}  // extern "C"

// ---- packed variable-length sequences
// On the tensor cores they run chunk-packed: every sequence a run of whole chunks of one row (fewer
// than C zero tokens each), the scans walking each sequence's chunks.  On the CUDA cores they run
// padded: sequence s as row s of a batch of rows of p->T tokens.
namespace {

// Bytes a token takes in each working tensor, in order.  Forward: q k v g beta (packed in) | o (unpacked
// out).  Backward: q k v g beta do (in) | dq dk dv dg dbeta (out).
constexpr int kVarlenAll[2] = {6, 11};

void varlen_rows(const gdr::Dims& d, bool backward, int64_t* rb) {
    const int64_t es = (d.bf16 || d.f16) ? 2 : 4;
    const int64_t qk = (int64_t)d.Hk * d.K * es, vv = (int64_t)d.H * d.V * es;
    const int64_t gg = (int64_t)d.H * (d.per_k ? d.K : 1) * 4, bb = (int64_t)d.H * es;
    const int64_t fw[6] = {qk, qk, vv, gg, bb, vv};
    const int64_t bw[11] = {qk, qk, vv, gg, bb, vv, qk, qk, vv, gg, bb};
    for (int i = 0; i < kVarlenAll[backward]; ++i) rb[i] = backward ? bw[i] : fw[i];
}

// The chunk-packed problem of at most `chunks` chunks: one row of whole chunks.
gdr::Dims chunk_packed(const gdr::Dims& d, int64_t chunks) {
    gdr::Dims v = d;
    v.B = 1;
    v.NT = (int)chunks;
    v.T = (int)(chunks * d.C);
    return v;
}

// chunks of the chunk-packed layout in the worst case for p: n sequences of p->T tokens
int64_t max_chunks(const gdr::Dims& d) { return (int64_t)d.B * d.NT; }

// the chunk-packed row's indices fit in int32
bool chunk_packed_fits(const gdr::Dims& d) { return max_chunks(d) * d.C * d.H <= INT32_MAX; }

struct VarlenWorkspace {
    size_t cu, co, cs, pad[11], inner, inner_bytes, total;
    int64_t rows;   // rows of every working tensor
};

VarlenWorkspace plan_varlen(const gdr::Dims& d, bool backward, bool chunked, size_t inner_bytes) {
    VarlenWorkspace ws{};
    int64_t rb[11];
    varlen_rows(d, backward, rb);
    ws.rows = chunked ? max_chunks(d) * d.C : (int64_t)d.B * d.T;
    size_t off = 0;
    ws.cu = off;
    off = round_up(off + (size_t)(d.B + 1) * sizeof(int32_t), 256);
    ws.co = ws.cs = off;
    if (chunked) {
        off = round_up(off + (size_t)(d.B + 1) * sizeof(int32_t), 256);
        ws.cs = off;
        off = round_up(off + (size_t)max_chunks(d) * sizeof(int32_t), 256);
    }
    for (int i = 0; i < kVarlenAll[backward]; ++i) {
        ws.pad[i] = off;
        off = round_up(off + (size_t)ws.rows * rb[i], 256);
    }
    ws.inner = off;
    ws.inner_bytes = inner_bytes;
    ws.total = off + inner_bytes;
    return ws;
}

// cu_seqlens on the host: cu[0] = 0, cu[n] = total, every length in [0, T]
gdr_status check_cu(const int32_t* cu, int64_t n, int64_t total, int64_t T) {
    if (!cu) return GDR_ERR_NULL;
    if (total < 0 || cu[0] != 0 || (int64_t)cu[n] != total) return GDR_ERR_ARG;
    for (int64_t s = 0; s < n; ++s) {
        const int64_t len = (int64_t)cu[s + 1] - cu[s];
        if (len < 0 || len > T) return GDR_ERR_ARG;
    }
    return GDR_OK;
}

// workspace of the inner call(s): the padded problem's, and on the tensor cores also the largest
// chunk-packed problem's
gdr_status varlen_inner_bytes(const gdr_problem* p, const gdr::Dims& d, bool backward, size_t* bytes,
                              bool* chunked) {
    gdr_status st;
    int S = 1;
    *chunked = false;
    if (backward) {
        BwdPath path;
        if ((st = pick_backward(p, d, &path)) != GDR_OK) return st;
        if ((st = resolve_segments(p, d, path != BwdPath::Simt, &S)) != GDR_OK) return st;
        *bytes = plan_backward(d, path, S).total;
        if (path != BwdPath::Simt && chunk_packed_fits(d)) {
            *chunked = true;
            const size_t c = plan_backward(chunk_packed(d, max_chunks(d)), path, 1).total;
            if (c > *bytes) *bytes = c;
        }
    } else {
        Path path;
        if ((st = pick_forward(p, d, &path)) != GDR_OK) return st;
        if (path == Path::FusedTc)   // packed sequences: the warp-level fused kernel, or the staged one (KDA)
            path = d.per_k ? Path::Tensor : Path::Fused;
        if ((st = resolve_segments(p, d, path != Path::Simt, &S)) != GDR_OK) return st;
        *bytes = plan_staged(d, path == Path::Fused, S).total;
        if (path != Path::Simt && chunk_packed_fits(d)) {
            *chunked = true;
            const size_t c = plan_staged(chunk_packed(d, max_chunks(d)), path == Path::Fused, 1).total;
            if (c > *bytes) *bytes = c;
        }
    }
    return GDR_OK;
}

// Validates a varlen call up to the workspace and returns its plan and the device cu to use
// (the caller's, or the host array copied into the workspace on `s`).
gdr_status varlen_setup(const gdr_problem* p, gdr::Dims* d, bool backward, const int32_t* cu_host,
                        const int32_t* cu_dev, int64_t total, void* workspace, size_t workspace_bytes,
                        cudaStream_t s, VarlenWorkspace* ws, const int** cu) {
    // p is the caller's problem with segments = 1 (see varlen_problem)
    gdr_status st = check_problem(p, d);
    if (st != GDR_OK) return st;
    if ((st = check_cu(cu_host, p->B, total, p->T)) != GDR_OK) return st;
    if (cu_dev && (reinterpret_cast<uintptr_t>(cu_dev) & 3u) != 0) return GDR_ERR_ALIGN;
    size_t inner = 0;
    bool chunked = false;
    if ((st = varlen_inner_bytes(p, *d, backward, &inner, &chunked)) != GDR_OK) return st;
    *ws = plan_varlen(*d, backward, chunked, inner);
    if (!workspace || workspace_bytes < ws->total) return GDR_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDR_ERR_ALIGN;
    if (cu_dev) {
        *cu = cu_dev;
    } else {
        int32_t* c = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + ws->cu);
        if ((st = from_cuda(cudaMemcpyAsync(c, cu_host, (size_t)(d->B + 1) * sizeof(int32_t),
                                            cudaMemcpyHostToDevice, s))) != GDR_OK)
            return st;
        *cu = c;
    }
    return GDR_OK;
}

// The varlen calls scan each sequence whole: the segment-parallel scan does not apply, so the caller's
// p->segments is replaced by 1 before anything else looks at the problem.
gdr_problem varlen_problem(const gdr_problem* p) {
    gdr_problem q = *p;
    q.segments = 1;
    return q;
}

size_t varlen_workspace_bytes(const gdr_problem* p_in, bool backward) {
    gdr::Dims d;
    size_t inner = 0;
    bool chunked = false;
    if (!p_in) return 0;
    const gdr_problem p1 = varlen_problem(p_in);
    const gdr_problem* p = &p1;
    if (check_problem(p, &d) != GDR_OK || varlen_inner_bytes(p, d, backward, &inner, &chunked) != GDR_OK) return 0;
    return plan_varlen(d, backward, chunked, inner).total;
}

}  // namespace

extern "C" {

size_t gdr_varlen_forward_workspace_bytes(const gdr_problem* p) { return varlen_workspace_bytes(p, false); }

size_t gdr_varlen_backward_workspace_bytes(const gdr_problem* p) { return varlen_workspace_bytes(p, true); }

gdr_status gdr_varlen_forward(const gdr_problem* p_in, const int32_t* cu_seqlens, const int32_t* cu_seqlens_device,
                              int64_t total, const void* q, const void* k, const void* v, const float* g,
                              const void* beta, const float* h0, void* o, float* h_final, void* workspace,
                              size_t workspace_bytes, void* stream) {
    if (!p_in) return GDR_ERR_NULL;
    const gdr_problem p1 = varlen_problem(p_in);
    const gdr_problem* p = &p1;
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if (total > 0 && (st = check_ptrs({q, k, v, g, beta, o}, {h0, h_final})) != GDR_OK) return st;
    if (total <= 0 && (st = check_ptrs({}, {q, k, v, g, beta, o, h0, h_final})) != GDR_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    VarlenWorkspace ws;
    const int* cu = nullptr;
    if ((st = varlen_setup(p, &d, false, cu_seqlens, cu_seqlens_device, total, workspace, workspace_bytes, s, &ws,
                           &cu)) != GDR_OK)
        return st;
    Path path;
    if ((st = pick_forward(p, d, &path)) != GDR_OK) return st;
    if (path == Path::FusedTc)   // packed sequences: the warp-level fused kernel, or the staged one (KDA)
        path = d.per_k ? Path::Tensor : Path::Fused;
    char* base = static_cast<char*>(workspace);
    int64_t rb[11];
    varlen_rows(d, false, rb);
    const void* packed[5] = {q, k, v, g, beta};
    gdr::RowCopy in[5];
    for (int i = 0; i < 5; ++i) in[i] = {packed[i], base + ws.pad[i], rb[i]};
    const gdr::RowCopy out[1] = {{base + ws.pad[5], o, rb[5]}};
    int64_t chunks = 0;   // the chunk-packed row's chunks, from the host lengths
    for (int64_t i = 0; i < d.B; ++i) chunks += ((int64_t)cu_seqlens[i + 1] - cu_seqlens[i] + d.C - 1) / d.C;
    if (path == Path::Fused && d.bf16 && d.C == 64 && chunk_packed_fits(d) && chunks > 0) {
        // the fused path reads q, k, v, g, beta in place and writes o in place: no copies (bf16; fp16
        // takes the chunk-packed copies below)
        int* co = reinterpret_cast<int*>(base + ws.co);
        int* cs = reinterpret_cast<int*>(base + ws.cs);
        const gdr::Dims d1 = chunk_packed(d, chunks);
        const StagedWorkspace iw = plan_staged(d1, true, 1);
        char* ib = base + ws.inner;
        float* g_cum = reinterpret_cast<float*>(ib + iw.g_cum);
        void *w = ib + iw.w, *u = ib + iw.u, *P = ib + iw.P;
        unsigned int* err = device_error_word();
        if ((st = from_cuda(gdr::varlen_plan(cu, d.B, total, d.C, (int)chunks, co, cs, s))) != GDR_OK) return st;
        if ((st = from_cuda(gdr::mma_prepare_packed(d1, q, k, v, g, beta, w, u, g_cum, P, cu, co, cs, d.B, (int)total,
                                                    s, err))) != GDR_OK)
            return st;
        if ((st = from_cuda(gdr::mma_scan_output(d1, q, k, w, u, g_cum, P, h0, o, h_final, s, err, co, d.B, cu,
                                                 (int)total))) != GDR_OK)
            return st;
        t_last_variant = path_name(path);
        return GDR_OK;
    }
    if (path != Path::Simt && chunk_packed_fits(d) && chunks > 0) {
        int* co = reinterpret_cast<int*>(base + ws.co);
        int* cs = reinterpret_cast<int*>(base + ws.cs);
        const gdr::VarlenMap m{cu, co, cs, d.B, total, 0, d.C, chunks * d.C};
        const gdr::Dims d1 = chunk_packed(d, chunks);
        const StagedWorkspace iw = plan_staged(d1, path == Path::Fused, 1);
        char* ib = base + ws.inner;
        float* g_cum = reinterpret_cast<float*>(ib + iw.g_cum);
        void *w = ib + iw.w, *u = ib + iw.u, *v_new = ib + iw.v_new, *h_ckpt = ib + iw.h_ckpt;
        void* P = (path == Path::Fused && d.C == 64) ? ib + iw.P : nullptr;
        void* pad[6];
        for (int i = 0; i < 6; ++i) pad[i] = base + ws.pad[i];
        unsigned int* err = device_error_word();
        if ((st = from_cuda(gdr::varlen_plan(cu, d.B, total, d.C, (int)chunks, co, cs, s))) != GDR_OK) return st;
        if ((st = from_cuda(gdr::varlen_pack(in, 5, m, s))) != GDR_OK) return st;
        if ((st = from_cuda(gdr::mma_prepare(d1, pad[1], pad[2], reinterpret_cast<const float*>(pad[3]), pad[4], w, u,
                                             g_cum, s, err, pad[0], P))) != GDR_OK)
            return st;
        if (path == Path::Fused) {
            if ((st = from_cuda(gdr::mma_scan_output(d1, pad[0], pad[1], w, u, g_cum, P, h0, pad[5], h_final, s, err,
                                                     co, d.B))) != GDR_OK)
                return st;
        } else {
            if ((st = from_cuda(gdr::mma_scan(d1, pad[1], w, u, g_cum, h0, h_ckpt, v_new, h_final, s, err, co,
                                              d.B))) != GDR_OK)
                return st;
            if ((st = from_cuda(gdr::tc_output(d1, pad[0], pad[1], v_new, h_ckpt, g_cum, pad[5], s, err))) != GDR_OK)
                return st;
        }
        if ((st = from_cuda(gdr::varlen_unpack(out, 1, m, s))) != GDR_OK) return st;
        t_last_variant = path_name(path);
        return GDR_OK;
    }
    const gdr::VarlenMap m{cu, nullptr, nullptr, d.B, total, d.T, d.C, (int64_t)d.B * d.T};
    if ((st = from_cuda(gdr::varlen_pack(in, 5, m, s))) != GDR_OK) return st;
    if ((st = gdr_forward(p, base + ws.pad[0], base + ws.pad[1], base + ws.pad[2],
                          reinterpret_cast<const float*>(base + ws.pad[3]), base + ws.pad[4], h0, base + ws.pad[5],
                          h_final, base + ws.inner, ws.inner_bytes, stream)) != GDR_OK)
        return st;
    if (total > 0 && (st = from_cuda(gdr::varlen_unpack(out, 1, m, s))) != GDR_OK) return st;
    return GDR_OK;
}

gdr_status gdr_varlen_backward(const gdr_problem* p_in, const int32_t* cu_seqlens, const int32_t* cu_seqlens_device,
                               int64_t total, const void* q, const void* k, const void* v, const float* g,
                               const void* beta, const float* h0, const void* d_o, const float* dh_final, void* dq,
                               void* dk, void* dv, float* dg, void* dbeta, float* dh0, void* workspace,
                               size_t workspace_bytes, void* stream) {
    if (!p_in) return GDR_ERR_NULL;
    const gdr_problem p1 = varlen_problem(p_in);
    const gdr_problem* p = &p1;
    gdr::Dims d;
    gdr_status st = check_problem(p, &d);
    if (st != GDR_OK) return st;
    if (total > 0 && (st = check_ptrs({q, k, v, g, beta, d_o, dq, dk, dv, dg, dbeta}, {h0, dh_final, dh0})) != GDR_OK)
        return st;
    if (total <= 0 &&
        (st = check_ptrs({}, {q, k, v, g, beta, d_o, dq, dk, dv, dg, dbeta, h0, dh_final, dh0})) != GDR_OK)
        return st;
    cudaStream_t s = (cudaStream_t)stream;
    VarlenWorkspace ws;
    const int* cu = nullptr;
    if ((st = varlen_setup(p, &d, true, cu_seqlens, cu_seqlens_device, total, workspace, workspace_bytes, s, &ws,
                           &cu)) != GDR_OK)
        return st;
    BwdPath path;
    if ((st = pick_backward(p, d, &path)) != GDR_OK) return st;
    char* base = static_cast<char*>(workspace);
    int64_t rb[11];
    varlen_rows(d, true, rb);
    const void* packed_in[6] = {q, k, v, g, beta, d_o};
    void* packed_out[5] = {dq, dk, dv, dg, dbeta};
    auto pad = [&](int i) { return static_cast<void*>(base + ws.pad[i]); };
    gdr::RowCopy in[6], out[5];
    for (int i = 0; i < 6; ++i) in[i] = {packed_in[i], pad(i), rb[i]};
    for (int i = 0; i < 5; ++i) out[i] = {pad(6 + i), packed_out[i], rb[6 + i]};
    int64_t chunks = 0;   // the chunk-packed row's chunks, from the host lengths
    for (int64_t i = 0; i < d.B; ++i) chunks += ((int64_t)cu_seqlens[i + 1] - cu_seqlens[i] + d.C - 1) / d.C;
    if (path != BwdPath::Simt && chunk_packed_fits(d) && chunks > 0) {
        int* co = reinterpret_cast<int*>(base + ws.co);
        int* cs = reinterpret_cast<int*>(base + ws.cs);
        const gdr::VarlenMap m{cu, co, cs, d.B, total, 0, d.C, chunks * d.C};
        const gdr::Dims d1 = chunk_packed(d, chunks);
        if ((st = from_cuda(gdr::varlen_plan(cu, d.B, total, d.C, (int)chunks, co, cs, s))) != GDR_OK) return st;
        if ((st = from_cuda(gdr::varlen_pack(in, 6, m, s))) != GDR_OK) return st;
        if ((st = run_backward(d1, path, 1, base + ws.inner, plan_backward(d1, path, 1), pad(0), pad(1), pad(2),
                               static_cast<const float*>(pad(3)), pad(4), h0, pad(5), dh_final, pad(6), pad(7),
                               pad(8), static_cast<float*>(pad(9)), pad(10), dh0, s, co, d.B)) != GDR_OK)
            return st;
        return from_cuda(gdr::varlen_unpack(out, 5, m, s));
    }
    const gdr::VarlenMap m{cu, nullptr, nullptr, d.B, total, d.T, d.C, (int64_t)d.B * d.T};
    if ((st = from_cuda(gdr::varlen_pack(in, 6, m, s))) != GDR_OK) return st;
    if ((st = gdr_backward(p, pad(0), pad(1), pad(2), static_cast<const float*>(pad(3)), pad(4), h0, pad(5), dh_final,
                           pad(6), pad(7), pad(8), static_cast<float*>(pad(9)), pad(10), dh0, base + ws.inner,
                           ws.inner_bytes, stream)) != GDR_OK)
        return st;
    if (total > 0 && (st = from_cuda(gdr::varlen_unpack(out, 5, m, s))) != GDR_OK) return st;
    return GDR_OK;
}

const char* gdr_status_string(gdr_status s) {
    switch (s) {
        case GDR_OK: return "ok";
        case GDR_ERR_NULL: return "a required pointer is NULL";
        case GDR_ERR_SHAPE: return "unsupported or inconsistent sizes";
        case GDR_ERR_DTYPE: return "unknown io dtype or gate kind";
        case GDR_ERR_ALIGN: return "a pointer is not 16-byte aligned (workspace: 256-byte)";
        case GDR_ERR_WORKSPACE: return "workspace missing or too small";
        case GDR_ERR_CUDA: return "a CUDA call or kernel launch failed";
        case GDR_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel gave up";
        case GDR_ERR_UNSUPPORTED: return "the requested variant cannot run this problem";
        case GDR_ERR_ARG: return "invalid argument";
    }
    return "unknown status";
}

gdr_status gdr_get_device_status(void* stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDR_ERR_CUDA;
    unsigned int code = 0;
    if (gdr::read_and_clear_device_error(&code) != cudaSuccess) return GDR_ERR_CUDA;
    return code == 0 ? GDR_OK : GDR_ERR_DEVICE_TIMEOUT;
}

const char* gdr_last_variant(void) { return t_last_variant.c_str(); }

int gdr_version(void) { return 100; }

}  // extern "C"
