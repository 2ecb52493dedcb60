// Internal interface between the C ABI (gdr_api.cpp) and the kernel files.
// Not installed; the public interface is include/gdr.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdr.h"

namespace gdr {

// Validated problem sizes, as every launcher receives them.
struct Dims {
    int B, T, H, K, V, C, NT;
    int Hk, G;      // q/k heads and the group size H / Hk: value head h reads q and k of head h / G
    int per_k;      // 1: per-key-dim gate (g is [B,T,H,K]); 0: scalar gate
    int bf16;       // 1: io tensors are bf16 (the tensor-core kernels take these)
    int f16;        // 1: io tensors are fp16 (CUDA-core kernels only); bf16 = f16 = 0: fp32
    float scale;    // resolved output scale
};

// ---- fp32 CUDA-core kernels (simt_kernels.cu): every K, V in {64,128}, C in {32,64}, both dtypes.
cudaError_t simt_prepare(const Dims& d, const void* k, const void* v, const float* g, const void* beta,
                         void* w, void* u, float* g_cum, cudaStream_t s);
cudaError_t simt_scan(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum,
                      const float* h0, void* h_ckpt, void* v_new, float* h_final, cudaStream_t s);
cudaError_t simt_output(const Dims& d, const void* q, const void* k, const void* v_new, const void* h_ckpt,
                        const float* g_cum, void* o, cudaStream_t s);

// ---- tensor-core kernels (bf16 io; the forward's also fp16 io, with d.f16)
// with q and P non-NULL (scalar gate, C = 64) it also writes P = tril_0(q k^T * exp(G_i - G_j))
// per chunk as [B, NT, H, C, C] bf16; with tinv non-NULL, (I + A)^{-1} per chunk, [B, NT, H, C, C] bf16
// pdl: launch as the programmatic dependent of the stream's previous kernel (see gdr_api.cpp's overlapped
// forward): it may start once every CTA of that kernel has signalled, and must read nothing it writes.
// tc_scores: S = k k^T and P = q k^T on tcgen05 (K = V = 128 with P, one q/k head per value head, no
// inverse; other calls ignore it).  The overlapped forward asks for it: beside the scan the forward
// measured faster with it, while a prepare on its own is faster on mma.sync.
cudaError_t mma_prepare(const Dims& d, const void* k, const void* v, const float* g, const void* beta, void* w,
                        void* u, float* g_cum, cudaStream_t s, unsigned int* err, const void* q = nullptr,
                        void* P = nullptr, void* tinv = nullptr, bool pdl = false, bool tc_scores = false);
// mma_prepare for fp16 io (d.f16): every shape and gate of the bf16 forms, no inverse.
cudaError_t mma_prepare_f16(const Dims& d, const void* k, const void* v, const float* g, const void* beta, void* w,
                            void* u, float* g_cum, cudaStream_t s, unsigned int* err, const void* q, void* P,
                            void* tinv, bool pdl, bool tc_scores);
// The prepare with P (scalar gate, C = 64) on the chunk-packed row d (B = 1) of packed variable-length
// sequences, reading q, k, v, g, beta in place from the caller's packed tensors of `total` tokens: chunk c of
// the row is chunk c - co[s] of sequence s = cs[c] (cu, co, cs as varlen_plan makes them).  w, u, g_cum and
// P fill the row as mma_prepare's would for the chunk-packed copy of the inputs.
cudaError_t mma_prepare_packed(const Dims& d, const void* q, const void* k, const void* v, const float* g,
                               const void* beta, void* w, void* u, float* g_cum, void* P, const int* cu,
                               const int* co, const int* cs, int nseq, int total, cudaStream_t s, unsigned int* err);
// the scan's recurrence runs on mma.sync (register-resident), see scan_mma.cu
// co (packed variable-length sequences, else NULL): d has B = 1 and whole chunks; sequence z of nseq runs
// the chunks co[z] .. co[z+1]-1 from h0[z] to h_final[z] (one CTA column per sequence)
cudaError_t mma_scan(const Dims& d, const void* k, const void* w, const void* u, const float* g_cum, const float* h0,
                     void* h_ckpt, void* v_new, float* h_final, cudaStream_t s, unsigned int* err,
                     const int* co = nullptr, int nseq = 0);
// the segment-parallel scan: on the segment view (B S sequences of T / S tokens), every segment's affine
// map h_end = M h_start + Z (M [B S, H, K, K], Z [B S, H, K, V], fp32), then the serial stitch of the maps
// into the segments' starting states h_start [B S, H, K, V] and h_final [B, H, K, V] (NULL: not written).
// reverse: the backward's stitch, end[S-1] = h0 (dh_final), end[s-1] = M_s^T end[s] + Z_s, into h_start
// (the segment ends) and h_final (dh0).
cudaError_t mma_scan_transfer(const Dims& d_view, const void* k, const void* w, const void* u, const float* g_cum,
                              float* m_out, float* z_out, cudaStream_t s, unsigned int* err);
cudaError_t segment_combine(const Dims& d, int S, const float* M, const float* Z, const float* h0, float* h_start,
                            float* h_final, cudaStream_t s, bool reverse = false);
cudaError_t tc_output(const Dims& d, const void* q, const void* k, const void* v_new, const void* h_ckpt,
                      const float* g_cum, void* o, cudaStream_t s, unsigned int* err);

// scan and output fused (scalar gate, bf16), see fused_mma.cu
// P: the prepare's [B, NT, H, C, C] tiles (C = 64), or NULL to compute q k^T in the kernel
cudaError_t mma_scan_output(const Dims& d, const void* q, const void* k, const void* w, const void* u,
                            const float* g_cum, const void* P, const float* h0, void* o, float* h_final,
                            cudaStream_t s, unsigned int* err, const int* co = nullptr, int nseq = 0,
                            const int* pcu = nullptr, int Tin = 0);
// pcu, Tin (with co and P): q, k and o are the caller's packed tensors of Tin tokens, sequence z starting at
// packed row pcu[z]; w, u, g_cum and P are the chunk-packed row's (see fused_mma.cu)

// The same scan and output on the tcgen05 tensor cores, one CTA per (batch, head) (fused_tc.cu): bf16 io,
// K = V = 128, C = 64 (any T, grouped value heads), and P from the prepare.  With a per-key-dim gate q and k
// are the gated operands qg and kg and P comes from tc_gated_operands.
bool tc_scan_output_supported(const Dims& d);
// Per (batch, value head, chunk) with a per-key-dim gate (bf16, K = V = 128, C = 64): P = tril_0(Q~) as the
// prepare with P writes it for a scalar gate, qg = q exp(G) and kg = k exp(G_last - G) [B, T, H, K] bf16
// (tc_output.cu, the output kernel's first half).
cudaError_t tc_gated_operands(const Dims& d, const void* q, const void* k, const float* g_cum, void* P, void* kg,
                              void* qg, cudaStream_t s, unsigned int* err);
// pdl: launch as the programmatic dependent of the stream's previous kernel (the prepare), which must
// trigger early (griddepcontrol.launch_dependents); the scan's setup then runs under its tail.
cudaError_t tc_scan_output(const Dims& d, const void* q, const void* k, const void* w, const void* u,
                           const float* g_cum, const void* P, const float* h0, void* o, float* h_final,
                           cudaStream_t s, unsigned int* err, bool pdl = false);

// ---- backward stages on the CUDA cores (simt_backward.cu): every shape and io dtype;
// intermediates fp32, see include/gdr.h for each stage's definition
cudaError_t simt_bwd_dv_local(const Dims& d, const void* q, const void* k, const float* g_cum, const void* d_o,
                              float* dv_loc, cudaStream_t s);
cudaError_t simt_bwd_scan_dh(const Dims& d, const void* q, const void* k, const void* w, const float* g_cum,
                             const void* d_o, const float* dv_loc, const float* dh_final, float* dh_ckpt,
                             float* dv_new, float* dh0, cudaStream_t s);
// inter16: dh_ckpt and dv_new (du) are in the io dtype (from the tensor-core reverse scan), else fp32.
// only: NULL, or per-chunk flags [B][NT][H]; a chunk whose flag is 0 is skipped (the tensor-core
// per-chunk stage for a per-key gate flags the chunks it leaves to these two).
cudaError_t simt_bwd_dqkwg(const Dims& d, const void* q, const void* k, const void* v_new, const float* g_cum,
                           const void* h_ckpt, const void* dh_ckpt, const void* d_o, const void* dv_new,
                           void* dq, float* dk_part, float* dw, float* dG_part, cudaStream_t s, bool inter16 = false,
                           const int* only = nullptr);
cudaError_t simt_bwd_wy(const Dims& d, const void* k, const void* v, const void* beta, const float* g_cum,
                        const float* dw, const void* du, const float* dk_part, const float* dG_part, void* dk,
                        void* dv, void* dbeta, float* dg, cudaStream_t s, bool inter16 = false,
                        const int* only = nullptr);

// grouped value heads: dq, dk [B,T,Hk,K] = sums over each group of dq_v, dk_v [B,T,H,K] (io dtype)
cudaError_t group_sum_heads(const Dims& d, const void* dq_v, const void* dk_v, void* dq, void* dk, cudaStream_t s);

// ---- backward on the tensor cores (bf16 io, scalar gate, C = 64)
// reverse scan: dv' = scale P^T do + (k gamma) dh, dh = e^(G_L) dh + scale (q e^G)^T do - w^T dv';
// co, nseq: packed variable-length sequences as for mma_scan (dh_final[z] back to dh0[z])
// dh_ckpt [B,NT,H,K,V] and dv_new [B,T,H,V] bf16 (bwd_scan_mma.cu)
cudaError_t mma_bwd_scan(const Dims& d, const void* q, const void* k, const void* w, const float* g_cum, const void* P,
                         const void* d_o, const float* dh_final, void* dh_ckpt, void* dv_new, float* dh0,
                         cudaStream_t s, unsigned int* err, const int* co = nullptr, int nseq = 0);
// the reverse scan with the local term precomputed: dv' = dv_loc + kg dh; dv_loc [B,T,H,V] bf16;
// either gate, C = 32 or 64 (bwd_scan_mma.cu)
cudaError_t mma_bwd_scan_dl(const Dims& d, const void* q, const void* k, const void* w, const float* g_cum,
                            const void* dv_loc, const void* d_o, const float* dh_final, void* dh_ckpt, void* dv_new,
                            float* dh0, cudaStream_t s, unsigned int* err, const int* co = nullptr, int nseq = 0);
// dv_loc = scale tril_0(Q~)^T do per chunk, bf16 (bwd_dvloc_mma.cu)
cudaError_t mma_bwd_dv_local(const Dims& d, const void* q, const void* k, const float* g_cum, const void* d_o,
                             void* dv_loc, cudaStream_t s);
// the per-chunk stage (dq, dk, dv, dbeta, dg) from the chunk's tiles and T = (I + A)^{-1} (bwd_chunk_mma.cu)
cudaError_t mma_bwd_chunk(const Dims& d, const void* q, const void* k, const void* v, const void* beta,
                          const float* g_cum, const void* w, const void* u, const void* tinv, const void* v_new,
                          const void* h_ckpt, const void* d_o, const void* dv_new, const void* dh_ckpt, void* dq,
                          void* dk, void* dv, void* dbeta, float* dg, cudaStream_t s);
// The same stage at C = 64 fed by TMA from swizzled tiles, persistent with the next chunk's tiles prefetched
// (bwd_chunk_tma.cu); err: the device error word for its bounded barrier waits.
cudaError_t mma_bwd_chunk_tma(const Dims& d, const void* q, const void* k, const void* v, const void* beta,
                              const float* g_cum, const void* w, const void* u, const void* tinv, const void* v_new,
                              const void* h_ckpt, const void* d_o, const void* dv_new, const void* dh_ckpt, void* dq,
                              void* dk, void* dv, void* dbeta, float* dg, cudaStream_t s, unsigned int* err);
// The same stage for a per-key-dim gate (bf16 io, C = 32 or 64).  exact_flags [B][NT][H]: set to 1 for a
// chunk whose gate moves more than the kernel's exponent bound from the chunk's middle row (nothing of that
// chunk is written; simt_bwd_dqkwg and simt_bwd_wy with only = exact_flags complete it), else 0.
cudaError_t mma_bwd_chunk_kda(const Dims& d, const void* q, const void* k, const void* v, const void* beta,
                              const float* g_cum, const void* w, const void* u, const void* tinv, const void* v_new,
                              const void* h_ckpt, const void* d_o, const void* dv_new, const void* dh_ckpt, void* dq,
                              void* dk, void* dv, void* dbeta, float* dg, int* exact_flags, cudaStream_t s);

// ---- packed variable-length sequences (varlen.cu)
// One tensor of token rows, row_bytes bytes a token: packed [total, row] <-> a working layout, either
//   padded:       [n, T, row], sequence s on the rows s T .. s T + len_s - 1 (co == NULL), or
//   chunk-packed: [NT C, row], sequence s on the rows C co[s] .. C co[s] + len_s - 1 (co, cs given);
// rows of the working layout past a sequence's length are zero after a pack and not read by an unpack.
struct RowCopy {
    const void* src;
    void* dst;
    int64_t row_bytes;
};
constexpr int kMaxCopies = 8;
struct VarlenMap {
    const int* cu;     // device int32 [n + 1]
    const int* co;     // chunk-packed: device int32 [n + 1] chunk offsets; NULL: padded
    const int* cs;     // chunk-packed: device int32 [NT], the sequence owning each chunk
    int n;
    int64_t total;     // packed rows
    int T;             // padded: tokens per row
    int C;             // chunk-packed: tokens per chunk
    int64_t rows;      // rows of the working layout: n T, or NT C
};
// pack: copies[i].src packed, .dst working layout; unpack: .src working layout, .dst packed.  The grid is
// capped at 8 CTAs per SM.
cudaError_t varlen_pack(const RowCopy* copies, int count, const VarlenMap& m, cudaStream_t s);
cudaError_t varlen_unpack(const RowCopy* copies, int count, const VarlenMap& m, cudaStream_t s);
// co[s] = sum over r < s of ceil(len_r / C), clamped to NT (co[n] too), and cs[c] = s for c in
// [co[s], co[s+1]): the chunk-packed layout of the sequences in cu.  One CTA.
cudaError_t varlen_plan(const int* cu, int n, int64_t total, int C, int NT, int* co, int* cs, cudaStream_t s);

// ---- device error word (device_status.cu)
// Bounded waits in kernels write a nonzero code here instead of trapping.
cudaError_t read_and_clear_device_error(unsigned int* code);
// Address of the error word on the current device (to pass to kernels).
cudaError_t device_error_ptr(unsigned int** ptr);
constexpr unsigned int kDeviceErrTimeout = 1u;

}  // namespace gdr
