/*
 * gdr.h -- C ABI of libgdr, the chunked gated-delta-rule forward on one GPU.
 *
 * The gated delta rule keeps, per (batch b, head h), a K x V state S and for
 * every token t applies
 *     S~ = D_t S_{t-1},  delta_t = beta_t (v_t - S~^T k_t),  S_t = S~ + k_t delta_t^T,
 *     o_t = scale * S_t^T q_t,
 * with D_t = exp(g_t) (scalar gate, GDN) or diag(exp(g_t[0..K))) (per-key-dim gate,
 * KDA).  The library computes this in chunks of C tokens in three stages:
 *
 *   gdr_prepare_wy   the fused WY prepare of "Reuse P as beta tiles in gated
 *                    deltanet fused prepare" (TileOPs-Metax PR #60): the gated
 *                    strictly-lower A, its inverse (I + A)^{-1}, w and u;
 *   gdr_scan_h       the serial inter-chunk state scan of
 *                    "kernel_fun/kda/_kernels/bwd_scan.py" (module docstring:
 *                    hck[c] = h before the update, v' = u - w h, h = decay*h + kg^T v');
 *   gdr_chunk_output the chunk output that the same page says the forward
 *                    assembled in its epilogue warps (module docstring, "the
 *                    warps that assembled o in the forward");
 *   gdr_forward      all three, (q, k, v, g, beta, h0) -> (o, h_final).
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *   never allocates device memory; gdr_forward takes its scratch from a caller
 *   workspace.  Every call is asynchronous on `stream` (a cudaStream_t passed
 *   as void*; NULL is the legacy default stream) and returns as soon as the
 *   launches are queued.
 * - Layouts are contiguous, head dim last ("head-last", as the re-scan page's
 *   host wrapper takes them): q, k [B,T,H,K]; w [B,T,HV,K]; v, u, v_new, o
 *   [B,T,HV,V]; g, g_cum [B,T,HV] (scalar gate) or [B,T,HV,K] (per-key-dim
 *   gate), always fp32; beta [B,T,HV]; h0, h_final [B,HV,K,V] fp32; h_ckpt
 *   [B,NT,HV,K,V] with NT = ceil(T/C).  Every per-head tensor below that is not
 *   q or k is indexed by the value head.
 * - Grouped value heads: HV = G H value heads share the H q/k heads, value
 *   head hv reading the q and k of head hv / G (the scan page indexes its
 *   tensors by value head this way).  HV = H (or 0) is the ungrouped case.
 * - "io" tensors (q, k, v, beta, w, u, v_new, o, h_ckpt) have the problem's
 *   io_dtype: fp32, bf16 or fp16.  g, g_cum, h0 and h_final are always fp32.
 * - g is the natural-log per-token decay (<= 0 for a decaying state); the
 *   library takes its chunk-local inclusive cumsum itself.
 * - Argument errors are detected before anything is launched and returned as a
 *   status code; nothing is written in that case.  A launch failure returns
 *   GDR_ERR_CUDA.  Waits inside kernels are bounded: if one gives up, the kernel
 *   records GDR_ERR_DEVICE_TIMEOUT in a device error word and exits; read it with
 *   gdr_get_device_status().
 * - Supported: K, V in {64, 128}; chunk C in {32, 64}; B, H, T >= 1, any T;
 *   every pointer 16-byte aligned.
 * - A T that is not a multiple of C ends in a partial chunk.  It is computed as
 *   if the sequence went on to a multiple of C with tokens of beta = 0, g = 0
 *   and zero q, k, v: each such token leaves the state as it is (S_t = S_{t-1}),
 *   so every result equals that of the unpadded delta rule.  Nothing past T is
 *   read or written; the partial chunk has its checkpoint (the state before its
 *   first token) like any other chunk.
 * - Thread safety: calls may be made from several host threads.  The only
 *   per-call host state is the name of the kernel variant that ran, which is
 *   kept per host thread (gdr_last_variant).
 */
#ifndef GDR_H
#define GDR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDR_API __attribute__((visibility("default")))
#else
#define GDR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdr_status {
    GDR_OK = 0,
    GDR_ERR_NULL = 1,            /* a required pointer is NULL */
    GDR_ERR_SHAPE = 2,           /* a size is <= 0, or K/V/chunk unsupported */
    GDR_ERR_DTYPE = 3,           /* io_dtype or gate kind not known */
    GDR_ERR_ALIGN = 4,           /* a pointer is not 16-byte aligned */
    GDR_ERR_WORKSPACE = 5,       /* workspace NULL or smaller than gdr_forward_workspace_bytes */
    GDR_ERR_CUDA = 6,            /* a CUDA call or launch failed */
    GDR_ERR_DEVICE_TIMEOUT = 7,  /* a bounded in-kernel wait gave up (read via gdr_get_device_status) */
    GDR_ERR_UNSUPPORTED = 8,     /* a variant hint that cannot run this problem */
    GDR_ERR_ARG = 9              /* another invalid argument (e.g. a NaN scale) */
} gdr_status;

/* fp16 io runs the forward's tensor-core kernels as bf16 does (q, k, v, beta, o and every
 * intermediate fp16, the state fp32), with three exceptions: FUSED_TC takes a scalar gate only, no
 * segmented scan runs (segments > 1 is GDR_ERR_UNSUPPORTED), and the backward runs the CUDA-core
 * kernels.  A per-key-dim gate keeps its gated copies of k and q for the scores in bf16 inside the
 * kernels, because their factors exceed fp16's range. */
typedef enum gdr_dtype { GDR_F32 = 0, GDR_BF16 = 1, GDR_F16 = 2 } gdr_dtype;

typedef enum gdr_gate {
    GDR_GATE_SCALAR = 0,  /* GDN: g [B,T,H] */
    GDR_GATE_PER_K = 1    /* KDA: g [B,T,H,K] */
} gdr_gate;

/* Which kernels to run.  AUTO picks the fastest measured variant that supports
 * the problem: for bf16 io with a scalar gate and 64-token chunks FUSED_TC when
 * K = V = 128 and either B * HV * V / 32 > 152 (the warp-level fused kernel's grid
 * would need more than one wave of the GPU's 152 SMs) or B = 1 with at least 128
 * chunks and no segmented scan (one long sequence, which FUSED_TC runs in pieces
 * whose scans overlap the next piece's prepare), else FUSED; with a per-key-dim
 * gate FUSED_TC when K = V = 128, C = 64 and no segmented scan applies; TENSOR for
 * other bf16 problems; SIMT for fp32 io.  fp16 io follows the bf16 rules (its
 * FUSED_TC taking a scalar gate only, see gdr_dtype).  The single-stage entry
 * points run their tensor-core kernel for AUTO, TENSOR, FUSED and FUSED_TC on
 * bf16 and fp16 io. */
typedef enum gdr_variant {
    GDR_VARIANT_AUTO = 0,
    GDR_VARIANT_SIMT = 1,     /* fp32 CUDA-core arithmetic throughout (exact-fp32 path) */
    GDR_VARIANT_TENSOR = 2,   /* staged kernels on the tensor cores (bf16 or fp16 io) */
    GDR_VARIANT_FUSED = 3,    /* WY prepare, then scan and output fused, warp-level MMA, one CTA per
                                 (batch, head, 32 value columns) (bf16 or fp16 io, scalar gate) */
    GDR_VARIANT_FUSED_TC = 4  /* the same with scan and output on the tcgen05 tensor cores, one CTA per
                                 (batch, head) (bf16 io, K = V = 128, chunk 64; a per-key-dim gate
                                 adds the gdr_gated_operands kernel; fp16 io with a scalar gate);
                                 packed sequences (gdr_varlen_*) run FUSED for it, TENSOR with a
                                 per-key-dim gate */
} gdr_variant;

typedef struct gdr_problem {
    int64_t B, T, H, K, V;
    int64_t chunk;      /* C: tokens per chunk */
    int32_t io_dtype;   /* gdr_dtype */
    int32_t gate;       /* gdr_gate */
    float scale;        /* output scale; <= 0 selects 1/sqrt(K) */
    int32_t variant;    /* gdr_variant */
    int64_t HV;         /* value heads, a multiple of H; 0 means HV = H (see below) */
    int32_t segments;   /* gdr_forward on the tensor cores: scan each sequence as this many segments
                           in parallel (see gdr_scan_transfer); 0 = chosen from the problem, 1 = off;
                           fp16 io scans whole (0 means 1; > 1 is GDR_ERR_UNSUPPORTED) */
} gdr_problem;

/*
 * Stage 1: WY prepare ("Reuse P as beta tiles in gated deltanet fused prepare":
 * A_g, the Neumann/substitution inverse, w = A_g^{-1} k_beta, u = A_g^{-1} v_beta).
 * Per (b, h, chunk), with G the chunk-local inclusive cumsum of g:
 *     A_ij  = beta_i sum_d k_id k_jd exp(G_id - G_jd)   for i > j, else 0
 *     w     = (I + A)^{-1} (k * beta * exp(G))          [C,K]
 *     u     = (I + A)^{-1} (v * beta)                   [C,V]
 * Inputs:  k [B,T,H,K] io, v [B,T,H,V] io, g fp32, beta [B,T,H] io.
 * Outputs: w [B,T,H,K] io, u [B,T,H,V] io, g_cum (same shape as g) fp32 = G.
 * The prepare page builds k_beta without exp(G); the form above is the one
 * under which v' = u - w h is the recurrence's delta, and it is the one used.
 */
GDR_API gdr_status gdr_prepare_wy(const gdr_problem* p, const void* k, const void* v, const float* g,
                          const void* beta, void* w, void* u, float* g_cum, void* stream);

/*
 * Stage 2: the serial state scan ("kernel_fun/kda/_kernels/bwd_scan.py", module
 * docstring).  Per (b, h), h = h0 (zero if h0 == NULL), then for c = 0 .. NT-1:
 *     h_ckpt[c] = h                          (rounded to io dtype)
 *     v'_c      = u_c - w_c h                -> v_new (io dtype)
 *     h         = exp(G_last) * h + (k * exp(G_last - G))^T v'_c
 * where G = g_cum of chunk c and G_last its last row (a K-vector for KDA that
 * scales the rows of h).  h is carried in fp32; h_final = h after the last chunk.
 * Inputs:  k, w [B,T,H,K] io; u [B,T,H,V] io; g_cum fp32; h0 [B,H,K,V] fp32 or NULL.
 * Outputs: h_ckpt [B,NT,H,K,V] io or NULL (not written); v_new [B,T,H,V] io;
 *          h_final [B,H,K,V] fp32 or NULL (not written).
 */
GDR_API gdr_status gdr_scan_h(const gdr_problem* p, const void* k, const void* w, const void* u,
                      const float* g_cum, const float* h0, void* h_ckpt, void* v_new,
                      float* h_final, void* stream);

/*
 * The segment-parallel scan, for few sequences and heads at long T.  One chunk of the
 * scan above is affine in h: h <- A_c h + B_c, A_c = diag(exp(G_last)) - kg^T w [K,K],
 * B_c = kg^T u [K,V].  So NT / S consecutive chunks are one map h_end = M h_start + Z,
 * and the S segments of a sequence can be scanned at once once their starting states
 * are known.  (The pages scan serially; this is the algebra of the recurrence they give.)
 *
 * gdr_scan_transfer: for every segment s of every (b, h), M [B,S,H,K,K] = the product of
 * its A_c (later chunks on the left) and Z [B,S,H,K,V] = the state the segment leaves from
 * a zero state, both fp32.  Inputs as gdr_scan_h; bf16 io, whole chunks (T % C == 0) and
 * NT % segments == 0 (GDR_ERR_ARG otherwise); the variant SIMT is GDR_ERR_UNSUPPORTED.
 *
 * gdr_scan_combine: h_start[b,0] = h0 (zero if NULL), h_start[b,s+1] = M_s h_start[b,s] + Z_s,
 * h_final = M_{S-1} h_start[b,S-1] + Z_{S-1}; h_start [B,S,H,K,V] fp32, h_final [B,H,K,V] fp32
 * or NULL.  fp32 on the CUDA cores; any io dtype (the maps are fp32).
 *
 * With h_start in hand, gdr_scan_h or gdr_scan_output run every segment at once on the
 * problem with B S sequences of T / S tokens and h0 = h_start: every [B,T,...] and
 * [B,NT,...] tensor has the same memory layout in that view.  gdr_forward does all of
 * this itself when gdr_forward_segments(p) > 1.
 */
GDR_API gdr_status gdr_scan_transfer(const gdr_problem* p, const void* k, const void* w, const void* u,
                                     const float* g_cum, int32_t segments, float* M, float* Z, void* stream);
GDR_API gdr_status gdr_scan_combine(const gdr_problem* p, int32_t segments, const float* M, const float* Z,
                                    const float* h0, float* h_start, float* h_final, void* stream);

/* The backward's stitch.  The reverse state scan (gdr_bwd_scan_dh and its tensor-core forms) is affine
 * the other way: a segment maps the state gradient at its end to the one at its start by M^T, M its
 * forward map from gdr_scan_transfer, plus Zb, the gradient it leaves at its start from a zero gradient
 * at its end (the reverse scan's dh0 on the segment problem with dh_final = NULL).  From the last
 * segment: ends[b,S-1] = dh_final (zero if NULL), ends[b,s-1] = M_s^T ends[b,s] + Zb_s, and
 * dh0 = M_0^T ends[b,0] + Zb_0.  ends [B,S,H,K,V] fp32 (each segment's dh_final for the reverse scan on
 * the segment problem), dh0 [B,H,K,V] fp32 or NULL; fp32 on the CUDA cores.  gdr_backward does all
 * of this itself when gdr_forward_segments(p) > 1. */
GDR_API gdr_status gdr_scan_combine_reverse(const gdr_problem* p, int32_t segments, const float* M, const float* Zb,
                                            const float* dh_final, float* ends, float* dh0, void* stream);

/* The number of segments gdr_forward (and, on the tensor cores, gdr_backward) scans this problem in: p->segments when that is > 1 (it must
 * divide NT, with T % C == 0), 1 for p->segments == 1 and on the CUDA-core path, and for 0 a choice
 * from the problem: when B * HV * V / 32 (the serial scan's CTAs) is at most 76, the largest divisor
 * of NT whose segments keep at least 16 chunks and whose segmented grid fits 152 SMs.  0 for a
 * problem gdr_forward would reject. */
GDR_API int gdr_forward_segments(const gdr_problem* p);

/*
 * Stage 3: chunk output.  Per (b, h, chunk c), with G = g_cum of the chunk:
 *     o_c = scale * [ (q * exp(G)) h_ckpt[c] + tril_0(Q~) v'_c ],
 *     Q~_ij = sum_d q_id k_jd exp(G_id - G_jd)   (diagonal included)
 * Inputs:  q, k [B,T,H,K] io; v_new [B,T,H,V] io; h_ckpt [B,NT,H,K,V] io; g_cum fp32.
 * Output:  o [B,T,H,V] io.
 */
GDR_API gdr_status gdr_chunk_output(const gdr_problem* p, const void* q, const void* k, const void* v_new,
                            const void* h_ckpt, const float* g_cum, void* o, void* stream);

/*
 * Stages 2 and 3 fused, for a scalar gate and bf16 or fp16 io: the state scan of
 * gdr_scan_h and the chunk output of gdr_chunk_output in one pass, so v' and the
 * checkpoints never reach device memory.  Per (b, h): h = h0 (zero if NULL); for
 * each chunk c, v'_c = u_c - w_c h, o_c = scale [ (q exp(G)) h + tril_0(Q~) v'_c ],
 * h = exp(G_last) h + (k exp(G_last - G))^T v'_c.
 * Inputs:  q, k, w [B,T,H,K] io; u [B,T,H,V] io; g_cum [B,T,H] fp32 (the
 *          chunk-local cumsum, as gdr_prepare_wy writes it); P [B,NT,H,C,C] io
 *          as gdr_prepare_wyp writes it, or NULL to form it here (C = 64 for a
 *          non-NULL P); h0 [B,H,K,V] fp32 or NULL.
 * Outputs: o [B,T,H,V] io; h_final [B,H,K,V] fp32 or NULL (not written).
 * Returns GDR_ERR_UNSUPPORTED for fp32 io.  The kernel is the tcgen05 one for
 * variant FUSED_TC (K = V = 128, C = 64, P required) and for AUTO where
 * gdr_forward's AUTO would take it; the warp-level one otherwise.
 * Per-key-dim gate: variant FUSED_TC only, with q, k, P replaced by the qg, kg
 * and P that gdr_gated_operands writes (GDR_ERR_UNSUPPORTED otherwise).
 */
GDR_API gdr_status gdr_scan_output(const gdr_problem* p, const void* q, const void* k, const void* w, const void* u,
                                   const float* g_cum, const void* P, const float* h0, void* o, float* h_final,
                                   void* stream);

/*
 * gdr_prepare_wy plus, per chunk, the gated causal score matrix of the chunk
 * output, P = tril_0(Q~) with Q~_ij = sum_d q_id k_jd exp(G_i - G_j) (no scale),
 * so that gdr_scan_output need not form q k^T once per value slice.
 * Scalar gate, bf16 or fp16 io and chunk C = 64 only (GDR_ERR_UNSUPPORTED otherwise).
 * Extra input: q [B,T,H,K] io.  Extra output: P [B,NT,H,C,C] io, row i of
 * chunk c holding the scores of query token c*C+i against key tokens c*C+j.
 */
GDR_API gdr_status gdr_prepare_wyp(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                                   const void* beta, void* w, void* u, float* g_cum, void* P, void* stream);

/*
 * For a per-key-dim gate, the operands the tcgen05 scan+output kernel takes in
 * place of q, k (gdr_scan_output, variant FUSED_TC), per (b, value head, chunk)
 * with G = g_cum of the chunk (a K-vector per token) and G_last its last row:
 *     P  = tril_0(Q~),  Q~_ij = sum_d q_id k_jd exp(G_id - G_jd)   [C,C] (no scale)
 *     qg = q * exp(G),  kg = k * exp(G_last - G)                    [C,K]
 * so that o_c = scale [qg h_c + P v'_c] and h <- exp(G_last) * h + kg^T v'_c are
 * the chunk output and the scan of gdr_chunk_output and gdr_scan_h.  P follows
 * the output page's form ("kernel_fun/kda/_kernels/bwd_scan.py", module
 * docstring: the o assembly); a chunk whose gate spreads by more than 40 within
 * it is formed in fp32 instead of from gated bf16 copies.
 * Inputs:  q, k [B,T,H,K] bf16; g_cum [B,T,HV,K] fp32 (gdr_prepare_wy's).
 * Outputs: P [B,NT,HV,C,C] bf16; qg, kg [B,T,HV,K] bf16 (value heads).
 * bf16, per-key-dim gate, K = V = 128, C = 64 only (GDR_ERR_UNSUPPORTED otherwise).
 */
GDR_API gdr_status gdr_gated_operands(const gdr_problem* p, const void* q, const void* k, const float* g_cum, void* P,
                                      void* kg, void* qg, void* stream);

/*
 * Bytes of device workspace gdr_forward needs for this problem (0 when the
 * variant it would run keeps every intermediate on chip).  Returns 0 for a
 * problem that gdr_forward would reject.
 */
GDR_API size_t gdr_forward_workspace_bytes(const gdr_problem* p);

/*
 * The whole forward: (q, k, v, g, beta, h0) -> (o, h_final).
 * Inputs:  q, k [B,T,H,K] io; v [B,T,H,V] io; g fp32; beta [B,T,H] io;
 *          h0 [B,H,K,V] fp32 or NULL (zero initial state).
 * Outputs: o [B,T,H,V] io; h_final [B,H,K,V] fp32 or NULL (not written).
 * workspace: device memory of at least gdr_forward_workspace_bytes(p) bytes,
 *          256-byte aligned, owned by the caller, not read before written;
 *          may be NULL when that size is 0.
 */
GDR_API gdr_status gdr_forward(const gdr_problem* p, const void* q, const void* k, const void* v,
                       const float* g, const void* beta, const float* h0, void* o,
                       float* h_final, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The whole forward over HOST tensors, for callers whose inputs and outputs live in
 * host memory.  The method pages have no counterpart to this call; it is a
 * deployment aid that hides the host link behind the computation.
 *
 * The sequence runs in `pieces` token ranges of whole chunks (every sequence of the
 * batch alike).  While piece i computes on `stream` (gdr_forward on the piece, from
 * the fp32 state piece i-1 left), the inputs of piece i+1 travel to the device and
 * the output of piece i-1 back to the host, each on a stream the call creates and
 * releases itself.  The chunking and the state carried between pieces are those of
 * one gdr_forward over the whole sequence, so the results equal gdr_forward's for
 * the variant the pieces run (each piece is its own problem of T_piece tokens, on
 * which AUTO may choose another variant than on the whole).
 * Inputs:  q, k, v, g, beta, h0 as gdr_forward's, in host memory.  Page-locked
 *          memory (cudaHostAlloc, cudaHostRegister) lets the copies overlap the
 *          computation; pageable memory works, with the copies serialised.
 * Outputs: o, h_final as gdr_forward's, in host memory (h_final NULL: not written).
 * pieces:  0 selects 8; at most 64 and at most the chunk count are used.
 * scratch: device memory of at least gdr_forward_host_scratch_bytes(p, pieces)
 *          bytes, 256-byte aligned, owned by the caller: two pieces' inputs and
 *          outputs, the states and one piece's gdr_forward workspace.
 * Asynchronous like every call: everything it queues is ordered after the work
 * already on `stream`, and the results are in host memory once `stream` has
 * completed (cudaStreamSynchronize).  The host buffers must stay valid until then.
 * Returns GDR_ERR_WORKSPACE for a missing or short scratch, GDR_ERR_ARG for
 * pieces < 0, and gdr_forward's codes for the problem.
 */
GDR_API size_t gdr_forward_host_scratch_bytes(const gdr_problem* p, int32_t pieces);
GDR_API gdr_status gdr_forward_host(const gdr_problem* p, const void* q, const void* k, const void* v,
                                   const float* g, const void* beta, const float* h0, void* o, float* h_final,
                                   int32_t pieces, void* scratch, size_t scratch_bytes, void* stream);

/*
 * gdr_forward without a workspace argument, for callers that cannot allocate
 * device memory themselves (for example a plugin whose host framework owns all
 * device memory, or a latency-critical loop that must not call cudaMalloc).
 * The method pages have no counterpart to this call; it is a deployment aid.
 *
 * It runs the staged forward (variant AUTO runs the tensor-core stages for
 * bf16 and fp16 io and the CUDA-core stages for fp32 io, as gdr_forward's AUTO
 * does with the fused path left out; SIMT and TENSOR are honoured; FUSED and
 * FUSED_TC are not offered here and return GDR_ERR_UNSUPPORTED -- call gdr_forward
 * for them) and
 * takes the scratch from an array of GDR_STATIC_SCRATCH_BYTES compiled into the
 * library.  Arguments and outputs are those of gdr_forward.
 * - A problem whose gdr_forward_workspace_bytes exceeds GDR_STATIC_SCRATCH_BYTES
 *   is rejected with GDR_ERR_WORKSPACE; nothing is launched.
 * - Every GPU that loads this part of the library holds that array until the
 *   process exits.
 * - All calls on a device share the array: calls whose kernels may overlap on
 *   the GPU (e.g. on unordered streams) race on it.  Issue them in order.
 * - The array keeps the previous call's contents; nothing needs clearing,
 *   because the stages write every scratch byte before reading it.
 * - The first call on each device looks up the array's device address with
 *   that device current; make it before any stream capture starts.  The address
 *   is kept for the life of the device's context: after a cudaDeviceReset of a
 *   device, do not call this entry point on that device again.
 */
#define GDR_STATIC_SCRATCH_BYTES (64ull << 20)
GDR_API gdr_status gdr_forward_static_scratch(const gdr_problem* p, const void* q, const void* k, const void* v,
                                              const float* g, const void* beta, const float* h0, void* o,
                                              float* h_final, void* stream);

/*
 * ---------------------------------------------------------------- backward
 * The gradient of the forward above.  Given do = dL/do [B,T,H,V] (io dtype)
 * and dh_final = dL/dh_final [B,H,K,V] (fp32, or NULL for zero), it returns
 * dq, dk [B,T,H,K], dv [B,T,H,V] and dbeta [B,T,H] in the io dtype,
 * dg (the shape of g) and dh0 [B,H,K,V] in fp32.
 *
 * Steps:
 * - The forward prepare (gdr_prepare_wy) and the forward re-scan (gdr_scan_h)
 *   run again. They rebuild G, w, the checkpoints h_c and v', as the backward
 *   page's first stage does ("kernel_fun/kda/_kernels/bwd_scan.py", module
 *   docstring: the forward re-scan that feeds the gradient stages).
 * - Then come the four stages below, each the derivative of one line of the
 *   chunked forward. Rows i, j are tokens of one chunk; G_L is the chunk's
 *   last row; dh_next = dL/d(state after the chunk).
 *   L(X, Y)_i = sum_j X_ij Y_j e^(G_i - G_j) and
 *   R(X, Y)_j = sum_i X_ij Y_i e^(G_i - G_j), elementwise over the key dim.
 *
 * A partial last chunk is read as in the forward. The gate gradient of its
 * padding goes to token T - 1, whose G the padding repeats.
 *
 * Two sets of kernels compute these stages.
 * - On the CUDA cores in fp32 (entry points gdr_bwd_dv_local, gdr_bwd_scan_dh,
 *   gdr_bwd_dqkwg, gdr_bwd_wy; fp32 intermediates): every shape, both dtypes.
 *   Variant SIMT re-scans on the CUDA cores too.  For bf16 io, variants AUTO
 *   and TENSOR re-scan on the tensor cores, then run these stages whenever the
 *   tensor-core set below does not apply.
 * - On the tensor cores (gdr_bwd_prepare, gdr_bwd_scan_dh_p or, for C = 32,
 *   gdr_bwd_dv_local_tc and gdr_bwd_scan_dh_tc, then gdr_bwd_wy_dqkg; bf16
 *   intermediates): bf16 io with a scalar gate, which variants AUTO and TENSOR
 *   take.
 * - For a per-key-dim gate with bf16 io, AUTO and TENSOR run gdr_bwd_prepare,
 *   gdr_bwd_dv_local_tc, gdr_bwd_scan_dh_tc and gdr_bwd_wy_dqkg on the tensor
 *   cores.  The last leaves a chunk whose gate moves too far within it for the
 *   split-gate products to gdr_bwd_dqkwg and gdr_bwd_wy (argument only), which
 *   compute that chunk exactly in fp32.
 * The variant FUSED is not offered here (GDR_ERR_UNSUPPORTED).
 */

/* dv_loc = scale tril_0(Q~)^T do per chunk.  Inputs q, k, do io; g_cum fp32.
 * Output dv_loc [B,T,H,V] fp32. */
GDR_API gdr_status gdr_bwd_dv_local(const gdr_problem* p, const void* q, const void* k, const float* g_cum,
                                    const void* d_o, float* dv_loc, void* stream);

/* The reverse state scan.  dh = dh_final (zero if NULL), then for c = NT-1 .. 0:
 *     dh_ckpt[c] = dh                               (gradient of the state after chunk c)
 *     dv'_c      = dv_loc_c + (k exp(G_L - G)) dh   -> dv_new
 *     dh         = exp(G_L) dh + scale (q exp(G))^T do_c - w_c^T dv'_c
 * and dh0 = dh.  Inputs q, k, w, do io; g_cum, dv_loc, dh_final fp32.
 * Outputs dh_ckpt [B,NT,H,K,V], dv_new [B,T,H,V], dh0 [B,H,K,V], all fp32;
 * dh0 may be NULL (not written). */
GDR_API gdr_status gdr_bwd_scan_dh(const gdr_problem* p, const void* q, const void* k, const void* w,
                                   const float* g_cum, const void* d_o, const float* dv_loc,
                                   const float* dh_final, float* dh_ckpt, float* dv_new, float* dh0, void* stream);

/* only: NULL (every chunk), or flags [B,NT,H] int32 as gdr_bwd_wy_dqkg writes them: gdr_bwd_dqkwg and
 * gdr_bwd_wy then compute, and write, only the chunks whose flag is nonzero. */

/* Per chunk, with h = h_ckpt[c], dhn = dh_ckpt[c], dqg = scale do h^T,
 * dQ~ = scale tril_0(do v'^T), dkg = v' dhn^T, kg = k exp(G_L - G):
 *     dq      = dqg exp(G) + L(dQ~, k)                                 (io; final)
 *     dk_part = R(dQ~, q) + dkg exp(G_L - G)                           fp32
 *     dw      = -dv' h^T                                               fp32
 *     dG_part = dqg q exp(G) + q L(dQ~, k) - k R(dQ~, q) - dkg kg      fp32, the shape of g
 *               (+ sum_i dkg_i kg_i + exp(G_L) sum_v h dhn on the chunk's last token;
 *                a scalar gate sums over the key dim)
 * Inputs q, k, v_new, h_ckpt, do io; g_cum fp32; dh_ckpt, dv_new fp32 (see below). */
GDR_API gdr_status gdr_bwd_dqkwg(const gdr_problem* p, const void* q, const void* k, const void* v_new,
                                 const float* g_cum, const void* h_ckpt, const void* dh_ckpt, const void* d_o,
                                 const void* dv_new, void* dq, float* dk_part, float* dw, float* dG_part,
                                 const int* only, void* stream);

/* The WY backward, with (I + A)^{-1} rebuilt from k, beta, g_cum and du = dv_new:
 *     dkb = Tinv^T dw, dvb = Tinv^T du, dA = strict_lower(-Tinv^T (dw kb^T + du vb^T) Tinv^T),
 *     Y = beta_i dA_ij, M = A with beta = 1
 *     dk    = dk_part + beta exp(G) dkb + L(Y, k) + R(Y, k)             (io)
 *     dv    = beta dvb                                                  (io)
 *     dbeta = sum_d dkb k exp(G) + sum_v dvb v + sum_j dA_ij M_ij      (io)
 *     dg    = reverse cumsum over each chunk of dG_part + dkb kb + k L(Y, k) - k R(Y, k)   (fp32)
 * Inputs k, v, beta io; g_cum, dw, dk_part, dG_part fp32; dv_new fp32 (see below). */
GDR_API gdr_status gdr_bwd_wy(const gdr_problem* p, const void* k, const void* v, const void* beta,
                              const float* g_cum, const float* dw, const void* dv_new, const float* dk_part,
                              const float* dG_part, void* dk, void* dv, void* dbeta, float* dg, const int* only,
                              void* stream);

/* dh_ckpt and dv_new of gdr_bwd_dqkwg and gdr_bwd_wy are fp32 (as gdr_bwd_scan_dh writes them), or,
 * for bf16 io with a variant other than SIMT, bf16 (as gdr_bwd_scan_dh_tc and gdr_bwd_scan_dh_p
 * write them). */

/* The tensor-core stages (bf16 io; GDR_ERR_UNSUPPORTED otherwise). */

/* gdr_prepare_wyp plus T = (I + A)^{-1} of every chunk: tinv [B,NT,H,C,C] bf16, row i of chunk c
 * holding row i of T.  Other arguments as gdr_prepare_wyp; P may be NULL (not written), and must
 * be for C = 32 or a per-key-dim gate (q is then unused). */
GDR_API gdr_status gdr_bwd_prepare(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                                   const void* beta, void* w, void* u, float* g_cum, void* P, void* tinv,
                                   void* stream);

/* The reverse scan of gdr_bwd_scan_dh with dv_loc = scale P^T do formed inside from the prepare's P.
 * Inputs q, k, w, do bf16; g_cum fp32; P [B,NT,H,C,C] bf16; dh_final fp32 or NULL.
 * Outputs dh_ckpt [B,NT,H,K,V] bf16, dv_new [B,T,H,V] bf16, dh0 fp32 or NULL. */
GDR_API gdr_status gdr_bwd_scan_dh_p(const gdr_problem* p, const void* q, const void* k, const void* w,
                                     const float* g_cum, const void* P, const void* d_o, const float* dh_final,
                                     void* dh_ckpt, void* dv_new, float* dh0, void* stream);

/* gdr_bwd_dqkwg and gdr_bwd_wy in one pass per chunk (the pages' wy_dqkg), T read from tinv
 * instead of rebuilt; the WY term of dA is -(dkb w^T + dvb u^T), which equals
 * -Tinv^T (dw kb^T + du vb^T) Tinv^T because w = Tinv kb and u = Tinv vb.
 * A per-key-dim gate enters every C x C product through q exp(G - G_ref), k exp(G_ref - G) and
 * k exp(G - G_ref), G_ref the chunk's middle row; exact_flags [B,NT,H] int32 (required for that gate,
 * ignored for a scalar one) gets 1 for a chunk whose gate moves more than 40 from that row (nothing
 * of it written: gdr_bwd_dqkwg and gdr_bwd_wy with only = exact_flags do it), else 0.
 * Inputs q, k, v, beta, w, u, tinv, v_new, h_ckpt, do, dv_new, dh_ckpt bf16; g_cum fp32.
 * Outputs dq, dk, dv, dbeta bf16; dg fp32. */
GDR_API gdr_status gdr_bwd_wy_dqkg(const gdr_problem* p, const void* q, const void* k, const void* v,
                                   const void* beta, const float* g_cum, const void* w, const void* u,
                                   const void* tinv, const void* v_new, const void* h_ckpt, const void* d_o,
                                   const void* dv_new, const void* dh_ckpt, void* dq, void* dk, void* dv,
                                   void* dbeta, float* dg, int* exact_flags, void* stream);

/* The local term and the reverse scan on the tensor cores for the problems the fused per-chunk
 * stage does not take (a per-key-dim gate, or C = 32); bf16 io, GDR_ERR_UNSUPPORTED otherwise.
 * gdr_bwd_dv_local_tc: dv_loc = scale tril_0(Q~)^T do per chunk, [B,T,H,V] bf16.  For a per-key-dim
 * gate Q~ is formed from q exp(G - G_ref) and k exp(G_ref - G) around the chunk's middle row, and
 * exactly in fp32 for a chunk whose gate moves further than that keeps bounded.
 * gdr_bwd_scan_dh_tc: the reverse scan of gdr_bwd_scan_dh with dv_loc in bf16 and dh_ckpt, dv_new
 * written in bf16.  gdr_backward runs these, then gdr_bwd_dqkwg and gdr_bwd_wy's kernels reading
 * the bf16 dh_ckpt and dv_new. */
GDR_API gdr_status gdr_bwd_dv_local_tc(const gdr_problem* p, const void* q, const void* k, const float* g_cum,
                                       const void* d_o, void* dv_loc, void* stream);
GDR_API gdr_status gdr_bwd_scan_dh_tc(const gdr_problem* p, const void* q, const void* k, const void* w,
                                      const float* g_cum, const void* dv_loc, const void* d_o,
                                      const float* dh_final, void* dh_ckpt, void* dv_new, float* dh0,
                                      void* stream);

/* Grouped value heads (HV > H): the stage entry points above (gdr_bwd_dqkwg's dq, gdr_bwd_wy's
 * dk, gdr_bwd_wy_dqkg's dq and dk) write these per value head, [B,T,HV,K] in the io dtype; the
 * gradient of a shared q/k head is the sum over its group, which this call forms:
 * dq [B,T,H,K] = sum over g < HV/H of dq_v[:, :, h*(HV/H) + g], and the same for dk.
 * gdr_backward does this itself. */
GDR_API gdr_status gdr_bwd_group_sum(const gdr_problem* p, const void* dq_v, const void* dk_v, void* dq, void* dk,
                                     void* stream);

/* Bytes of device workspace gdr_backward needs (0 for a problem it would reject). */
GDR_API size_t gdr_backward_workspace_bytes(const gdr_problem* p);

/*
 * The whole backward: every stage above in order.
 * Inputs:  q, k, v, g, beta, h0 as gdr_forward took them; do [B,T,H,V] io;
 *          dh_final [B,H,K,V] fp32 or NULL (zero).
 * Outputs: dq, dk [B,T,H,K] io; dv [B,T,H,V] io; dg (shape of g) fp32;
 *          dbeta [B,T,H] io; dh0 [B,H,K,V] fp32 or NULL (not written).
 * workspace: at least gdr_backward_workspace_bytes(p) bytes, 256-byte aligned.
 */
GDR_API gdr_status gdr_backward(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                                const void* beta, const float* h0, const void* d_o, const float* dh_final,
                                void* dq, void* dk, void* dv, float* dg, void* dbeta, float* dh0,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Packed variable-length sequences.  The pages take equal-length batches only
 * (the scan's host wrapper in "kernel_fun/kda/_kernels/bwd_scan.py" asserts a
 * whole number of chunks).  A packed batch is read here as n independent
 * problems of the same recurrence, each sequence starting from its own initial
 * state; the n sequences of one packed token axis are the batch rows of p:
 *   p->B = n, p->T = a row length at least the longest sequence.
 *   cu_seqlens:        host int32 [n + 1], cu[0] = 0, non-decreasing, cu[n] = total,
 *                      every length cu[s+1] - cu[s] <= p->T; otherwise GDR_ERR_ARG.
 *   cu_seqlens_device: the same numbers in device memory (4-byte aligned), or NULL:
 *                      the call then copies cu_seqlens into the workspace on `stream`
 *                      (cudaMemcpyAsync; from pinned memory the host array must stay
 *                      unchanged until the stream has passed the call, and a stream
 *                      being captured into a graph needs cu_seqlens_device).
 *   total:             packed tokens; 0 allowed (the packed pointers may then be NULL).
 * Packed tensors have the batched layouts with B = 1 and T = total: q, k
 * [total,H,K] io; v [total,HV,V] io; g [total,HV] or [total,HV,K] fp32; beta
 * [total,HV] io; o like v.  Per-sequence tensors keep the batched layouts:
 * h0, h_final, dh_final, dh0 [n,HV,K,V] fp32 (sequence s starts from h0[s]).
 * The sequences are computed in a working layout in the workspace, the rest of
 * it zero tokens (beta = 0, g = 0, q = k = v = 0: the state passes unchanged and
 * their outputs are dropped).  On the tensor cores (bf16 or fp16 io) it is chunk-packed:
 * one row of whole chunks, sequence s taking ceil(len_s / C) of them, each run
 * scanned from h0[s]; the work is the real tokens plus fewer than C per
 * sequence.  The fused forward at C = 64 with bf16 io reads q, k, v, g, beta and writes o
 * in place; the other tensor-core paths copy the inputs into the row and the
 * results back.  The CUDA-core paths use padded rows, sequence s as row s of p,
 * through gdr_forward / gdr_backward on p: the work is n * p->T tokens.  A
 * sequence's results never depend on another sequence's tokens, finite or not.
 * p->segments is not used: every sequence is scanned whole.
 * workspace: at least gdr_varlen_*_workspace_bytes(p), 256-byte aligned, owned by the caller.
 */
GDR_API size_t gdr_varlen_forward_workspace_bytes(const gdr_problem* p);
GDR_API gdr_status gdr_varlen_forward(const gdr_problem* p, const int32_t* cu_seqlens, const int32_t* cu_seqlens_device,
                                      int64_t total, const void* q, const void* k, const void* v, const float* g,
                                      const void* beta, const float* h0, void* o, float* h_final, void* workspace,
                                      size_t workspace_bytes, void* stream);
/* The gradient of gdr_varlen_forward's (o, h_final): do packed like o, dh_final [n,HV,K,V]
 * fp32 or NULL; dq, dk, dv, dg, dbeta packed like q, k, v, g, beta; dh0 [n,HV,K,V] or NULL. */
GDR_API size_t gdr_varlen_backward_workspace_bytes(const gdr_problem* p);
GDR_API gdr_status gdr_varlen_backward(const gdr_problem* p, const int32_t* cu_seqlens,
                                       const int32_t* cu_seqlens_device, int64_t total, const void* q, const void* k,
                                       const void* v, const float* g, const void* beta, const float* h0,
                                       const void* d_o, const float* dh_final, void* dq, void* dk, void* dv, float* dg,
                                       void* dbeta, float* dh0, void* workspace, size_t workspace_bytes, void* stream);

/* Static, human-readable text for a status code. */
GDR_API const char* gdr_status_string(gdr_status s);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device.  Returns GDR_OK, GDR_ERR_DEVICE_TIMEOUT, or GDR_ERR_CUDA when
 * the synchronisation itself failed.
 */
GDR_API gdr_status gdr_get_device_status(void* stream);

/*
 * A check of the failure detection above, on the GPU, with nothing else in flight.
 * One CTA initialises an mbarrier that expects one arrival and waits on it with a
 * limit of `polls` polls (1 .. 4194304; GDR_ERR_ARG otherwise).  With arrive == 0
 * nothing arrives: the wait runs out, the kernel records GDR_ERR_DEVICE_TIMEOUT in
 * the device error word and exits normally, so the next gdr_get_device_status
 * reports it (and clears it).  With arrive != 0 the thread arrives first and the
 * wait succeeds.  No tensor-core work or TMA copy is issued, so nothing is left
 * running when the wait gives up.  The method pages have no counterpart to this
 * call; it exists to exercise the library's bounded waits.
 */
GDR_API gdr_status gdr_selftest_bounded_wait(int32_t polls, int32_t arrive, void* stream);

/*
 * Name of the kernel variant the last successful call on this host thread
 * launched (e.g. "simt", "tensor", "fused"); "" before any call.  The pointer
 * stays valid until the next call on the same thread.
 */
GDR_API const char* gdr_last_variant(void);

/* Library version, major * 10000 + minor * 100 + patch. */
GDR_API int gdr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H */
