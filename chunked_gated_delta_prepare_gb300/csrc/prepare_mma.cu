// WY prepare launchers for bf16 io (the kernel and its design: prepare_mma.cuh; fp16 io:
// prepare_mma_f16.cu).
#include "prepare_mma.cuh"

namespace gdr {
namespace {

template <int K, int V, int C, bool PER_K, bool WITH_P>
cudaError_t launch_prepare(const Dims& d, const void* q, const void* k, const void* v, const float* g,
                           const void* beta, void* w, void* u, float* g_cum, void* P, void* tinv, cudaStream_t s,
                           unsigned int* err, bool pdl, bool tc_scores) {
    if constexpr (K == 128 && V == 128 && C == 64 && !PER_K && WITH_P) {
        if (tc_scores && d.G == 1 && !tinv)
            return launch_prepare_v<K, V, C, PER_K, WITH_P, false, false, true>(d, q, k, v, g, beta, w, u, g_cum, P,
                                                                                tinv, s, err, PackedIn{}, pdl);
    }
    if (d.G != 1 || tinv)
        return launch_prepare_v<K, V, C, PER_K, WITH_P, true>(d, q, k, v, g, beta, w, u, g_cum, P, tinv, s, err,
                                                              PackedIn{}, pdl);
    return launch_prepare_v<K, V, C, PER_K, WITH_P, false>(d, q, k, v, g, beta, w, u, g_cum, P, tinv, s, err,
                                                           PackedIn{}, pdl);
}

template <int K, int V, int C>
cudaError_t pick_gate(const Dims& d, const void* q, const void* k, const void* v, const float* g, const void* beta,
                      void* w, void* u, float* g_cum, void* P, void* tinv, cudaStream_t s, unsigned int* err,
                      bool pdl, bool tc) {
    if (d.per_k)
        return launch_prepare<K, V, C, true, false>(d, q, k, v, g, beta, w, u, g_cum, P, tinv, s, err, pdl, tc);
    if constexpr (C == 64) {
        if (P) return launch_prepare<K, V, C, false, true>(d, q, k, v, g, beta, w, u, g_cum, P, tinv, s, err, pdl, tc);
    }
    return launch_prepare<K, V, C, false, false>(d, q, k, v, g, beta, w, u, g_cum, P, tinv, s, err, pdl, tc);
}

template <int K, int V>
cudaError_t pick_chunk(const Dims& d, const void* q, const void* k, const void* v, const float* g, const void* beta,
                       void* w, void* u, float* g_cum, void* P, void* tinv, cudaStream_t s, unsigned int* err,
                       bool pdl, bool tc) {
    return d.C == 32 ? pick_gate<K, V, 32>(d, q, k, v, g, beta, w, u, g_cum, P, tinv, s, err, pdl, tc)
                     : pick_gate<K, V, 64>(d, q, k, v, g, beta, w, u, g_cum, P, tinv, s, err, pdl, tc);
}

template <int K, int V>
cudaError_t packed_prepare(const Dims& d, const void* q, const void* k, const void* v, const float* g,
                           const void* beta, void* w, void* u, float* g_cum, void* P, cudaStream_t s,
                           unsigned int* err, PackedIn pin) {
    if (d.G != 1)
        return launch_prepare_v<K, V, 64, false, true, true, true>(d, q, k, v, g, beta, w, u, g_cum, P, nullptr, s,
                                                                   err, pin);
    return launch_prepare_v<K, V, 64, false, true, false, true>(d, q, k, v, g, beta, w, u, g_cum, P, nullptr, s, err,
                                                                pin);
}

}  // namespace

cudaError_t mma_prepare_packed(const Dims& d, const void* q, const void* k, const void* v, const float* g,
                               const void* beta, void* w, void* u, float* g_cum, void* P, const int* cu,
                               const int* co, const int* cs, int nseq, int total, cudaStream_t s, unsigned int* err) {
    if (!d.bf16 || d.per_k || d.C != 64 || d.B != 1 || !q || !P || !cu || !co || !cs || nseq < 1 || total < 1)
        return cudaErrorInvalidValue;
    const PackedIn pin{cu, co, cs, nseq, total};
    if (d.K == 64 && d.V == 64) return packed_prepare<64, 64>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pin);
    if (d.K == 64 && d.V == 128) return packed_prepare<64, 128>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pin);
    if (d.K == 128 && d.V == 64) return packed_prepare<128, 64>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pin);
    return packed_prepare<128, 128>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pin);
}

cudaError_t mma_prepare(const Dims& d, const void* k, const void* v, const float* g, const void* beta, void* w,
                        void* u, float* g_cum, cudaStream_t s, unsigned int* err, const void* q, void* P,
                        void* tinv, bool pdl, bool tc_scores) {
    if (P && (d.per_k || d.C != 64 || !q)) return cudaErrorInvalidValue;
    if (d.f16) return mma_prepare_f16(d, k, v, g, beta, w, u, g_cum, s, err, q, P, tinv, pdl, tc_scores);
    if (!d.bf16) return cudaErrorInvalidValue;
    const bool tc = tc_scores;
    if (d.K == 64 && d.V == 64) return pick_chunk<64, 64>(d, q, k, v, g, beta, w, u, g_cum, P, tinv, s, err, pdl, tc);
    if (d.K == 64 && d.V == 128) return pick_chunk<64, 128>(d, q, k, v, g, beta, w, u, g_cum, P, tinv, s, err, pdl, tc);
    if (d.K == 128 && d.V == 64) return pick_chunk<128, 64>(d, q, k, v, g, beta, w, u, g_cum, P, tinv, s, err, pdl, tc);
    return pick_chunk<128, 128>(d, q, k, v, g, beta, w, u, g_cum, P, tinv, s, err, pdl, tc);
}

}  // namespace gdr
