// WY prepare launchers for fp16 io (the kernel and its design: prepare_mma.cuh), in a translation
// unit of their own so that the two io types compile side by side.  Every fp16 form takes the
// grouped-head indexing (EXTRA), which is the plain one when G = 1; none writes the inverse, which
// only the bf16 backward reads.
#include "prepare_mma.cuh"

namespace gdr {
namespace {

template <int K, int V, int C, bool PER_K, bool WITH_P, bool EXTRA, bool UMMA = false>
cudaError_t f16_launch(const Dims& d, const void* q, const void* k, const void* v, const float* g, const void* beta,
                       void* w, void* u, float* g_cum, void* P, cudaStream_t s, unsigned int* err, bool pdl) {
    return launch_prepare_v<K, V, C, PER_K, WITH_P, EXTRA, false, UMMA, true>(d, q, k, v, g, beta, w, u, g_cum, P,
                                                                              nullptr, s, err, PackedIn{}, pdl);
}

template <int K, int V, int C>
cudaError_t f16_gate(const Dims& d, const void* q, const void* k, const void* v, const float* g, const void* beta,
                     void* w, void* u, float* g_cum, void* P, cudaStream_t s, unsigned int* err, bool pdl, bool tc) {
    if (d.per_k) return f16_launch<K, V, C, true, false, true>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pdl);
    if constexpr (C == 64) {
        if (P) {
            if constexpr (K == 128 && V == 128) {
                // the tcgen05 scan's operands: S and P on tcgen05 when asked, else the plain form for one
                // q/k head per value head (both measured on the bf16 twins of these kernels)
                if (d.G == 1)
                    return tc ? f16_launch<K, V, C, false, true, false, true>(d, q, k, v, g, beta, w, u, g_cum, P, s,
                                                                             err, pdl)
                              : f16_launch<K, V, C, false, true, false>(d, q, k, v, g, beta, w, u, g_cum, P, s, err,
                                                                        pdl);
            }
            return f16_launch<K, V, C, false, true, true>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pdl);
        }
    }
    return f16_launch<K, V, C, false, false, true>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pdl);
}

template <int K, int V>
cudaError_t f16_chunk(const Dims& d, const void* q, const void* k, const void* v, const float* g, const void* beta,
                      void* w, void* u, float* g_cum, void* P, cudaStream_t s, unsigned int* err, bool pdl, bool tc) {
    return d.C == 32 ? f16_gate<K, V, 32>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pdl, tc)
                     : f16_gate<K, V, 64>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pdl, tc);
}

}  // namespace

cudaError_t mma_prepare_f16(const Dims& d, const void* k, const void* v, const float* g, const void* beta, void* w,
                            void* u, float* g_cum, cudaStream_t s, unsigned int* err, const void* q, void* P,
                            void* tinv, bool pdl, bool tc_scores) {
    if (!d.f16 || tinv || (P && (d.per_k || d.C != 64 || !q))) return cudaErrorInvalidValue;
    if (d.K == 64 && d.V == 64) return f16_chunk<64, 64>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pdl, tc_scores);
    if (d.K == 64) return f16_chunk<64, 128>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pdl, tc_scores);
    if (d.V == 64) return f16_chunk<128, 64>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pdl, tc_scores);
    return f16_chunk<128, 128>(d, q, k, v, g, beta, w, u, g_cum, P, s, err, pdl, tc_scores);
}

}  // namespace gdr
