// decode_sv.cu -- the sparse-V (eps mode) instances of decode_kernel
// (decode_dev.cuh), in their own translation unit: the plain kernels carry
// none of their code, and the two units compile in parallel.
#include "decode_dev.cuh"

namespace kvd {

cudaError_t launch_decode_sv(const kvd_cache &c, const Geom &g, const DecodePlan &p,
                             const float *q, float scale, const int32_t *sel_idx,
                             const int32_t *sel_cnt, float *out, float *partials,
                             uint32_t *counters, cudaStream_t st, bool pdl, bool early_q,
                             float sv_eps) {
    return launch_decode_any<true>(c, g, p, q, scale, sel_idx, sel_cnt, out, partials,
                                   counters, st, pdl, early_q, sv_eps);
}

}  // namespace kvd
