// decode_tail.cu -- the moment-tail instances of decode_kernel (decode_dev.cuh):
// the listed blocks attended exactly, every other block by its count, key mean
// and value mean ("SCSA: Self-Calibrating Subquadratic Attention", "2.
// Mechanism", moment tail).  Their own translation unit keeps that code out of
// the plain kernels and compiles in parallel with them.
#include "decode_dev.cuh"

namespace kvd {

cudaError_t launch_decode_tail(const kvd_cache &c, const Geom &g, const DecodePlan &p,
                               const float *q, float scale, const int32_t *sel_idx,
                               const int32_t *sel_cnt, float *out, float *partials,
                               uint32_t *counters, cudaStream_t st, bool pdl) {
    DecodeArgs a = make_decode_args(c, g, p, q, scale, sel_idx, sel_cnt, out, partials,
                                    counters, false, 0.0f);
    a.moments = static_cast<const __half *>(c.moments);
    const int P_sub = g.B * g.Hkv * p.subgroups;
    const int gc = p.heads_per_cta;
    if (p.wide) {  // quantized caches only (plan_decode)
        if (g.dtype == KVD_INT8)
            return launch_decode_gc<KVD_INT8, false, false, true, true>(gc, a, P_sub, st, pdl);
        if (g.dtype == KVD_Q8_0)
            return launch_decode_gc<KVD_Q8_0, false, false, true, true>(gc, a, P_sub, st, pdl);
        return launch_decode_gc<KVD_Q4_0, false, false, true, true>(gc, a, P_sub, st, pdl);
    }
    if (g.dtype == KVD_INT8)
        return launch_decode_gc<KVD_INT8, false, false, true>(gc, a, P_sub, st, pdl);
    if (g.dtype == KVD_Q8_0)
        return launch_decode_gc<KVD_Q8_0, false, false, true>(gc, a, P_sub, st, pdl);
    if (g.dtype == KVD_Q4_0)
        return launch_decode_gc<KVD_Q4_0, false, false, true>(gc, a, P_sub, st, pdl);
    return launch_decode_gc<KVD_F16, false, false, true>(gc, a, P_sub, st, pdl);
}

}  // namespace kvd
