// decode_fused.cu -- decode_kernel instances that select their blocks
// themselves (decode_dev.cuh, fused_select): for small f16 problems a decode
// step is then the token's append and this one kernel, without the selection
// kernel's launch and ticket between them.
#include "decode_dev.cuh"

namespace kvd {

cudaError_t launch_decode_fused(const kvd_cache &c, const Geom &g, const DecodePlan &p,
                                const float *q, float scale, int se, int rb, int keff,
                                int32_t *sel_idx, int32_t *sel_cnt, float *out,
                                float *partials, uint32_t *counters, cudaStream_t st,
                                bool pdl) {
    DecodeArgs a = make_decode_args(c, g, p, q, scale, sel_idx, sel_cnt, out, partials,
                                    counters, true, 0.0f);
    a.kbounds = static_cast<const __half *>(c.kbounds);
    a.sel_out_idx = sel_idx;
    a.sel_out_cnt = sel_cnt;
    a.fuse_se = se;
    a.fuse_rb = rb;
    a.fuse_keff = keff;
    const int P_sub = g.B * g.Hkv * p.subgroups;
    return launch_decode_gc<KVD_F16, false, false, false, false, true>(p.heads_per_cta, a,
                                                                        P_sub, st, pdl);
}

}  // namespace kvd
