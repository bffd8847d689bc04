// decode.cu -- decode launches: decode_kernel (split-KV decode over the
// selected or all blocks; decode_dev.cuh) without sparse-V, the int8 q.k test
// export, and the split plan.  decode_sv.cu holds the sparse-V kernels.
#include "decode_dev.cuh"

namespace kvd {
namespace {

// ----------------------------------------------------------------------------
// Test export: exact int32 q.k dots of every cached token, computed with the
// decode kernel's query quantization and row-dot routines.
template <int GC>
__global__ void __launch_bounds__(256) qk_debug_kernel(DecodeArgs a, int32_t *dots,
                                                       int8_t *q_codes, float *q_scales) {
    __shared__ __align__(16) int8_t ks[kBlock * kHeadDim];
    __shared__ __align__(16) uint32_t q_s[GC * 32];
    __shared__ float coef[GC];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int blk = blockIdx.x;
    const int prob = blockIdx.y;
    const int sub = prob % a.subgroups;
    const int bg = prob / a.subgroups;
    const int b = bg / a.Hkv, g = bg % a.Hkv;
    const int h0 = g * a.G + sub * GC;
    load_query<KVD_INT8, GC>(a, b, h0, warp, lane, q_s, coef, blk == 0 ? q_codes : nullptr,
                             q_scales);
    const int8_t *src = static_cast<const int8_t *>(a.k) +
                        (static_cast<size_t>(bg) * a.max_seq + static_cast<size_t>(blk) * kBlock) *
                            kHeadDim;
    for (int i = tid; i < kBlock * kHeadDim / 16; i += 256)
        reinterpret_cast<uint4 *>(ks)[i] = reinterpret_cast<const uint4 *>(src)[i];
    __syncthreads();
    QRegsI8<GC> qr;
    const int t = lane >> 2, c = lane & 3;
    load_qregs_i8<GC>(q_s, t, c, qr);
    const int tok = 8 * warp + t;
    const int dot = qk_int8_row<GC>(ks + tok * kHeadDim, qr, t, c);
    const int hq = (c * GC) >> 2;
    const int pos = blk * kBlock + tok;
    if ((c % (4 / GC)) == 0 && pos < a.len)
        dots[(static_cast<size_t>(b) * a.H + h0 + hq) * a.len + pos] = dot;
}

}  // namespace

DecodePlan plan_decode(const Geom &g, int max_blocks, int sm_count, bool one_head,
                       bool allow_wide) {
    DecodePlan p;
    p.heads_per_cta = one_head ? 1 : g.G < 4 ? g.G : 4;
    p.subgroups = g.G / p.heads_per_cta;
    const long P = static_cast<long>(g.B) * g.Hkv * p.subgroups;
    // the wide tile when every problem still gets at least 8 CTAs with one CTA
    // per SM (long single sequences); the f16 tile has no wide form
    p.wide = allow_wide && g.dtype != KVD_F16 && P * 8 <= sm_count;
    const int per_sm = p.wide                ? 1
                       : g.dtype == KVD_F16  ? Tile<KVD_F16>::kMinCtas
                       : g.dtype == KVD_Q8_0 ? Tile<KVD_Q8_0>::kMinCtas
                       : g.dtype == KVD_Q4_0 ? Tile<KVD_Q4_0>::kMinCtas
                                             : Tile<KVD_INT8>::kMinCtas;
    const long target = static_cast<long>(sm_count) * per_sm;  // one wave of resident CTAs
    long s = P >= target ? 1 : target / P;
    const long by_work = (static_cast<long>(max_blocks) + 3) / 4;  // >= 4 blocks per split
    if (s > by_work) s = by_work;
    if (s < 1) s = 1;
    if (s > kMaxSplits) s = kMaxSplits;
    p.splits = static_cast<int>(s);
    p.blocks = max_blocks;
    return p;
}

size_t decode_partials_bytes(const Geom &g, const DecodePlan &p) {
    if (p.splits <= 1) return 0;
    return static_cast<size_t>(g.B) * g.Hkv * p.subgroups * p.splits * p.heads_per_cta *
           kPartStride * sizeof(float);
}

cudaError_t launch_decode(const kvd_cache &c, const Geom &g, const DecodePlan &p,
                          const float *q, float scale, const int32_t *sel_idx,
                          const int32_t *sel_cnt, float *out, float *partials,
                          uint32_t *counters, cudaStream_t st, bool pdl, bool early_q,
                          float sv_eps) {
    if (sv_eps > 0.0f)
        return launch_decode_sv(c, g, p, q, scale, sel_idx, sel_cnt, out, partials, counters,
                                st, pdl, early_q, sv_eps);
    return launch_decode_any<false>(c, g, p, q, scale, sel_idx, sel_cnt, out, partials,
                                    counters, st, pdl, early_q, 0.0f);
}

cudaError_t launch_decode_per_head(const kvd_cache &c, const Geom &g, const DecodePlan &p,
                                   const float *q, float scale, const int32_t *sel_idx,
                                   const int32_t *sel_cnt, float *out, float *partials,
                                   uint32_t *counters, cudaStream_t st, bool pdl) {
    DecodeArgs a = make_decode_args(c, g, p, q, scale, sel_idx, sel_cnt, out, partials,
                                    counters, false, 0.0f);
    a.per_head = 1;  // p.heads_per_cta is 1: CTA problem b * H + h reads list row b * H + h
    const int P_sub = g.B * g.Hkv * p.subgroups;
    if (p.wide) {  // quantized caches only (plan_decode)
        if (g.dtype == KVD_INT8)
            return launch_decode_t<KVD_INT8, 1, false, false, false, true>(a, P_sub, st, pdl);
        if (g.dtype == KVD_Q8_0)
            return launch_decode_t<KVD_Q8_0, 1, false, false, false, true>(a, P_sub, st, pdl);
        return launch_decode_t<KVD_Q4_0, 1, false, false, false, true>(a, P_sub, st, pdl);
    }
    if (g.dtype == KVD_INT8)
        return launch_decode_t<KVD_INT8, 1, false, false, false>(a, P_sub, st, pdl);
    if (g.dtype == KVD_Q8_0)
        return launch_decode_t<KVD_Q8_0, 1, false, false, false>(a, P_sub, st, pdl);
    if (g.dtype == KVD_Q4_0)
        return launch_decode_t<KVD_Q4_0, 1, false, false, false>(a, P_sub, st, pdl);
    return launch_decode_t<KVD_F16, 1, false, false, false>(a, P_sub, st, pdl);
}

cudaError_t launch_qk_debug(const kvd_cache &c, const Geom &g, const float *q, int32_t *dots,
                            int8_t *q_codes, float *q_scales, cudaStream_t st) {
    DecodeArgs a = {};
    a.k = c.k;
    a.q = q;
    a.Hkv = g.Hkv;
    a.H = g.H;
    a.G = g.G;
    a.max_seq = g.max_seq;
    a.nbmax = g.nbmax;
    a.len = g.len;
    a.NB = g.NB;
    a.scale_log2 = 1.0f;
    const int gc = g.G < 4 ? g.G : 4;
    a.subgroups = g.G / gc;
    dim3 grid(g.NB, g.B * g.Hkv * a.subgroups);
    switch (gc) {
        case 1: qk_debug_kernel<1><<<grid, 256, 0, st>>>(a, dots, q_codes, q_scales); break;
        case 2: qk_debug_kernel<2><<<grid, 256, 0, st>>>(a, dots, q_codes, q_scales); break;
        default: qk_debug_kernel<4><<<grid, 256, 0, st>>>(a, dots, q_codes, q_scales); break;
    }
    return cudaGetLastError();
}

}  // namespace kvd
