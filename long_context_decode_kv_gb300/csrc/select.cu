// select.cu -- the selection launches: select_kernel (scoring, then the
// radix select by the last CTA of each problem; select_dev.cuh) and
// fill_kernel, for the selections that need no bounds (no candidates to
// rank: K_SEL = 0, or at least as large as the candidate count).
#include "select_dev.cuh"

namespace kvd {
namespace {

template <int G, int MODE>
__global__ void __launch_bounds__(kScoreThreads, 1) select_kernel(SelArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ SelShared ss;
    select_body<G, MODE>(a, blockIdx.x, gridDim.x, blockIdx.y, smem, ss);
}

// Selections that rank nothing: sink blocks, all candidates (take_all) or
// none, recent blocks.
__global__ void __launch_bounds__(256) fill_kernel(int32_t *sel_idx, int32_t *sel_cnt, int nbmax,
                                                   int NB, int se, int rb, int take_all) {
    pdl_wait();
    pdl_launch_dependents();
    const int p = blockIdx.x;
    int32_t *dst = sel_idx + static_cast<size_t>(p) * nbmax;
    const int n_take = take_all ? rb - se : 0;
    for (int j = threadIdx.x; j < se + n_take; j += blockDim.x) dst[j] = j;
    for (int j = rb + threadIdx.x; j < NB; j += blockDim.x) dst[se + n_take + (j - rb)] = j;
    if (threadIdx.x == 0) sel_cnt[p] = se + n_take + (NB - rb);
}

// fill_kernel under per-sequence lengths: each problem's own forced blocks
// and candidates (every candidate when k_sel reaches the longest sequence's
// count, none when k_sel is 0).
__global__ void __launch_bounds__(256) fill_kernel_varlen(SelArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int p = blockIdx.x;
    SelArgs v;
    const int take = problem_args(a, p, v);
    fill_list(v, p, take >= 1, threadIdx.x, blockDim.x);  // one row per problem of the grid
}

template <int G, int MODE>
cudaError_t launch_select_t(const SelArgs &a0, int P, cudaStream_t st, bool pdl) {
    constexpr int smem = select_smem_bytes<G>();
    int occupancy = 1;
    const cudaError_t e = prepare_kernel(reinterpret_cast<const void *>(select_kernel<G, MODE>),
                                         kScoreThreads, smem, &occupancy);
    if (e != cudaSuccess) return e;
    SelArgs a = a0;
    a.marks = mark_region(kMarkSelect);
    // CTAs per problem: as many as fit on the GPU at once, split evenly (a
    // small problem still gains from many CTAs streaming its bounds)
    const long cap = static_cast<long>(occupancy) * device_sm_count();
    long X = cap / P;
    if (X > kMaxCtasPerProblem) X = kMaxCtasPerProblem;
    if (X < 1) X = 1;
    long R = (static_cast<long>(a.n) + X - 1) / X;
    X = (a.n + R - 1) / R;
    a.R = static_cast<int>(R);
    const dim3 grid(static_cast<unsigned>(X), static_cast<unsigned>(P));
    return launch_ex(select_kernel<G, MODE>, grid, dim3(kScoreThreads), smem, st, pdl, a);
}

template <int MODE>
cudaError_t launch_select_any(const SelArgs &a, int G, int P, cudaStream_t st, bool pdl) {
    switch (G) {
        case 1: return launch_select_t<1, MODE>(a, P, st, pdl);
        case 2: return launch_select_t<2, MODE>(a, P, st, pdl);
        case 4: return launch_select_t<4, MODE>(a, P, st, pdl);
        case 8: return launch_select_t<8, MODE>(a, P, st, pdl);
        case 16: return launch_select_t<16, MODE>(a, P, st, pdl);
        default: return cudaErrorInvalidValue;
    }
}

// The selection kernel for P problems, with per-sequence geometry on the
// device when the cache carries sequence lengths; per_head: one query head
// of each group (a.head_sub).
cudaError_t launch_select_mode(const SelArgs &a, int G, int P, cudaStream_t st, bool pdl,
                               bool per_head = false) {
    if (per_head)  // G = 1 problems: one head at a time
        return a.seq_lens ? launch_select_t<1, kSelect | kVarlen | kPerHead>(a, P, st, pdl)
                          : launch_select_t<1, kSelect | kPerHead>(a, P, st, pdl);
    return a.seq_lens ? launch_select_any<kSelect | kVarlen>(a, G, P, st, pdl)
                      : launch_select_any<kSelect>(a, G, P, st, pdl);
}

SelArgs base_args(const kvd_cache &c, const Geom &g, const float *q) {
    SelArgs a = {};
    a.q = q;
    a.kbounds = static_cast<const __half *>(c.kbounds);
    a.Hkv = g.Hkv;
    a.H = g.H;
    a.nbmax = g.nbmax;
    a.NB = g.NB;
    a.dev_status = c.dev_status;
    a.head_sub = -1;
    a.G_all = g.G;
    a.seq_lens = c.seq_lens;
    a.len_max = g.len;
    a.seq_add = g.seq_add;
    return a;
}

// The arguments of a ranking selection over the longest sequence's geometry.
SelArgs rank_args(const kvd_cache &c, const Geom &g, const float *q, const ForcedRange &f,
                  int k_sel, int sink_tokens, int recent_tokens, int32_t *sel_idx,
                  int32_t *sel_cnt, const SelScratch &scr) {
    SelArgs a = base_args(c, g, q);
    a.se = f.se;
    a.n = f.rb - f.se;
    a.keys = scr.keys;
    a.ldk = (a.n + 3) / 4 * 4;
    a.ldn = a.ldk;
    a.range = scr.range;
    a.ticket = scr.ticket;
    a.sel_idx = sel_idx;
    a.sel_cnt = sel_cnt;
    a.rb = f.rb;
    a.keff = k_sel < a.n ? k_sel : a.n;
    a.k_sel = k_sel;
    a.sink_tokens = sink_tokens;
    a.recent_tokens = recent_tokens;
    return a;
}

}  // namespace

int max_select_blocks() { return kMaxSelectBlocks; }

cudaError_t launch_select(const kvd_cache &c, const Geom &g, const float *q, int k_sel,
                          int sink_tokens, int recent_tokens, int32_t *sel_idx,
                          int32_t *sel_cnt, const SelScratch &scr, cudaStream_t st, bool pdl,
                          const StepToken *tok) {
    const ForcedRange f = forced_range(g.len, sink_tokens, recent_tokens);
    const int n_cand = f.rb - f.se;
    const int keff = k_sel < n_cand ? k_sel : n_cand;
    const int P = g.B * g.Hkv;
    // a decode step's token rides in the selection kernel when its block is
    // forced (a recent window) and there is a top-K to find; otherwise it is
    // appended by its own launch first
    const bool topk = keff > 0 && keff < n_cand;
    // the fused append writes rows and bounds only: a cache that keeps block
    // means appends through the append kernel, which recomputes them
    // with per-sequence lengths some problems may rank nothing (filled without
    // the fused path), so their tokens are appended by the append kernel too
    const bool fuse = tok && topk && recent_tokens > 0 && c.moments == nullptr && !c.seq_lens;
    if (tok && !fuse) {
        kvd_cache c0 = c;
        c0.len = tok->len0;
        const cudaError_t e = launch_append(c0, tok->k_new, tok->v_new, 1, st, pdl);
        if (e != cudaSuccess) return e;
    }
    SelArgs a = rank_args(c, g, q, f, k_sel, sink_tokens, recent_tokens, sel_idx, sel_cnt, scr);
    if (!topk) {
        if (c.seq_lens)  // shorter sequences may still rank: the same rule per problem
            return launch_ex(fill_kernel_varlen, dim3(P), dim3(256), 0, st, pdl, a);
        return launch_ex(fill_kernel, dim3(P), dim3(256), 0, st, pdl, sel_idx, sel_cnt, g.nbmax,
                         f.NB, f.se, f.rb, keff > 0 ? 1 : 0);
    }
    if (fuse) {
        a.app_cache = c;
        a.app_cache.len = tok->len0;
        a.app_k = static_cast<const __half *>(tok->k_new);
        a.app_v = static_cast<const __half *>(tok->v_new);
    }
    // the step's token block is the last one; it is never a candidate while
    // the recent window is non-empty, so scoring may start before the
    // upstream kernels finish
    a.overlap = fuse ? 1 : 0;
    return launch_select_mode(a, g.G, P, st, pdl);
}

// Per-query-head selection: query head h of KV head g ranks the blocks by its
// own bound, not the group's maximum.  One launch per head of the group, each
// a G = 1 selection over the B * Hkv problems (the same scratch, reused in
// stream order), writing rows [B, H] of sel_idx / sel_cnt.
cudaError_t launch_select_per_head(const kvd_cache &c, const Geom &g, const float *q, int k_sel,
                                   int sink_tokens, int recent_tokens, int32_t *sel_idx,
                                   int32_t *sel_cnt, const SelScratch &scr, cudaStream_t st,
                                   bool pdl) {
    const ForcedRange f = forced_range(g.len, sink_tokens, recent_tokens);
    const int n_cand = f.rb - f.se;
    const int keff = k_sel < n_cand ? k_sel : n_cand;
    const int P = g.B * g.Hkv;
    SelArgs a = rank_args(c, g, q, f, k_sel, sink_tokens, recent_tokens, sel_idx, sel_cnt, scr);
    if (!(keff > 0 && keff < n_cand)) {  // nothing to rank: every head gets the same list
        if (c.seq_lens) {
            a.head_sub = 0;
            a.G_all = 1;  // rows are (b, h) = problem index over B * H
            a.Hkv = g.H;  // problem b * H + h belongs to sequence b
            return launch_ex(fill_kernel_varlen, dim3(P * g.G), dim3(256), 0, st, pdl, a);
        }
        return launch_ex(fill_kernel, dim3(P * g.G), dim3(256), 0, st, pdl, sel_idx, sel_cnt,
                         g.nbmax, f.NB, f.se, f.rb, keff > 0 ? 1 : 0);
    }
    for (int sub = 0; sub < g.G; ++sub) {
        a.head_sub = sub;
        const cudaError_t e = launch_select_mode(a, 1, P, st, pdl, true);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_scores_debug(const kvd_cache &c, const Geom &g, const float *q, float *ub,
                                cudaStream_t st) {
    SelArgs a = base_args(c, g, q);
    a.se = 0;
    a.n = g.NB;
    a.ub = ub;
    return launch_select_any<kExport>(a, g.G, g.B * g.Hkv, st, false);
}

}  // namespace kvd
