// internal.h -- launchers shared between the kernel translation units and the
// C-ABI front end (api.cu).  Arguments are already validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "kvdecode.h"

namespace kvd {

// Geometry shared by the launchers (all sizes validated).
struct Geom {
    int dtype, B, Hkv, max_seq, len;  // len = tokens to read / after append
    int H, G;                         // query heads, group size
    int NB;                           // ceil(len / 64)
    int nbmax;                        // max_seq / 64
    int seq_add;  // tokens a decode step appended that the caller's seq_lens lacks
};

// Decode split plan: grid = (splits, B * Hkv * subgroups).  Split s attends
// the list positions [s * blocks / splits, (s + 1) * blocks / splits), and
// positions past `blocks` (a sel_cnt above the planned bound) round-robin.
struct DecodePlan {
    int heads_per_cta;  // query heads handled by one CTA (<= 4)
    int subgroups;      // G / heads_per_cta
    int splits;         // CTAs per (sequence, KV head, subgroup)
    int blocks;         // list length planned for (max_sel, at most NB)
    bool wide;          // one CTA per SM with twice the consumer groups
};

// one_head: one query head per CTA (lists per query head).  allow_wide: the
// launch may take the wide tile (quantized caches, few problems); every
// decode call allows it, so they all plan the same tile and splits.
DecodePlan plan_decode(const Geom &g, int max_blocks, int sm_count, bool one_head = false,
                       bool allow_wide = false);
size_t decode_partials_bytes(const Geom &g, const DecodePlan &p);
// SM count of the current device (cached per device ordinal; safe to call
// from several host threads).
int device_sm_count();
// Opens kernel fn to smem bytes of dynamic shared memory on the current device
// and returns (in occ, when not null) how many of its CTAs of `threads`
// threads fit on one SM.  The driver calls run once per (kernel, device, smem);
// later calls read a table under a lock, so host threads driving different
// devices may launch at the same time.
cudaError_t prepare_kernel(const void *fn, int threads, size_t smem, int *occ = nullptr);

// Stage marks of kernel kind `kind` (0 selection, 1 decode, 2 other):
// kMarkCtas * kMarkSlots words, or null when marks are off (every build
// without -DKVD_MARKS, or no buffer given to kvd_debug_stage_marks).
enum MarkKind { kMarkSelect = 0, kMarkDecode = 1, kMarkOther = 2, kMarkKinds = 3 };
unsigned long long *mark_region(int kind);

// Host argument rules shared by the entry points (api.cu): the cache
// descriptor, and the query-head count against it.
kvd_status check_cache(const kvd_cache *c);
kvd_status check_heads(const kvd_cache *c, int n_heads);

cudaError_t launch_append(const kvd_cache &c, const void *k_new, const void *v_new, int n_new,
                          cudaStream_t st, bool pdl, bool f32_in = false);

// Scratch of the selection (workspace regions; range and ticket are zero
// between calls, and every completed call leaves them zero).
struct SelScratch {
    uint32_t *keys;    // [B*Hkv][round_up(candidates, 4)] keys
    unsigned *range;   // [range_rows][2] key range of the problem (max, ~min)
    unsigned *ticket;  // [range_rows] arrival counters
    int range_rows;    // problems that may split over several CTAs need a row each
};

// The one token a decode step appends ([B, 1, Hkv, 128] f16 each) and the
// cache length before it.
struct StepToken {
    const void *k_new, *v_new;
    int len0;
};

// tok: inside a decode step, the token to append before the selection (g and
// c.len then describe the cache after it); the selection kernel appends it
// when the token's block is forced, else a separate append launch does.
cudaError_t launch_select(const kvd_cache &c, const Geom &g, const float *q, int k_sel,
                          int sink_tokens, int recent_tokens, int32_t *sel_idx,
                          int32_t *sel_cnt, const SelScratch &scr, cudaStream_t st, bool pdl,
                          const StepToken *tok);
// Per-query-head selection (sel_idx [B, H, nbmax], sel_cnt [B, H]).
cudaError_t launch_select_per_head(const kvd_cache &c, const Geom &g, const float *q, int k_sel,
                                   int sink_tokens, int recent_tokens, int32_t *sel_idx,
                                   int32_t *sel_cnt, const SelScratch &scr, cudaStream_t st,
                                   bool pdl);

cudaError_t launch_scores_debug(const kvd_cache &c, const Geom &g, const float *q, float *ub,
                                cudaStream_t st);

// early_q: the query may be read before the upstream kernels complete (true
// only when the caller's own earlier kernels in the same chain wrote nothing
// the query depends on, as inside kvd_decode_step).  sv_eps > 0: sparse-V in
// eps mode (0: every V term is accumulated).
cudaError_t launch_decode(const kvd_cache &c, const Geom &g, const DecodePlan &p,
                          const float *q, float scale, const int32_t *sel_idx,
                          const int32_t *sel_cnt, float *out, float *partials,
                          uint32_t *counters, cudaStream_t st, bool pdl, bool early_q,
                          float sv_eps = 0.0f);

// The sparse-V (sv_eps > 0) kernels behind launch_decode (decode_sv.cu).
cudaError_t launch_decode_sv(const kvd_cache &c, const Geom &g, const DecodePlan &p,
                             const float *q, float scale, const int32_t *sel_idx,
                             const int32_t *sel_cnt, float *out, float *partials,
                             uint32_t *counters, cudaStream_t st, bool pdl, bool early_q,
                             float sv_eps);
// Decode over lists per query head (sel_idx [B, H, nbmax], sel_cnt [B, H]);
// p planned with one_head.
cudaError_t launch_decode_per_head(const kvd_cache &c, const Geom &g, const DecodePlan &p,
                                   const float *q, float scale, const int32_t *sel_idx,
                                   const int32_t *sel_cnt, float *out, float *partials,
                                   uint32_t *counters, cudaStream_t st, bool pdl);

// Head dims other than 128 (general_d.cu, general_d_decode.cu; f16 and int8
// caches without block means or per-sequence lengths).  The append writes
// tokens [len0, len0 + n_new); the selection takes the candidate range
// [se, rb) and scratch keys rows of round_up(max_seq / 64, 4); the decode
// writes the splits' partials (gd_partials_bytes) and then out.
cudaError_t launch_append_gd(const kvd_cache &c, const void *k_new, const void *v_new,
                             int n_new, int len0, cudaStream_t st, bool f32_in);
cudaError_t launch_select_gd(const kvd_cache &c, const float *q, int n_heads, int k_sel, int se,
                             int rb, int32_t *sel_idx, int32_t *sel_cnt, uint32_t *keys,
                             cudaStream_t st);
int gd_splits(int problems, int max_blocks, int sm_count, int per_sm);
size_t gd_partials_bytes(int problems, int G, int D, int splits);
// Head dims 64, 256 and 512 with G in {1, 2, 4, 8, 16}: the warp-specialised
// kernel (general_d_fast.cu), its splits merged by the last CTA of each
// problem into out (counters: B * H words, zero between calls).
bool gd_fast_supported(const kvd_cache &c, int G);
cudaError_t launch_decode_gd_fast(const kvd_cache &c, const float *q, int n_heads,
                                  float scale_log2, const int32_t *sel_idx,
                                  const int32_t *sel_cnt, int max_blocks, float *out,
                                  float *partials, uint32_t *counters, cudaStream_t st);
cudaError_t launch_decode_gd(const kvd_cache &c, const float *q, int n_heads, float scale,
                             const int32_t *sel_idx, const int32_t *sel_cnt, int max_blocks,
                             float *out, float *partials, uint32_t *counters, cudaStream_t st);
// A kernel whose one mbarrier wait runs out after limit_ns (selftest.cu).
cudaError_t launch_wait_probe(int32_t *status, uint64_t limit_ns, cudaStream_t st);

// The listed blocks exactly plus the moment tail of every other block
// (decode_tail.cu); c.moments must be set.
cudaError_t launch_decode_tail(const kvd_cache &c, const Geom &g, const DecodePlan &p,
                               const float *q, float scale, const int32_t *sel_idx,
                               const int32_t *sel_cnt, float *out, float *partials,
                               uint32_t *counters, cudaStream_t st, bool pdl);

cudaError_t launch_qk_debug(const kvd_cache &c, const Geom &g, const float *q, int32_t *dots,
                            int8_t *q_codes, float *q_scales, cudaStream_t st);

// Launch helper: cudaLaunchKernelEx with optional programmatic stream
// serialization (the kernel must call pdl_wait() before reading upstream data).
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t st, bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Cooperative launch: every CTA of the grid is resident at once (the launch
// fails otherwise), as kernels whose CTAs wait on one another require.
template <typename... KArgs, typename... Args>
cudaError_t launch_coop(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                        cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace kvd
