/*
 * kvdecode.h -- C ABI of libkvdecode.so: single-token decode attention over a
 * long KV cache that reads only part of it (Quest-style block selection),
 * for NVIDIA GB300 (sm_103a), one GPU.
 *
 * Sources, by page title and section:
 *  [QUEST]  "Sparse Attention -- Quest-style block-selector for long-context
 *           decode (#551)": "Method: Quest-style min/max block bounds",
 *           "S2/S3 engineering design" (fill op, selector op, FA-VEC block
 *           skip), "Knobs", "Gate ladder", "All-KV-types composition
 *           (bug-747)".
 *  [CPUATT] "cpu-attn" (Hugging Face kernels card): "Usage", "Method",
 *           "Correctness", "Requirements and limits".
 *  [SCSA]   "SCSA: Self-Calibrating Subquadratic Attention": "2. Mechanism"
 *           (the moment tail of the key groups not read exactly).
 *  [CERT]   "Certified Sparse Attention via Perturbed Retrieval": Appendix
 *           Table 4 (GQA-shared scan against one scan per query head).
 *
 * Conventions for every entry point
 *  - All device memory is allocated and owned by the caller.  The library
 *    never allocates or frees device memory and never synchronizes: every
 *    call enqueues its kernels on `stream` (a cudaStream_t passed as void*;
 *    NULL means the legacy default stream) and returns.
 *  - Arguments are checked on the host before anything is enqueued.  A call
 *    that returns anything but KVD_OK has enqueued nothing (the one
 *    exception, KVD_ERR_CUDA from a failed launch, is documented there).
 *  - Device pointers must be 16-byte aligned.  Layouts are dense row-major
 *    with the shapes given; no strides.
 *  - Faults found on the device (a bounded wait that ran out) are written to
 *    the cache's optional `dev_status` word (0 = fine); the kernels never
 *    trap.  Read the word after the stream has finished.
 *  - No call is thread-safe on the same cache or workspace; calls on one
 *    stream are ordered by the stream.  The library's own host state (per
 *    device: the SM count, the kernels' shared-memory attributes and
 *    occupancy, the workspace-free decode's array address) is filled once
 *    per device under a lock, so host threads driving different devices, or
 *    different caches on one device, may call at the same time.
 */
#ifndef KVDECODE_H
#define KVDECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVD_ABI_VERSION 3

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define KVD_API __attribute__((visibility("default")))
#else
#define KVD_API
#endif

typedef enum {
    KVD_OK = 0,
    KVD_ERR_INVALID = 1,      /* bad argument: NULL/misaligned pointer, bad size */
    KVD_ERR_UNSUPPORTED = 2,  /* legal but not built: block != 64, a head_dim that is not
                                 a multiple of 16 in [16, 1024], ... */
    KVD_ERR_CAPACITY = 3,     /* append would pass max_seq */
    KVD_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    KVD_ERR_TIMEOUT = 5,      /* device only: a bounded wait ran out (dev_status) */
    KVD_ERR_WORKSPACE = 6     /* workspace NULL, misaligned or too small */
} kvd_status;

typedef enum { KVD_F16 = 0, KVD_INT8 = 1, KVD_Q8_0 = 2, KVD_Q4_0 = 3 } kvd_kv_dtype;

/*
 * The cache: a plain descriptor of caller-owned device memory.
 *
 * Layout is head-major, so one block of `block` tokens of one (sequence,
 * KV head) is one contiguous run of memory:
 *   k, v        [batch, n_kv_heads, max_seq, head_dim]   f16 or int8 codes,
 *               or [.., head_dim / 2] bytes of 4-bit codes (q4_0)
 *   k_scale,    int8: [batch, n_kv_heads, max_seq] f32;
 *   v_scale     q8_0, q4_0: [batch, n_kv_heads, max_seq, head_dim / 32] f16
 *               (NULL for f16)
 *   kbounds     [batch, n_kv_heads, max_seq / block, head_dim, 2]  f16
 * kbounds holds the per-(KV head, block) channel-wise key envelope (QUEST,
 * Method: one minimum and one maximum per channel for every block) as interleaved
 * pairs: kbounds[..., d, 0] = kmin[d], kbounds[..., d, 1] = kmax[d] (one
 * contiguous 512-byte row per block).  It is always taken from the f16 keys
 * before quantization [QUEST All-KV-types composition].
 * int8 rows hold per-token per-head absmax codes [CPUATT Method]: scale =
 * absmax/127 (f32), code = round-half-even(x / scale) clamped to +-127, and
 * a row whose scale is 0 holds zero codes.
 * q8_0 rows hold the same codes per group of 32 channels (the llama.cpp
 * cache type of [QUEST] "All-KV-types composition"), each group with its
 * own f16 scale d = fl16(fl32(absmax_group / 127)); code = round-half-even
 * of the f32 quotient x / d, clamped to +-127 (zero codes when d is 0).
 * q4_0 rows hold 4-bit codes per group of 32 channels: m is the group's
 * value of largest magnitude (the first in channel order), the f16 scale is
 * d = fl16(fl32(m / -8)), code = clamp(round-half-even(fl32(x / d)) + 8,
 * 0, 15) (all 8 when d is 0), and the value is d * (code - 8); byte i of a
 * group holds channels 2i (low nibble) and 2i+1 (high nibble).
 * The bounds come from the f16 keys on every cache type.
 *
 * `len` (tokens cached; the same for every sequence) is host state, advanced
 * by kvd_kv_append.  Rows at or beyond `len` are never read by a decode
 * call's arithmetic (they may hold anything).
 * `dev_status` may be NULL; if set it is one device int32 that kernels set
 * to a kvd_status code when a bounded device wait runs out.
 * `moments` may be NULL; if set, [batch, n_kv_heads, max_seq / block, 2,
 * head_dim] f16: per block the mean of its stored keys, then of its stored
 * values (dequantized: code * scale for int8, code * d for q8_0, (code - 8)
 * * d for q4_0), over the block's tokens below len, each channel's f32 sum
 * in token order divided by the count and rounded to f16.  kvd_kv_append
 * and kvd_decode_step keep them for every block they write; they feed the
 * moment tail of kvd_decode_attn_tail.  Rewinding len inside a block and
 * appending again recomputes that block's means from its rows.
 * `seq_lens` may be NULL (every sequence holds len tokens); if set, a device
 * int32 [batch] with sequence b's own length, 0 <= seq_lens[b] <= len, and
 * `len` is the batch's maximum (it sizes the grids).  Every call then works
 * per sequence: kvd_kv_append writes sequence b's new rows from position
 * seq_lens[b] (the caller adds n_new to seq_lens afterwards; the library
 * never writes it), the selection ranks blocks below ceil(seq_lens[b] / block)
 * with the recent window ending at seq_lens[b], and the decode calls attend
 * tokens below seq_lens[b] (a sequence of length 0 gets a zero output).
 * kvd_decode_step appends sequence b's token at seq_lens[b] and then selects
 * and attends over its seq_lens[b] + 1 tokens (the caller adds 1 to seq_lens
 * after the step).  kvd_debug_scores does not take it (UNSUPPORTED).
 */
typedef struct kvd_cache {
    int32_t dtype;        /* kvd_kv_dtype */
    int32_t batch;        /* independent sequences, >= 1 */
    int32_t n_kv_heads;   /* Hkv >= 1 */
    int32_t head_dim;     /* D: 128 (every cache type and call), or any other multiple
                             of 16 up to 1024 ("cpu-attn", Requirements and limits)
                             for f16 and int8 caches without moments or seq_lens,
                             through kvd_kv_append(_f32), kvd_select_blocks,
                             kvd_decode_attn(_dense), kvd_decode_step(_host) and
                             kvd_workspace_bytes; other calls return UNSUPPORTED */
    int32_t max_seq;      /* capacity in tokens, a multiple of `block` */
    int32_t block;        /* B_SEL; only 64 is built [QUEST Knobs: default 64] */
    int32_t len;          /* tokens currently cached, 0 <= len <= max_seq */
    int32_t reserved;     /* must be 0 */
    void *k;
    void *v;
    void *k_scale;        /* f32 (int8) or f16 (q8_0, q4_0) scales, see above */
    void *v_scale;
    void *kbounds;
    int32_t *dev_status;
    void *moments;        /* optional block means (moment tail), see above */
    const int32_t *seq_lens;  /* optional per-sequence lengths, see above */
} kvd_cache;

/* ---------------------------------------------------------------------- */
/* Append n_new tokens to every sequence  [QUEST S2/S3 "Fill op" and       */
/* All-KV-types composition; CPUATT Method "quantize at append time"].     */
/*   k_new, v_new: device, [batch, n_new, n_kv_heads, head_dim] f16.        */
/* Writes rows len .. len+n_new-1 (f16 verbatim, or int8 codes + scales)   */
/* and the bounds of every block those rows touch: a block that already   */
/* held tokens is min/max-merged, a block that starts in the new range is  */
/* overwritten.  With cache->moments set, the key and value means of every */
/* touched block are recomputed over its rows below the new len.          */
/* On KVD_OK, cache->len += n_new (host side; the kernels                  */
/* are only enqueued).  n_new == 0 is a no-op.                             */
/* Errors: INVALID, UNSUPPORTED, CAPACITY (len + n_new > max_seq), CUDA.   */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_kv_append(kvd_cache *cache, const void *k_new, const void *v_new,
                         int32_t n_new, void *stream);

/* ---------------------------------------------------------------------- */
/* kvd_kv_append from f32 input  [CPUATT Usage: the cache takes each       */
/* token's K and V as f32; QUEST All-KV-types composition: the bounds come */
/* from the keys before quantization].                                      */
/*   k_new, v_new: device, [batch, n_new, n_kv_heads, head_dim] f32.         */
/*   f16 cache: stores each value's nearest f16 (ties to even), exactly as  */
/*   kvd_kv_append of those f16 values would.                               */
/*   int8 / q8_0 / q4_0: the rows are quantized from the f32 values; a       */
/*   block's bounds are the f32 keys' channel envelope rounded outward to   */
/*   f16 (kmin toward -inf, kmax toward +inf), merged as usual, so they     */
/*   hold every key.  Block means (when kept) come from the stored rows.    */
/* Errors and len: as kvd_kv_append.                                        */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_kv_append_f32(kvd_cache *cache, const float *k_new, const float *v_new,
                             int32_t n_new, void *stream);

/* ---------------------------------------------------------------------- */
/* Quest block selection for one query token per sequence  [QUEST Method   */
/* "Per-query upper bound", "Top-K block selection"; S2/S3 selector op:    */
/* "GQA -> max UB over the query group per KV-head"].                      */
/*   q: device [batch, n_heads, head_dim] f32; query head h belongs to KV   */
/*      head h / (n_heads / n_kv_heads) [CPUATT Usage].                    */
/*   For each (sequence, KV head) and block j < NB = ceil(len / block):    */
/*     UB(j) = max over the group's heads h of                             */
/*             sum_d max(q_h[d] * kmin_j[d], q_h[d] * kmax_j[d])            */
/*   Forced blocks: those meeting [0, sink_tokens) (sink) and those        */
/*   meeting [len - recent_tokens, len) (recent window).  Of the other     */
/*   blocks the k_sel with the largest UB are taken (all of them if fewer),*/
/*   equal bounds going to the lower block index.                          */
/*   sel_idx: device [batch, n_kv_heads, max_seq / block] int32; row r     */
/*            receives its selected block ids ascending in its first        */
/*            sel_cnt[r] entries (the rest is left untouched).             */
/*   sel_cnt: device [batch, n_kv_heads] int32; every row gets the same     */
/*            count, kvd_selected_count(len, block, k_sel, sink, recent).  */
/*   workspace: device scratch of kvd_workspace_bytes(...) bytes.          */
/* Errors: INVALID (len == 0, k_sel/sink/recent < 0, n_heads not a         */
/* multiple of n_kv_heads), UNSUPPORTED (group size not 1, 2, 4, 8 or 16;  */
/* more than 49152 blocks), WORKSPACE, CUDA.                               */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_select_blocks(const kvd_cache *cache, const float *q, int32_t n_heads,
                             int32_t k_sel, int32_t sink_tokens, int32_t recent_tokens,
                             int32_t *sel_idx, int32_t *sel_cnt,
                             void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* Per-query-head selection: the ablation of the GQA-shared one  [CERT      */
/* Appendix Table 4: one scan per query head against the GQA-shared scan;   */
/* QUEST "GQA": the shared block set avoids per-head divergence].           */
/*   As kvd_select_blocks, except that query head h ranks the blocks by its  */
/*   own bound UB_h(j) (no maximum over the group), and its list is row      */
/*   (b, h) of sel_idx [batch, n_heads, max_seq / block] int32, its count    */
/*   sel_cnt[b, h] ([batch, n_heads] int32).  Forced blocks and ties as      */
/*   there.  One launch per head of a group.                                  */
/* Errors: as kvd_select_blocks.                                              */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_select_blocks_per_head(const kvd_cache *cache, const float *q,
                                      int32_t n_heads, int32_t k_sel, int32_t sink_tokens,
                                      int32_t recent_tokens, int32_t *sel_idx,
                                      int32_t *sel_cnt, void *workspace,
                                      size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* Decode attention over lists per query head (kvd_select_blocks_per_head's  */
/* rows): as kvd_decode_attn, with query head h attending the blocks of row  */
/* (b, h) of sel_idx [batch, n_heads, max_seq / block] (sel_cnt [batch,      */
/* n_heads]).  Each CTA serves one query head, so a block listed for several */
/* heads of a group is read once per head.                                    */
/* Errors: as kvd_decode_attn.                                                */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_decode_attn_per_head(const kvd_cache *cache, const float *q,
                                    int32_t n_heads, float softmax_scale,
                                    const int32_t *sel_idx, const int32_t *sel_cnt,
                                    int32_t max_sel, float *out, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* Split-KV decode attention over selected blocks only  [QUEST S3 FA-VEC   */
/* block skip: unselected blocks are not read; CPUATT Method].             */
/*   For query head h of KV head g, over the tokens t < len of the blocks  */
/*   listed in sel_idx[b, g, :sel_cnt[b, g]] (ascending or not; each block */
/*   once):                                                                 */
/*     f16:  logit_t = softmax_scale * sum_d q[d] * k_t[d]                  */
/*     int8: q is quantized once per head like a cache row; logit_t =      */
/*           dot_int32(q_code, k_code_t) * q_scale * k_scale_t * softmax_scale */
/*           and v_t = v_scale_t * v_code_t                                 */
/*     q8_0: q as for int8; logit_t = q_scale * softmax_scale *             */
/*           sum_g d_g(k_t) * dot_int32 over group g (32 channels), and     */
/*           v_t[c] = d_g(v_t) * v_code_t[c] with g = c / 32                */
/*     q4_0: as q8_0 with (code - 8) in place of the code                   */
/*     out_h = sum_t softmax(logit)_t * v_t       (f32 accumulation)       */
/*   An empty selection gives a zero output row.                           */
/*   out: device [batch, n_heads, head_dim] f32.                            */
/*   max_sel: an upper bound of every sel_cnt row (it only sizes the split  */
/*   grid; sel_cnt values above max_sel are still attended in full), e.g.  */
/*   kvd_selected_count(...).                                              */
/*   workspace: as for kvd_select_blocks; holds split partials and the      */
/*   per-problem arrival counters.  The workspace must be zero-filled      */
/*   before its first use; every call that completes leaves the counters   */
/*   at zero again.  After a call that reported a device fault, zero it.  */
/* Errors: INVALID, UNSUPPORTED, WORKSPACE, CUDA.                          */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_decode_attn(const kvd_cache *cache, const float *q, int32_t n_heads,
                           float softmax_scale, const int32_t *sel_idx,
                           const int32_t *sel_cnt, int32_t max_sel, float *out,
                           void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* Dense decode attention over all len tokens (no bounds, no selection):  */
/* the no-skip reference arm  [QUEST Gate ladder "select-all ... sparse    */
/* must equal dense"; CPUATT Method].  Same arithmetic and arguments as    */
/* kvd_decode_attn with every block selected.                              */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_decode_attn_dense(const kvd_cache *cache, const float *q, int32_t n_heads,
                                 float softmax_scale, float *out,
                                 void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* Decode attention with sparse-V in eps mode  [QUEST "Adaptive tau (the   */
/* eps mode)", "Compose" item 3: inside the attended blocks, skip the V    */
/* work of positions whose weight is negligible, so that the dropped share */
/* of the softmax mass stays below eps].                                    */
/*   As kvd_decode_attn (sel_idx/sel_cnt/max_sel as there), or over every  */
/*   block when sel_idx is NULL (then sel_cnt and max_sel are ignored),     */
/*   except that, for each query head, the V term of position t is left out */
/*   of the numerator when                                                  */
/*     p_t < sparse_v_eps * mean_{u in c} p_u,   p_u = exp(s_u - max_c s)   */
/*   where c is t's chunk: the attended positions u with u / 16 == t / 16   */
/*   (a 16-token quarter of a 64-token block).  Every position stays in the */
/*   softmax denominator, so out_h = sum_{kept t} w_t v_t / sum_{all t} w_t */
/*   and the dropped share of sum_t w_t is below sparse_v_eps.              */
/*   sparse_v_eps = 0 gives kvd_decode_attn's (or the dense call's) output  */
/*   bit for bit; values above 16 drop every V term (out = 0).               */
/*   The comparison runs in f32 on the GPU: a position whose p_t lies within */
/*   rounding of the threshold may fall on either side.                     */
/* Errors: as kvd_decode_attn; INVALID also for a negative, NaN or infinite */
/* sparse_v_eps.                                                            */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_decode_attn_sv(const kvd_cache *cache, const float *q, int32_t n_heads,
                              float softmax_scale, const int32_t *sel_idx,
                              const int32_t *sel_cnt, int32_t max_sel, float sparse_v_eps,
                              float *out, void *workspace, size_t workspace_bytes,
                              void *stream);

/* ---------------------------------------------------------------------- */
/* Decode attention over the selected blocks plus the moment tail of every */
/* other block  [SCSA "2. Mechanism": a group that is not read exactly     */
/* contributes its count m times exp(a), a = softmax_scale * q . c_K, at   */
/* its value mean c_V, inside the shared normalizer; here the groups are   */
/* the Quest blocks the selection leaves out].                              */
/*   As kvd_decode_attn (same arguments), plus, for each query head h and   */
/*   each block j < NB = ceil(len / block) not listed in its row:           */
/*     term weight m_j * exp(softmax_scale * q_h . c_K(j)), value c_V(j)    */
/*   with m_j = min(block, len - j * block), c_K/c_V the f16 block means of */
/*   cache->moments, and q_h the f32 query (unquantized on every cache      */
/*   type).  out_h = (sum over listed tokens w_t v_t + sum over the other   */
/*   blocks of their terms) / (the same sum of weights).                    */
/*   Every listed row must be strictly ascending (as kvd_select_blocks      */
/*   writes it); otherwise a block may be counted both ways or not at all  */
/*   (wrong output, no fault).  Every row listing all NB blocks gives        */
/*   kvd_decode_attn's output bit for bit.                                   */
/*   Each launch reads all NB moment rows (512 bytes per block and KV head) */
/*   besides the listed blocks.                                              */
/* Errors: as kvd_decode_attn; INVALID also when cache->moments is NULL or  */
/* misaligned, or sel_idx/sel_cnt is NULL.                                  */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_decode_attn_tail(const kvd_cache *cache, const float *q,
                                int32_t n_heads, float softmax_scale,
                                const int32_t *sel_idx, const int32_t *sel_cnt,
                                int32_t max_sel, float *out, void *workspace,
                                size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* kvd_decode_attn without a workspace: the paper has no counterpart; this  */
/* is a convenience of this library.  Same arguments, arithmetic and output */
/* as kvd_decode_attn, minus workspace/workspace_bytes, for head_dim 128    */
/* only (the tuned kernels; other head dims return UNSUPPORTED).            */
/*   For callers that cannot allocate device memory when they decode: a    */
/*   plugin that an engine hands only its input and output buffers, or     */
/*   code whose device memory is owned by another allocator.  The split     */
/*   partials and arrival counters live in one array of                     */
/*   KVD_STATIC_SCRATCH_BYTES compiled into the library; every GPU that     */
/*   loads the library holds that array until the process exits.  The call */
/*   allocates nothing (no cudaMalloc/cudaFree, no library allocator).      */
/*   The first call on a device looks up the array's device address (once  */
/*   per device, with that device current); make that first call before    */
/*   any stream capture.  cudaDeviceReset drops that address: after a reset */
/*   of a device, do not call this entry point on it again in the same      */
/*   process.  Each call zeroes the counters on `stream` before             */
/*   its kernel.  All calls on a device share the array: two calls that    */
/*   may overlap on the GPU (different streams, no ordering) race and give  */
/*   wrong outputs; order them on one stream or with events.                */
/* Errors: as kvd_decode_attn (the same cache and head checks);             */
/* UNSUPPORTED for a head_dim other than 128; WORKSPACE when this call's     */
/* partials and counters would pass KVD_STATIC_SCRATCH_BYTES (on a 152-SM   */
/* GPU every accepted shape needs under 0.7 MiB, so WORKSPACE does not      */
/* occur there).                                                            */
/* ---------------------------------------------------------------------- */
#define KVD_STATIC_SCRATCH_BYTES (1u << 20)
KVD_API kvd_status kvd_decode_attn_static(const kvd_cache *cache, const float *q,
                                  int32_t n_heads, float softmax_scale,
                                  const int32_t *sel_idx, const int32_t *sel_cnt,
                                  int32_t max_sel, float *out, void *stream);

/* ---------------------------------------------------------------------- */
/* One whole decode step on device buffers: append one token per sequence */
/* (k_new, v_new: [batch, 1, n_kv_heads, head_dim] f16), then select and   */
/* attend over the len+1 cached tokens.  Equivalent to kvd_kv_append,      */
/* kvd_select_blocks and kvd_decode_attn in that order on `stream`; with   */
/* k_sel < 0 the attention is dense.  sel_idx/sel_cnt may be NULL, and then */
/* the selection lives in the workspace.  On KVD_OK cache->len has grown by */
/* one (also when a later launch failed with KVD_ERR_CUDA after the append */
/* was enqueued).                                                           */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_decode_step(kvd_cache *cache, const float *q, const void *k_new,
                           const void *v_new, int32_t n_heads, float softmax_scale,
                           int32_t k_sel, int32_t sink_tokens, int32_t recent_tokens,
                           int32_t *sel_idx, int32_t *sel_cnt, float *out,
                           void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* kvd_decode_step with HOST inputs and output: q_host ([batch, n_heads,   */
/* head_dim] f32), k_new_host/v_new_host ([batch, 1, n_kv_heads, head_dim] */
/* f16) in, out_host ([batch, n_heads, head_dim] f32) out, all enqueued on */
/* `stream`.  A buffer in page-locked host memory that CUDA maps into the  */
/* device's address space (16-byte aligned) is read or written in place by */
/* the kernels, over the host link; any other buffer is staged through    */
/* the workspace with cudaMemcpyAsync (pageable memory makes those copies   */
/* synchronous).  out_host is valid once the stream has finished, and the  */
/* host must not change the inputs before then.                             */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_decode_step_host(kvd_cache *cache, const float *q_host,
                                const void *k_new_host, const void *v_new_host,
                                int32_t n_heads, float softmax_scale, int32_t k_sel,
                                int32_t sink_tokens, int32_t recent_tokens,
                                int32_t *sel_idx, int32_t *sel_cnt, float *out_host,
                                void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* Workspace bytes that every call above needs for this cache geometry    */
/* (batch, n_kv_heads, max_seq, dtype) and n_heads query heads, for any   */
/* len <= max_seq and any selection.  One zero-filled workspace of this    */
/* size serves all the calls (they use disjoint regions: split partials,   */
/* per-problem arrival counters, selection keys, a selection for           */
/* kvd_decode_step when the caller passes none, and the host-step staging  */
/* buffers).  The split grid follows the current device's SM count, so    */
/* query it with the device that will run the calls current.  0 on        */
/* invalid arguments.                                                       */
/* ---------------------------------------------------------------------- */
KVD_API size_t kvd_workspace_bytes(const kvd_cache *cache, int32_t n_heads);

/* Blocks selected per (sequence, KV head) for a cache of len tokens:      */
/* forced sink and recent blocks plus min(k_sel, other blocks).  -1 on     */
/* invalid arguments.  Host only.                                          */
KVD_API int32_t kvd_selected_count(int32_t len, int32_t block, int32_t k_sel,
                           int32_t sink_tokens, int32_t recent_tokens);

/* Static description of a status code.  Host only. */
KVD_API const char *kvd_status_string(kvd_status status);

/* KVD_ABI_VERSION of the built library.  Host only. */
KVD_API int32_t kvd_abi_version(void);

/* ---------------------------------------------------------------------- */
/* Test exports: the exact integer q.k dots and the block bounds, computed */
/* by the same device routines the decode and select kernels use.         */
/*   kvd_debug_qk_int8: dots [batch, n_heads, len] int32, q_codes [batch,   */
/*   n_heads, head_dim] int8, q_scales [batch, n_heads] f32 (int8 cache     */
/*   only)  [CPUATT Method: integer logit dots, exact].                      */
/*   kvd_debug_scores: ub [batch, n_kv_heads, NB] f32, the group bound UB(j)*/
/*   of every block j < NB = ceil(len / block)  [QUEST Method].             */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_debug_qk_int8(const kvd_cache *cache, const float *q, int32_t n_heads,
                             int32_t *dots, int8_t *q_codes, float *q_scales, void *stream);
KVD_API kvd_status kvd_debug_scores(const kvd_cache *cache, const float *q, int32_t n_heads,
                            float *ub, void *stream);

/* ---------------------------------------------------------------------- */
/* Test export of the bounded-wait path: one kernel waits on an mbarrier    */
/* phase that nothing completes, gives up after limit_us microseconds of    */
/* wall time (the decode and selection kernels give up after 2 s), and      */
/* writes KVD_ERR_TIMEOUT to *dev_status (a device int32) unless it holds a */
/* code already.  The kernel then returns normally: the context stays       */
/* usable.  Errors: INVALID (dev_status NULL or misaligned, limit_us 0 or   */
/* above 1,000,000), CUDA.                                                  */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_debug_wait_timeout(int32_t *dev_status, int32_t limit_us, void *stream);

/* ---------------------------------------------------------------------- */
/* Profiling export (no counterpart on the pages): stage marks.  In a      */
/* library built with KVD_MARKS (build.py: environment KVD_MARKS=1) the    */
/* kernels write the GPU's global nanosecond timer at numbered points of   */
/* their work into `marks`, a caller-owned device buffer of at least       */
/* 3 * 4096 * 16 * 8 bytes (16-byte aligned): region k (0 selection,       */
/* 1 decode, 2 other kernels) holds 16 slots per CTA for up to 4096 CTAs,  */
/* numbered x-fastest.  Later launches write into it until it is replaced; */
/* marks = NULL turns recording off.  Host only; nothing is launched.      */
/* Errors: UNSUPPORTED in every build without marks (the default);         */
/* INVALID when the buffer is too small or misaligned.                     */
/* ---------------------------------------------------------------------- */
KVD_API kvd_status kvd_debug_stage_marks(void *marks, size_t bytes);

#ifdef __cplusplus
}
#endif
#endif /* KVDECODE_H */
