// api.cu -- the extern "C" entry points of libkvdecode.so: argument checks on
// the host, workspace layout, and kernel dispatch on the caller's stream.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "internal.h"

namespace kvd {

int max_select_blocks();

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // 0: not asked yet

struct KernelKey {
    const void *fn;
    int dev;
    size_t smem;  // 0 in the table of attribute values
    bool operator==(const KernelKey &o) const {
        return fn == o.fn && dev == o.dev && smem == o.smem;
    }
};
struct KernelKeyHash {
    size_t operator()(const KernelKey &k) const {
        return std::hash<const void *>()(k.fn) ^ (static_cast<size_t>(k.dev) << 48) ^
               (k.smem << 20);
    }
};

}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 152;  // GB300
    }
    int sms = g_sm_count[dev].load(std::memory_order_relaxed);
    if (sms > 0) return sms;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0) {
        cudaGetLastError();
        return 152;
    }
    g_sm_count[dev].store(sms, std::memory_order_relaxed);  // every writer stores the same value
    return sms;
}

cudaError_t prepare_kernel(const void *fn, int threads, size_t smem, int *occ) {
    static std::mutex mu;
    // per (kernel, device): the largest dynamic shared memory opened so far
    // (the attribute is only raised, so a launch sized below it stays valid);
    // per (kernel, device, size): the occupancy
    static std::unordered_map<KernelKey, size_t, KernelKeyHash> opened;
    static std::unordered_map<KernelKey, int, KernelKeyHash> occupancy;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    size_t &top = opened[KernelKey{fn, dev, 0}];
    if (smem > top) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        top = smem;
    }
    const KernelKey key{fn, dev, smem};
    auto it = occupancy.find(key);
    if (it == occupancy.end()) {
        int o = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, fn, threads, smem);
        if (e != cudaSuccess) return e;
        it = occupancy.emplace(key, o > 0 ? o : 1).first;
    }
    if (occ) *occ = it->second;
    return cudaSuccess;
}

namespace {
std::atomic<unsigned long long *> g_marks{nullptr};
}  // namespace

unsigned long long *mark_region(int kind) {
#ifdef KVD_MARKS
    unsigned long long *m = g_marks.load(std::memory_order_relaxed);
    return m ? m + static_cast<size_t>(kind) * kMarkCtas * kMarkSlots : nullptr;
#else
    (void)kind;
    return nullptr;
#endif
}

namespace {
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) % 16) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) % 4) == 0; }
}  // namespace

kvd_status check_cache(const kvd_cache *c) {
    if (!c) return KVD_ERR_INVALID;
    if (c->dtype != KVD_F16 && c->dtype != KVD_INT8 && c->dtype != KVD_Q8_0 &&
        c->dtype != KVD_Q4_0)
        return KVD_ERR_INVALID;
    if (c->batch < 1 || c->n_kv_heads < 1) return KVD_ERR_INVALID;
    if (c->head_dim != kHeadDim) {
        // other head dims: multiples of 16 up to 1024, f16 and int8 caches,
        // without block means or per-sequence lengths
        if (c->head_dim < 16 || c->head_dim > 1024 || c->head_dim % 16 != 0)
            return KVD_ERR_UNSUPPORTED;
        if (c->dtype != KVD_F16 && c->dtype != KVD_INT8) return KVD_ERR_UNSUPPORTED;
        if (c->moments || c->seq_lens) return KVD_ERR_UNSUPPORTED;
    }
    if (c->block != kBlock) return KVD_ERR_UNSUPPORTED;
    if (c->max_seq < kBlock || c->max_seq % kBlock != 0) return KVD_ERR_INVALID;
    if (c->len < 0 || c->len > c->max_seq) return KVD_ERR_INVALID;
    if (c->reserved != 0) return KVD_ERR_INVALID;
    const void *ptrs[3] = {c->k, c->v, c->kbounds};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return KVD_ERR_INVALID;
    if (c->dtype != KVD_F16) {
        if (!c->k_scale || !c->v_scale || !aligned16(c->k_scale) || !aligned16(c->v_scale))
            return KVD_ERR_INVALID;
    }
    if (c->dev_status && !aligned4(c->dev_status)) return KVD_ERR_INVALID;
    if (c->moments && !aligned16(c->moments)) return KVD_ERR_INVALID;
    if (c->seq_lens && !aligned4(c->seq_lens)) return KVD_ERR_INVALID;
    if (static_cast<long long>(c->batch) * c->n_kv_heads * 16 > 65535) return KVD_ERR_UNSUPPORTED;
    return KVD_OK;
}

kvd_status check_heads(const kvd_cache *c, int n_heads) {
    if (n_heads < 1 || n_heads % c->n_kv_heads != 0) return KVD_ERR_INVALID;
    const int G = n_heads / c->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return KVD_ERR_UNSUPPORTED;
    return KVD_OK;
}

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A head dim the general kernels serve (the tuned ones take 128).
bool general_d(const kvd_cache *c) { return c->head_dim != kHeadDim; }

Geom make_geom(const kvd_cache *c, int n_heads, int len) {
    Geom g;
    g.dtype = c->dtype;
    g.B = c->batch;
    g.Hkv = c->n_kv_heads;
    g.max_seq = c->max_seq;
    g.len = len;
    g.H = n_heads;
    g.G = n_heads / c->n_kv_heads;
    g.NB = (len + kBlock - 1) / kBlock;
    g.nbmax = c->max_seq / kBlock;
    g.seq_add = 0;
    return g;
}

// Workspace regions (byte offsets; every region 256-byte aligned).
struct WsLayout {
    size_t counters, partials, keys, sel_range, sel_ticket, sel_idx, sel_cnt, q, k_new, v_new,
        out, total;
    int range_rows;
    DecodePlan plan;
};

WsLayout ws_layout(const kvd_cache *c, int n_heads) {
    WsLayout w;
    const Geom g = make_geom(c, n_heads, c->max_seq);
    // splits never exceed the plan for a selection of every block
    w.plan = plan_decode(g, g.nbmax, device_sm_count());
    const size_t P = static_cast<size_t>(g.B) * g.Hkv;
    size_t off = 0;
    w.counters = off;  // one per query head: enough for one-head-per-CTA plans too
    off += align_up(static_cast<size_t>(g.B) * g.H * sizeof(uint32_t));
    const size_t D = static_cast<size_t>(c->head_dim);
    w.partials = off;
    off += align_up(general_d(c) ? gd_partials_bytes(static_cast<int>(P), g.G, c->head_dim,
                                                     gd_splits(static_cast<int>(P), g.nbmax,
                                                               device_sm_count(), 0))
                                 : decode_partials_bytes(g, w.plan));
    w.keys = off;  // key rows padded to 16 bytes
    off += align_up(P * ((g.nbmax + 3) / 4 * 4) * sizeof(uint32_t));
    // key ranges and tickets: only problems split over several CTAs use
    // them, and there are fewer of those than 2 * SMs
    const size_t sms = static_cast<size_t>(device_sm_count());
    const size_t hrows = P < 2 * sms ? P : 2 * sms;
    w.range_rows = static_cast<int>(hrows);
    w.sel_range = off;
    off += align_up(hrows * 2 * sizeof(unsigned));
    w.sel_ticket = off;
    off += align_up(hrows * sizeof(unsigned));
    w.sel_idx = off;
    off += align_up(P * g.nbmax * sizeof(int32_t));
    w.sel_cnt = off;
    off += align_up(P * sizeof(int32_t));
    w.q = off;
    off += align_up(static_cast<size_t>(g.B) * g.H * D * sizeof(float));
    w.k_new = off;
    off += align_up(P * D * sizeof(__half));
    w.v_new = off;
    off += align_up(P * D * sizeof(__half));
    w.out = off;
    off += align_up(static_cast<size_t>(g.B) * g.H * D * sizeof(float));
    w.total = off;
    return w;
}

kvd_status check_ws(void *ws, size_t bytes, size_t need) {
    if (!ws || !aligned(ws, kAlign) || bytes < need) return KVD_ERR_WORKSPACE;
    return KVD_OK;
}

template <typename T>
T *ws_at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

kvd_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVD_OK : KVD_ERR_CUDA; }

void forced_range(int len, int sink, int recent, int *se, int *rb) {
    const int NB = (len + kBlock - 1) / kBlock;
    int s = (sink + kBlock - 1) / kBlock;
    if (s > NB) s = NB;
    int r = NB;
    if (recent > 0) {
        long start = static_cast<long>(len) - recent;
        if (start < 0) start = 0;
        r = static_cast<int>(start / kBlock);
    }
    if (r < s) r = s;
    *se = s;
    *rb = r;
}

SelScratch sel_scratch(void *ws, const WsLayout &w) {
    SelScratch scr;
    scr.keys = ws_at<uint32_t>(ws, w.keys);
    scr.range = ws_at<unsigned>(ws, w.sel_range);
    scr.ticket = ws_at<unsigned>(ws, w.sel_ticket);
    scr.range_rows = w.range_rows;
    return scr;
}

// tok: inside a decode step, the token to append first (c->len already counts it)
kvd_status select_impl(const kvd_cache *c, const float *q, int n_heads, int k_sel, int sink,
                       int recent, int32_t *sel_idx, int32_t *sel_cnt, void *ws,
                       const WsLayout &w, cudaStream_t st, const StepToken *tok = nullptr) {
    if (general_d(c)) {
        if (tok && launch_append_gd(*c, tok->k_new, tok->v_new, 1, tok->len0, st, false) !=
                       cudaSuccess)
            return KVD_ERR_CUDA;
        int se, rb;
        forced_range(c->len, sink, recent, &se, &rb);
        return cuda_status(launch_select_gd(*c, q, n_heads, k_sel, se, rb, sel_idx, sel_cnt,
                                            ws_at<uint32_t>(ws, w.keys), st));
    }
    Geom g = make_geom(c, n_heads, c->len);
    g.seq_add = tok ? 1 : 0;  // a step's token: seq_lens does not count it yet
    const SelScratch scr = sel_scratch(ws, w);
    return cuda_status(launch_select(*c, g, q, k_sel, sink, recent, sel_idx, sel_cnt, scr, st,
                                     true, tok));
}

kvd_status decode_impl(const kvd_cache *c, const float *q, int n_heads, float scale,
                       const int32_t *sel_idx, const int32_t *sel_cnt, int max_sel, float *out,
                       void *ws, const WsLayout &w, cudaStream_t st, bool in_step = false,
                       float sv_eps = 0.0f) {
    Geom g = make_geom(c, n_heads, c->len);
    g.seq_add = in_step ? 1 : 0;  // the step's token: seq_lens does not count it yet
    const bool dense = sel_idx == nullptr;
    int max_blocks = dense ? g.NB : max_sel;
    if (max_blocks > g.NB) max_blocks = g.NB;
    if (max_blocks < 1) max_blocks = 1;
    if (general_d(c)) {
        if (sv_eps > 0.0f) return KVD_ERR_UNSUPPORTED;
        return cuda_status(launch_decode_gd(*c, q, n_heads, scale, sel_idx, sel_cnt, max_blocks,
                                            out, ws_at<float>(ws, w.partials),
                                            ws_at<uint32_t>(ws, w.counters), st));
    }
    // the wide tile for listed blocks only: over every block (a long stream) the
    // two-CTA tile keeps two producers per SM and streams faster
    const DecodePlan p = plan_decode(g, max_blocks, device_sm_count(), false, !dense);
    return cuda_status(launch_decode(*c, g, p, q, scale, sel_idx, sel_cnt, out,
                                     ws_at<float>(ws, w.partials),
                                     ws_at<uint32_t>(ws, w.counters), st, true, in_step,
                                     sv_eps));
}

// The listed blocks plus the moment tail of the others.  The split grid is
// planned for the larger of the two streams: the listed blocks, or the
// moment rows counted as one block per 32 rows (about the same bytes).
kvd_status decode_tail_impl(const kvd_cache *c, const float *q, int n_heads, float scale,
                            const int32_t *sel_idx, const int32_t *sel_cnt, int max_sel,
                            float *out, void *ws, const WsLayout &w, cudaStream_t st) {
    const Geom g = make_geom(c, n_heads, c->len);
    int max_blocks = max_sel < g.NB ? max_sel : g.NB;
    if (max_blocks < 1) max_blocks = 1;
    const int tail_work = (g.NB + 31) / 32;
    DecodePlan p = plan_decode(g, max_blocks > tail_work ? max_blocks : tail_work,
                               device_sm_count(), false, true);
    p.blocks = max_blocks;
    return cuda_status(launch_decode_tail(*c, g, p, q, scale, sel_idx, sel_cnt, out,
                                          ws_at<float>(ws, w.partials),
                                          ws_at<uint32_t>(ws, w.counters), st, true));
}

// Lists per query head (an ablation of the GQA-shared selection).
kvd_status decode_per_head_impl(const kvd_cache *c, const float *q, int n_heads, float scale,
                                const int32_t *sel_idx, const int32_t *sel_cnt, int max_sel,
                                float *out, void *ws, const WsLayout &w, cudaStream_t st) {
    const Geom g = make_geom(c, n_heads, c->len);
    int max_blocks = max_sel < g.NB ? max_sel : g.NB;
    if (max_blocks < 1) max_blocks = 1;
    const DecodePlan p = plan_decode(g, max_blocks, device_sm_count(), true, true);
    return cuda_status(launch_decode_per_head(*c, g, p, q, scale, sel_idx, sel_cnt, out,
                                              ws_at<float>(ws, w.partials),
                                              ws_at<uint32_t>(ws, w.counters), st, true));
}

kvd_status check_select_args(const kvd_cache *c, int n_heads, int k_sel, int sink, int recent) {
    kvd_status s = check_cache(c);
    if (s != KVD_OK) return s;
    if ((s = check_heads(c, n_heads)) != KVD_OK) return s;
    if (c->len < 1 || k_sel < 0 || sink < 0 || recent < 0) return KVD_ERR_INVALID;
    if ((c->len + kBlock - 1) / kBlock > max_select_blocks()) return KVD_ERR_UNSUPPORTED;
    return KVD_OK;
}

}  // namespace
}  // namespace kvd

using namespace kvd;

extern "C" {

int32_t kvd_abi_version(void) { return KVD_ABI_VERSION; }

const char *kvd_status_string(kvd_status s) {
    switch (s) {
        case KVD_OK: return "ok";
        case KVD_ERR_INVALID: return "invalid argument";
        case KVD_ERR_UNSUPPORTED: return "unsupported configuration";
        case KVD_ERR_CAPACITY: return "append would pass max_seq";
        case KVD_ERR_CUDA: return "CUDA runtime error";
        case KVD_ERR_TIMEOUT: return "device wait timed out";
        case KVD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        default: return "unknown status";
    }
}

int32_t kvd_selected_count(int32_t len, int32_t block, int32_t k_sel, int32_t sink_tokens,
                           int32_t recent_tokens) {
    if (len < 1 || block != kBlock || k_sel < 0 || sink_tokens < 0 || recent_tokens < 0)
        return -1;
    int se, rb;
    forced_range(len, sink_tokens, recent_tokens, &se, &rb);
    const int NB = (len + kBlock - 1) / kBlock;
    const int n_cand = rb - se;
    return (NB - n_cand) + (k_sel < n_cand ? k_sel : n_cand);
}

size_t kvd_workspace_bytes(const kvd_cache *cache, int32_t n_heads) {
    if (check_cache(cache) != KVD_OK || check_heads(cache, n_heads) != KVD_OK) return 0;
    return ws_layout(cache, n_heads).total;
}

}  // extern "C"

namespace {

kvd_status append_impl(kvd_cache *cache, const void *k_new, const void *v_new, int32_t n_new,
                       void *stream, bool f32_in) {
    kvd_status s = check_cache(cache);
    if (s != KVD_OK) return s;
    if (n_new < 0) return KVD_ERR_INVALID;
    if (n_new == 0) return KVD_OK;
    if (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)) return KVD_ERR_INVALID;
    if (static_cast<long long>(cache->len) + n_new > cache->max_seq) return KVD_ERR_CAPACITY;
    const cudaError_t e =
        general_d(cache)
            ? launch_append_gd(*cache, k_new, v_new, n_new, cache->len,
                               static_cast<cudaStream_t>(stream), f32_in)
            : launch_append(*cache, k_new, v_new, n_new, static_cast<cudaStream_t>(stream), true,
                            f32_in);
    if (e != cudaSuccess) return KVD_ERR_CUDA;
    cache->len += n_new;
    return KVD_OK;
}

}  // namespace

extern "C" {

kvd_status kvd_kv_append(kvd_cache *cache, const void *k_new, const void *v_new, int32_t n_new,
                         void *stream) {
    return append_impl(cache, k_new, v_new, n_new, stream, false);
}

kvd_status kvd_kv_append_f32(kvd_cache *cache, const float *k_new, const float *v_new,
                             int32_t n_new, void *stream) {
    return append_impl(cache, k_new, v_new, n_new, stream, true);
}

kvd_status kvd_select_blocks(const kvd_cache *cache, const float *q, int32_t n_heads,
                             int32_t k_sel, int32_t sink_tokens, int32_t recent_tokens,
                             int32_t *sel_idx, int32_t *sel_cnt, void *workspace,
                             size_t workspace_bytes, void *stream) {
    kvd_status s = check_select_args(cache, n_heads, k_sel, sink_tokens, recent_tokens);
    if (s != KVD_OK) return s;
    if (!q || !aligned(q, 16) || !sel_idx || !aligned(sel_idx, 4) || !sel_cnt ||
        !aligned(sel_cnt, 4))
        return KVD_ERR_INVALID;
    const WsLayout w = ws_layout(cache, n_heads);
    if ((s = check_ws(workspace, workspace_bytes, w.total)) != KVD_OK) return s;
    return select_impl(cache, q, n_heads, k_sel, sink_tokens, recent_tokens, sel_idx, sel_cnt,
                       workspace, w, static_cast<cudaStream_t>(stream));
}

kvd_status kvd_decode_attn(const kvd_cache *cache, const float *q, int32_t n_heads,
                           float softmax_scale, const int32_t *sel_idx, const int32_t *sel_cnt,
                           int32_t max_sel, float *out, void *workspace, size_t workspace_bytes,
                           void *stream) {
    kvd_status s = check_cache(cache);
    if (s != KVD_OK) return s;
    if ((s = check_heads(cache, n_heads)) != KVD_OK) return s;
    if (cache->len < 1 || max_sel < 0) return KVD_ERR_INVALID;
    if (!q || !aligned(q, 16) || !out || !aligned(out, 16)) return KVD_ERR_INVALID;
    if (!sel_idx || !aligned(sel_idx, 4) || !sel_cnt || !aligned(sel_cnt, 4))
        return KVD_ERR_INVALID;
    const WsLayout w = ws_layout(cache, n_heads);
    if ((s = check_ws(workspace, workspace_bytes, w.total)) != KVD_OK) return s;
    return decode_impl(cache, q, n_heads, softmax_scale, sel_idx, sel_cnt, max_sel, out,
                       workspace, w, static_cast<cudaStream_t>(stream));
}

kvd_status kvd_decode_attn_sv(const kvd_cache *cache, const float *q, int32_t n_heads,
                              float softmax_scale, const int32_t *sel_idx,
                              const int32_t *sel_cnt, int32_t max_sel, float sparse_v_eps,
                              float *out, void *workspace, size_t workspace_bytes,
                              void *stream) {
    kvd_status s = check_cache(cache);
    if (s != KVD_OK) return s;
    if ((s = check_heads(cache, n_heads)) != KVD_OK) return s;
    if (cache->len < 1) return KVD_ERR_INVALID;
    if (!(sparse_v_eps >= 0.0f) || !std::isfinite(sparse_v_eps)) return KVD_ERR_INVALID;
    if (!q || !aligned(q, 16) || !out || !aligned(out, 16)) return KVD_ERR_INVALID;
    if (sel_idx) {
        if (max_sel < 0 || !aligned(sel_idx, 4) || !sel_cnt || !aligned(sel_cnt, 4))
            return KVD_ERR_INVALID;
    }
    const WsLayout w = ws_layout(cache, n_heads);
    if ((s = check_ws(workspace, workspace_bytes, w.total)) != KVD_OK) return s;
    return decode_impl(cache, q, n_heads, softmax_scale, sel_idx, sel_idx ? sel_cnt : nullptr,
                       sel_idx ? max_sel : 0, out, workspace, w,
                       static_cast<cudaStream_t>(stream), false, sparse_v_eps);
}

kvd_status kvd_select_blocks_per_head(const kvd_cache *cache, const float *q, int32_t n_heads,
                                      int32_t k_sel, int32_t sink_tokens,
                                      int32_t recent_tokens, int32_t *sel_idx,
                                      int32_t *sel_cnt, void *workspace, size_t workspace_bytes,
                                      void *stream) {
    kvd_status s = check_select_args(cache, n_heads, k_sel, sink_tokens, recent_tokens);
    if (s != KVD_OK) return s;
    if (general_d(cache)) return KVD_ERR_UNSUPPORTED;  // per-head lists: D = 128 only
    if (!q || !aligned(q, 16)) return KVD_ERR_INVALID;
    if (!sel_idx || !aligned(sel_idx, 4) || !sel_cnt || !aligned(sel_cnt, 4))
        return KVD_ERR_INVALID;
    const WsLayout w = ws_layout(cache, n_heads);
    if ((s = check_ws(workspace, workspace_bytes, w.total)) != KVD_OK) return s;
    const Geom g = make_geom(cache, n_heads, cache->len);
    return cuda_status(launch_select_per_head(*cache, g, q, k_sel, sink_tokens, recent_tokens,
                                              sel_idx, sel_cnt, sel_scratch(workspace, w),
                                              static_cast<cudaStream_t>(stream), true));
}

kvd_status kvd_decode_attn_per_head(const kvd_cache *cache, const float *q, int32_t n_heads,
                                    float softmax_scale, const int32_t *sel_idx,
                                    const int32_t *sel_cnt, int32_t max_sel, float *out,
                                    void *workspace, size_t workspace_bytes, void *stream) {
    kvd_status s = check_cache(cache);
    if (s != KVD_OK) return s;
    if ((s = check_heads(cache, n_heads)) != KVD_OK) return s;
    if (general_d(cache)) return KVD_ERR_UNSUPPORTED;  // per-head lists: D = 128 only
    if (cache->len < 1 || max_sel < 0) return KVD_ERR_INVALID;
    if (!q || !aligned(q, 16) || !out || !aligned(out, 16)) return KVD_ERR_INVALID;
    if (!sel_idx || !aligned(sel_idx, 4) || !sel_cnt || !aligned(sel_cnt, 4))
        return KVD_ERR_INVALID;
    const WsLayout w = ws_layout(cache, n_heads);
    if ((s = check_ws(workspace, workspace_bytes, w.total)) != KVD_OK) return s;
    return decode_per_head_impl(cache, q, n_heads, softmax_scale, sel_idx, sel_cnt, max_sel,
                                out, workspace, w, static_cast<cudaStream_t>(stream));
}

kvd_status kvd_decode_attn_tail(const kvd_cache *cache, const float *q, int32_t n_heads,
                                float softmax_scale, const int32_t *sel_idx,
                                const int32_t *sel_cnt, int32_t max_sel, float *out,
                                void *workspace, size_t workspace_bytes, void *stream) {
    kvd_status s = check_cache(cache);
    if (s != KVD_OK) return s;
    if ((s = check_heads(cache, n_heads)) != KVD_OK) return s;
    if (general_d(cache)) return KVD_ERR_UNSUPPORTED;  // block means: D = 128 only
    if (cache->len < 1 || max_sel < 0 || !cache->moments) return KVD_ERR_INVALID;
    if (!q || !aligned(q, 16) || !out || !aligned(out, 16)) return KVD_ERR_INVALID;
    if (!sel_idx || !aligned(sel_idx, 4) || !sel_cnt || !aligned(sel_cnt, 4))
        return KVD_ERR_INVALID;
    const WsLayout w = ws_layout(cache, n_heads);
    if ((s = check_ws(workspace, workspace_bytes, w.total)) != KVD_OK) return s;
    return decode_tail_impl(cache, q, n_heads, softmax_scale, sel_idx, sel_cnt, max_sel, out,
                            workspace, w, static_cast<cudaStream_t>(stream));
}

kvd_status kvd_decode_attn_dense(const kvd_cache *cache, const float *q, int32_t n_heads,
                                 float softmax_scale, float *out, void *workspace,
                                 size_t workspace_bytes, void *stream) {
    kvd_status s = check_cache(cache);
    if (s != KVD_OK) return s;
    if ((s = check_heads(cache, n_heads)) != KVD_OK) return s;
    if (cache->len < 1) return KVD_ERR_INVALID;
    if (!q || !aligned(q, 16) || !out || !aligned(out, 16)) return KVD_ERR_INVALID;
    const WsLayout w = ws_layout(cache, n_heads);
    if ((s = check_ws(workspace, workspace_bytes, w.total)) != KVD_OK) return s;
    return decode_impl(cache, q, n_heads, softmax_scale, nullptr, nullptr, 0, out, workspace, w,
                       static_cast<cudaStream_t>(stream));
}

kvd_status kvd_decode_step(kvd_cache *cache, const float *q, const void *k_new,
                           const void *v_new, int32_t n_heads, float softmax_scale,
                           int32_t k_sel, int32_t sink_tokens, int32_t recent_tokens,
                           int32_t *sel_idx, int32_t *sel_cnt, float *out, void *workspace,
                           size_t workspace_bytes, void *stream) {
    kvd_status s = check_cache(cache);
    if (s != KVD_OK) return s;
    if ((s = check_heads(cache, n_heads)) != KVD_OK) return s;
    if (!q || !aligned(q, 16) || !out || !aligned(out, 16)) return KVD_ERR_INVALID;
    if (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)) return KVD_ERR_INVALID;
    if (cache->len + 1 > cache->max_seq) return KVD_ERR_CAPACITY;
    const bool dense = k_sel < 0;
    if (!dense) {
        if (sink_tokens < 0 || recent_tokens < 0) return KVD_ERR_INVALID;
        if ((cache->len + 1 + kBlock - 1) / kBlock > max_select_blocks())
            return KVD_ERR_UNSUPPORTED;
        if ((sel_idx && !aligned(sel_idx, 4)) || (sel_cnt && !aligned(sel_cnt, 4)))
            return KVD_ERR_INVALID;
    }
    const WsLayout w = ws_layout(cache, n_heads);
    if ((s = check_ws(workspace, workspace_bytes, w.total)) != KVD_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dense) {
        const cudaError_t e = general_d(cache)
                                  ? launch_append_gd(*cache, k_new, v_new, 1, cache->len, st, false)
                                  : launch_append(*cache, k_new, v_new, 1, st, true);
        if (e != cudaSuccess) return KVD_ERR_CUDA;
        cache->len += 1;
        return decode_impl(cache, q, n_heads, softmax_scale, nullptr, nullptr, 0, out, workspace,
                           w, st, true);
    }
    if (!sel_idx) sel_idx = ws_at<int32_t>(workspace, w.sel_idx);
    if (!sel_cnt) sel_cnt = ws_at<int32_t>(workspace, w.sel_cnt);
    // the selection appends the token (in its own kernel when the token's
    // block is forced, else by an append launch just before)
    const StepToken tok = {k_new, v_new, cache->len};
    cache->len += 1;
    s = select_impl(cache, q, n_heads, k_sel, sink_tokens, recent_tokens, sel_idx, sel_cnt,
                    workspace, w, st, &tok);
    if (s != KVD_OK) {
        cache->len -= 1;
        return s;
    }
    const int max_sel =
        kvd_selected_count(cache->len, kBlock, k_sel, sink_tokens, recent_tokens);
    return decode_impl(cache, q, n_heads, softmax_scale, sel_idx, sel_cnt, max_sel, out,
                       workspace, w, st, true);
}

}  // extern "C"

namespace kvd {
namespace {

// The device-side address of host buffer p when the GPU can reach it
// directly: pinned host memory mapped into the device's address space (on a
// Grace host the kernels then read and write it over the chip-to-chip link).
// nullptr for pageable or unknown memory, or an address not 16-byte aligned.
void *device_view(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();  // not a CUDA-known pointer: clear the error
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
    return aligned(at.devicePointer, 16) ? at.devicePointer : nullptr;
}

}  // namespace
}  // namespace kvd

extern "C" {

kvd_status kvd_decode_step_host(kvd_cache *cache, const float *q_host, const void *k_new_host,
                                const void *v_new_host, int32_t n_heads, float softmax_scale,
                                int32_t k_sel, int32_t sink_tokens, int32_t recent_tokens,
                                int32_t *sel_idx, int32_t *sel_cnt, float *out_host,
                                void *workspace, size_t workspace_bytes, void *stream) {
    kvd_status s = check_cache(cache);
    if (s != KVD_OK) return s;
    if ((s = check_heads(cache, n_heads)) != KVD_OK) return s;
    if (!q_host || !k_new_host || !v_new_host || !out_host) return KVD_ERR_INVALID;
    const WsLayout w = ws_layout(cache, n_heads);
    if ((s = check_ws(workspace, workspace_bytes, w.total)) != KVD_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t qb = static_cast<size_t>(cache->batch) * n_heads * cache->head_dim * sizeof(float);
    const size_t kb = static_cast<size_t>(cache->batch) * cache->n_kv_heads * cache->head_dim * 2;
    // Buffers the GPU can reach directly are used in place by the kernels;
    // the others are staged through the workspace by copies on the stream.
    float *q_dev = static_cast<float *>(device_view(q_host));
    void *k_dev = device_view(k_new_host);
    void *v_dev = device_view(v_new_host);
    float *o_map = static_cast<float *>(device_view(out_host));
    if (!q_dev) {
        q_dev = ws_at<float>(workspace, w.q);
        if (cudaMemcpyAsync(q_dev, q_host, qb, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return KVD_ERR_CUDA;
    }
    if (!k_dev) {
        k_dev = ws_at<void>(workspace, w.k_new);
        if (cudaMemcpyAsync(k_dev, k_new_host, kb, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return KVD_ERR_CUDA;
    }
    if (!v_dev) {
        v_dev = ws_at<void>(workspace, w.v_new);
        if (cudaMemcpyAsync(v_dev, v_new_host, kb, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return KVD_ERR_CUDA;
    }
    float *o_dev = o_map ? o_map : ws_at<float>(workspace, w.out);
    s = kvd_decode_step(cache, q_dev, k_dev, v_dev, n_heads, softmax_scale, k_sel, sink_tokens,
                        recent_tokens, sel_idx, sel_cnt, o_dev, workspace, workspace_bytes,
                        stream);
    if (s != KVD_OK) return s;
    if (!o_map &&
        cudaMemcpyAsync(out_host, o_dev, qb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return KVD_ERR_CUDA;
    return KVD_OK;
}

kvd_status kvd_debug_qk_int8(const kvd_cache *cache, const float *q, int32_t n_heads,
                             int32_t *dots, int8_t *q_codes, float *q_scales, void *stream) {
    kvd_status s = check_cache(cache);
    if (s != KVD_OK) return s;
    if ((s = check_heads(cache, n_heads)) != KVD_OK) return s;
    if (general_d(cache)) return KVD_ERR_UNSUPPORTED;  // the tuned decode only
    if (cache->dtype != KVD_INT8 || cache->len < 1) return KVD_ERR_INVALID;
    if (!q || !aligned(q, 16) || !dots || !aligned(dots, 4) || !q_codes ||
        !aligned(q_codes, 4) || !q_scales || !aligned(q_scales, 4))
        return KVD_ERR_INVALID;
    const Geom g = make_geom(cache, n_heads, cache->len);
    return cuda_status(launch_qk_debug(*cache, g, q, dots, q_codes, q_scales,
                                       static_cast<cudaStream_t>(stream)));
}

kvd_status kvd_debug_stage_marks(void *marks, size_t bytes) {
#ifdef KVD_MARKS
    const size_t need = static_cast<size_t>(kMarkKinds) * kMarkCtas * kMarkSlots * 8;
    if (marks && (bytes < need || !aligned16(marks))) return KVD_ERR_INVALID;
    g_marks.store(static_cast<unsigned long long *>(marks), std::memory_order_relaxed);
    return KVD_OK;
#else
    (void)marks;
    (void)bytes;
    return KVD_ERR_UNSUPPORTED;
#endif
}

kvd_status kvd_debug_wait_timeout(int32_t *dev_status, int32_t limit_us, void *stream) {
    if (!dev_status || !aligned(dev_status, 4)) return KVD_ERR_INVALID;
    if (limit_us < 1 || limit_us > 1000000) return KVD_ERR_INVALID;
    return cuda_status(launch_wait_probe(dev_status, static_cast<uint64_t>(limit_us) * 1000u,
                                         static_cast<cudaStream_t>(stream)));
}

kvd_status kvd_debug_scores(const kvd_cache *cache, const float *q, int32_t n_heads, float *ub,
                            void *stream) {
    kvd_status s = check_cache(cache);
    if (s != KVD_OK) return s;
    if (cache->seq_lens) return KVD_ERR_UNSUPPORTED;
    if ((s = check_heads(cache, n_heads)) != KVD_OK) return s;
    if (general_d(cache)) return KVD_ERR_UNSUPPORTED;  // the tuned scorer only
    if (cache->len < 1) return KVD_ERR_INVALID;
    if (!q || !aligned(q, 16) || !ub || !aligned(ub, 4)) return KVD_ERR_INVALID;
    const Geom g = make_geom(cache, n_heads, cache->len);
    return cuda_status(launch_scores_debug(*cache, g, q, ub, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
