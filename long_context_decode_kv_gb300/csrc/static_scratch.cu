// static_scratch.cu -- kvd_decode_attn_static: the split-KV decode of
// kvd_decode_attn with its scratch (split partials and per-problem arrival
// counters) held in a fixed device array inside the library, so the caller
// passes no workspace and nothing is allocated per call.
//
// Why it exists: some callers cannot allocate device memory when they call
// the decode -- a plugin inside a host engine that hands it only the input and
// output buffers and owns every allocation itself, or code running where a
// cudaMalloc would synchronize the device or fail because the memory pool is
// already carved up.  They pay with a fixed KVD_STATIC_SCRATCH_BYTES on every
// GPU that loads the library, and with one rule: calls that share the array
// must not run at the same time on the GPU.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace kvd {
namespace {

static_assert(KVD_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte regions");

// Shared by every kvd_decode_attn_static call on a device; each GPU that
// loads the library holds it until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[KVD_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};  // device address, per device ordinal (under the lock)

// In host code g_static_scratch names a host-side stand-in; the array's device
// address is asked of the runtime once per device, with that device current.
// cudaDeviceReset on a device drops the module holding the array, so the
// address kept here is then stale: a process that resets a device must not
// call this entry point on it again.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

bool aligned_to(const void *p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// The argument rules of kvd_decode_attn (the same cache and head checks),
// minus the workspace; only the tuned head dim (128) is served here.
kvd_status check_args(const kvd_cache *c, const float *q, int n_heads, const int32_t *sel_idx,
                      const int32_t *sel_cnt, int max_sel, const float *out) {
    kvd_status s = check_cache(c);
    if (s != KVD_OK) return s;
    if ((s = check_heads(c, n_heads)) != KVD_OK) return s;
    if (c->head_dim != kHeadDim) return KVD_ERR_UNSUPPORTED;
    if (c->len < 1 || max_sel < 0) return KVD_ERR_INVALID;
    if (!q || !aligned_to(q, 16) || !out || !aligned_to(out, 16)) return KVD_ERR_INVALID;
    if (!sel_idx || !aligned_to(sel_idx, 4) || !sel_cnt || !aligned_to(sel_cnt, 4))
        return KVD_ERR_INVALID;
    return KVD_OK;
}

}  // namespace
}  // namespace kvd

using namespace kvd;

extern "C" kvd_status kvd_decode_attn_static(const kvd_cache *cache, const float *q,
                                             int32_t n_heads, float softmax_scale,
                                             const int32_t *sel_idx, const int32_t *sel_cnt,
                                             int32_t max_sel, float *out, void *stream) {
    const kvd_status s = check_args(cache, q, n_heads, sel_idx, sel_cnt, max_sel, out);
    if (s != KVD_OK) return s;

    Geom g;
    g.dtype = cache->dtype;
    g.B = cache->batch;
    g.Hkv = cache->n_kv_heads;
    g.max_seq = cache->max_seq;
    g.len = cache->len;
    g.H = n_heads;
    g.G = n_heads / cache->n_kv_heads;
    g.NB = (cache->len + kBlock - 1) / kBlock;
    g.nbmax = cache->max_seq / kBlock;
    g.seq_add = 0;
    int max_blocks = max_sel < g.NB ? max_sel : g.NB;
    if (max_blocks < 1) max_blocks = 1;
    const DecodePlan p = plan_decode(g, max_blocks, device_sm_count(), false, true);
    const size_t counter_bytes =
        round256(static_cast<size_t>(g.B) * g.Hkv * p.subgroups * sizeof(uint32_t));
    if (counter_bytes + decode_partials_bytes(g, p) > KVD_STATIC_SCRATCH_BYTES)
        return KVD_ERR_WORKSPACE;

    void *base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return KVD_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The array holds what the last call left there; the arrival counters must
    // start at zero (the partials are written before they are read).
    if (cudaMemsetAsync(base, 0, counter_bytes, st) != cudaSuccess) return KVD_ERR_CUDA;
    uint32_t *counters = static_cast<uint32_t *>(base);
    float *partials = reinterpret_cast<float *>(static_cast<unsigned char *>(base) + counter_bytes);
    const cudaError_t e = launch_decode(*cache, g, p, q, softmax_scale, sel_idx, sel_cnt, out,
                                        partials, counters, st, false, false);
    return e == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}
