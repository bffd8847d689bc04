// append.cu -- KV append: copy (f16) or quantize (int8, q8_0, q4_0) the new
// rows, from f16 or f32 input, and fill the per-block key envelope (and the
// block means, when kept) in the same pass (append_dev.cuh).
//
// One warp per (sequence, KV head, touched block).
#include "append_dev.cuh"
#include "common.cuh"
#include "internal.h"

namespace kvd {
namespace {

constexpr int kAppendWarps = 4;

template <int DT, typename IN>
__global__ void __launch_bounds__(32 * kAppendWarps)
append_kernel(kvd_cache c, const IN *__restrict__ k_new, const IN *__restrict__ v_new,
              int n_new, int len0, int first_blk, int n_aff) {
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int a = blockIdx.x * kAppendWarps + warp;
    const int p = blockIdx.y;
    const int b = p / c.n_kv_heads;
    if (c.seq_lens) {  // this sequence's own position: its touched blocks
        len0 = seq_len_of(c.seq_lens, b, c.len, c.dev_status);
        first_blk = len0 / kBlock;
        n_aff = (len0 + n_new - 1) / kBlock - first_blk + 1;
    }
    if (a >= n_aff) return;
    append_block_warp<DT, true, IN>(c, k_new, v_new, n_new, len0, first_blk + a, b,
                                    p % c.n_kv_heads, lane);
}

template <typename IN>
cudaError_t launch_append_in(const kvd_cache &c, const void *k_new, const void *v_new,
                             int n_new, cudaStream_t st, bool pdl) {
    const int len0 = c.len;
    const int first = len0 / kBlock;
    const int last = (len0 + n_new - 1) / kBlock;
    // with per-sequence lengths a sequence's n_new rows touch at most this many
    const int n_aff = c.seq_lens ? (n_new + kBlock - 1) / kBlock + 1 : last - first + 1;
    dim3 grid((n_aff + kAppendWarps - 1) / kAppendWarps, c.batch * c.n_kv_heads);
    dim3 block(32 * kAppendWarps);
    const IN *kn = static_cast<const IN *>(k_new);
    const IN *vn = static_cast<const IN *>(v_new);
    if (c.dtype == KVD_F16)
        return launch_ex(append_kernel<KVD_F16, IN>, grid, block, 0, st, pdl, c, kn, vn, n_new,
                         len0, first, n_aff);
    if (c.dtype == KVD_Q8_0)
        return launch_ex(append_kernel<KVD_Q8_0, IN>, grid, block, 0, st, pdl, c, kn, vn, n_new,
                         len0, first, n_aff);
    if (c.dtype == KVD_Q4_0)
        return launch_ex(append_kernel<KVD_Q4_0, IN>, grid, block, 0, st, pdl, c, kn, vn, n_new,
                         len0, first, n_aff);
    return launch_ex(append_kernel<KVD_INT8, IN>, grid, block, 0, st, pdl, c, kn, vn, n_new,
                     len0, first, n_aff);
}

}  // namespace

cudaError_t launch_append(const kvd_cache &c, const void *k_new, const void *v_new, int n_new,
                          cudaStream_t st, bool pdl, bool f32_in) {
    return f32_in ? launch_append_in<float>(c, k_new, v_new, n_new, st, pdl)
                  : launch_append_in<__half>(c, k_new, v_new, n_new, st, pdl);
}

}  // namespace kvd
