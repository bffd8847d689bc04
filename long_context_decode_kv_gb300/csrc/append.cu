// append.cu -- KV append: copy (f16) or absmax-quantize (int8) the new rows
// and fill the per-block key envelope in the same pass (append_dev.cuh).
//
// One warp per (sequence, KV head, touched block).
#include "append_dev.cuh"
#include "common.cuh"
#include "internal.h"

namespace kvd {
namespace {

constexpr int kAppendWarps = 4;

template <int DT>
__global__ void __launch_bounds__(32 * kAppendWarps)
append_kernel(kvd_cache c, const __half *__restrict__ k_new, const __half *__restrict__ v_new,
              int n_new, int len0, int first_blk, int n_aff) {
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int a = blockIdx.x * kAppendWarps + warp;
    if (a >= n_aff) return;
    const int p = blockIdx.y;
    append_block_warp<DT>(c, k_new, v_new, n_new, len0, first_blk + a, p / c.n_kv_heads,
                          p % c.n_kv_heads, lane);
}

}  // namespace

cudaError_t launch_append(const kvd_cache &c, const void *k_new, const void *v_new, int n_new,
                          cudaStream_t st, bool pdl) {
    const int len0 = c.len;
    const int first = len0 / kBlock;
    const int last = (len0 + n_new - 1) / kBlock;
    const int n_aff = last - first + 1;
    dim3 grid((n_aff + kAppendWarps - 1) / kAppendWarps, c.batch * c.n_kv_heads);
    dim3 block(32 * kAppendWarps);
    const __half *kn = static_cast<const __half *>(k_new);
    const __half *vn = static_cast<const __half *>(v_new);
    if (c.dtype == KVD_F16)
        return launch_ex(append_kernel<KVD_F16>, grid, block, 0, st, pdl, c, kn, vn, n_new, len0,
                         first, n_aff);
    if (c.dtype == KVD_Q8_0)
        return launch_ex(append_kernel<KVD_Q8_0>, grid, block, 0, st, pdl, c, kn, vn, n_new,
                         len0, first, n_aff);
    if (c.dtype == KVD_Q4_0)
        return launch_ex(append_kernel<KVD_Q4_0>, grid, block, 0, st, pdl, c, kn, vn, n_new,
                         len0, first, n_aff);
    return launch_ex(append_kernel<KVD_INT8>, grid, block, 0, st, pdl, c, kn, vn, n_new, len0,
                     first, n_aff);
}

}  // namespace kvd
