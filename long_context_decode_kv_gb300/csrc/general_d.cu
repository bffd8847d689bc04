// general_d.cu -- append and block selection for head dims other than 128.
//
// "cpu-attn", Requirements and limits: the head dim may be any multiple of 16
// up to 1024.  The tuned kernels give every lane of a warp 4 of 128
// channels; these loop over the channels of a row instead, for the f16 and
// int8 caches (the group-quantized types, block means and per-sequence
// lengths stay at 128).  They compute what the tuned ones do:
//
//  * append -- "cpu-attn", Method: per token and head, absmax int8 codes of
//    K and V (scale = absmax / 127, code = round-half-even(x / scale)), or the
//    f16 values as given; "Sparse Attention -- Quest-style block-selector for
//    long-context decode (#551)", "Fill op": the channel-wise min and max of
//    the f16 keys before quantization, merged into a block that held tokens;
//  * selection -- same page, "Selection": UB = sum over channels of
//    max(q * kmin, q * kmax), the max over the query heads of a KV head
//    (GQA), the top K_SEL of the candidate blocks by UB with ties to the lower
//    block index, plus every sink and recent block, listed ascending.
//
// Layouts are those of the header with head_dim = D: rows of D channels, the
// bounds [.., D, 2] f16.

#include "common.cuh"
#include "internal.h"

namespace kvd {
namespace {

constexpr int kRankThreads = 1024;
constexpr int kScoreWarps = 8;
constexpr int kScoreBlocksPerCta = 16;  // two per warp: many loads in flight


__device__ __forceinline__ float in_value(const __half *p, size_t i) { return __half2float(p[i]); }
__device__ __forceinline__ float in_value(const float *p, size_t i) { return p[i]; }

__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    return a;
}

// One warp: the new tokens of one (sequence b, KV head h) that fall in cache
// block blk0 + blockIdx.x, rows first, then that block's bounds.
template <int DT, typename IN>
__global__ void __launch_bounds__(32) gd_append_kernel(kvd_cache c, const IN *k_new,
                                                       const IN *v_new, int n_new, int len0,
                                                       int blk0) {
    constexpr bool kF32In = sizeof(IN) == 4;
    const int blk = blk0 + static_cast<int>(blockIdx.x);
    const int h = blockIdx.y, b = blockIdx.z, lane = threadIdx.x;
    const int D = c.head_dim;
    const long lo = static_cast<long>(blk) * kBlock;
    const long end = static_cast<long>(len0) + n_new;
    const long nlo = lo > len0 ? lo : len0;
    const long nhi = lo + kBlock < end ? lo + kBlock : end;
    const bool merge = lo < len0;
    const size_t row0 = (static_cast<size_t>(b) * c.n_kv_heads + h) * c.max_seq;
    auto src_row = [&](long t) {
        return ((static_cast<size_t>(b) * n_new + (t - len0)) * c.n_kv_heads + h) * D;
    };
    for (long t = nlo; t < nhi; ++t) {
        const size_t src = src_row(t), dst = (row0 + t) * D;
        if constexpr (DT == KVD_F16) {
            __half *K = static_cast<__half *>(c.k), *V = static_cast<__half *>(c.v);
            for (int d = lane; d < D; d += 32) {
                if constexpr (kF32In) {  // the nearest f16
                    K[dst + d] = __float2half_rn(k_new[src + d]);
                    V[dst + d] = __float2half_rn(v_new[src + d]);
                } else {  // the f16 bits as given
                    K[dst + d] = k_new[src + d];
                    V[dst + d] = v_new[src + d];
                }
            }
        } else {
            float ak = 0.0f, av = 0.0f;
            for (int d = lane; d < D; d += 32) {
                ak = fmaxf(ak, fabsf(in_value(k_new, src + d)));
                av = fmaxf(av, fabsf(in_value(v_new, src + d)));
            }
            const float ks = __fdiv_rn(warp_max(ak), 127.0f);
            const float vs = __fdiv_rn(warp_max(av), 127.0f);
            int8_t *K = static_cast<int8_t *>(c.k), *V = static_cast<int8_t *>(c.v);
            for (int d = lane; d < D; d += 32) {
                int kc = 0, vc = 0;
                if (ks != 0.0f) kc = max(-127, min(127, __float2int_rn(__fdiv_rn(in_value(k_new, src + d), ks))));
                if (vs != 0.0f) vc = max(-127, min(127, __float2int_rn(__fdiv_rn(in_value(v_new, src + d), vs))));
                K[dst + d] = static_cast<int8_t>(kc);
                V[dst + d] = static_cast<int8_t>(vc);
            }
            if (lane == 0) {
                static_cast<float *>(c.k_scale)[row0 + t] = ks;
                static_cast<float *>(c.v_scale)[row0 + t] = vs;
            }
        }
    }
    const size_t nbmax = static_cast<size_t>(c.max_seq / kBlock);
    __half2 *bounds = reinterpret_cast<__half2 *>(c.kbounds) +
                      ((static_cast<size_t>(b) * c.n_kv_heads + h) * nbmax + blk) * D;
    for (int d = lane; d < D; d += 32) {
        float mn = __int_as_float(0x7f800000), mx = -mn;
        for (long t = nlo; t < nhi; ++t) {
            float x = in_value(k_new, src_row(t) + d);
            if (kF32In && DT == KVD_F16) x = __half2float(__float2half_rn(x));
            mn = fminf(mn, x);
            mx = fmaxf(mx, x);
        }
        if (merge) {
            const float2 f = __half22float2(bounds[d]);
            mn = fminf(mn, f.x);
            mx = fmaxf(mx, f.y);
        }
        // f32 keys of a quantized cache: the envelope rounded outward; else
        // every value is an f16 already and converts back exactly
        bounds[d] = (kF32In && DT != KVD_F16)
                        ? __halves2half2(__float2half_rd(mn), __float2half_ru(mx))
                        : __floats2half2_rn(mn, mx);
    }
}

// An order-preserving u32 key of a bound (+0 and -0 give one key).
__device__ __forceinline__ uint32_t gd_key(float x) {
    const uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Keys of blocks [16 * blockIdx.x, +16) of problem p = blockIdx.y (sequence
// p / Hkv, KV head p % Hkv): warp w scores blocks w, w + 8, ..; lane l takes
// channels l, l + 32, .. of the G query heads (query in shared memory).
// DC: the head dim fixed at compile time (its loops then fold), or 0 to read
// it from the cache.
template <int G, int DC>
__global__ void __launch_bounds__(kScoreWarps * 32) gd_score_kernel(kvd_cache c, const float *q,
                                                                    int H, int NB, uint32_t *keys,
                                                                    int key_stride) {
    extern __shared__ float sq[];  // [G][D]
    const int D = DC > 0 ? DC : c.head_dim;
    const int p = blockIdx.y, b = p / c.n_kv_heads, h = p % c.n_kv_heads;
    const float *qp = q + (static_cast<size_t>(b) * H + static_cast<size_t>(h) * G) * D;
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) sq[i] = qp[i];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t nbmax = static_cast<size_t>(c.max_seq / kBlock);
    const __half2 *bnd = reinterpret_cast<const __half2 *>(c.kbounds) + p * nbmax * D;
    for (int i = warp; i < kScoreBlocksPerCta; i += kScoreWarps) {
        const int j = blockIdx.x * kScoreBlocksPerCta + i;
        if (j >= NB) break;
        const __half2 *row = bnd + static_cast<size_t>(j) * D;
        float acc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = 0.0f;
        for (int d = lane; d < D; d += 32) {
            const float2 f = __half22float2(row[d]);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float qv = sq[g * D + d];
                acc[g] += fmaxf(qv * f.x, qv * f.y);
            }
        }
        float ub = -__int_as_float(0x7f800000);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float a = acc[g];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            ub = fmaxf(ub, a);
        }
        if (lane == 0) keys[static_cast<size_t>(p) * key_stride + j] = gd_key(ub);
    }
}

// Exclusive rank of this thread's flag among the CTA's flags (thread order);
// *total = the CTA's count.  sh: 33 ints of shared memory.
__device__ __forceinline__ int cta_scan_flag(bool f, int *total, int *sh) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const unsigned m = __ballot_sync(0xffffffffu, f);
    if (lane == 0) sh[w] = __popc(m);
    __syncthreads();
    if (w == 0) {
        const int v = lane < nw ? sh[lane] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane < nw) sh[lane] = incl - v;
        if (lane == 31) sh[32] = incl;
    }
    __syncthreads();
    const int r = sh[w] + __popc(m & ((1u << lane) - 1u));
    *total = sh[32];
    __syncthreads();  // sh is reused by the next call
    return r;
}

// One CTA per problem: the K_SEL-th largest candidate key T by a 4-pass
// radix select (8 bits a pass, counted in shared memory), then one ascending
// pass that lists the forced blocks, the candidates above T, and the first
// (by index) candidates equal to T that complete K_SEL.
__global__ void __launch_bounds__(kRankThreads) gd_rank_kernel(const uint32_t *keys,
                                                               int key_stride, int NB, int nbmax,
                                                               int k_sel, int se, int rb,
                                                               int32_t *sel_idx,
                                                               int32_t *sel_cnt) {
    __shared__ unsigned hist[256];
    __shared__ int scan_sh[33];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;
    const int p = blockIdx.x, tid = threadIdx.x;
    const uint32_t *kp = keys + static_cast<size_t>(p) * key_stride;
    const int n_cand = rb - se;
    const bool all = k_sel >= n_cand, none = k_sel == 0;
    uint32_t T = 0;
    int take_eq = 0;
    if (!all && !none) {
        uint32_t prefix = 0, mask = 0;
        int need = k_sel;  // rank of T among the keys that match prefix on mask
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
            __syncthreads();
            for (int j = se + tid; j < rb; j += blockDim.x) {
                const uint32_t k = kp[j];
                if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (tid < 32) {
                // the bin holding the need-th largest: lane l sums bins
                // 8 (31 - l) .. +7, an inclusive scan over lanes counts the
                // keys from the top, and the first lane to reach need walks
                // its own 8 bins downward
                const int lo = 8 * (31 - tid);
                int own = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) own += static_cast<int>(hist[lo + i]);
                int incl = own;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += y;
                }
                const unsigned reach = __ballot_sync(0xffffffffu, incl >= need);
                if (tid == __ffs(reach) - 1) {
                    int above = incl - own, bin = lo + 7;
                    for (; bin > lo; --bin) {
                        if (above + static_cast<int>(hist[bin]) >= need) break;
                        above += static_cast<int>(hist[bin]);
                    }
                    s_need = need - above;
                    s_prefix = prefix | (static_cast<uint32_t>(bin) << shift);
                }
            }
            __syncthreads();
            need = s_need;
            prefix = s_prefix;
            mask |= 255u << shift;
            __syncthreads();
        }
        T = prefix;
        take_eq = need;
    }
    int32_t *out = sel_idx + static_cast<size_t>(p) * nbmax;
    int base = 0, eq_base = 0;
    for (int j0 = 0; j0 < NB; j0 += blockDim.x) {
        const int j = j0 + tid;
        bool in = false, eq = false;
        if (j < NB) {
            if (j < se || j >= rb || all) {
                in = true;
            } else if (!none) {
                const uint32_t k = kp[j];
                in = k > T;
                eq = k == T;
            }
        }
        int eq_total, in_total;
        const int eq_rank = cta_scan_flag(eq, &eq_total, scan_sh);
        if (eq && eq_base + eq_rank < take_eq) in = true;
        const int pos = cta_scan_flag(in, &in_total, scan_sh);
        if (in) out[base + pos] = j;
        base += in_total;
        eq_base += eq_total;
    }
    if (tid == 0) sel_cnt[p] = base;
}

template <int DT>
cudaError_t append_dt(const kvd_cache &c, const void *k_new, const void *v_new, int n_new,
                      int len0, cudaStream_t st, bool f32_in) {
    const int blk0 = len0 / kBlock, blk1 = (len0 + n_new - 1) / kBlock;
    const dim3 grid(blk1 - blk0 + 1, c.n_kv_heads, c.batch);
    if (f32_in)
        gd_append_kernel<DT, float><<<grid, 32, 0, st>>>(
            c, static_cast<const float *>(k_new), static_cast<const float *>(v_new), n_new, len0,
            blk0);
    else
        gd_append_kernel<DT, __half><<<grid, 32, 0, st>>>(
            c, static_cast<const __half *>(k_new), static_cast<const __half *>(v_new), n_new,
            len0, blk0);
    return cudaGetLastError();
}

template <int G, int DC = 0>
cudaError_t score_g(const kvd_cache &c, const float *q, int H, int NB, uint32_t *keys,
                    int key_stride, cudaStream_t st) {
    const size_t smem = static_cast<size_t>(G) * c.head_dim * sizeof(float);
    auto kern = gd_score_kernel<G, DC>;
    cudaError_t e = prepare_kernel(reinterpret_cast<const void *>(kern), kScoreWarps * 32, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((NB + kScoreBlocksPerCta - 1) / kScoreBlocksPerCta,
                    c.batch * c.n_kv_heads);
    kern<<<grid, kScoreWarps * 32, smem, st>>>(c, q, H, NB, keys, key_stride);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append_gd(const kvd_cache &c, const void *k_new, const void *v_new,
                             int n_new, int len0, cudaStream_t st, bool f32_in) {
    if (n_new < 1) return cudaSuccess;
    return c.dtype == KVD_F16 ? append_dt<KVD_F16>(c, k_new, v_new, n_new, len0, st, f32_in)
                              : append_dt<KVD_INT8>(c, k_new, v_new, n_new, len0, st, f32_in);
}

cudaError_t launch_select_gd(const kvd_cache &c, const float *q, int n_heads, int k_sel, int se,
                             int rb, int32_t *sel_idx, int32_t *sel_cnt, uint32_t *keys,
                             cudaStream_t st) {
    const int NB = (c.len + kBlock - 1) / kBlock;
    const int nbmax = c.max_seq / kBlock;
    const int key_stride = (nbmax + 3) / 4 * 4;
    const int G = n_heads / c.n_kv_heads;
    const bool rank = k_sel > 0 && k_sel < rb - se;
    if (rank) {  // the keys of every candidate (only candidates are ranked)
        cudaError_t e;
        const int D = c.head_dim;
        // common head dims (64, 96, 256) of GQA groups of 4 and 8, with folded loops
        if (G == 4 && D == 64) e = score_g<4, 64>(c, q, n_heads, NB, keys, key_stride, st);
        else if (G == 8 && D == 64) e = score_g<8, 64>(c, q, n_heads, NB, keys, key_stride, st);
        else if (G == 4 && D == 96) e = score_g<4, 96>(c, q, n_heads, NB, keys, key_stride, st);
        else if (G == 8 && D == 96) e = score_g<8, 96>(c, q, n_heads, NB, keys, key_stride, st);
        else if (G == 4 && D == 256) e = score_g<4, 256>(c, q, n_heads, NB, keys, key_stride, st);
        else if (G == 8 && D == 256) e = score_g<8, 256>(c, q, n_heads, NB, keys, key_stride, st);
        else switch (G) {
            case 1: e = score_g<1>(c, q, n_heads, NB, keys, key_stride, st); break;
            case 2: e = score_g<2>(c, q, n_heads, NB, keys, key_stride, st); break;
            case 4: e = score_g<4>(c, q, n_heads, NB, keys, key_stride, st); break;
            case 8: e = score_g<8>(c, q, n_heads, NB, keys, key_stride, st); break;
            default: e = score_g<16>(c, q, n_heads, NB, keys, key_stride, st); break;
        }
        if (e != cudaSuccess) return e;
    }
    gd_rank_kernel<<<c.batch * c.n_kv_heads, kRankThreads, 0, st>>>(
        keys, key_stride, NB, nbmax, k_sel, se, rb, sel_idx, sel_cnt);
    return cudaGetLastError();
}

}  // namespace kvd
