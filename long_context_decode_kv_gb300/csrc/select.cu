// select.cu -- Quest block selection: block bounds, GQA max, top-K with the
// sink and recent blocks forced in.
//
// "Sparse Attention -- Quest-style block-selector for long-context decode
// (#551)":
//  - Method, "Per-query upper bound": UB_h(j) = sum_d max(q_d kmin_j[d],
//    q_d kmax_j[d]) (kmax where q_d > 0, kmin where q_d < 0);
//  - S2/S3 selector op: "GQA -> max UB over the query group per KV-head"
//    (one block set per KV head);
//  - Method, "Top-K block selection": the top-K_SEL blocks by bound plus the
//    recent window and the attention-sink block.
// Equal bounds go to the lower block index; the top-K budget counts only the
// blocks that are not forced.
//
// Two kernels:
//  score_kernel  spreads the bound reads (512 B per block) over every SM and
//                writes one order-preserving u32 key per candidate block;
//  topk_kernel   one CTA per (sequence, KV head): radix select of the K-th
//                largest key in shared memory, then an ascending compaction
//                that merges forced blocks, larger keys, and the lowest-index
//                blocks among those equal to the K-th key.
#include "common.cuh"
#include "internal.h"

namespace kvd {
namespace {

constexpr int kScoreWarps = 8;
constexpr int kScoreSlots = 4;                    // blocks per warp per pass (8 lanes each)
constexpr int kScorePasses = 4;
constexpr int kBlocksPerScoreCta = kScoreWarps * kScoreSlots * kScorePasses;  // 128
constexpr int kTopkThreads = 1024;
constexpr int kMaxSelectBlocks = 49152;

__device__ __forceinline__ void half8_to_float(const uint4 &w, float *f) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 v = __half22float2(h[i]);
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}

// Bound of one head over 16 channels held by this lane.
__device__ __forceinline__ float head_bound16(const float *qv, const float *lo, const float *hi) {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s = fmaf(qv[i], qv[i] >= 0.0f ? hi[i] : lo[i], s);
    return s;
}

// Sum over the 8 lanes of a slot (lane bits 0..2) of NH per-head partials,
// returning to each lane the full sum of head (e * NH) / 8 (NH in 1, 2, 4).
template <int NH>
__device__ __forceinline__ float reduce8_scatter(float (&v)[NH], int e) {
    constexpr unsigned full = 0xffffffffu;
    if constexpr (NH == 4) {
        const bool up = (e & 4) != 0;
        float k0 = up ? v[2] : v[0], k1 = up ? v[3] : v[1];
        const float s0 = up ? v[0] : v[2], s1 = up ? v[1] : v[3];
        k0 += __shfl_xor_sync(full, s0, 4);
        k1 += __shfl_xor_sync(full, s1, 4);
        const bool mid = (e & 2) != 0;
        float k = mid ? k1 : k0;
        k += __shfl_xor_sync(full, mid ? k0 : k1, 2);
        k += __shfl_xor_sync(full, k, 1);
        return k;
    } else if constexpr (NH == 2) {
        const bool up = (e & 4) != 0;
        float k = up ? v[1] : v[0];
        k += __shfl_xor_sync(full, up ? v[0] : v[1], 4);
        k += __shfl_xor_sync(full, k, 2);
        k += __shfl_xor_sync(full, k, 1);
        return k;
    } else {
        float k = v[0];
        k += __shfl_xor_sync(full, k, 4);
        k += __shfl_xor_sync(full, k, 2);
        k += __shfl_xor_sync(full, k, 1);
        return k;
    }
}

// Group bound of the 4 blocks of this warp pass.  Lane = slot * 8 + e; lane e
// holds channels [8e, 8e+8) and [64+8e, 64+8e+8) of its slot's block.  The
// group's query heads are processed 4 at a time from q_s (shared, [G][128]).
template <int G>
__device__ __forceinline__ float group_bound(const float *__restrict__ q_s, const float *lo,
                                             const float *hi, int e) {
    constexpr int NH = G < 4 ? G : 4;
    float best = kNegBig;
#pragma unroll
    for (int h0 = 0; h0 < G; h0 += NH) {
        float part[NH];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
            float qv[16];
            const float *qh = q_s + (h0 + hh) * kHeadDim;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                qv[i] = qh[8 * e + i];
                qv[8 + i] = qh[64 + 8 * e + i];
            }
            part[hh] = head_bound16(qv, lo, hi);
        }
        float s = reduce8_scatter<NH>(part, e);
        // max over the NH heads spread over the slot's lanes
        if constexpr (NH == 4) {
            s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 2));
            s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 4));
        } else if constexpr (NH == 2) {
            s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 4));
        }
        best = fmaxf(best, s);
    }
    return best;
}

// keys != nullptr: write u32 keys of blocks [blk_lo, blk_lo + n) to keys[p*n + j - blk_lo].
// ub != nullptr: write f32 bounds of blocks [0, n) to ub[p*n + j] (blk_lo = 0).
template <int G>
__global__ void __launch_bounds__(32 * kScoreWarps)
score_kernel(const float *__restrict__ q, const __half *__restrict__ kmin,
             const __half *__restrict__ kmax, int Hkv, int H, int nbmax, int blk_lo, int n,
             uint32_t *__restrict__ keys, float *__restrict__ ub) {
    __shared__ __align__(16) float q_s[G * kHeadDim];
    const int p = blockIdx.y;               // (sequence, KV head)
    const int b = p / Hkv, g = p % Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = lane >> 3, e = lane & 7;
    pdl_wait();
    pdl_launch_dependents();
    const float *qg = q + (static_cast<size_t>(b) * H + static_cast<size_t>(g) * G) * kHeadDim;
    for (int i = threadIdx.x; i < G * kHeadDim; i += blockDim.x) q_s[i] = qg[i];
    __syncthreads();

    const size_t base = static_cast<size_t>(p) * nbmax;
    const int cta0 = blockIdx.x * kBlocksPerScoreCta;
#pragma unroll 1
    for (int pass = 0; pass < kScorePasses; ++pass) {
        const int jr = cta0 + pass * kScoreWarps * kScoreSlots + warp * kScoreSlots + slot;
        const bool valid = jr < n;
        float lo[16], hi[16];
        if (valid) {
            const __half *pl = kmin + (base + blk_lo + jr) * kHeadDim;
            const __half *ph = kmax + (base + blk_lo + jr) * kHeadDim;
            half8_to_float(*reinterpret_cast<const uint4 *>(pl + 8 * e), lo);
            half8_to_float(*reinterpret_cast<const uint4 *>(pl + 64 + 8 * e), lo + 8);
            half8_to_float(*reinterpret_cast<const uint4 *>(ph + 8 * e), hi);
            half8_to_float(*reinterpret_cast<const uint4 *>(ph + 64 + 8 * e), hi + 8);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) lo[i] = hi[i] = 0.0f;
        }
        const float s = group_bound<G>(q_s, lo, hi, e);
        if (valid && e == 0) {
            const size_t o = static_cast<size_t>(p) * n + jr;
            if (keys) keys[o] = float_to_key(s);
            if (ub) ub[o] = s;
        }
    }
}

// Exclusive scan of one int per thread over a 1024-thread CTA; *total gets the sum.
__device__ __forceinline__ int cta_exclusive_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
        int s = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s - w;  // exclusive prefix of warp totals
        if (lane == 31) *total = s;
    }
    __syncthreads();
    const int r = warp_sums[warp] + x - v;
    __syncthreads();
    return r;
}

enum TopkMode { kTakeNone = 0, kTakeAll = 1, kTakeTopK = 2 };

// One CTA per (sequence, KV head).
//   forced blocks: [0, se) and [rb, NB); candidates: [se, rb)
//   mode kTakeTopK: keys [P, rb - se] hold the candidates' keys and keff of
//   them are taken; kTakeAll / kTakeNone take every / no candidate.
__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const uint32_t *__restrict__ keys, int mode, int keff, int NB, int se, int rb,
            int nbmax, int32_t *__restrict__ sel_idx, int32_t *__restrict__ sel_cnt) {
    const int cand_lo = se;
    const int n_cand = mode == kTakeTopK ? rb - se : 0;
    extern __shared__ __align__(16) uint32_t s_keys[];
    __shared__ int hist[256];
    __shared__ int warp_sums[32];
    __shared__ int s_total;
    __shared__ uint32_t s_red[2][32];
    __shared__ int s_digit, s_above;
    const int p = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_launch_dependents();

    const uint32_t *kp = keys + static_cast<size_t>(p) * n_cand;
    uint32_t kmn = 0xffffffffu, kmx = 0u;
    for (int i = tid; i < n_cand; i += kTopkThreads) {
        const uint32_t k = kp[i];
        s_keys[i] = k;
        kmn = min(kmn, k);
        kmx = max(kmx, k);
    }
    // CTA min / max of the keys
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        kmn = min(kmn, __shfl_xor_sync(0xffffffffu, kmn, o));
        kmx = max(kmx, __shfl_xor_sync(0xffffffffu, kmx, o));
    }
    if (lane == 0) { s_red[0][warp] = kmn; s_red[1][warp] = kmx; }
    __syncthreads();
    if (warp == 0) {
        kmn = s_red[0][lane];
        kmx = s_red[1][lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            kmn = min(kmn, __shfl_xor_sync(0xffffffffu, kmn, o));
            kmx = max(kmx, __shfl_xor_sync(0xffffffffu, kmx, o));
        }
        if (lane == 0) { s_red[0][0] = kmn; s_red[1][0] = kmx; }
    }
    __syncthreads();
    kmn = s_red[0][0];
    kmx = s_red[1][0];

    // ---- radix select: T = K-th largest key, need_eq = keys equal to T to take
    uint32_t T = 0u;
    int need_eq = 0;
    const bool take_all = mode == kTakeAll;
    const bool take_none = mode == kTakeNone;
    if (mode == kTakeTopK) {
        const uint32_t diff = kmn ^ kmx;
        if (diff == 0u) {
            T = kmn;
            need_eq = keff;
        } else {
            const int nbits = 32 - __clz(diff);
            uint32_t mask = nbits >= 32 ? 0u : (0xffffffffu << nbits);
            uint32_t prefix = kmn & mask;
            int krem = keff;
            for (int hi = nbits; hi > 0; hi -= 8) {
                const int lo = hi > 8 ? hi - 8 : 0;
                const uint32_t dmask = (1u << (hi - lo)) - 1u;
                for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
                __syncthreads();
                for (int i0 = 0; i0 < n_cand; i0 += kTopkThreads) {
                    const int i = i0 + tid;
                    bool in = false;
                    int d = 0;
                    if (i < n_cand) {
                        const uint32_t k = s_keys[i];
                        in = (k & mask) == prefix;
                        d = static_cast<int>((k >> lo) & dmask);
                    }
                    // one shared atomic per distinct digit per warp
                    const unsigned act = __ballot_sync(0xffffffffu, in);
                    if (in) {
                        const unsigned peers = __match_any_sync(act, d);
                        if ((__ffs(peers) - 1) == lane) atomicAdd(&hist[d], __popc(peers));
                    }
                }
                __syncthreads();
                if (warp == 0) {
                    // lane l owns digits 8l..8l+7; find the digit holding the krem-th largest
                    int s = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) s += hist[8 * lane + i];
                    int incl = s;  // sum over lanes >= lane
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_down_sync(0xffffffffu, incl, o);
                        if (lane + o < 32) incl += y;
                    }
                    const int above = incl - s;
                    if (above < krem && krem <= incl) {
                        int acc = above;
                        for (int i = 7; i >= 0; --i) {
                            const int c = hist[8 * lane + i];
                            if (krem <= acc + c) { s_digit = 8 * lane + i; s_above = acc; break; }
                            acc += c;
                        }
                    }
                }
                __syncthreads();
                prefix |= static_cast<uint32_t>(s_digit) << lo;
                mask |= dmask << lo;
                krem -= s_above;
                __syncthreads();
            }
            T = prefix;
            need_eq = krem;
        }
    }

    // ---- ascending compaction over [0, NB)
    const int chunk = (NB + kTopkThreads - 1) / kTopkThreads;
    const int j0 = tid * chunk;
    const int j1 = min(NB, j0 + chunk);
    auto is_cand = [&](int j) { return j >= se && j < rb; };
    int eq_here = 0;
    if (mode == kTakeTopK)
        for (int j = j0; j < j1; ++j)
            if (is_cand(j) && s_keys[j - cand_lo] == T) ++eq_here;
    int eq_rank = cta_exclusive_scan(eq_here, warp_sums, &s_total);
    int n_here = 0;
    {
        int r = eq_rank;
        for (int j = j0; j < j1; ++j) {
            bool take;
            if (!is_cand(j)) take = true;
            else if (take_all) take = true;
            else if (take_none) take = false;
            else {
                const uint32_t k = s_keys[j - cand_lo];
                take = k > T || (k == T && r < need_eq);
                if (k == T) ++r;
            }
            n_here += take;
        }
    }
    const int out0 = cta_exclusive_scan(n_here, warp_sums, &s_total);
    int32_t *dst = sel_idx + static_cast<size_t>(p) * nbmax;
    {
        int r = eq_rank, o = out0;
        for (int j = j0; j < j1; ++j) {
            bool take;
            if (!is_cand(j)) take = true;
            else if (take_all) take = true;
            else if (take_none) take = false;
            else {
                const uint32_t k = s_keys[j - cand_lo];
                take = k > T || (k == T && r < need_eq);
                if (k == T) ++r;
            }
            if (take) dst[o++] = j;
        }
    }
    if (tid == 0) sel_cnt[p] = s_total;
}

template <int G>
cudaError_t launch_score(const kvd_cache &c, const Geom &g, const float *q, int blk_lo, int n,
                         uint32_t *keys, float *ub, cudaStream_t st, bool pdl) {
    dim3 grid((n + kBlocksPerScoreCta - 1) / kBlocksPerScoreCta, g.B * g.Hkv);
    return launch_ex(score_kernel<G>, grid, dim3(32 * kScoreWarps), 0, st, pdl, q,
                     static_cast<const __half *>(c.kmin), static_cast<const __half *>(c.kmax),
                     g.Hkv, g.H, g.nbmax, blk_lo, n, keys, ub);
}

cudaError_t launch_score_any(const kvd_cache &c, const Geom &g, const float *q, int blk_lo,
                             int n, uint32_t *keys, float *ub, cudaStream_t st, bool pdl) {
    switch (g.G) {
        case 1: return launch_score<1>(c, g, q, blk_lo, n, keys, ub, st, pdl);
        case 2: return launch_score<2>(c, g, q, blk_lo, n, keys, ub, st, pdl);
        case 4: return launch_score<4>(c, g, q, blk_lo, n, keys, ub, st, pdl);
        case 8: return launch_score<8>(c, g, q, blk_lo, n, keys, ub, st, pdl);
        case 16: return launch_score<16>(c, g, q, blk_lo, n, keys, ub, st, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int max_select_blocks() { return kMaxSelectBlocks; }

cudaError_t launch_select(const kvd_cache &c, const Geom &g, const float *q, int k_sel,
                          int sink_tokens, int recent_tokens, int32_t *sel_idx,
                          int32_t *sel_cnt, uint32_t *keys, cudaStream_t st, bool pdl) {
    const int NB = g.NB;
    int se = (sink_tokens + kBlock - 1) / kBlock;
    if (se > NB) se = NB;
    int rb = NB;
    if (recent_tokens > 0) {
        long start = static_cast<long>(g.len) - recent_tokens;
        if (start < 0) start = 0;
        rb = static_cast<int>(start / kBlock);
    }
    if (rb < se) rb = se;
    const int n_cand = rb - se;
    const int keff = k_sel < n_cand ? k_sel : n_cand;
    cudaError_t err = cudaSuccess;
    const bool need_scores = keff > 0 && keff < n_cand;
    if (need_scores) {
        err = launch_score_any(c, g, q, se, n_cand, keys, nullptr, st, pdl);
        if (err != cudaSuccess) return err;
    }
    static bool attr_set = false;
    if (!attr_set) {
        err = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kMaxSelectBlocks * static_cast<int>(sizeof(uint32_t)));
        if (err != cudaSuccess) return err;
        attr_set = true;
    }
    const int mode = need_scores ? kTakeTopK : (keff == 0 ? kTakeNone : kTakeAll);
    const size_t smem = static_cast<size_t>(need_scores ? n_cand : 0) * sizeof(uint32_t);
    return launch_ex(topk_kernel, dim3(g.B * g.Hkv), dim3(kTopkThreads), smem, st, pdl,
                     static_cast<const uint32_t *>(keys), mode, keff, NB, se, rb, g.nbmax,
                     sel_idx, sel_cnt);
}

cudaError_t launch_scores_debug(const kvd_cache &c, const Geom &g, const float *q, float *ub,
                                cudaStream_t st) {
    return launch_score_any(c, g, q, 0, g.NB, nullptr, ub, st, false);
}

}  // namespace kvd
