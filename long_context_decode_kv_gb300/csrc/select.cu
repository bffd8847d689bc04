// select.cu -- Quest block selection: block bounds, GQA max, top-K with the
// sink and recent blocks forced in.
//
// "Sparse Attention -- Quest-style block-selector for long-context decode
// (#551)":
//  - Method, "Per-query upper bound": UB_h(j) = sum_d max(q_d kmin_j[d],
//    q_d kmax_j[d]) (kmax where q_d > 0, kmin where q_d < 0);
//  - S2/S3 selector op: the group's query heads reduce to one bound per
//    (KV head, block) by a max, so the whole group shares one block set;
//  - Method, "Top-K block selection": the top-K_SEL blocks by bound plus the
//    recent window and the attention-sink block.
// Equal bounds go to the lower block index; the top-K budget counts only the
// blocks that are not forced.
//
// score_kernel: streams the bounds (512 B per block) of a contiguous range of
// candidate blocks through a TMA ring in shared memory, over every SM, and
// writes one order-preserving u32 key per block (or the f32 bound itself,
// for the test export).
//
// topk_kernel: one 1024-thread CTA per (sequence, KV head) holds the keys
// (L2-resident) in shared memory, finds the K-th largest key with
// range-adaptive 12-bit radix passes, and writes the ascending list: forced
// sink blocks, the taken candidates (larger keys, then the lowest-index
// blocks equal to the K-th key), forced recent blocks.
#include "common.cuh"
#include "internal.h"

namespace kvd {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;

constexpr int kScoreWarps = 8;                       // consumers; warp 8 produces
constexpr int kScoreThreads = 32 * (kScoreWarps + 1);
constexpr int kScoreSlots = 4;                       // blocks per warp per stage (8 lanes each)
constexpr int kStageBlocks = kScoreWarps * kScoreSlots;  // 32
constexpr int kBoundRowBytes = kHeadDim * 2 * 2;      // (kmin, kmax) f16 pairs: 512 B
constexpr int kScoreStages = 4;
constexpr int kScoreStageBytes = kStageBlocks * kBoundRowBytes;  // 16 KiB

constexpr int kMaxSelectBlocks = 49152;  // candidate keys held in shared memory
constexpr int kDigitBits = 12;
constexpr int kBins = 1 << kDigitBits;

enum TopkMode { kTakeNone = 0, kTakeAll = 1, kTakeTopK = 2 };

// ------------------------------------------------------ bound math ---
// Scoring lane layout: 16 lanes per block; lane e (0..15) of a block holds
// channels [8e, 8e+8), as (kmin, kmax) pairs.  A warp scores two blocks at a
// time.  Per channel and head the bound's term is one packed FMA:
//   max(q*kmin, q*kmax) = min(q,0)*kmin + max(q,0)*kmax   (exact: the other
// product is a signed zero), accumulated as a pair and summed at the end.

// The 16-byte chunk order of lane e: lanes 4..7 (mod 8) take their two
// chunks swapped so that the 8 lanes of a quarter-warp hit distinct banks.
__device__ __forceinline__ int chunk_swap(int e) { return (e >> 2) & 1; }

// Query pairs (min(q,0), max(q,0)) of this lane's 8 channels, in the order
// the lane reads its bound pairs.
template <int NH>
__device__ __forceinline__ void load_qpairs(const float *q_s, int h0, int e,
                                            float2 (&qp)[NH][8]) {
    const int sw = chunk_swap(e);
#pragma unroll
    for (int hh = 0; hh < NH; ++hh)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = ((i >> 2) ^ sw) * 4 + (i & 3);  // channel within the lane's 8
            const float x = q_s[(h0 + hh) * kHeadDim + 8 * e + c];
            qp[hh][i] = make_float2(fminf(x, 0.0f), fmaxf(x, 0.0f));
        }
}

// Sum over the 16 lanes of a block (lane bits 0..3) of NH per-head partials,
// returning to each lane the full sum of head (e * NH) / 16 (NH in 1, 2, 4).
template <int NH>
__device__ __forceinline__ float reduce16_scatter(float (&v)[NH], int e) {
    if constexpr (NH == 4) {
        const bool up = (e & 8) != 0;
        float k0 = up ? v[2] : v[0], k1 = up ? v[3] : v[1];
        const float s0 = up ? v[0] : v[2], s1 = up ? v[1] : v[3];
        k0 += __shfl_xor_sync(kFullMask, s0, 8);
        k1 += __shfl_xor_sync(kFullMask, s1, 8);
        const bool mid = (e & 4) != 0;
        float k = mid ? k1 : k0;
        k += __shfl_xor_sync(kFullMask, mid ? k0 : k1, 4);
        k += __shfl_xor_sync(kFullMask, k, 2);
        k += __shfl_xor_sync(kFullMask, k, 1);
        return k;
    } else if constexpr (NH == 2) {
        const bool up = (e & 8) != 0;
        float k = up ? v[1] : v[0];
        k += __shfl_xor_sync(kFullMask, up ? v[0] : v[1], 8);
        k += __shfl_xor_sync(kFullMask, k, 4);
        k += __shfl_xor_sync(kFullMask, k, 2);
        k += __shfl_xor_sync(kFullMask, k, 1);
        return k;
    } else {
        float k = v[0];
        k += __shfl_xor_sync(kFullMask, k, 8);
        k += __shfl_xor_sync(kFullMask, k, 4);
        k += __shfl_xor_sync(kFullMask, k, 2);
        k += __shfl_xor_sync(kFullMask, k, 1);
        return k;
    }
}

// Max over the NH heads spread over the block's lanes (after reduce16_scatter).
template <int NH>
__device__ __forceinline__ float max_over_heads(float s) {
    if constexpr (NH == 4) {
        s = fmaxf(s, __shfl_xor_sync(kFullMask, s, 4));
        s = fmaxf(s, __shfl_xor_sync(kFullMask, s, 8));
    } else if constexpr (NH == 2) {
        s = fmaxf(s, __shfl_xor_sync(kFullMask, s, 8));
    }
    return s;
}

// Bound of one head over the lane's 8 channels: kb holds (kmin, kmax) pairs.
__device__ __forceinline__ float head_bound8(const float2 *qp, const float2 *kb) {
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = __ffma2_rn(qp[i], kb[i], acc);
    return acc.x + acc.y;
}

// Group bound of one block from this lane's 8 channels: the max over the
// group's heads of each head's bound.
template <int G>
__device__ __forceinline__ float group_bound(const float *q_s,
                                             const float2 (&qreg)[G < 4 ? G : 4][8],
                                             const float2 *kb, int e) {
    constexpr int NH = G < 4 ? G : 4;
    float best = kNegBig;
#pragma unroll 1
    for (int h0 = 0; h0 < G; h0 += NH) {
        float part[NH];
        if constexpr (G <= 4) {
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) part[hh] = head_bound8(qreg[hh], kb);
        } else {
            float2 qv[NH][8];
            load_qpairs<NH>(q_s, h0, e, qv);
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) part[hh] = head_bound8(qv[hh], kb);
        }
        best = fmaxf(best, max_over_heads<NH>(reduce16_scatter<NH>(part, e)));
    }
    return best;
}

// CTA (x, p) of score_kernel: candidate blocks [x*R, min(n, (x+1)*R)) of
// problem p = (sequence, KV head), i.e. cache blocks blk_lo + j.  Their
// bounds stream through a TMA ring (stages of 32 blocks; warp 8 produces,
// warps 0..7 consume, warp w scoring blocks 4w..4w+3 of each stage two at a
// time).  keys != nullptr: keys[p*n + j] = order-preserving key of the bound;
// ub != nullptr: ub[p*n + j] = the f32 bound (test export).
template <int G>
__global__ void __launch_bounds__(kScoreThreads, 2)
score_kernel(const float *__restrict__ q, const __half *__restrict__ kbounds, int Hkv, int H,
             int nbmax, int blk_lo, int n,
             int R, uint32_t *__restrict__ keys, float *__restrict__ ub,
             int32_t *__restrict__ dev_status, int overlap) {
    constexpr int NH = G < 4 ? G : 4;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kScoreStages * kScoreStageBytes);
    uint64_t *empty = full + kScoreStages;
    float *q_s = reinterpret_cast<float *>(empty + kScoreStages);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(q_s + G * kHeadDim);
    int *issued_s = const_cast<int *>(abort_flag) + 1;

    const int p = blockIdx.y;
    const int b = p / Hkv, g = p % Hkv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = lane >> 4, e = lane & 15;
    const int j0 = blockIdx.x * R;
    const int j1 = min(n, j0 + R);
    const int nstage = (j1 - j0 + kStageBlocks - 1) / kStageBlocks;

    if (tid == 0) {
        for (int i = 0; i < kScoreStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kScoreWarps);
        }
        *abort_flag = 0;
        *issued_s = 0;
        fence_barrier_init();
    }
    // overlap: inside a decode step whose appended token lands in a forced
    // block, the candidate bounds and the query are complete before the
    // upstream append runs, so scoring overlaps it; the grid-dependency wait
    // then moves to the end, so this grid still completes after the append.
    if (!overlap) pdl_wait();
    const float *qg = q + (static_cast<size_t>(b) * H + static_cast<size_t>(g) * G) * kHeadDim;
    for (int i = tid; i < G * kHeadDim; i += blockDim.x) q_s[i] = qg[i];
    __syncthreads();
    pdl_launch_dependents();

    const size_t base = static_cast<size_t>(p) * nbmax + blk_lo;  // row of candidate 0
    if (warp == kScoreWarps) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int issued = 0;
            for (int si = 0; si < nstage; ++si) {
                const int s = si % kScoreStages;
                if (si >= kScoreStages &&
                    !mbar_wait(&empty[s], ((si / kScoreStages) - 1) & 1, abort_flag)) {
                    *abort_flag = 1;
                    report_status(dev_status, KVD_ERR_TIMEOUT);
                    break;
                }
                const int jb = j0 + si * kStageBlocks;
                const int cnt = min(kStageBlocks, j1 - jb);
                const uint32_t bytes = static_cast<uint32_t>(cnt) * kBoundRowBytes;
                mbar_arrive_expect_tx(&full[s], bytes);
                tma_load_1d(ring + s * kScoreStageBytes, kbounds + (base + jb) * kHeadDim * 2,
                            bytes, &full[s], pol);
                issued = si + 1;
            }
            *issued_s = issued;
        }
    } else {
        float2 qreg[NH][8];
        if constexpr (G <= 4) load_qpairs<NH>(q_s, 0, e, qreg);
        const int sw = chunk_swap(e);
        for (int si = 0; si < nstage; ++si) {
            const int s = si % kScoreStages;
            const bool ok = mbar_wait(&full[s], (si / kScoreStages) & 1, abort_flag);
            if (!__all_sync(kFullMask, ok)) {
                if (lane == 0) {
                    *abort_flag = 1;
                    report_status(dev_status, KVD_ERR_TIMEOUT);
                }
                break;
            }
            const uint8_t *st = ring + s * kScoreStageBytes;
            float sc[2];
            int jr[2];
#pragma unroll
            for (int ps = 0; ps < 2; ++ps) {
                const int k = warp * kScoreSlots + 2 * ps + half;  // block within the stage
                jr[ps] = j0 + si * kStageBlocks + k;
                float2 kb[8];
                if (jr[ps] < j1) {
                    const uint4 *row = reinterpret_cast<const uint4 *>(st + k * kBoundRowBytes);
                    const uint4 c0 = row[2 * e + sw], c1 = row[2 * e + 1 - sw];
                    const __half2 *h0 = reinterpret_cast<const __half2 *>(&c0);
                    const __half2 *h1 = reinterpret_cast<const __half2 *>(&c1);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        kb[i] = __half22float2(h0[i]);
                        kb[4 + i] = __half22float2(h1[i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) kb[i] = make_float2(0.0f, 0.0f);
                }
                sc[ps] = group_bound<G>(q_s, qreg, kb, e);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
            for (int ps = 0; ps < 2; ++ps) {
                if (jr[ps] < j1 && e == 0) {
                    const size_t o = static_cast<size_t>(p) * n + jr[ps];
                    if (keys) keys[o] = float_to_key(sc[ps]);
                    if (ub) ub[o] = sc[ps];
                }
            }
        }
    }
    __syncthreads();
    if (*abort_flag && warp == kScoreWarps && lane == 0) {
        // wind down: wait (bounded) for the copies still landing in the ring
        const int issued = *issued_s;
        volatile int never = 0;
        for (int i = max(0, issued - kScoreStages); i < issued; ++i)
            (void)mbar_wait(&full[i % kScoreStages], (i / kScoreStages) & 1, &never);
    }
    if (overlap) pdl_wait();
}

// ------------------------------------------------------------- top-K ---
constexpr int kTopkThreads = 1024;

struct TopkArgs {
    const uint32_t *keys;   // [P, rb - se] candidate keys (score_kernel)
    int32_t *sel_idx, *sel_cnt;
    int nbmax, NB;
    int se, rb;        // forced: [0, se) and [rb, NB); candidates [se, rb)
    int keff, mode;    // candidates to take, TopkMode
};

// Exclusive scan of one int per thread over a 1024-thread CTA; *total gets
// the sum.  All threads must call it.
__device__ __forceinline__ int cta_exclusive_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFullMask, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int w = warp_sums[lane];
        int s = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFullMask, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s - w;  // exclusive prefix of the warp totals
        if (lane == 31) *total = s;
    }
    __syncthreads();
    const int r = warp_sums[warp] + x - v;
    __syncthreads();
    return r;
}

// One CTA per (sequence, KV head).  Thread t owns the C = ceil(n / 1024)
// consecutive candidates [tC, tC + C); their keys sit in shared memory
// transposed (key tC + i at i*1024 + t), so that every shared access below is
// conflict-free.  The K-th largest key T comes from range-adaptive 12-bit
// radix passes; the ascending list then needs one CTA scan of the packed
// per-thread counts of keys above and equal to T.
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(TopkArgs a) {
    extern __shared__ __align__(16) uint32_t s_keys[];
    __shared__ int hist[kBins];
    __shared__ int warp_sums[32];
    __shared__ int s_total;
    __shared__ uint32_t s_red[2][32];
    __shared__ int s_digit, s_above;
    const int n_cand = a.rb - a.se;
    const int n_keys = a.mode == kTakeTopK ? n_cand : 0;
    const int C = (n_cand + kTopkThreads - 1) / kTopkThreads;  // candidates per thread
    const int p = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c0 = min(n_cand, tid * C), c1 = min(n_cand, c0 + C);
    pdl_wait();
    pdl_launch_dependents();

    const uint32_t *kp = a.keys + static_cast<size_t>(p) * n_keys;
    uint32_t kmn = 0xffffffffu, kmx = 0u;
    if (a.mode == kTakeTopK) {
        for (int j = c0; j < c1; ++j) {
            const uint32_t k = __ldcg(kp + j);
            s_keys[(j - c0) * kTopkThreads + tid] = k;
            kmn = min(kmn, k);
            kmx = max(kmx, k);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        kmn = min(kmn, __shfl_xor_sync(kFullMask, kmn, o));
        kmx = max(kmx, __shfl_xor_sync(kFullMask, kmx, o));
    }
    if (lane == 0) {
        s_red[0][warp] = kmn;
        s_red[1][warp] = kmx;
    }
    __syncthreads();
    if (warp == 0) {
        kmn = s_red[0][lane];
        kmx = s_red[1][lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            kmn = min(kmn, __shfl_xor_sync(kFullMask, kmn, o));
            kmx = max(kmx, __shfl_xor_sync(kFullMask, kmx, o));
        }
        if (lane == 0) {
            s_red[0][0] = kmn;
            s_red[1][0] = kmx;
        }
    }
    __syncthreads();
    kmn = s_red[0][0];
    kmx = s_red[1][0];

    // ---- T = the keff-th largest key; need_eq = keys equal to T to take.
    // Digits of 12 bits from the top of the bits where the keys differ.
    uint32_t T = 0u;
    int need_eq = 0;
    if (a.mode == kTakeTopK) {
        const uint32_t diff = kmn ^ kmx;
        if (diff == 0u) {
            T = kmn;
            need_eq = a.keff;
        } else {
            const int nbits = 32 - __clz(diff);
            uint32_t mask = nbits >= 32 ? 0u : (0xffffffffu << nbits);
            uint32_t prefix = kmn & mask;
            int krem = a.keff;
            for (int hi = nbits; hi > 0; hi -= kDigitBits) {
                const int lo = hi > kDigitBits ? hi - kDigitBits : 0;
                const int nb = 1 << (hi - lo);
                const uint32_t dmask = static_cast<uint32_t>(nb - 1);
                for (int i = tid; i < nb; i += kTopkThreads) hist[i] = 0;
                __syncthreads();
                for (int i = 0; i < c1 - c0; ++i) {
                    const uint32_t k = s_keys[i * kTopkThreads + tid];
                    if ((k & mask) == prefix) atomicAdd(&hist[(k >> lo) & dmask], 1);
                }
                __syncthreads();
                // thread t owns the 4 digits nb-1-4t .. nb-4-4t (descending order)
                int c4[4];
                int here = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int d = nb - 1 - 4 * tid - j;
                    c4[j] = d >= 0 ? hist[d] : 0;
                    here += c4[j];
                }
                const int above = cta_exclusive_scan(here, warp_sums, &s_total);
                if (above < krem && krem <= above + here) {
                    int acc = above;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (krem <= acc + c4[j]) {
                            s_digit = nb - 1 - 4 * tid - j;
                            s_above = acc;
                            break;
                        }
                        acc += c4[j];
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

    // ---- ascending list: sink blocks, taken candidates, recent blocks
    int32_t *dst = a.sel_idx + static_cast<size_t>(p) * a.nbmax;
    for (int j = tid; j < a.se; j += kTopkThreads) dst[j] = j;
    int gt_here = 0, eq_here = 0;
    if (a.mode == kTakeAll) {
        gt_here = c1 - c0;
    } else if (a.mode == kTakeTopK) {
        for (int i = 0; i < c1 - c0; ++i) {
            const uint32_t k = s_keys[i * kTopkThreads + tid];
            gt_here += k > T;
            eq_here += k == T;
        }
    }
    // counts stay below 2^16 (n <= 49152): greater in the low half, equal in the high
    const int pre = cta_exclusive_scan(gt_here | (eq_here << 16), warp_sums, &s_total);
    const int tot = s_total;
    const int gt_pre = pre & 0xffff, eq_pre = pre >> 16;
    // equal keys are taken in index order: the first need_eq of them
    int o = a.se + gt_pre + min(eq_pre, need_eq);
    if (a.mode == kTakeAll) {
        for (int j = c0; j < c1; ++j) dst[o++] = a.se + j;
    } else if (a.mode == kTakeTopK) {
        int r = eq_pre;
        for (int i = 0; i < c1 - c0; ++i) {
            const uint32_t k = s_keys[i * kTopkThreads + tid];
            const bool take = k > T || (k == T && r < need_eq);
            r += k == T;
            if (take) dst[o++] = a.se + c0 + i;
        }
    }
    const int taken = (tot & 0xffff) + min(tot >> 16, need_eq);
    for (int j = a.rb + tid; j < a.NB; j += kTopkThreads) dst[a.se + taken + (j - a.rb)] = j;
    if (tid == 0) a.sel_cnt[p] = a.se + taken + (a.NB - a.rb);
}

constexpr int score_smem_bytes(int G) {
    return kScoreStages * kScoreStageBytes + 2 * kScoreStages * 8 + G * kHeadDim * 4 + 16;
}

template <int G>
cudaError_t launch_score(const kvd_cache &c, const Geom &g, const float *q, int blk_lo, int n,
                         uint32_t *keys, float *ub, cudaStream_t st, bool pdl, bool overlap) {
    static bool attr_set = false;
    constexpr int smem = score_smem_bytes(G);
    if (!attr_set) {
        const cudaError_t e = cudaFuncSetAttribute(
            score_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // blocks per CTA: about two CTAs per SM in total, at least one stage each
    const long P = static_cast<long>(g.B) * g.Hkv;
    const long want = 2L * device_sm_count();
    long R = (static_cast<long>(n) * P + want - 1) / want;
    R = (R + kStageBlocks - 1) / kStageBlocks * kStageBlocks;
    if (R < kStageBlocks) R = kStageBlocks;
    dim3 grid(static_cast<unsigned>((n + R - 1) / R), static_cast<unsigned>(P));
    return launch_ex(score_kernel<G>, grid, dim3(kScoreThreads), smem, st, pdl, q,
                     static_cast<const __half *>(c.kbounds), g.Hkv, g.H, g.nbmax, blk_lo, n,
                     static_cast<int>(R), keys, ub, c.dev_status, overlap ? 1 : 0);
}

cudaError_t launch_score_any(const kvd_cache &c, const Geom &g, const float *q, int blk_lo,
                             int n, uint32_t *keys, float *ub, cudaStream_t st, bool pdl,
                             bool overlap) {
    switch (g.G) {
        case 1: return launch_score<1>(c, g, q, blk_lo, n, keys, ub, st, pdl, overlap);
        case 2: return launch_score<2>(c, g, q, blk_lo, n, keys, ub, st, pdl, overlap);
        case 4: return launch_score<4>(c, g, q, blk_lo, n, keys, ub, st, pdl, overlap);
        case 8: return launch_score<8>(c, g, q, blk_lo, n, keys, ub, st, pdl, overlap);
        case 16: return launch_score<16>(c, g, q, blk_lo, n, keys, ub, st, pdl, overlap);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_topk(const TopkArgs &a, int P, int n_cand, cudaStream_t st, bool pdl) {
    static bool attr_set = false;
    if (!attr_set) {
        const cudaError_t e =
            cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kMaxSelectBlocks * static_cast<int>(sizeof(uint32_t)));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // transposed key layout: ceil(n / 1024) * 1024 slots (<= kMaxSelectBlocks)
    const size_t slots = (static_cast<size_t>(n_cand) + kTopkThreads - 1) / kTopkThreads *
                         kTopkThreads;
    const size_t smem = (a.mode == kTakeTopK ? slots : 0) * sizeof(uint32_t);
    return launch_ex(topk_kernel, dim3(P), dim3(kTopkThreads), smem, st, pdl, a);
}

}  // namespace

int max_select_blocks() { return kMaxSelectBlocks; }

cudaError_t launch_select(const kvd_cache &c, const Geom &g, const float *q, int k_sel,
                          int sink_tokens, int recent_tokens, int32_t *sel_idx,
                          int32_t *sel_cnt, uint32_t *keys, cudaStream_t st, bool pdl,
                          bool after_step_append) {
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
    TopkArgs a;
    a.keys = keys;
    a.sel_idx = sel_idx;
    a.sel_cnt = sel_cnt;
    a.nbmax = g.nbmax;
    a.NB = NB;
    a.se = se;
    a.rb = rb;
    a.keff = keff;
    a.mode = (keff > 0 && keff < n_cand) ? kTakeTopK : (keff == 0 ? kTakeNone : kTakeAll);
    if (a.mode == kTakeTopK) {
        // the appended token's block is the last one; it is never a candidate
        // while the recent window is non-empty
        const bool overlap = after_step_append && recent_tokens > 0;
        const cudaError_t e =
            launch_score_any(c, g, q, se, n_cand, keys, nullptr, st, pdl, overlap);
        if (e != cudaSuccess) return e;
    }
    return launch_topk(a, g.B * g.Hkv, n_cand, st, pdl);
}

cudaError_t launch_scores_debug(const kvd_cache &c, const Geom &g, const float *q, float *ub,
                                cudaStream_t st) {
    return launch_score_any(c, g, q, 0, g.NB, nullptr, ub, st, false, false);
}

}  // namespace kvd
