// select_dev.cuh -- device side of the Quest block selection: block bounds,
// GQA max, top-K with the sink and recent blocks forced in.  Used by
// select_kernel and fill_kernel_varlen (select.cu).
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
// select_kernel: the candidate blocks of a problem (sequence, KV head) are
// split over X CTAs.  Each CTA streams the bounds (512 B per block) of its
// range through a TMA ring in shared memory, turns every block's group bound
// into an order-preserving u32 key (written to global scratch), and folds
// the keys' range [kmin, kmax] into the problem's.  It then takes a ticket;
// the last CTA of the problem to arrive finishes the selection alone, with
// the problem's keys in shared memory: the keff-th largest key T by a radix
// select whose first digit bins (key - kmin) over the keys' actual range
// (bounds of one problem are close together, so the top bits of the keys
// barely differ), one pass that marks the keys above T's bin and collects
// the few keys inside it, digits of those keys' low bits, then the
// ascending list written in index order.  No CTA waits for another.
// A problem of at most kSmallRank candidates skips the copy and the radix
// passes over the whole ring: its last CTA holds one key per thread and finds
// T from 8-bit radix digits over the keys' range (select_small).
//
// Modes (template MODE): kExport writes the bounds for the tests; kSelect
// selects; kVarlen finds each problem's geometry from its own sequence length
// on the device; kPerHead serves one query head of each group per launch
// (lists per query head, the ablation of the shared block set).
#pragma once

#include "append_dev.cuh"
#include "common.cuh"
#include "internal.h"

namespace kvd {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;

constexpr int kScoreWarps = 16;                      // consumers; warp 16 produces
constexpr int kScoreThreads = 32 * (kScoreWarps + 1);
constexpr int kConsumerThreads = 32 * kScoreWarps;
constexpr int kScoreSlots = 4;                       // blocks per warp per stage (8 lanes each)
constexpr int kStageBlocks = kScoreWarps * kScoreSlots;  // 64
constexpr int kBoundRowBytes = kHeadDim * 2 * 2;      // (kmin, kmax) f16 pairs: 512 B
constexpr int kScoreStages = 6;
constexpr int kScoreStageBytes = kStageBlocks * kBoundRowBytes;  // 32 KiB

constexpr int kMaxSelectBlocks = 49152;
constexpr int kMaxCtasPerProblem = 1024;
// The last CTA of a problem of at most this many candidates ranks them one
// key per thread (select_small): no key copy, no radix passes.
constexpr int kSmallRank = 512;

// Radix select over v = key - kmin: the first digit is v >> shift with
// shift the least that leaves at most kBins1 bins; later digits take up to
// kSubBits of the bits below.
constexpr int kBins1Bits = 11;
constexpr int kBins1 = 1 << kBins1Bits;
constexpr int kSubBits = 11;
constexpr int kSubBins = 1 << kSubBits;
// Keys the last CTA keeps in shared memory (the rest of the ring is its
// scratch); a larger problem's keys are read from L2.
constexpr int kRingKeys = 32768;
constexpr int kMaxWords = (kMaxSelectBlocks + 31) / 32;
// Keys of the threshold bin collected for the later digits, and the most
// that are ranked directly (against each other) instead.
constexpr int kCandCap = 2560;
constexpr int kRankMax = 256;
constexpr int kScratchBytes = kBins1 * 4 + 2 * kMaxWords * 4 + kCandCap * 8;
static_assert(kRingKeys * 4 + kScratchBytes <= kScoreStages * kScoreStageBytes,
              "keys and tail scratch must fit the ring");

enum TopkMode { kTakeNone = 0, kTakeAll = 1, kTakeTopK = 2 };
// Modes: kExport (bounds out), kSelect, and kSelect with the flags kVarlen
// (per-sequence lengths: each problem's own candidates, forced blocks and
// budget, found on the device) and kPerHead (one query head of each group per
// launch, head_sub; problem p writes list row p * G_all + head_sub).
enum SelMode { kExport = 0, kSelect = 1, kVarlen = 2, kPerHead = 4 };

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

struct SelArgs {
    const float *q;
    const __half *kbounds;
    int Hkv, H, nbmax;
    int se, n, R;          // candidates: blocks se .. se+n-1; R per CTA
    uint32_t *keys;        // [P][ldk] keys (scratch)
    int ldk;
    float *ub;             // kExport: [P][n] bounds
    unsigned *range;       // [P][2] max key, ~min key (zero between calls)
    unsigned *ticket;      // [P] arrival counters (zero between calls)
    int32_t *sel_idx, *sel_cnt;
    int NB, rb, keff;
    int32_t *dev_status;
    int overlap;
    // per-query-head selection (kPerHead, an ablation of the GQA-shared one):
    // this launch serves query head head_sub of every group of G_all heads
    int head_sub, G_all;
    int ldn;  // keys of a problem's row its last CTA copies: n rounded up to 4
    // per-sequence lengths (kVarlen): the rules the host applies to len
    const int32_t *seq_lens;
    int len_max, k_sel, sink_tokens, recent_tokens;
    int seq_add;  // tokens a decode step appended that seq_lens lacks
    // decode step: the token to append (app_k non-null), fused here because
    // its block is forced (never scored); app_cache.len is the length before
    kvd_cache app_cache;
    const __half *app_k, *app_v;
    unsigned long long *marks;  // stage marks (KVD_MARKS builds), or null
};

__device__ __forceinline__ int warp_inclusive_scan(int x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFullMask, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

struct RadixShared {
    int wsum[kScoreWarps + 1];
    int digit, above, last, first;
    unsigned kmin, kmax;  // the CTA's, then the problem's, key range
    int ccount;           // keys collected from the threshold bin
};

// Digit of the krem-th largest key from a shared-memory histogram of NBINS
// bins (left zeroed); krem becomes the rank within that digit.  The consumer
// thread t owns the digits NBINS-1-c*t .. NBINS-c*(t+1) (c = NBINS/256,
// descending).  All threads call it.
template <int NBINS>
__device__ int radix_digit(int *hist, int &krem, RadixShared &rs) {
    constexpr int c = NBINS / kConsumerThreads;
    static_assert(c >= 1 && (c < 4 || c % 4 == 0), "bins per thread");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __syncthreads();  // histogram complete
    int cnt[c];
    int here = 0;
    if (warp < kScoreWarps) {
        const int base = NBINS - c * (tid + 1);
        int v[c];
        if constexpr (c % 4 == 0) {
            // 4 bins per 16-byte access (base is a multiple of 4)
#pragma unroll
            for (int i = 0; i < c; i += 4) {
                int4 *h4 = reinterpret_cast<int4 *>(hist + base + i);
                const int4 w = *h4;
                *h4 = make_int4(0, 0, 0, 0);
                v[i] = w.x; v[i + 1] = w.y; v[i + 2] = w.z; v[i + 3] = w.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < c; ++i) {
                v[i] = hist[base + i];
                hist[base + i] = 0;
            }
        }
#pragma unroll
        for (int jj = 0; jj < c; ++jj) {
            cnt[jj] = v[c - 1 - jj];
            here += cnt[jj];
        }
    }
    const int incl = warp_inclusive_scan(here, lane);
    if (lane == 31 && warp < kScoreWarps) rs.wsum[warp] = incl;
    __syncthreads();
    if (warp < kScoreWarps) {
        const int wv = lane < kScoreWarps ? rs.wsum[lane] : 0;
        const int winc = warp_inclusive_scan(wv, lane);
        const int wex = __shfl_sync(kFullMask, winc - wv, warp);
        const int above = wex + incl - here;
        if (above < krem && krem <= above + here) {
            int acc = above;
#pragma unroll
            for (int jj = 0; jj < c; ++jj) {
                if (krem <= acc + cnt[jj]) {
                    rs.digit = NBINS - 1 - c * tid - jj;
                    rs.above = acc;
                    break;
                }
                acc += cnt[jj];
            }
        }
    }
    __syncthreads();
    krem -= rs.above;
    return rs.digit;
}

struct SelShared {
    RadixShared rs;
    int abort, issued;
};

// Count, into hist, the digit ((key - kmin) >> lo) & dmask of every key
// j < n whose bits above hi, (key - kmin) >> hi, equal prefix (hi < 32).
// PADDED: the row's keys up to the next multiple of 4 are counted too.
// Keys are read 16 per thread per round into registers before any atomic is
// issued, so the loads overlap and the shared atomics pipeline.
template <bool ALL, bool PADDED = false>
__device__ __forceinline__ void count_digits(const uint32_t *keys, int n, uint32_t kmin, int hi,
                                             uint32_t prefix, int lo, uint32_t dmask,
                                             int *hist) {
    const int nq = (n + 3) / 4;
    const uint4 *k4p = reinterpret_cast<const uint4 *>(keys);
    for (int q0 = threadIdx.x; q0 < nq; q0 += 4 * kScoreThreads) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int q = q0 + u * kScoreThreads;
            w[u] = q < nq ? k4p[q] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = 4 * (q0 + u * kScoreThreads);
            const uint32_t kk[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t v = kk[c] - kmin;
                // padded rows: whole 16-byte groups of the row count (the
                // padding keys are taken back out by the caller)
                if ((PADDED ? j < 4 * nq : j + c < n) && (ALL || (v >> hi) == prefix))
                    atomicAdd(&hist[(v >> lo) & dmask], 1);
            }
        }
    }
}

// Phase 4: the ascending list from the bitmaps of the keys above T (gtw)
// and equal to T (eqw; the need_eq lowest-index ones are taken), plus the
// forced sink and recent blocks, and the count.
__device__ __forceinline__ void select_write_list(const SelArgs &a, size_t row, int n,
                                                  const uint32_t *gtw, const uint32_t *eqw,
                                                  int need_eq, RadixShared &rs) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nw = (n + 31) / 32;
    // thread t owns words [t*wpt, (t+1)*wpt): an exclusive scan of the
    // packed counts (above | equal << 16; both below 2^16) orders them
    const int wpt = (nw + kScoreThreads - 1) / kScoreThreads;
    const int w0 = min(nw, tid * wpt), w1 = min(nw, w0 + wpt);
    unsigned mine = 0;
    for (int wi = w0; wi < w1; ++wi)
        mine += static_cast<unsigned>(__popc(gtw[wi])) | (static_cast<unsigned>(__popc(eqw[wi])) << 16);
    const unsigned incl = static_cast<unsigned>(warp_inclusive_scan(static_cast<int>(mine), lane));
    if (lane == 31) rs.wsum[warp] = static_cast<int>(incl);
    __syncthreads();
    if (tid == 0) KVD_MARK(a.marks, 12);  // list offsets scanned
    unsigned before = incl - mine;
    for (int w = 0; w < warp; ++w) before += static_cast<unsigned>(rs.wsum[w]);
    int g_before = static_cast<int>(before & 0xffffu), e_before = static_cast<int>(before >> 16);
    int32_t *dst = a.sel_idx + row * a.nbmax;
    for (int wi = w0; wi < w1; ++wi) {
        const uint32_t gm = gtw[wi], em = eqw[wi];
        uint32_t take = gm;
        int r = min(max(need_eq - e_before, 0), __popc(em));  // equal keys taken here
        for (uint32_t m = em; r > 0; --r) {
            take |= m & (0u - m);  // lowest remaining equal key
            m &= m - 1;
        }
        int o = a.se + g_before + min(e_before, need_eq);
        for (uint32_t m = take; m; m &= m - 1) dst[o++] = a.se + 32 * wi + (__ffs(m) - 1);
        g_before += __popc(gm);
        e_before += __popc(em);
    }
    for (int j = tid; j < a.se; j += kScoreThreads) dst[j] = j;
    for (int j = a.rb + tid; j < a.NB; j += kScoreThreads) dst[a.se + a.keff + (j - a.rb)] = j;
    if (tid == 0) a.sel_cnt[row] = a.se + a.keff + (a.NB - a.rb);
    if (lane == 0) KVD_MARK_LAST(a.marks, 13);  // the last warp's list entries written
}

// Phases 3-4 of the last CTA of a problem, with the problem's key range
// [kmin, kmax] in rs: the keff-th largest key T, then the ascending list
// from bitmaps of the keys above and equal to T.  ksrc: the keys (shared
// memory when IN_SMEM, else global); scratch: kScratchBytes of shared memory
// whose histogram part is zero.
template <bool IN_SMEM>
__device__ __forceinline__ void select_finish(const SelArgs &a, size_t row, int n,
                                              const uint32_t *ksrc, uint8_t *scratch,
                                              RadixShared &rs) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kWarps = kScoreWarps + 1;
    int *hist = reinterpret_cast<int *>(scratch);
    uint32_t *gtw = reinterpret_cast<uint32_t *>(scratch + kBins1 * 4);  // [nw] keys above T
    const int nw = (n + 31) / 32;
    uint32_t *eqw = gtw + nw;                                           // [nw] keys equal to T
    uint32_t *ck = gtw + 2 * kMaxWords;                                 // threshold-bin keys
    int *ci = reinterpret_cast<int *>(ck + kCandCap);                   // and their indices
    const uint32_t kmin = rs.kmin;
    const uint32_t range = rs.kmax - kmin;
    const int bits = range ? 32 - __clz(static_cast<int>(range)) : 0;
    const int shift = bits > kBins1Bits ? bits - kBins1Bits : 0;

    // ---- digit 1: the bin v >> shift of T (krem: keys still to take from it)
    count_digits<true, IN_SMEM>(ksrc, n, kmin, 31, 0u, shift, kBins1 - 1, hist);
    if (tid == 0) KVD_MARK(a.marks, 11);  // thread 0's keys counted
    int krem = a.keff;
    if (IN_SMEM && tid == 0) atomicAdd(&hist[0], n - (n + 3) / 4 * 4);  // padding keys (kmin)
    if (tid == 0) rs.ccount = 0;
    const int d1 = radix_digit<kBins1>(hist, krem, rs);
    if (tid == 0) KVD_MARK(a.marks, 7);  // first digit found

    // ---- one pass: keys in bins above d1 are in; keys in bin d1 are collected.
    // Thread t builds word t (keys 32t .. 32t+31) in registers, reading its
    // eight 16-byte chunks in a rotated order so that the eight lanes of a
    // quarter-warp hit distinct banks; a warp scan places the collected keys.
    // bin d1 holds the keys in [k_lo, k_hi): v >> shift == d1
    const uint64_t k_lo64 = static_cast<uint64_t>(kmin) + (static_cast<uint64_t>(d1) << shift);
    const uint64_t k_hi64 = k_lo64 + (1ull << shift);
    const uint32_t k_lo = static_cast<uint32_t>(k_lo64);          // <= kmax
    const bool none_above = k_hi64 > 0xffffffffull;
    const uint32_t k_hi = none_above ? 0xffffffffu : static_cast<uint32_t>(k_hi64);
    for (int w0 = 0; w0 < nw; w0 += kScoreThreads) {
        const int wi = w0 + tid;
        uint32_t gmask = 0u, cmask = 0u;
        if (wi < nw) {
            uint32_t lmask = 0u;
            const uint4 *k4 = reinterpret_cast<const uint4 *>(ksrc + 32 * wi);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int ch = (i + wi) & 7;
                const int jb = 32 * wi + 4 * ch;
                const uint4 w = jb < n ? k4[ch] : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t kk[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (kk[e] >= k_hi) gmask |= 1u << (4 * ch + e);
                    if (kk[e] >= k_lo) lmask |= 1u << (4 * ch + e);
                }
            }
            // keys past n (padding or beyond the row) are dropped here
            const int valid = n - 32 * wi;
            const uint32_t vmask = valid >= 32 ? 0xffffffffu : ((1u << valid) - 1u);
            if (none_above) gmask = 0u;
            gmask &= vmask;
            cmask = lmask & ~gmask & vmask;
            gtw[wi] = gmask;
            eqw[wi] = 0u;
        }
        const int cn = __popc(cmask);
        if (__any_sync(kFullMask, cn != 0)) {
            const int incl = warp_inclusive_scan(cn, lane);
            int at = 0;
            if (lane == 31) at = atomicAdd(&rs.ccount, incl);
            at = __shfl_sync(kFullMask, at, 31) + incl - cn;
            for (uint32_t mm = cmask; mm; mm &= mm - 1u, ++at) {
                const int j = 32 * wi + (__ffs(mm) - 1);
                if (at < kCandCap) {
                    ck[at] = ksrc[j];
                    ci[at] = j;
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0) KVD_MARK(a.marks, 8);  // above-bitmap written, threshold bin collected
    const int m = rs.ccount;
    const bool compact = m <= kCandCap;
    if (m <= kRankMax) {
        // few keys in the bin: each one's rank among them (key descending,
        // index ascending) decides it; the krem best join the list
        for (int c = warp; c < m; c += kWarps) {
            const uint32_t kc = ck[c];
            const int jc = ci[c];
            int beats = 0;
            for (int o = lane; o < m; o += 32) {
                const uint32_t ko = ck[o];
                beats += ko > kc || (ko == kc && ci[o] < jc);
            }
            beats = __reduce_add_sync(kFullMask, beats);
            if (lane == 0 && beats < krem) atomicOr(&gtw[jc >> 5], 1u << (jc & 31));
        }
        __syncthreads();
        if (tid == 0) KVD_MARK(a.marks, 9);  // threshold bin ranked
        select_write_list(a, row, n, gtw, eqw, 0, rs);
        return;
    }

    // ---- the bits of v below the bin, kSubBits at a time, over bin d1's keys
    // (the collected ones, or every key again when too many were in the bin)
    uint32_t prefix = static_cast<uint32_t>(d1);
    int hi = shift;
    while (hi > 0) {
        const int db = hi < kSubBits ? hi : kSubBits;
        const int lo = hi - db;
        const uint32_t dmask = (1u << db) - 1u;
        if (compact) {
            for (int c = tid; c < m; c += kScoreThreads) {
                const uint32_t v = ck[c] - kmin;
                if ((v >> hi) == prefix) atomicAdd(&hist[(v >> lo) & dmask], 1);
            }
        } else {
            count_digits<false>(ksrc, n, kmin, hi, prefix, lo, dmask, hist);
        }
        const int d = radix_digit<kSubBins>(hist, krem, rs);
        prefix = (prefix << db) | static_cast<uint32_t>(d);
        hi = lo;
    }
    const uint32_t T = kmin + prefix;
    const int need_eq = krem;  // keys equal to T to take, lowest index first

    // ---- bin d1's keys above / equal to T join the bitmaps
    if (compact) {
        for (int c = tid; c < m; c += kScoreThreads) {
            const uint32_t k = ck[c];
            const int j = ci[c];
            if (k > T)
                atomicOr(&gtw[j >> 5], 1u << (j & 31));
            else if (k == T)
                atomicOr(&eqw[j >> 5], 1u << (j & 31));
        }
    } else {
        for (int wi = warp; wi < nw; wi += kWarps) {
            const int j = 32 * wi + lane;
            const uint32_t k = j < n ? ksrc[j] : 0u;
            const bool inbin = j < n && ((k - kmin) >> shift) == static_cast<uint32_t>(d1);
            const unsigned gm = __ballot_sync(kFullMask, inbin && k > T);
            const unsigned em = __ballot_sync(kFullMask, inbin && k == T);
            if (lane == 0) {
                gtw[wi] |= gm;
                eqw[wi] = em;
            }
        }
    }
    __syncthreads();
    if (tid == 0) KVD_MARK(a.marks, 9);  // threshold found by the later digits

    // ================================================= phase 4: the list
    select_write_list(a, row, n, gtw, eqw, need_eq, rs);
}

// Out of line: code the common path does not run stays off its instruction
// stream (after an L2 flush each kernel's instructions come from HBM again).
// The decode step's token, appended by one warp of the first tile.
__device__ __noinline__ void fused_append(const SelArgs &a, int b, int g, int lane) {
    const int len0 = a.app_cache.len, blk = len0 / kBlock;
    const kvd_cache &c = a.app_cache;
    if (c.dtype == KVD_Q8_0)
        append_block_warp<KVD_Q8_0, false>(c, a.app_k, a.app_v, 1, len0, blk, b, g, lane);
    else if (c.dtype == KVD_Q4_0)
        append_block_warp<KVD_Q4_0, false>(c, a.app_k, a.app_v, 1, len0, blk, b, g, lane);
    else if (c.dtype == KVD_F16)
        append_block_warp<KVD_F16, false>(c, a.app_k, a.app_v, 1, len0, blk, b, g, lane);
    else
        append_block_warp<KVD_INT8, false>(c, a.app_k, a.app_v, 1, len0, blk, b, g, lane);
}

// The tail of a problem too large for its keys to fit the ring.
__device__ __noinline__ void select_finish_from_l2(const SelArgs &a, size_t row, int n,
                                                   const uint32_t *keys, uint8_t *scratch,
                                                   RadixShared &rs) {
    select_finish<false>(a, row, n, keys, scratch, rs);
}

// Exclusive sum, over the CTA's threads in order, of v; every thread calls
// (wsum: kScoreWarps + 1 ints of shared memory).
__device__ __forceinline__ int block_exclusive_sum(int v, int *wsum) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int incl = warp_inclusive_scan(v, lane);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = incl - v;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    __syncthreads();  // wsum free for the next call
    return before;
}

// The list of a problem of n <= kSmallRank candidates, by its last CTA once
// every key of row kp is in: thread t holds key t.  With v = key - kmin over
// the keys' range, the keff-th largest v, T, comes from 8-bit radix digits,
// top down: each pass counts the digit of every key that matches the digits
// found so far into a 256-bin histogram in shared memory (keys visited 37
// apart, so that neighbouring blocks' close keys do not pile onto one bin in
// one instruction), and warp 0 finds the digit by a warp scan.  Keys above T
// are in, and of the keys equal to T the lowest indices fill the rest; one
// scan of packed counts places them.  Two CTA barriers a pass (the histograms
// alternate between two buffers, the idle one cleared by warp 1), where
// building T bit by bit took 32 block-wide counts.  scratch: 4.3 KiB of
// shared memory.  All threads call.
__device__ __forceinline__ void select_small(const SelArgs &a, size_t row, int n,
                                             const uint32_t *kp, uint8_t *scratch,
                                             RadixShared &rs) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int *hist = reinterpret_cast<int *>(scratch);                       // [2][256]
    uint32_t *ks = reinterpret_cast<uint32_t *>(scratch + 2048);        // [kSmallRank]
    uint32_t *wmm = ks + kSmallRank;                                    // [2][kScoreWarps + 1]
    constexpr int kWarps = kScoreWarps + 1;
    const bool have = tid < n;
    const uint32_t key = have ? __ldcg(kp + tid) : 0u;
    if (have) ks[tid] = key;
    for (int i = tid; i < 512; i += kScoreThreads) hist[i] = 0;
    const uint32_t lo = __reduce_min_sync(kFullMask, have ? key : 0xffffffffu);
    const uint32_t hi = __reduce_max_sync(kFullMask, have ? key : 0u);
    if (lane == 0) {
        wmm[warp] = lo;
        wmm[kWarps + warp] = hi;
    }
    __syncthreads();
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int w = 0; w < kWarps; ++w) {
        kmin = min(kmin, wmm[w]);
        kmax = max(kmax, wmm[kWarps + w]);
    }
    const uint32_t range = kmax - kmin;
    int hb = range ? 32 - __clz(static_cast<int>(range)) : 0;  // v < 2^hb
    // the key this thread counts (37 is odd: a permutation of 0 .. 511)
    const int jc = (tid * 37) & 511;
    const bool counts = tid < 512 && jc < n;
    const uint32_t vc = counts ? ks[jc] - kmin : 0u;
    int krem = a.keff;  // keys still to take among those matching prefix
    uint32_t prefix = 0u;
    for (int pass = 0; hb > 0; ++pass) {
        const int db = hb < 8 ? hb : 8, lo_b = hb - db;
        int *h = hist + 256 * (pass & 1);
        if (counts && (hb >= 32 || (vc >> hb) == prefix))
            atomicAdd(&h[(vc >> lo_b) & ((1u << db) - 1u)], 1);
        __syncthreads();  // (A) the pass's histogram is complete
        if (warp == 0) {
            // lane l takes bins 255 - 8l down to 248 - 8l: a scan counts from the top
            int c8[8], sum = 0;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                c8[jj] = h[255 - 8 * lane - jj];
                sum += c8[jj];
            }
            const int incl = warp_inclusive_scan(sum, lane);
            const int above = incl - sum;
            if (above < krem && krem <= incl) {
                int acc = above;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    if (krem > acc && krem <= acc + c8[jj]) {
                        rs.digit = 255 - 8 * lane - jj;
                        rs.above = acc;
                    }
                    acc += c8[jj];
                }
            }
        } else if (warp == 1) {
            // the other buffer (read by warp 0 in the previous pass) for the next
            int *hn = hist + 256 * ((pass + 1) & 1);
            for (int i = lane; i < 256; i += 32) hn[i] = 0;
        }
        __syncthreads();  // (B) the digit is known; the next buffer is clear
        prefix = (prefix << db) | static_cast<uint32_t>(rs.digit);
        krem -= rs.above;
        hb = lo_b;
    }
    // prefix = T - kmin; krem of the keys equal to T are taken, lowest index first.
    // One scan of (keys above T) | (keys equal to T) << 16 places every key:
    // position = above-T keys before it + min(equal keys before it, krem).
    const uint32_t v = key - kmin;
    const bool gt = have && v > prefix, eq = have && v == prefix;
    const int packed = (gt ? 1 : 0) | (eq ? 1 << 16 : 0);
    const int before = block_exclusive_sum(packed, rs.wsum);
    const int g_before = before & 0xffff, e_before = before >> 16;
    int32_t *dst = a.sel_idx + row * a.nbmax;
    if (gt || (eq && e_before < krem)) dst[a.se + g_before + min(e_before, krem)] = a.se + tid;
    for (int j = tid; j < a.se; j += kScoreThreads) dst[j] = j;
    for (int j = a.rb + tid; j < a.NB; j += kScoreThreads) dst[a.se + a.keff + (j - a.rb)] = j;
    if (tid == 0) a.sel_cnt[row] = a.se + a.keff + (a.NB - a.rb);
}

// Phases 3-4 by the last CTA of problem p: the problem's keys into the ring
// (when they fit), the key range, then the radix select and the list.
__device__ __forceinline__ void select_rank(const SelArgs &a, int p, size_t row, int n, int X,
                                            const uint32_t *kp, bool in_smem, uint8_t *ring,
                                            RadixShared &rs) {
    const int tid = threadIdx.x;
    // the problem's key range: loads issued ahead of the copy, used after it
    unsigned *rg = a.range + 2 * static_cast<size_t>(p);
    unsigned r_max = 0u, r_nmin = 0u;
    if (X > 1 && tid == 0) {
        r_max = __ldcg(rg);
        r_nmin = __ldcg(rg + 1);
    }
    if (in_smem) {
        // the problem's keys (L2-resident) into the ring, 16 bytes per thread
        // and load, eight loads in flight per thread before any store
        const int nq = a.ldn / 4;
        const uint4 *src = reinterpret_cast<const uint4 *>(kp);
        uint4 *dst = reinterpret_cast<uint4 *>(ring);
        for (int i0 = tid; i0 < nq; i0 += 8 * kScoreThreads) {
            uint4 w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * kScoreThreads;
                w[u] = i < nq ? __ldcg(src + i) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * kScoreThreads;
                if (i < nq) dst[i] = w[u];
            }
        }
    }
    // tail scratch: the ring past the keys (the histogram part zeroed)
    uint8_t *scratch = ring + (in_smem ? kRingKeys * 4 : 0);
    {
        int4 *h4 = reinterpret_cast<int4 *>(scratch);
        for (int i = tid; i < kBins1 / 4; i += kScoreThreads) h4[i] = make_int4(0, 0, 0, 0);
    }
    if (X > 1 && tid == 0) {
        rs.kmax = r_max;
        rs.kmin = ~r_nmin;
        __stcg(rg, 0u);  // leave the words ready for the next call
        __stcg(rg + 1, 0u);
        a.ticket[p] = 0u;
    }

    // ================================================= phase 3: T
    __syncthreads();  // keys copied; the range in rs
    if (tid == 0) KVD_MARK(a.marks, 6);  // keys in shared memory
    // the row's padding keys (up to 3 past n) read as kmin: bin 0, taken back out
    if (in_smem && tid < a.ldn - n) reinterpret_cast<uint32_t *>(ring)[n + tid] = rs.kmin;
    __syncthreads();
    // the rest reads the keys from shared memory, or from L2 for a problem too
    // large for the ring; each variant is compiled with its address space known
    if (in_smem)
        select_finish<true>(a, row, n, reinterpret_cast<const uint32_t *>(ring), scratch, rs);
    else
        select_finish_from_l2(a, row, n, kp, scratch, rs);
}

// Problem p's own selection geometry under per-sequence lengths.  take: 0
// ranks nothing beyond the forced blocks, 1 takes every candidate, 2 ranks.
__device__ __forceinline__ int problem_args(const SelArgs &a, int p, SelArgs &v) {
    v = a;
    const int L =
        seq_len_of(a.seq_lens, p / a.Hkv, a.len_max - a.seq_add, a.dev_status) + a.seq_add;
    const ForcedRange f = forced_range(L, a.sink_tokens, a.recent_tokens);
    v.NB = f.NB;
    v.se = f.se;
    v.rb = f.rb;
    v.n = f.rb - f.se;
    v.keff = a.k_sel < v.n ? a.k_sel : v.n;
    v.ldn = (v.n + 3) / 4 * 4;
    return v.keff == 0 ? 0 : v.keff == v.n ? 1 : 2;
}

// The list of a problem that ranks nothing: sink blocks, every candidate when
// take_all, recent blocks; threads tid of nthr.
__device__ __forceinline__ void fill_list(const SelArgs &v, size_t row, bool take_all, int tid,
                                          int nthr) {
    int32_t *dst = v.sel_idx + row * v.nbmax;
    const int n_take = take_all ? v.rb - v.se : 0;
    for (int j = tid; j < v.se + n_take; j += nthr) dst[j] = j;
    for (int j = v.rb + tid; j < v.NB; j += nthr) dst[v.se + n_take + (j - v.rb)] = j;
    if (tid == 0) v.sel_cnt[row] = v.se + n_take + (v.NB - v.rb);
}

// CTA (x, p): candidate blocks j in [x*R, min(n, (x+1)*R)) of problem p,
// i.e. cache blocks se + j.  Their bounds stream through a TMA ring (stages
// of 64 blocks; warp 16 produces, warps 0..15 consume, warp w scoring blocks
// 4w..4w+3 of each stage two at a time).
template <int G, int MODE>
__device__ void select_body(const SelArgs &a_in, int x_tile, int n_tiles, int p, uint8_t *smem,
                            SelShared &ss) {
    // per-sequence lengths: this problem's own geometry (a copy of the args)
    constexpr bool kVar = (MODE & kVarlen) != 0, kOneHead = (MODE & kPerHead) != 0;
    SelArgs av;
    int take = 2;
    if constexpr (kVar) take = problem_args(a_in, p, av);
    const SelArgs &a = kVar ? av : a_in;
    // the list row this problem writes
    const size_t row = kOneHead ? static_cast<size_t>(p) * a_in.G_all + a_in.head_sub
                                : static_cast<size_t>(p);
    constexpr int NH = G < 4 ? G : 4;
    RadixShared &rs = ss.rs;
    int &s_abort = ss.abort;
    int &s_issued = ss.issued;
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kScoreStages * kScoreStageBytes);
    uint64_t *empty = full + kScoreStages;
    float *q_s = reinterpret_cast<float *>(empty + kScoreStages);
    volatile int *abort_flag = &s_abort;

    const int b = p / a.Hkv, g = p % a.Hkv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = lane >> 4, e = lane & 15;
    const int j0 = x_tile * a.R;
    const int j1 = min(a.n, j0 + a.R);
    const int nstage = (j1 - j0 + kStageBlocks - 1) / kStageBlocks;

    if (tid == 0) {
        for (int i = 0; i < kScoreStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kScoreWarps);
        }
        s_abort = 0;
        s_issued = 0;
        rs.kmin = 0xffffffffu;
        rs.kmax = 0u;
        fence_barrier_init();
        KVD_MARK(a_in.marks, 0);  // entry
    }
    __syncthreads();
    // overlap: inside a decode step whose appended token lands in a forced
    // block, the candidate bounds and the query are complete before the
    // upstream append runs, so scoring overlaps it; the grid-dependency wait
    // then comes before anything shared with earlier kernels is written.
    if (!a.overlap) pdl_wait();
    pdl_launch_dependents();
    if constexpr (kVar) {
        if (take < 2) {  // nothing to rank in this sequence: the first CTA fills
            if (x_tile == 0) fill_list(a, row, take == 1, tid, kScoreThreads);
            return;
        }
    }

    // ================================================= phase 1: keys
    const size_t base = static_cast<size_t>(p) * a.nbmax + a.se;  // row of candidate 0
    if (warp == kScoreWarps) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int issued = 0;
            for (int si = 0; si < nstage; ++si) {
                const int s = si % kScoreStages;
                if (si >= kScoreStages &&
                    !mbar_wait(&empty[s], ((si / kScoreStages) - 1) & 1, abort_flag)) {
                    s_abort = 1;
                    report_status(a.dev_status, KVD_ERR_TIMEOUT);
                    break;
                }
                const int jb = j0 + si * kStageBlocks;
                const int cnt = min(kStageBlocks, j1 - jb);
                const uint32_t bytes = static_cast<uint32_t>(cnt) * kBoundRowBytes;
                mbar_arrive_expect_tx(&full[s], bytes);
                tma_load_1d(ring + s * kScoreStageBytes, a.kbounds + (base + jb) * kHeadDim * 2,
                            bytes, &full[s], pol);
                issued = si + 1;
            }
            s_issued = issued;
        }
    } else {
        // the producer's first copies are in flight while the query loads
        const size_t h0 = kOneHead ? static_cast<size_t>(g) * a.G_all + a.head_sub
                                   : static_cast<size_t>(g) * G;
        const float *qg = a.q + (static_cast<size_t>(b) * a.H + h0) * kHeadDim;
        for (int i = tid; i < G * kHeadDim; i += kConsumerThreads) q_s[i] = qg[i];
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
        float2 qreg[NH][8];
        if constexpr (G <= 4) load_qpairs<NH>(q_s, 0, e, qreg);
        const int sw = chunk_swap(e);
        uint32_t tmin = 0xffffffffu, tmax = 0u;  // range of this thread's keys
        for (int si = 0; si < nstage; ++si) {
            const int s = si % kScoreStages;
            const bool ok = mbar_wait(&full[s], (si / kScoreStages) & 1, abort_flag);
            if (!__all_sync(kFullMask, ok)) {
                if (lane == 0) {
                    s_abort = 1;
                    report_status(a.dev_status, KVD_ERR_TIMEOUT);
                }
                break;
            }
            if (si == 0 && tid == 0) KVD_MARK(a.marks, 1);  // first bounds in
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
                    if constexpr (MODE != kExport) {
                        const uint32_t key = float_to_key(sc[ps]);
                        a.keys[static_cast<size_t>(p) * a.ldk + jr[ps]] = key;
                        tmin = min(tmin, key);
                        tmax = max(tmax, key);
                    } else {
                        a.ub[static_cast<size_t>(p) * a.n + jr[ps]] = sc[ps];
                    }
                }
            }
        }
        if (tid == 0) KVD_MARK(a.marks, 2);  // warp 0 scored its blocks
        if constexpr (MODE != kExport) {
            tmin = __reduce_min_sync(kFullMask, tmin);
            tmax = __reduce_max_sync(kFullMask, tmax);
            if (lane == 0) {
                atomicMin(&rs.kmin, tmin);
                atomicMax(&rs.kmax, tmax);
            }
        }
    }
    __syncthreads();
    if (s_abort) {
        if (warp == kScoreWarps && lane == 0) {
            // wind down: wait (bounded) for the copies still landing in the ring
            const int issued = s_issued;
            volatile int never = 0;
            for (int i = max(0, issued - kScoreStages); i < issued; ++i)
                (void)mbar_wait(&full[i % kScoreStages], (i / kScoreStages) & 1, &never);
        }
        if (a.overlap) pdl_wait();
        return;
    }
    if (a.overlap) pdl_wait();  // the upstream kernels are complete past here
    if constexpr (MODE == kExport) return;
    // The decode step's token for (b, g) is appended by warp 0 of the first
    // CTA of the problem to take its ticket, after the dependency wait (the
    // previous step's kernels may still read the row it replaces) and off the
    // way to the ranking, which the last CTA does (a problem of one CTA
    // appends after its ranking).  The step's decode kernel waits for this
    // whole grid, so it sees the token.

    // ================================================= phase 2: ticket
    const int X = n_tiles;
    const int n = a.n;
    const uint32_t *kp = a.keys + static_cast<size_t>(p) * a.ldk;
    const bool in_smem = n <= kRingKeys;
    if (X > 1) {
        // this CTA's key range into the problem's (max key, ~min key: both
        // zero-based maxima), then the ticket; its release covers the keys
        __syncthreads();
        if (tid == 0) {
            KVD_MARK(a.marks, 3);  // every warp scored
            if (n > kSmallRank) {  // the radix tail bins over the keys' range
                unsigned *rg = a.range + 2 * static_cast<size_t>(p);
                atomicMax(rg, rs.kmax);
                atomicMax(rg + 1, ~rs.kmin);
            }
            const unsigned t = atomic_add_acq_rel_gpu(a.ticket + p, 1u);
            rs.last = t == static_cast<unsigned>(X - 1);
            rs.first = t == 0u;
            KVD_MARK(a.marks, 4);  // ticket taken
        }
        __syncthreads();
    }
    // the first CTA to arrive appends the step's token; the last (every key
    // is in) ranks
    const bool appends = a.app_k && warp == 0 && (X == 1 || rs.first);
    if (appends && X > 1) fused_append(a, b, g, lane);
    if (X == 1 || rs.last) {
        if (n <= kSmallRank) {
            __syncthreads();  // (X == 1) this CTA's key stores, seen by all its threads
            if (X > 1 && tid == 0) a.ticket[p] = 0u;  // ready for the next call
            select_small(a, row, n, kp, ring, rs);
        } else {
            select_rank(a, p, row, n, X, kp, in_smem, ring, rs);
        }
        if (tid == 0) KVD_MARK(a.marks, 5);  // list written
    }
    if (appends && X == 1) fused_append(a, b, g, lane);
    if (tid == 0) KVD_MARK(a.marks, 10);  // exit
}


template <int G>
constexpr int select_smem_bytes() {
    return kScoreStages * kScoreStageBytes + 2 * kScoreStages * 8 + G * kHeadDim * 4;
}

}  // namespace
}  // namespace kvd
