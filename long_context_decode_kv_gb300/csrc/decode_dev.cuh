// decode_dev.cuh -- device side of the split-KV decode (decode_kernel) over
// the selected KV blocks (or all of them for the dense arm).
//
// "Sparse Attention -- Quest-style block-selector for long-context decode
// (#551)", S3 "FA-VEC block-skip": unselected blocks are skipped before the
// K read, the q.k product and the V accumulation; the long-context decode hot
// path is the vector kernel, not MMA -- no tensor cores: the work is 2-4
// multiply-adds per byte read, so HBM bandwidth bounds it.
// "cpu-attn", Method: int8 rows with per-token scales, exact int32 q.k dots
// on the query quantized once per head, f32 softmax and f32 accumulation.
// "SCSA", Mechanism: an online-softmax (max, sum, accumulator) gauge over an
// ascending sweep, merged across splits.
//
// CTA = (split s of the block list, sequence b, KV head g, head subgroup).
// The last warp is the producer: one lane streams each
// listed 64-token block (K, V and, for int8, both scale rows) into a ring of
// shared-memory stages with 1-D TMA bulk copies completing on an mbarrier.
// The other warps form two consumer groups of four (four groups in the wide
// tile, one CTA per SM) that take blocks in turn, so more warps hide each
// other's latencies; within a group warp w owns
// tokens 16w..16w+15 of the block and keeps its own online-softmax state for
// the CTA's query heads, so no CTA-wide barrier is needed per block.  PV runs
// on packed f32x2 FMAs.  At the end the warp states merge in shared memory
// and the CTA writes a partial (m, l, acc[128]) per head; the last CTA of the
// problem to arrive merges all splits.  Variants: sparse-V (SV), the moment
// tail of the unlisted blocks (TAIL), per-sequence lengths and per-head lists
// (run-time arguments).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace kvd {
namespace {


constexpr int kWarpsPerGroup = 4;
constexpr int kTokensPerWarp = kBlock / kWarpsPerGroup;    // 16
// q4_0 PV weights: floats from one token's [4 groups][4 heads] pairs to the
// next token's; 40 (not 32) puts tokens t and t + 1..3 on distinct banks, so
// the pair stores of a QK pass take two wavefronts, not eight.
constexpr int kQ4PwTok = 40;
// Partial rows: m, l, two pad words, acc[128] (acc 16-byte aligned).
constexpr int kPartStride = kHeadDim + 4;
constexpr int kAccOff = 4;
constexpr int kMaxSplits = 256;
constexpr unsigned kFull = 0xffffffffu;
// Stage marker that ends a consumer group's loop.
constexpr int kEndMark = -2;
// Moment-tail stages carry kTailBase - chunk (chunk >= 0) as their block.
constexpr int kTailBase = -16;
// One block's moment row: the f16 key mean, then the f16 value mean.
constexpr int kMomentBytes = 2 * kHeadDim * 2;

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

template <int DT>
struct Tile;
template <>
struct Tile<KVD_INT8> {
    static constexpr int kRowBytes = kHeadDim;                        // int8 codes
    static constexpr int kKBytes = kBlock * kRowBytes;                // 8192
    static constexpr int kStageBytes = 2 * kKBytes + 2 * kBlock * 4;  // + both scale rows
    static constexpr int kGroups = 2;   // consumer groups (4 warps each)
    static constexpr int kStages = 6;   // a multiple of kGroups
    static constexpr int kTailRecs = 32;  // moment rows per tail stage
    static constexpr int kMinCtas = 2;
    static constexpr int kConsumerWarps = kGroups * kWarpsPerGroup;
    static constexpr int kThreads = 32 * (kConsumerWarps + 1);
};
template <>
struct Tile<KVD_Q8_0> {
    static constexpr int kRowBytes = kHeadDim;                        // int8 codes
    static constexpr int kKBytes = kBlock * kRowBytes;                // 8192
    static constexpr int kScaleBytes = kBlock * (kHeadDim / 32) * 2;  // f16 group scales: 512
    static constexpr int kStageBytes = 2 * kKBytes + 2 * kScaleBytes;
    static constexpr int kGroups = 2;
    static constexpr int kStages = 6;   // a multiple of kGroups
    static constexpr int kTailRecs = 32;
    static constexpr int kMinCtas = 2;
    static constexpr int kConsumerWarps = kGroups * kWarpsPerGroup;
    static constexpr int kThreads = 32 * (kConsumerWarps + 1);
};
template <>
struct Tile<KVD_Q4_0> {
    static constexpr int kRowBytes = kHeadDim / 2;                    // 4-bit codes
    static constexpr int kKBytes = kBlock * kRowBytes;                // 4096
    static constexpr int kScaleBytes = kBlock * (kHeadDim / 32) * 2;  // f16 group scales: 512
    static constexpr int kStageBytes = 2 * kKBytes + 2 * kScaleBytes;
    static constexpr int kGroups = 2;
    static constexpr int kStages = 10;  // a multiple of kGroups
    static constexpr int kTailRecs = 16;  // 8 KiB of a 9 KiB stage
    static constexpr int kMinCtas = 2;
    static constexpr int kConsumerWarps = kGroups * kWarpsPerGroup;
    static constexpr int kThreads = 32 * (kConsumerWarps + 1);
};
template <>
struct Tile<KVD_F16> {
    static constexpr int kRowBytes = 2 * kHeadDim;                    // f16
    static constexpr int kKBytes = kBlock * kRowBytes;                // 16384
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kGroups = 2;
    static constexpr int kStages = 4;   // a multiple of kGroups
    static constexpr int kTailRecs = 32;
    static constexpr int kMinCtas = 1;
    static constexpr int kConsumerWarps = kGroups * kWarpsPerGroup;
    static constexpr int kThreads = 32 * (kConsumerWarps + 1);
};

// The wide variant of a tile: twice the consumer groups and stages in one CTA
// per SM.  With few problems (long single sequences) one CTA per SM keeps its
// warps at one scheduling priority, where two CTAs per SM let the older one
// finish its share first and the younger one set the launch's end.
template <int DT, bool WIDE>
struct TileW : Tile<DT> {
    static constexpr int kGroups = (WIDE ? 2 : 1) * Tile<DT>::kGroups;
    static constexpr int kStages = (WIDE ? 2 : 1) * Tile<DT>::kStages;
    static constexpr int kMinCtas = WIDE ? 1 : Tile<DT>::kMinCtas;
    static constexpr int kConsumerWarps = kGroups * kWarpsPerGroup;
    static constexpr int kThreads = 32 * (kConsumerWarps + 1);
};

struct DecodeArgs {
    const void *k, *v;
    const void *k_scale, *v_scale;  // f32 per token (int8) or f16 per group (q8_0, q4_0)
    const __half *moments;          // block means (moment tail), or null
    const float *q;
    float *out;
    const int32_t *sel_idx, *sel_cnt;
    float *partials;
    uint32_t *counters;  // [problems] split arrivals
    int32_t *dev_status;
    int Hkv, H, G, max_seq, nbmax, len, NB, splits, subgroups;
    int plan_blocks;     // list length the splits were planned for (<= NB)
    float sv_eps;        // sparse-V (eps mode): 0 = every V term accumulated
    float scale_log2;  // softmax_scale * log2(e): logits live in base 2
    int early_q;       // q is complete before the upstream kernels finish
    int per_head;      // lists per query head ([B, H] rows; one head per CTA)
    const int32_t *seq_lens;  // per-sequence lengths (<= len), or null
    int seq_add;              // tokens appended by this step that seq_lens lacks
    unsigned long long *marks;  // stage marks (KVD_MARKS builds), or null
};

template <int DT, int GC, bool TAIL = false, bool WIDE = false>
struct SmemLayout {
    using T = TileW<DT, WIDE>;
    static constexpr int kStageBytes = T::kStageBytes;
    static constexpr int kStages = T::kStages;
    static constexpr int kStagesOff = 0;
    static constexpr int kRing = kStages * kStageBytes;
    static_assert(T::kTailRecs * kMomentBytes <= kStageBytes, "tail stage overflows");
    // merge rows: one state per consumer warp and head (two with the tail)
    static constexpr int kRows = (TAIL ? 2 : 1) * T::kConsumerWarps;
    // after the loop the ring holds the warp merge, then the split weights
    static constexpr int kMergeBytes = kRows * GC * kPartStride * 4;
    // split merge: (m, l) and the accumulators of every thread part
    static constexpr int kWeightBytes = T::kConsumerWarps * 32 * (16 + 8);
    static constexpr int kScratch = kMergeBytes > kWeightBytes ? kMergeBytes : kWeightBytes;
    static constexpr int kBarOff = (kRing > kScratch ? kRing : kScratch);
    static constexpr int kFullOff = kBarOff;
    static constexpr int kEmptyOff = kFullOff + 8 * kStages;
    static constexpr int kBlkOff = kEmptyOff + 8 * kStages;
    static constexpr int kQOff = (kBlkOff + 4 * kStages + 15) / 16 * 16;
    static constexpr int kQBytes = GC * kHeadDim * 4;  // f32 q (f16 cache) or codes
    static constexpr int kCoefOff = kQOff + kQBytes;
    static constexpr int kQsumOff = kCoefOff + 16;  // q4_0: [GC][4] group sums of the codes
    static constexpr int kPwOff = kQsumOff + 64;
    // per warp: [16 tokens][4 heads] pairs (p, p); q4_0: [16 tokens][4 groups]
    // [4 heads] pairs (w, w / 16), w = p times the group's value scale
    static constexpr int kPwWarpFloats = kTokensPerWarp * (DT == KVD_Q4_0 ? kQ4PwTok : 4 * 2);
    static constexpr int kPwBytes = T::kConsumerWarps * kPwWarpFloats * 4;
    static constexpr int kLOff = kPwOff + kPwBytes;  // split merge: L per head
    static constexpr int kFlagOff = kLOff + 16;
    // moment tail: the listed-block mask of each stage
    static constexpr int kMaskOff = kFlagOff + 16;
    static constexpr int kTotal = kMaskOff + (TAIL ? 4 * kStages : 0);
};

// ----------------------------------------------------------------------------
// Reductions (int32 or f32) over the 4 quarter lanes (lane bits 0..1)
// returning to each lane the total of head (c * GC) / 4.
template <int GC, typename T>
__device__ __forceinline__ T reduce4_scatter(T (&v)[GC], int c) {
    if constexpr (GC == 4) {
        const bool up = (c & 2) != 0;
        T k0 = up ? v[2] : v[0], k1 = up ? v[3] : v[1];
        const T s0 = up ? v[0] : v[2], s1 = up ? v[1] : v[3];
        k0 += __shfl_xor_sync(kFull, s0, 2);
        k1 += __shfl_xor_sync(kFull, s1, 2);
        const bool lo = (c & 1) != 0;
        T k = lo ? k1 : k0;
        k += __shfl_xor_sync(kFull, lo ? k0 : k1, 1);
        return k;
    } else if constexpr (GC == 2) {
        const bool up = (c & 2) != 0;
        T k = up ? v[1] : v[0];
        k += __shfl_xor_sync(kFull, up ? v[0] : v[1], 2);
        k += __shfl_xor_sync(kFull, k, 1);
        return k;
    } else {
        T k = v[0];
        k += __shfl_xor_sync(kFull, k, 2);
        k += __shfl_xor_sync(kFull, k, 1);
        return k;
    }
}

// f32 version over the 8 eighth lanes (lane bits 0..2): head (e * GC) / 8.
template <int GC>
__device__ __forceinline__ float reduce8_scatter(float (&v)[GC], int e) {
    if constexpr (GC == 4) {
        const bool up = (e & 4) != 0;
        float k0 = up ? v[2] : v[0], k1 = up ? v[3] : v[1];
        const float s0 = up ? v[0] : v[2], s1 = up ? v[1] : v[3];
        k0 += __shfl_xor_sync(kFull, s0, 4);
        k1 += __shfl_xor_sync(kFull, s1, 4);
        const bool mid = (e & 2) != 0;
        float k = mid ? k1 : k0;
        k += __shfl_xor_sync(kFull, mid ? k0 : k1, 2);
        k += __shfl_xor_sync(kFull, k, 1);
        return k;
    } else if constexpr (GC == 2) {
        const bool up = (e & 4) != 0;
        float k = up ? v[1] : v[0];
        k += __shfl_xor_sync(kFull, up ? v[0] : v[1], 4);
        k += __shfl_xor_sync(kFull, k, 2);
        k += __shfl_xor_sync(kFull, k, 1);
        return k;
    } else {
        float k = v[0];
        k += __shfl_xor_sync(kFull, k, 4);
        k += __shfl_xor_sync(kFull, k, 2);
        k += __shfl_xor_sync(kFull, k, 1);
        return k;
    }
}

// ----------------------------------------------------------------------------
// Query prologue, one warp per head hh < GC of the CTA.
//  int8: the row is quantized like a cache row (absmax, per head, once); the
//        packed codes go to q_s ([GC][32] words) and the logit coefficient
//        q_scale * softmax_scale * log2(e) to coef[hh].
//  f16:  q * softmax_scale * log2(e) in f32 goes to q_s ([GC][128] floats).
template <int DT, int GC>
__device__ __forceinline__ void load_query(const DecodeArgs &a, int b, int h0, int warp, int lane,
                                           uint32_t *q_s, float *coef, int8_t *q_codes_out,
                                           float *q_scales_out) {
    if (warp >= GC) return;
    const int hq = h0 + warp;
    const float4 x4 = *reinterpret_cast<const float4 *>(
        a.q + (static_cast<size_t>(b) * a.H + hq) * kHeadDim + 4 * lane);
    const float x[4] = {x4.x, x4.y, x4.z, x4.w};
    if constexpr (DT != KVD_F16) {
        float s;
        const uint32_t packed = quantize_row_warp(x, &s);
        q_s[warp * 32 + lane] = packed;
        if (lane == 0) coef[warp] = s * a.scale_log2;
        if constexpr (DT == KVD_Q4_0) {
            // sum of the head's codes over each 32-channel group (lanes 8g..8g+7)
            int qs = __dp4a(static_cast<int>(packed), 0x01010101, 0);
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) qs += __shfl_xor_sync(kFull, qs, o);
            if ((lane & 7) == 0)
                reinterpret_cast<int *>(coef + 4)[warp * 4 + (lane >> 3)] = qs;
        }
        if (q_codes_out) {
            *reinterpret_cast<uint32_t *>(q_codes_out +
                                          (static_cast<size_t>(b) * a.H + hq) * kHeadDim +
                                          4 * lane) = packed;
            if (lane == 0) q_scales_out[static_cast<size_t>(b) * a.H + hq] = s;
        }
    } else {
        float *qf = reinterpret_cast<float *>(q_s) + warp * kHeadDim + 4 * lane;
#pragma unroll
        for (int j = 0; j < 4; ++j) qf[j] = x[j] * a.scale_log2;
    }
}

// int8 QK mapping: lane = 4 t + c (t: token slot 0..7, c: quarter 0..3 of the
// 128 channels).  The lane reads 16-byte chunks 2c and 2c+1 of its token row,
// odd tokens in swapped order so that the 8 lanes of each quarter-warp hit
// distinct banks.  qr holds the matching query words in that order.
template <int GC>
struct QRegsI8 {
    uint32_t w[GC][8];
};

template <int GC>
__device__ __forceinline__ void load_qregs_i8(const uint32_t *q_s, int t, int c, QRegsI8<GC> &r) {
#pragma unroll
    for (int h = 0; h < GC; ++h)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int chunk = 2 * c + (i ^ (t & 1));
#pragma unroll
            for (int j = 0; j < 4; ++j) r.w[h][4 * i + j] = q_s[h * 32 + 4 * chunk + j];
        }
}

// Exact int32 dot of one token row with the query of head (c*GC)/4.
template <int GC>
__device__ __forceinline__ int qk_int8_row(const int8_t *row, const QRegsI8<GC> &r, int t, int c) {
    const uint4 ka = *reinterpret_cast<const uint4 *>(row + 16 * (2 * c + (t & 1)));
    const uint4 kb = *reinterpret_cast<const uint4 *>(row + 16 * (2 * c + 1 - (t & 1)));
    const uint32_t kw[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
    int d[GC];
#pragma unroll
    for (int h = 0; h < GC; ++h) {
        int s = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            s = __dp4a(static_cast<int>(kw[j]), static_cast<int>(r.w[h][j]), s);
        d[h] = s;
    }
    return reduce4_scatter<GC>(d, c);
}

// q8_0: the lane's quarter c of the channels is exactly the cache's group c,
// so its exact int32 dot takes the group's key scale before the quarters
// are summed (in f32) into the logit of head (c*GC)/4.
template <int GC>
__device__ __forceinline__ float qk_q8_row(const int8_t *row, const QRegsI8<GC> &r, int t, int c,
                                           float kscale) {
    const uint4 ka = *reinterpret_cast<const uint4 *>(row + 16 * (2 * c + (t & 1)));
    const uint4 kb = *reinterpret_cast<const uint4 *>(row + 16 * (2 * c + 1 - (t & 1)));
    const uint32_t kw[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
    float d[GC];
#pragma unroll
    for (int h = 0; h < GC; ++h) {
        int s = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            s = __dp4a(static_cast<int>(kw[j]), static_cast<int>(r.w[h][j]), s);
        d[h] = static_cast<float>(s) * kscale;  // |s| <= 32*127*127: exact in f32
    }
    return reduce4_scatter<GC>(d, c);
}

// q4_0: lane (t, c) reads its token row's 16 bytes of group c (32 channels,
// two per byte).  Its word i holds channels 8i..8i+7 of the group; the low
// nibbles are channels 8i, 8i+2, 8i+4, 8i+6 and the high ones the odd
// channels, so the query words are held in that even/odd order.  The codes
// (0..15) are non-negative as signed bytes, so dp4a gives sum(q * code), and
// q * (code - 8) subtracts 8 times the group's query sum.
template <int GC>
struct QRegsQ4 {
    uint32_t lo[GC][4], hi[GC][4];
    int qsum[GC];  // sum of the head's codes over this lane's group
};

template <int GC>
__device__ __forceinline__ void load_qregs_q4(const uint32_t *q_s, const int *qsum_s, int c,
                                              QRegsQ4<GC> &r) {
#pragma unroll
    for (int h = 0; h < GC; ++h) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w0 = q_s[h * 32 + 8 * c + 2 * i];      // channels 8i .. 8i+3
            const uint32_t w1 = q_s[h * 32 + 8 * c + 2 * i + 1];  // channels 8i+4 .. 8i+7
            r.lo[h][i] = __byte_perm(w0, w1, 0x6420);
            r.hi[h][i] = __byte_perm(w0, w1, 0x7531);
        }
        r.qsum[h] = qsum_s[h * 4 + c];
    }
}

template <int GC>
__device__ __forceinline__ float qk_q4_row(const uint8_t *row, const QRegsQ4<GC> &r, int c,
                                           float kscale) {
    const uint4 kw = *reinterpret_cast<const uint4 *>(row + 16 * c);
    const uint32_t w[4] = {kw.x, kw.y, kw.z, kw.w};
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        lo[i] = w[i] & 0x0f0f0f0fu;
        hi[i] = (w[i] >> 4) & 0x0f0f0f0fu;
    }
    float d[GC];
#pragma unroll
    for (int h = 0; h < GC; ++h) {
        int s = -8 * r.qsum[h];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s = __dp4a(static_cast<int>(lo[i]), static_cast<int>(r.lo[h][i]), s);
            s = __dp4a(static_cast<int>(hi[i]), static_cast<int>(r.hi[h][i]), s);
        }
        d[h] = static_cast<float>(s) * kscale;  // |s| <= 32*127*8: exact in f32
    }
    return reduce4_scatter<GC>(d, c);
}

// Two 4-bit codes per byte of w16 (channels 4l .. 4l+3 of the lane) -> exact
// floats, as pairs: code - 8 for the low nibbles (channels 4l and 4l+2) and
// 16 (code - 8) for the high ones (4l+1 and 4l+3), which are masked where
// they stand instead of shifted down; their PV weights carry the 1/16.
__device__ __forceinline__ void u4x4_to_f32x2(uint32_t w16, float2 &f01, float2 &f23) {
    const uint32_t lo = w16 & 0x0f0fu;  // codes of channels 4l and 4l+2
    const uint32_t hi = w16 & 0xf0f0u;  // 16 x the codes of channels 4l+1 and 4l+3
    const float2 bias = make_float2(-8388616.0f, -8388736.0f);  // -(2^23 + 8), -(2^23 + 128)
    f01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7650)),
                                 __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7650))),
                     bias);
    f23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7651)),
                                 __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7651))),
                     bias);
}

// f16 QK mapping: lane = 8 t4 + e (t4: token slot 0..3 per pass, e: eighth
// 0..7 of the channels).  The lane reads chunks 2e and 2e+1 (8 halves each) of
// its token row, lanes e >= 4 in swapped order (bank-conflict free).  The
// query pairs are held in that order.
template <int GC>
struct QRegsF16 {
    float2 f[GC][8];
};

template <int GC>
__device__ __forceinline__ void load_qregs_f16(const uint32_t *q_s, int e, QRegsF16<GC> &r) {
    const float *qf = reinterpret_cast<const float *>(q_s);
#pragma unroll
    for (int h = 0; h < GC; ++h)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int chunk = 2 * e + (i ^ (e >> 2));
#pragma unroll
            for (int j = 0; j < 4; ++j)
                r.f[h][4 * i + j] = make_float2(qf[h * kHeadDim + 8 * chunk + 2 * j],
                                                qf[h * kHeadDim + 8 * chunk + 2 * j + 1]);
        }
}

template <int GC>
__device__ __forceinline__ float qk_f16_row(const __half *row, const QRegsF16<GC> &r, int e) {
    const uint4 ka = *reinterpret_cast<const uint4 *>(row + 8 * (2 * e + (e >> 2)));
    const uint4 kb = *reinterpret_cast<const uint4 *>(row + 8 * (2 * e + 1 - (e >> 2)));
    float2 kf[8];
    const __half2 *ha = reinterpret_cast<const __half2 *>(&ka);
    const __half2 *hb = reinterpret_cast<const __half2 *>(&kb);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        kf[i] = __half22float2(ha[i]);
        kf[4 + i] = __half22float2(hb[i]);
    }
    float d[GC];
#pragma unroll
    for (int h = 0; h < GC; ++h) {
        float2 s = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < 8; ++j) s = __ffma2_rn(r.f[h][j], kf[j], s);
        d[h] = s.x + s.y;
    }
    return reduce8_scatter<GC>(d, e);
}

// Running softmax state of one consumer warp for the CTA's GC heads.
template <int GC>
struct WarpState {
    float m;             // running max (base-2 logits) of this lane's QK head
    float l;             // this lane's share of the running sum
    float2 acc[GC][2];   // channels 4*lane .. 4*lane+3 of every head, as pairs
};

template <int GC>
__device__ __forceinline__ void rescale(WarpState<GC> &st, float alpha_own, int lanes_per_head) {
    if (__any_sync(kFull, alpha_own != 1.0f)) {
#pragma unroll
        for (int h = 0; h < GC; ++h) {
            const float al = __shfl_sync(kFull, alpha_own, h * lanes_per_head);
            const float2 a2 = make_float2(al, al);
            st.acc[h][0] = __fmul2_rn(st.acc[h][0], a2);
            st.acc[h][1] = __fmul2_rn(st.acc[h][1], a2);
        }
    }
}

// acc[h] += p[h] * v (4 channels) for one token; pw_tok holds (p, p) pairs.
template <int GC>
__device__ __forceinline__ void pv_token(WarpState<GC> &st, const float *pw_tok, float2 v01,
                                         float2 v23) {
    if constexpr (GC >= 2) {
        const float4 p01 = *reinterpret_cast<const float4 *>(pw_tok);
        const float2 pa = make_float2(p01.x, p01.y), pb = make_float2(p01.z, p01.w);
        st.acc[0][0] = __ffma2_rn(v01, pa, st.acc[0][0]);
        st.acc[0][1] = __ffma2_rn(v23, pa, st.acc[0][1]);
        st.acc[1][0] = __ffma2_rn(v01, pb, st.acc[1][0]);
        st.acc[1][1] = __ffma2_rn(v23, pb, st.acc[1][1]);
        if constexpr (GC == 4) {
            const float4 p23 = *reinterpret_cast<const float4 *>(pw_tok + 4);
            const float2 pc = make_float2(p23.x, p23.y), pd = make_float2(p23.z, p23.w);
            st.acc[2][0] = __ffma2_rn(v01, pc, st.acc[2][0]);
            st.acc[2][1] = __ffma2_rn(v23, pc, st.acc[2][1]);
            st.acc[3][0] = __ffma2_rn(v01, pd, st.acc[3][0]);
            st.acc[3][1] = __ffma2_rn(v23, pd, st.acc[3][1]);
        }
    } else {
        const float2 pa = *reinterpret_cast<const float2 *>(pw_tok);
        st.acc[0][0] = __ffma2_rn(v01, pa, st.acc[0][0]);
        st.acc[0][1] = __ffma2_rn(v23, pa, st.acc[0][1]);
    }
}

// Bits b*w of x (b = 0..n-1) that have any of their w bits set, packed into
// bits 0..n-1: which tokens of a ballot (w lanes per token) are live.
template <int N, int W>
__device__ __forceinline__ uint32_t any_per_group(uint32_t x) {
    uint32_t r = 0;
#pragma unroll
    for (int b = 0; b < N; ++b)
        if ((x >> (W * b)) & ((1u << W) - 1u)) r |= 1u << b;
    return r;
}

// Sparse-V, eps mode ("Sparse Attention -- Quest-style block-selector ...",
// "Adaptive tau (the eps mode)"): a position's V term is dropped when its
// weight is below eps times the mean weight of its 16-token chunk (the
// warp's share of the block), both relative to the chunk's maximum, so the
// dropped share of the softmax mass stays below eps.  The position stays in
// the softmax denominator.  x: this lane's base-2 logits of NT tokens (-inf
// past the valid ones), bm: the chunk maximum of the lane's head, nvc: the
// chunk's valid tokens; the reduction runs over the lanes of one head
// (lane bits RED0 and up).  Returns, per token, whether V is kept.
template <int NT, int RED0>
__device__ __forceinline__ void sparse_v_keep(const float (&x)[NT], float bm, int nvc, float eps,
                                              bool (&keep)[NT]) {
    float c[NT];
    float cs = 0.0f;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        c[i] = exp2f(x[i] - bm);
        cs += c[i];
    }
#pragma unroll
    for (int o = RED0; o < 32; o <<= 1) cs += __shfl_xor_sync(kFull, cs, o);
    const float thr = nvc > 0 ? eps * cs / static_cast<float>(nvc) : 0.0f;
#pragma unroll
    for (int i = 0; i < NT; ++i) keep[i] = !(c[i] < thr);
}

// Four signed bytes -> two exact float pairs, one integer-to-float
// conversion per byte (fewer instructions than building each float from
// the byte's bits: this loop is the consumers' largest cost).
__device__ __forceinline__ void s8x4_to_f32x2(uint32_t w, float2 &f01, float2 &f23) {
    f01 = make_float2(static_cast<float>(static_cast<int8_t>(w & 0xffu)),
                      static_cast<float>(static_cast<int8_t>((w >> 8) & 0xffu)));
    f23 = make_float2(static_cast<float>(static_cast<int8_t>((w >> 16) & 0xffu)),
                      static_cast<float>(static_cast<int8_t>(w >> 24)));
}

// One stage (64-token block) for one consumer warp (wg = its index in the
// group), int8 cache: two QK passes of 8 tokens, one softmax update, 16
// tokens of PV.
template <int GC, bool SV>
__device__ __forceinline__ void consume_int8(const uint8_t *stage, int n_valid, const float *coef,
                                             const QRegsI8<GC> &qr, float *pw, int wg, int lane,
                                             WarpState<GC> &st, float sv_eps) {
    const int8_t *Ks = reinterpret_cast<const int8_t *>(stage);
    const int8_t *Vs = Ks + Tile<KVD_INT8>::kKBytes;
    const float *ksc = reinterpret_cast<const float *>(stage + 2 * Tile<KVD_INT8>::kKBytes);
    const float *vsc = ksc + kBlock;
    const int t = lane >> 2, c = lane & 3;
    const int tok0 = kTokensPerWarp * wg + t, tok1 = tok0 + 8;
    const int hq = (c * GC) >> 2;
    const float ninf = -__int_as_float(0x7f800000);
    const int d0 = qk_int8_row<GC>(Ks + tok0 * kHeadDim, qr, t, c);
    const int d1 = qk_int8_row<GC>(Ks + tok1 * kHeadDim, qr, t, c);
    const float cf = coef[hq];
    const float x0 = tok0 < n_valid ? static_cast<float>(d0) * cf * ksc[tok0] : ninf;
    const float x1 = tok1 < n_valid ? static_cast<float>(d1) * cf * ksc[tok1] : ninf;
    float bm = fmaxf(x0, x1);
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
    const float m_new = fmaxf(st.m, bm);
    const float alpha = exp2f(st.m - m_new);
    const float p0 = exp2f(x0 - m_new), p1 = exp2f(x1 - m_new);
    st.l = st.l * alpha + (p0 + p1);
    st.m = m_new;
    bool keep[2] = {true, true};
    uint32_t live = 0xffffu;  // tokens whose V some head still needs
    if constexpr (SV) {
        const float xs[2] = {x0, x1};
        sparse_v_keep<2, 4>(xs, bm, min(max(n_valid - kTokensPerWarp * wg, 0), kTokensPerWarp),
                            sv_eps, keep);
        const uint32_t b0 = __ballot_sync(kFull, keep[0] && tok0 < n_valid);  // lane 4t + c
        const uint32_t b1 = __ballot_sync(kFull, keep[1] && tok1 < n_valid);
        live = any_per_group<8, 4>(b0) | (any_per_group<8, 4>(b1) << 8);
    }
    constexpr int lph = 4 / GC;  // lanes per head among the quarters
    if ((c % lph) == 0) {
        const float w0 = tok0 < n_valid && keep[0] ? p0 * vsc[tok0] : 0.0f;
        const float w1 = tok1 < n_valid && keep[1] ? p1 * vsc[tok1] : 0.0f;
        *reinterpret_cast<float2 *>(pw + (t * 4 + hq) * 2) = make_float2(w0, w0);
        *reinterpret_cast<float2 *>(pw + ((t + 8) * 4 + hq) * 2) = make_float2(w1, w1);
    }
    rescale<GC>(st, alpha, lph);
    __syncwarp();
    const int nt = min(kTokensPerWarp, n_valid - kTokensPerWarp * wg);
    const int8_t *vrow = Vs + kTokensPerWarp * wg * kHeadDim + 4 * lane;
    if (SV && live != 0xffffu) {
        // sparse-V dropped some tokens for every head: only the live ones
        for (uint32_t m = live; m; m &= m - 1u) {
            const int t2 = __ffs(m) - 1;
            float2 f01, f23;
            s8x4_to_f32x2(*reinterpret_cast<const uint32_t *>(vrow + t2 * kHeadDim), f01, f23);
            pv_token<GC>(st, pw + t2 * 8, f01, f23);
        }
    } else if (nt == kTokensPerWarp) {
#pragma unroll
        for (int t2 = 0; t2 < kTokensPerWarp; ++t2) {
            float2 f01, f23;
            s8x4_to_f32x2(*reinterpret_cast<const uint32_t *>(vrow + t2 * kHeadDim), f01, f23);
            pv_token<GC>(st, pw + t2 * 8, f01, f23);
        }
    } else {
        for (int t2 = 0; t2 < nt; ++t2) {
            float2 f01, f23;
            s8x4_to_f32x2(*reinterpret_cast<const uint32_t *>(vrow + t2 * kHeadDim), f01, f23);
            pv_token<GC>(st, pw + t2 * 8, f01, f23);
        }
    }
}

// One stage for one consumer warp, q8_0 cache: as consume_int8, with the
// key scales per (token, group) inside the logit and the value scale of the
// lane's group (lanes 8g..8g+7 hold channels of group g) applied to the
// converted values.
template <int GC, bool SV>
__device__ __forceinline__ void consume_q8(const uint8_t *stage, int n_valid, const float *coef,
                                           const QRegsI8<GC> &qr, float *pw, int wg, int lane,
                                           WarpState<GC> &st, float sv_eps) {
    using TQ = Tile<KVD_Q8_0>;
    const int8_t *Ks = reinterpret_cast<const int8_t *>(stage);
    const int8_t *Vs = Ks + TQ::kKBytes;
    const __half *kd = reinterpret_cast<const __half *>(stage + 2 * TQ::kKBytes);  // [64][4]
    const __half *vd = kd + kBlock * (kHeadDim / 32);
    const int t = lane >> 2, c = lane & 3;
    const int tok0 = kTokensPerWarp * wg + t, tok1 = tok0 + 8;
    const int hq = (c * GC) >> 2;
    const float ninf = -__int_as_float(0x7f800000);
    const float dot0 = qk_q8_row<GC>(Ks + tok0 * kHeadDim, qr, t, c,
                                     __half2float(kd[tok0 * (kHeadDim / 32) + c]));
    const float dot1 = qk_q8_row<GC>(Ks + tok1 * kHeadDim, qr, t, c,
                                     __half2float(kd[tok1 * (kHeadDim / 32) + c]));
    const float cf = coef[hq];
    const float x0 = tok0 < n_valid ? dot0 * cf : ninf;
    const float x1 = tok1 < n_valid ? dot1 * cf : ninf;
    float bm = fmaxf(x0, x1);
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
    const float m_new = fmaxf(st.m, bm);
    const float alpha = exp2f(st.m - m_new);
    const float p0 = exp2f(x0 - m_new), p1 = exp2f(x1 - m_new);
    st.l = st.l * alpha + (p0 + p1);
    st.m = m_new;
    bool keep[2] = {true, true};
    uint32_t live = 0xffffu;
    if constexpr (SV) {
        const float xs[2] = {x0, x1};
        sparse_v_keep<2, 4>(xs, bm, min(max(n_valid - kTokensPerWarp * wg, 0), kTokensPerWarp),
                            sv_eps, keep);
        const uint32_t b0 = __ballot_sync(kFull, keep[0] && tok0 < n_valid);
        const uint32_t b1 = __ballot_sync(kFull, keep[1] && tok1 < n_valid);
        live = any_per_group<8, 4>(b0) | (any_per_group<8, 4>(b1) << 8);
    }
    constexpr int lph = 4 / GC;
    if ((c % lph) == 0) {
        const float w0 = tok0 < n_valid && keep[0] ? p0 : 0.0f;
        const float w1 = tok1 < n_valid && keep[1] ? p1 : 0.0f;
        *reinterpret_cast<float2 *>(pw + (t * 4 + hq) * 2) = make_float2(w0, w0);
        *reinterpret_cast<float2 *>(pw + ((t + 8) * 4 + hq) * 2) = make_float2(w1, w1);
    }
    rescale<GC>(st, alpha, lph);
    __syncwarp();
    const int nt = min(kTokensPerWarp, n_valid - kTokensPerWarp * wg);
    const int8_t *vrow = Vs + kTokensPerWarp * wg * kHeadDim + 4 * lane;
    const __half *vdl = vd + kTokensPerWarp * wg * (kHeadDim / 32) + (lane >> 3);
    if (live != 0xffffu || nt != kTokensPerWarp) {
        uint32_t m = live & ((nt >= 32 ? 0u : (1u << max(nt, 0))) - 1u);
        for (; m; m &= m - 1u) {
            const int t2 = __ffs(m) - 1;
            float2 f01, f23;
            s8x4_to_f32x2(*reinterpret_cast<const uint32_t *>(vrow + t2 * kHeadDim), f01, f23);
            const float dv = __half2float(vdl[t2 * (kHeadDim / 32)]);
            const float2 d2 = make_float2(dv, dv);
            pv_token<GC>(st, pw + t2 * 8, __fmul2_rn(f01, d2), __fmul2_rn(f23, d2));
        }
    } else {
#pragma unroll
        for (int t2 = 0; t2 < kTokensPerWarp; ++t2) {
            float2 f01, f23;
            s8x4_to_f32x2(*reinterpret_cast<const uint32_t *>(vrow + t2 * kHeadDim), f01, f23);
            const float dv = __half2float(vdl[t2 * (kHeadDim / 32)]);
            const float2 d2 = make_float2(dv, dv);
            pv_token<GC>(st, pw + t2 * 8, __fmul2_rn(f01, d2), __fmul2_rn(f23, d2));
        }
    }
}

// One stage for one consumer warp, q4_0 cache: consume_q8 with the 4-bit
// rows unpacked in registers, and the value scale of each (token, group)
// folded into that group's PV weights: lane (t, c) writes, for its head, the
// weights of GC of the four groups, and the lanes of group g (8g .. 8g+7)
// read group g's.  pw: [16 tokens, kQ4PwTok floats apart][4 groups][4 heads]
// pairs (w, w / 16).
template <int GC, bool SV>
__device__ __forceinline__ void consume_q4(const uint8_t *stage, int n_valid, const float *coef,
                                           const QRegsQ4<GC> &qr, float *pw, int wg, int lane,
                                           WarpState<GC> &st, float sv_eps) {
    using TQ = Tile<KVD_Q4_0>;
    const uint8_t *Ks = stage;
    const uint8_t *Vs = Ks + TQ::kKBytes;
    const __half *kd = reinterpret_cast<const __half *>(stage + 2 * TQ::kKBytes);  // [64][4]
    const __half *vd = kd + kBlock * (kHeadDim / 32);
    const int t = lane >> 2, c = lane & 3;
    const int tok0 = kTokensPerWarp * wg + t, tok1 = tok0 + 8;
    const int hq = (c * GC) >> 2;
    const float ninf = -__int_as_float(0x7f800000);
    const float dot0 = qk_q4_row<GC>(Ks + tok0 * TQ::kRowBytes, qr, c,
                                     __half2float(kd[tok0 * (kHeadDim / 32) + c]));
    const float dot1 = qk_q4_row<GC>(Ks + tok1 * TQ::kRowBytes, qr, c,
                                     __half2float(kd[tok1 * (kHeadDim / 32) + c]));
    const float cf = coef[hq];
    const float x0 = tok0 < n_valid ? dot0 * cf : ninf;
    const float x1 = tok1 < n_valid ? dot1 * cf : ninf;
    float bm = fmaxf(x0, x1);
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
    const float m_new = fmaxf(st.m, bm);
    const float alpha = exp2f(st.m - m_new);
    const float p0 = exp2f(x0 - m_new), p1 = exp2f(x1 - m_new);
    st.l = st.l * alpha + (p0 + p1);
    st.m = m_new;
    bool keep[2] = {true, true};
    uint32_t live = 0xffffu;
    if constexpr (SV) {
        const float xs[2] = {x0, x1};
        sparse_v_keep<2, 4>(xs, bm, min(max(n_valid - kTokensPerWarp * wg, 0), kTokensPerWarp),
                            sv_eps, keep);
        const uint32_t b0 = __ballot_sync(kFull, keep[0] && tok0 < n_valid);
        const uint32_t b1 = __ballot_sync(kFull, keep[1] && tok1 < n_valid);
        live = any_per_group<8, 4>(b0) | (any_per_group<8, 4>(b1) << 8);
    }
    constexpr int lph = 4 / GC;
    {
        const int g0 = (c % lph) * GC;  // this lane's groups g0 .. g0 + GC - 1
        const bool u0 = tok0 < n_valid && keep[0], u1 = tok1 < n_valid && keep[1];
#pragma unroll
        for (int j = 0; j < GC; ++j) {
            const float a0 = u0 ? p0 * __half2float(vd[tok0 * (kHeadDim / 32) + g0 + j]) : 0.0f;
            const float a1 = u1 ? p1 * __half2float(vd[tok1 * (kHeadDim / 32) + g0 + j]) : 0.0f;
            *reinterpret_cast<float2 *>(pw + t * kQ4PwTok + (g0 + j) * 8 + 2 * hq) =
                make_float2(a0, a0 * 0.0625f);
            *reinterpret_cast<float2 *>(pw + (t + 8) * kQ4PwTok + (g0 + j) * 8 + 2 * hq) =
                make_float2(a1, a1 * 0.0625f);
        }
    }
    rescale<GC>(st, alpha, lph);
    __syncwarp();
    const int nt = min(kTokensPerWarp, n_valid - kTokensPerWarp * wg);
    const uint8_t *vrow = Vs + kTokensPerWarp * wg * TQ::kRowBytes + 2 * lane;
    const float *pwg = pw + (lane >> 3) * 8;  // the lane's group, token 0
    if ((SV && live != 0xffffu) || nt != kTokensPerWarp) {
        uint32_t m = live & ((1u << max(nt, 0)) - 1u);
        for (; m; m &= m - 1u) {
            const int t2 = __ffs(m) - 1;
            float2 f01, f23;
            u4x4_to_f32x2(*reinterpret_cast<const uint16_t *>(vrow + t2 * TQ::kRowBytes), f01,
                          f23);
            pv_token<GC>(st, pwg + t2 * kQ4PwTok, f01, f23);
        }
    } else {
#pragma unroll
        for (int t2 = 0; t2 < kTokensPerWarp; ++t2) {
            float2 f01, f23;
            u4x4_to_f32x2(*reinterpret_cast<const uint16_t *>(vrow + t2 * TQ::kRowBytes), f01,
                          f23);
            pv_token<GC>(st, pwg + t2 * kQ4PwTok, f01, f23);
        }
    }
}

// One stage for one consumer warp (wg = its index in the group), f16 cache:
// four QK passes of 4 tokens.
template <int GC, bool SV>
__device__ __forceinline__ void consume_f16(const uint8_t *stage, int n_valid,
                                            const QRegsF16<GC> &qr, float *pw, int wg,
                                            int lane, WarpState<GC> &st, float sv_eps) {
    const __half *Ks = reinterpret_cast<const __half *>(stage);
    const __half *Vs = Ks + kBlock * kHeadDim;
    const int t4 = lane >> 3, e = lane & 7;
    const int hq = (e * GC) >> 3;
    const float ninf = -__int_as_float(0x7f800000);
    float x[4];
#pragma unroll
    for (int ps = 0; ps < 4; ++ps) {
        const int tok = kTokensPerWarp * wg + 4 * ps + t4;
        const float d = qk_f16_row<GC>(Ks + tok * kHeadDim, qr, e);
        x[ps] = tok < n_valid ? d : ninf;
    }
    float bm = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
    const float m_new = fmaxf(st.m, bm);
    const float alpha = exp2f(st.m - m_new);
    float p[4];
#pragma unroll
    for (int ps = 0; ps < 4; ++ps) p[ps] = exp2f(x[ps] - m_new);
    st.l = st.l * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
    st.m = m_new;
    bool keep[4] = {true, true, true, true};
    uint32_t live = 0xffffu;  // tokens whose V some head still needs
    if constexpr (SV) {
        sparse_v_keep<4, 8>(x, bm, min(max(n_valid - kTokensPerWarp * wg, 0), kTokensPerWarp),
                            sv_eps, keep);
        live = 0u;
#pragma unroll
        for (int ps = 0; ps < 4; ++ps) {
            const int tok = kTokensPerWarp * wg + 4 * ps + t4;
            const uint32_t bp = __ballot_sync(kFull, keep[ps] && tok < n_valid);  // lane 8 t4 + e
            live |= any_per_group<4, 8>(bp) << (4 * ps);
        }
    }
    constexpr int lph = 8 / GC;
    if ((e % lph) == 0) {
#pragma unroll
        for (int ps = 0; ps < 4; ++ps) {
            const float w = keep[ps] ? p[ps] : 0.0f;
            *reinterpret_cast<float2 *>(pw + ((4 * ps + t4) * 4 + hq) * 2) = make_float2(w, w);
        }
    }
    rescale<GC>(st, alpha, lph);
    __syncwarp();
    const int nt = min(kTokensPerWarp, n_valid - kTokensPerWarp * wg);
    const __half *vrow = Vs + kTokensPerWarp * wg * kHeadDim + 4 * lane;
    if (SV && live != 0xffffu) {
        // sparse-V dropped some tokens for every head: only the live ones
        for (uint32_t m = live; m; m &= m - 1u) {
            const int t2 = __ffs(m) - 1;
            const uint2 vw = *reinterpret_cast<const uint2 *>(vrow + t2 * kHeadDim);
            const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&vw.x));
            const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&vw.y));
            pv_token<GC>(st, pw + t2 * 8, v01, v23);
        }
        return;
    }
#pragma unroll 4
    for (int t2 = 0; t2 < nt; ++t2) {
        const uint2 vw = *reinterpret_cast<const uint2 *>(vrow + t2 * kHeadDim);
        const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&vw.x));
        const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&vw.y));
        pv_token<GC>(st, pw + t2 * 8, v01, v23);
    }
}

// ----------------------------------------------------------------------------
// Moment tail  ("SCSA: Self-Calibrating Subquadratic Attention", "2.
// Mechanism": a group of keys that is not read exactly contributes its count
// m times exp(a), a = scale * q . c_K, at its value mean c_V, inside the
// shared softmax normalizer).  Here the groups are the cache blocks the list
// leaves out.  Each split streams the moment rows of its share of all blocks
// through the same ring after its listed blocks; the producer marks which
// rows are listed (the list must be ascending), and the consumers fold the
// others into a second online softmax state per warp, merged with the exact
// states at the end.

// First position p in the ascending list[0, n) with list[p] >= target (n when
// none), by a 32-way search: one round of loads per factor of 32.
__device__ __forceinline__ int first_at_least(const int32_t *list, int n, int target, int lane) {
    int lo = 0, hi = n;
    while (hi - lo > 32) {
        const int step = (hi - lo + 31) / 32;
        const int p = lo + lane * step;
        const int v = p < hi ? list[p] : 0x7fffffff;
        const int k = __popc(__ballot_sync(kFull, v < target));
        if (k == 0) return lo;
        const int nhi = lo + k * step;
        lo += (k - 1) * step + 1;
        hi = nhi < hi ? nhi : hi;
    }
    const int p = lo + lane;
    const int v = p < hi ? list[p] : 0x7fffffff;
    return lo + __popc(__ballot_sync(kFull, v < target));
}

// Producer: the moment rows of chunks [c0, c1) of this split (chunk c holds
// blocks [c R, c R + R)), each stage tagged with its chunk and the mask of
// its listed blocks.  The list is walked once, 32 entries per load: ent holds
// entries cur .. cur + 31, of which the first o lanes are used up.
// i: the stage sequence number, advanced per stage.
template <int DT, bool WIDE>
__device__ __forceinline__ bool produce_tail(const DecodeArgs &a, int NB, int split, int bg,
                                             int cnt,
                                             const int32_t *list, int &i, uint64_t *full,
                                             uint64_t *empty, int *stage_blk,
                                             uint32_t *stage_mask, uint8_t *ring,
                                             volatile int *abort_flag, int lane, uint64_t pol) {
    using TL = TileW<DT, WIDE>;
    constexpr int R = TL::kTailRecs;
    const int nch = (NB + R - 1) / R;
    const int c0 = static_cast<int>((static_cast<long long>(split) * nch) / a.splits);
    const int c1 = static_cast<int>((static_cast<long long>(split + 1) * nch) / a.splits);
    if (c0 >= c1) return true;
    const __half *mom = a.moments + static_cast<size_t>(bg) * a.nbmax * (2 * kHeadDim);
    int cur = first_at_least(list, cnt, c0 * R, lane);
    int ent = cur + lane < cnt ? list[cur + lane] : 0x7fffffff;
    int o = 0;
    bool ok = true;
    for (int c = c0; c < c1; ++c) {
        const int lo = c * R, hi = lo + R;
        uint32_t m = 0;
        for (;;) {
            const bool live = lane >= o;
            const bool in = live && ent >= lo && ent < hi;
            m |= __reduce_or_sync(kFull, in ? 1u << (ent - lo) : 0u);
            o += __popc(__ballot_sync(kFull, live && ent < hi));
            if (o < 32) break;
            cur += 32;  // the batch is used up: the next 32 entries
            o = 0;
            ent = cur + lane < cnt ? list[cur + lane] : 0x7fffffff;
        }
        const int s = i % TL::kStages;
        if (lane == 0) {
            if (i >= TL::kStages)
                ok = mbar_wait(&empty[s], ((i / TL::kStages) - 1) & 1, abort_flag);
            if (ok) {
                const int nrec = min(R, NB - lo);
                stage_blk[s] = kTailBase - c;
                stage_mask[s] = m;
                mbar_arrive_expect_tx(&full[s], nrec * kMomentBytes);
                tma_load_1d(ring + s * TL::kStageBytes,
                            mom + static_cast<size_t>(lo) * (2 * kHeadDim), nrec * kMomentBytes,
                            &full[s], pol);
            } else {
                *abort_flag = 1;
                report_status(a.dev_status, KVD_ERR_TIMEOUT);
            }
        }
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;
        ++i;
    }
    return ok;
}

// Sum over the 32 lanes of each of v[0..N) (N a power of two <= 32), left
// scattered: lane l receives the total of index l >> (5 - log2 N).
template <int N>
__device__ __forceinline__ float reduce_scatter_n(float (&v)[N], int lane) {
#pragma unroll
    for (int len = N, o = 16; len > 1; len >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < len / 2; ++j) {
            const float keep = up ? v[len / 2 + j] : v[j];
            const float send = up ? v[j] : v[len / 2 + j];
            v[j] = keep + __shfl_xor_sync(kFull, send, o);
        }
    }
    float x = v[0];
#pragma unroll
    for (int o = 16 >> ilog2(N); o >= 1; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

// Lanes per (record, head) value of a warp's tail stage.
template <int DT, int GC>
constexpr int tail_shift() {
    return 5 - ilog2(Tile<DT>::kTailRecs / kWarpsPerGroup * GC);
}

// Consumer: the tail stages of this warp's group, from stage i (already
// waited for) to the group's end marker.  Warp wg takes records
// [wg RW, wg RW + RW) of each stage; ts.m and ts.l belong to the lane's head
// h = (lane >> SH) % GC, ts.acc to channels 4 lane .. 4 lane + 3 of every head.
template <int DT, int GC, bool WIDE>
__device__ __forceinline__ void tail_loop(const DecodeArgs &a, int len, int NB, int b, int h0,
                                          int i,
                                       uint64_t *full, uint64_t *empty, const int *stage_blk,
                                       const uint32_t *stage_mask, const uint8_t *ring, float *pw,
                                       int wg, int lane, volatile int *abort_flag,
                                       WarpState<GC> &ts) {
    using TL = TileW<DT, WIDE>;
    constexpr int R = TL::kTailRecs, RW = R / kWarpsPerGroup, N = RW * GC;
    constexpr int SH = tail_shift<DT, GC>(), LGC = ilog2(GC);
    float qf[GC][4];  // the f32 query in base-2 logit units
#pragma unroll
    for (int h = 0; h < GC; ++h) {
        const float4 v = *reinterpret_cast<const float4 *>(
            a.q + (static_cast<size_t>(b) * a.H + h0 + h) * kHeadDim + 4 * lane);
        qf[h][0] = v.x * a.scale_log2;
        qf[h][1] = v.y * a.scale_log2;
        qf[h][2] = v.z * a.scale_log2;
        qf[h][3] = v.w * a.scale_log2;
    }
    const int idx = lane >> SH, r_own = idx / GC, h_own = idx % GC;
    for (bool first = true;; i += TL::kGroups, first = false) {
        const int s = i % TL::kStages;
        if (!first) {
            const bool ok = mbar_wait(&full[s], (i / TL::kStages) & 1, abort_flag);
            if (!__all_sync(kFull, ok)) {
                if (lane == 0) {
                    *abort_flag = 1;
                    report_status(a.dev_status, KVD_ERR_TIMEOUT);
                }
                return;
            }
        }
        const int code = stage_blk[s];
        if (code == kEndMark) return;
        const int j0 = (kTailBase - code) * R + wg * RW;  // block of this warp's first record
        const uint32_t listed = stage_mask[s] >> (wg * RW);
        const uint8_t *rec = ring + s * TL::kStageBytes + wg * RW * kMomentBytes;
        uint32_t vm = 0;  // records to fold: present and not listed
#pragma unroll
        for (int r = 0; r < RW; ++r)
            if (j0 + r < NB && !((listed >> r) & 1u)) vm |= 1u << r;
        if (vm) {
            float d[N];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const uint2 w = *reinterpret_cast<const uint2 *>(rec + r * kMomentBytes + 8 * lane);
                const float2 k01 = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
                const float2 k23 = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
#pragma unroll
                for (int h = 0; h < GC; ++h)
                    d[r * GC + h] = fmaf(qf[h][3], k23.y,
                                         fmaf(qf[h][2], k23.x,
                                              fmaf(qf[h][1], k01.y, qf[h][0] * k01.x)));
            }
            float x = reduce_scatter_n<N>(d, lane);
            const int j = j0 + r_own;
            const int m = min(kBlock, len - j * kBlock);
            x = ((vm >> r_own) & 1u) ? x + (m == kBlock ? 6.0f : log2f(static_cast<float>(m)))
                                     : -INFINITY;
            // over this warp's records of the lane's head (lane bits above LGC + SH)
            float mx = x;
#pragma unroll
            for (int o = 1 << (SH + LGC); o < 32; o <<= 1)
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
            const float m_new = fmaxf(ts.m, mx);
            const float alpha = exp2f(ts.m - m_new);
            const float p = exp2f(x - m_new);
            float ps = p;
#pragma unroll
            for (int o = 1 << (SH + LGC); o < 32; o <<= 1) ps += __shfl_xor_sync(kFull, ps, o);
            ts.l = fmaf(ts.l, alpha, ps);
            ts.m = m_new;
            if ((lane & ((1 << SH) - 1)) == 0)
                *reinterpret_cast<float2 *>(pw + r_own * 8 + 2 * h_own) = make_float2(p, p);
            rescale<GC>(ts, alpha, 1 << SH);
            __syncwarp();
            for (uint32_t mm = vm; mm; mm &= mm - 1u) {
                const int r = __ffs(mm) - 1;
                const uint2 w = *reinterpret_cast<const uint2 *>(rec + r * kMomentBytes +
                                                                 2 * kHeadDim + 8 * lane);
                const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
                const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
                pv_token<GC>(ts, pw + r * 8, v01, v23);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

template <int DT, int GC, bool DENSE, bool SV, bool TAIL, bool WIDE>
__device__ void decode_body(const DecodeArgs &a, int split, int prob, uint8_t *smem) {
    static_assert(!TAIL || (!DENSE && !SV), "the moment tail runs on a listed selection alone");
    using SL = SmemLayout<DT, GC, TAIL, WIDE>;
    using TL = TileW<DT, WIDE>;
    static_assert(TL::kStages % TL::kGroups == 0, "stages must split evenly over the groups");
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + SL::kFullOff);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + SL::kEmptyOff);
    int *stage_blk = reinterpret_cast<int *>(smem + SL::kBlkOff);
    uint32_t *q_s = reinterpret_cast<uint32_t *>(smem + SL::kQOff);
    float *coef = reinterpret_cast<float *>(smem + SL::kCoefOff);
    float *pw_all = reinterpret_cast<float *>(smem + SL::kPwOff);
    float *l_tot = reinterpret_cast<float *>(smem + SL::kLOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SL::kFlagOff);
    int *last_flag = reinterpret_cast<int *>(smem + SL::kFlagOff + 4);
    int *issued_s = reinterpret_cast<int *>(smem + SL::kFlagOff + 8);
    uint32_t *stage_mask = reinterpret_cast<uint32_t *>(smem + SL::kMaskOff);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // prob = ((b * Hkv) + g) * subgroups + sub
    const int sub = prob % a.subgroups;
    const int bg = prob / a.subgroups;  // b * Hkv + g
    const int b = bg / a.Hkv, g = bg % a.Hkv;
    const int h0 = g * a.G + sub * GC;

    if (tid == 0) {
        for (int i = 0; i < TL::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWarpsPerGroup);
        }
        *abort_flag = 0;
        *issued_s = 0;
        fence_barrier_init();
        KVD_MARK(a.marks, 0);  // entry
    }
    __syncthreads();
    // Inside a decode step the query was written before the step's first
    // kernel, so it may be read while the selection is still finishing.
    if (a.early_q) load_query<DT, GC>(a, b, h0, warp, lane, q_s, coef, nullptr, nullptr);
    pdl_wait();  // upstream kernels (append, select) are complete past here
    if (tid == 0) KVD_MARK(a.marks, 1);  // dependency wait over
    pdl_launch_dependents();
    // the list row: the KV head's, or with per-head lists the CTA's one head's
    const int lrow = a.per_head ? prob : bg;
    // this sequence's own length (per-sequence lengths) and blocks
    const int len = seq_len_of(a.seq_lens, b, a.len - a.seq_add, a.dev_status) + a.seq_add;
    const int NB = (len + kBlock - 1) / kBlock;
    int cnt = DENSE ? NB : a.sel_cnt[lrow];
    cnt = max(0, min(cnt, NB));

    const size_t row0 = static_cast<size_t>(bg) * a.max_seq;  // first token row of (b, g)
    WarpState<GC> st;
    st.m = kNegBig;
    st.l = 0.0f;
#pragma unroll
    for (int h = 0; h < GC; ++h) st.acc[h][0] = st.acc[h][1] = make_float2(0.0f, 0.0f);
    WarpState<GC> ts = st;  // the moment tail's state (TAIL only)
    if (warp == TL::kConsumerWarps) {
        // ------------------------------------------------------ producer
        // The split's list positions: its share [pb, pe) of the planned
        // length, then (only when sel_cnt passes that length) every
        // splits-th position beyond it, from plan_blocks + split on.
        const uint64_t pol = l2_policy_evict_first();
        const int32_t *list = a.sel_idx + static_cast<size_t>(lrow) * a.nbmax;
        const int S = a.splits, MB = a.plan_blocks;
        const int pb = static_cast<int>((static_cast<long long>(split) * MB) / S);
        const int pe = static_cast<int>((static_cast<long long>(split + 1) * MB) / S);
        // the share's first list entries, read while cnt is in flight (pe <= NB <= nbmax)
        int pre = 0;
        if (!DENSE && lane < pe - pb) pre = list[pb + lane];
        const int n_own = max(0, min(pe, cnt) - pb);
        const int x0 = MB + split;
        const int n = n_own + (cnt > x0 ? (cnt - x0 + S - 1) / S : 0);
        int i = 0;  // stage sequence number
        bool ok = true;
        for (int i0 = 0; i0 < n && ok; i0 += 32) {
            const int m = min(32, n - i0);
            const int idx = i0 + lane;
            int mine = 0;
            if (idx < n) {
                const int pos = idx < n_own ? pb + idx : x0 + (idx - n_own) * S;
                mine = DENSE ? pos : (i0 == 0 && idx < n_own ? pre : list[pos]);
            }
            for (int j = 0; j < m; ++j) {
                const int blk = __shfl_sync(kFull, mine, j);
                const int s = i % TL::kStages;
                if (lane == 0) {
                    if (i >= TL::kStages)
                        ok = mbar_wait(&empty[s], ((i / TL::kStages) - 1) & 1, abort_flag);
                    if (ok) {
                        if (blk >= 0 && blk < NB) {
                            if (i == 0) KVD_MARK(a.marks, 8);  // first copy issued
                            stage_blk[s] = blk;
                            uint8_t *dst = smem + SL::kStagesOff + s * TL::kStageBytes;
                            const size_t r = row0 + static_cast<size_t>(blk) * kBlock;
                            mbar_arrive_expect_tx(&full[s], TL::kStageBytes);
                            tma_load_1d(dst, static_cast<const uint8_t *>(a.k) + r * TL::kRowBytes,
                                        TL::kKBytes, &full[s], pol);
                            tma_load_1d(dst + TL::kKBytes,
                                        static_cast<const uint8_t *>(a.v) + r * TL::kRowBytes,
                                        TL::kKBytes, &full[s], pol);
                            if constexpr (DT == KVD_INT8) {
                                tma_load_1d(dst + 2 * TL::kKBytes,
                                            static_cast<const float *>(a.k_scale) + r,
                                            kBlock * 4, &full[s], pol);
                                tma_load_1d(dst + 2 * TL::kKBytes + kBlock * 4,
                                            static_cast<const float *>(a.v_scale) + r,
                                            kBlock * 4, &full[s], pol);
                            } else if constexpr (DT == KVD_Q8_0 || DT == KVD_Q4_0) {
                                constexpr int kSB = TL::kScaleBytes;
                                tma_load_1d(dst + 2 * TL::kKBytes,
                                            static_cast<const __half *>(a.k_scale) +
                                                r * (kHeadDim / 32),
                                            kSB, &full[s], pol);
                                tma_load_1d(dst + 2 * TL::kKBytes + kSB,
                                            static_cast<const __half *>(a.v_scale) +
                                                r * (kHeadDim / 32),
                                            kSB, &full[s], pol);
                            }
                        } else {
                            // an id outside the cache: report it, skip the block
                            stage_blk[s] = -1;
                            report_status(a.dev_status, KVD_ERR_INVALID);
                            mbar_arrive(&full[s]);
                        }
                    } else {
                        *abort_flag = 1;
                        report_status(a.dev_status, KVD_ERR_TIMEOUT);
                    }
                }
                ok = __shfl_sync(kFull, ok, 0);
                if (!ok) break;
                ++i;
            }
        }
        if constexpr (TAIL) {
            if (ok)
                ok = produce_tail<DT, WIDE>(a, NB, split, bg, cnt, list, i, full, empty, stage_blk,
                                      stage_mask, smem + SL::kStagesOff, abort_flag, lane, pol);
        }
        const int issued = i;
        // one end marker per consumer group (stages i, i+1, ...)
        for (int j = 0; j < TL::kGroups && ok; ++j, ++i) {
            const int s = i % TL::kStages;
            if (lane == 0) {
                if (i >= TL::kStages)
                    ok = mbar_wait(&empty[s], ((i / TL::kStages) - 1) & 1, abort_flag);
                if (ok) {
                    stage_blk[s] = kEndMark;
                    mbar_arrive(&full[s]);
                } else {
                    *abort_flag = 1;
                    report_status(a.dev_status, KVD_ERR_TIMEOUT);
                }
            }
            ok = __shfl_sync(kFull, ok, 0);
        }
        if (lane == 0) *issued_s = issued;
    } else {
        // ------------------------------------------------------ consumers
        if (!a.early_q) load_query<DT, GC>(a, b, h0, warp, lane, q_s, coef, nullptr, nullptr);
        // the query words and coefficients are visible to every consumer warp
        asm volatile("bar.sync 1, %0;" ::"r"(TL::kConsumerWarps * 32) : "memory");
        float *pw = pw_all + warp * SL::kPwWarpFloats;
        const int group = warp / kWarpsPerGroup, wg = warp % kWarpsPerGroup;
        int i = group;         // stage sequence number of this group
        bool at_tail = false;  // stage i is the group's first moment-tail stage
        if constexpr (DT == KVD_Q4_0) {
            QRegsQ4<GC> qr;
            load_qregs_q4<GC>(q_s, reinterpret_cast<const int *>(coef + 4), lane & 3, qr);
            for (;; i += TL::kGroups) {
                const int s = i % TL::kStages;
                const bool ok = mbar_wait(&full[s], (i / TL::kStages) & 1, abort_flag);
                if (!__all_sync(kFull, ok)) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report_status(a.dev_status, KVD_ERR_TIMEOUT);
                    }
                    break;
                }
                const int blk = stage_blk[s];
                if (i == group && tid == 0) KVD_MARK(a.marks, 2);  // first stage in
                if (blk == kEndMark) break;
                if (TAIL && blk <= kTailBase) {
                    at_tail = true;
                    break;
                }
                if (blk >= 0) {
                    const int n_valid = min(kBlock, len - blk * kBlock);
                    consume_q4<GC, SV>(smem + SL::kStagesOff + s * TL::kStageBytes, n_valid,
                                       coef, qr, pw, wg, lane, st, a.sv_eps);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
        } else if constexpr (DT != KVD_F16) {
            QRegsI8<GC> qr;
            load_qregs_i8<GC>(q_s, lane >> 2, lane & 3, qr);
            for (;; i += TL::kGroups) {
                const int s = i % TL::kStages;
                const bool ok = mbar_wait(&full[s], (i / TL::kStages) & 1, abort_flag);
                if (!__all_sync(kFull, ok)) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report_status(a.dev_status, KVD_ERR_TIMEOUT);
                    }
                    break;
                }
                const int blk = stage_blk[s];
                if (i == group && tid == 0) KVD_MARK(a.marks, 2);  // first stage in
                if (blk == kEndMark) break;
                if (TAIL && blk <= kTailBase) {
                    at_tail = true;
                    break;
                }
                if (blk >= 0) {
                    const int n_valid = min(kBlock, len - blk * kBlock);
                    if constexpr (DT == KVD_INT8)
                        consume_int8<GC, SV>(smem + SL::kStagesOff + s * TL::kStageBytes,
                                             n_valid, coef, qr, pw, wg, lane, st, a.sv_eps);
                    else
                        consume_q8<GC, SV>(smem + SL::kStagesOff + s * TL::kStageBytes, n_valid,
                                           coef, qr, pw, wg, lane, st, a.sv_eps);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
        } else {
            QRegsF16<GC> qr;
            load_qregs_f16<GC>(q_s, lane & 7, qr);
            for (;; i += TL::kGroups) {
                const int s = i % TL::kStages;
                const bool ok = mbar_wait(&full[s], (i / TL::kStages) & 1, abort_flag);
                if (!__all_sync(kFull, ok)) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report_status(a.dev_status, KVD_ERR_TIMEOUT);
                    }
                    break;
                }
                const int blk = stage_blk[s];
                if (i == group && tid == 0) KVD_MARK(a.marks, 2);  // first stage in
                if (blk == kEndMark) break;
                if (TAIL && blk <= kTailBase) {
                    at_tail = true;
                    break;
                }
                if (blk >= 0) {
                    const int n_valid = min(kBlock, len - blk * kBlock);
                    consume_f16<GC, SV>(smem + SL::kStagesOff + s * TL::kStageBytes, n_valid,
                                        qr, pw, wg, lane, st, a.sv_eps);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
        }
        if constexpr (TAIL) {
            if (at_tail)
                tail_loop<DT, GC, WIDE>(a, len, NB, b, h0, i, full, empty, stage_blk, stage_mask,
                                  smem + SL::kStagesOff, pw, wg, lane, abort_flag, ts);
        }
        // per-warp totals: l summed over the lanes of each head
        if constexpr (DT != KVD_F16) {
            st.l += __shfl_xor_sync(kFull, st.l, 4);
            st.l += __shfl_xor_sync(kFull, st.l, 8);
            st.l += __shfl_xor_sync(kFull, st.l, 16);
        } else {
            st.l += __shfl_xor_sync(kFull, st.l, 8);
            st.l += __shfl_xor_sync(kFull, st.l, 16);
        }
    }
    __syncthreads();  // (A) every stage consumed: the ring becomes scratch
    if (tid == 0) KVD_MARK(a.marks, 3);  // every stage consumed
    const bool aborted = *abort_flag != 0;
    if (!aborted && warp < TL::kConsumerWarps) {
        float *mg = reinterpret_cast<float *>(smem + SL::kStagesOff);
        constexpr int lph = (DT != KVD_F16 ? 4 : 8) / GC;
#pragma unroll
        for (int h = 0; h < GC; ++h) {
            float *row = mg + (warp * GC + h) * kPartStride;
            if (lane == h * lph) {
                row[0] = st.m;
                row[1] = st.l;
            }
            *reinterpret_cast<float4 *>(row + kAccOff + 4 * lane) =
                make_float4(st.acc[h][0].x, st.acc[h][0].y, st.acc[h][1].x, st.acc[h][1].y);
        }
        if constexpr (TAIL) {
            constexpr int SH = tail_shift<DT, GC>();
#pragma unroll
            for (int h = 0; h < GC; ++h) {
                float *row = mg + ((TL::kConsumerWarps + warp) * GC + h) * kPartStride;
                if (lane == (h << SH)) {
                    row[0] = ts.m;
                    row[1] = ts.l;
                }
                *reinterpret_cast<float4 *>(row + kAccOff + 4 * lane) = make_float4(
                    ts.acc[h][0].x, ts.acc[h][0].y, ts.acc[h][1].x, ts.acc[h][1].y);
            }
        }
    }
    __syncthreads();  // (B) merge area written
    if (aborted) {
        // wind down: wait (bounded) for the copies still landing in the ring
        if (warp == TL::kConsumerWarps && lane == 0) {
            const int issued = *issued_s;
            volatile int never = 0;
            for (int i = max(0, issued - TL::kStages); i < issued; ++i)
                (void)mbar_wait(&full[i % TL::kStages], (i / TL::kStages) & 1, &never);
        }
        return;
    }

    // ---- CTA merge of the warp states: thread (h, 4 channels)
    const float *mg = reinterpret_cast<const float *>(smem + SL::kStagesOff);
    const bool single = a.splits == 1;
    float *part = a.partials + (static_cast<size_t>(prob) * a.splits + split) * GC * kPartStride;
    if (tid < GC * 32) {
        const int h = tid >> 5, d4 = tid & 31;
        float M = kNegBig;
#pragma unroll
        for (int w = 0; w < SL::kRows; ++w) M = fmaxf(M, mg[(w * GC + h) * kPartStride]);
        float L = 0.0f;
        float4 A = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int w = 0; w < SL::kRows; ++w) {
            const float *row = mg + (w * GC + h) * kPartStride;
            const float sc = exp2f(row[0] - M);
            L = fmaf(sc, row[1], L);
            const float4 r4 = *reinterpret_cast<const float4 *>(row + kAccOff + 4 * d4);
            A.x = fmaf(sc, r4.x, A.x);
            A.y = fmaf(sc, r4.y, A.y);
            A.z = fmaf(sc, r4.z, A.z);
            A.w = fmaf(sc, r4.w, A.w);
        }
        if (single) {
            const float inv = L > 0.0f ? 1.0f / L : 0.0f;
            *reinterpret_cast<float4 *>(a.out + (static_cast<size_t>(b) * a.H + h0 + h) *
                                                    kHeadDim + 4 * d4) =
                make_float4(A.x * inv, A.y * inv, A.z * inv, A.w * inv);
        } else {
            float *pr = part + h * kPartStride;
            if (d4 == 0) {
                pr[0] = M;
                pr[1] = L;
            }
            *reinterpret_cast<float4 *>(pr + kAccOff + 4 * d4) = A;
        }
    }
    if (single) return;

    // ---- the last CTA of this problem to arrive merges all splits
    __syncthreads();  // every partial store of the CTA precedes the release
    if (tid == 0) {
        KVD_MARK(a.marks, 4);  // partial written
        *last_flag = atomic_add_acq_rel_gpu(&a.counters[prob], 1u) ==
                     static_cast<unsigned>(a.splits - 1);
        KVD_MARK(a.marks, 5);  // arrival counted
    }
    __syncthreads();
    if (!*last_flag) return;
    // Thread (part, h, 4 channels) merges the splits of its part online:
    // one batch of loads (maxima, sums, accumulators of kMergeBatch splits)
    // in flight at a time, rescaled onto the running maximum.  The parts
    // then merge in shared memory (the ring).
    const int S = a.splits;
    const float *p0 = a.partials + static_cast<size_t>(prob) * S * GC * kPartStride;
    constexpr int kParts = TL::kConsumerWarps / GC;
    constexpr int kMergeBatch = 10;
    float *mrow = reinterpret_cast<float *>(smem + SL::kStagesOff);  // [kParts][GC] m, l
    float4 *arow = reinterpret_cast<float4 *>(mrow + 2 * TL::kConsumerWarps * 4);
    if (warp < TL::kConsumerWarps) {
        const int hd = tid % (GC * 32), part = tid / (GC * 32);
        const int h = hd >> 5, d4 = hd & 31;
        const int s_beg = (S * part) / kParts, s_end = (S * (part + 1)) / kParts;
        const float *base = p0 + h * kPartStride;
        float M = kNegBig, L = 0.0f;
        float4 A = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int s0 = s_beg; s0 < s_end; s0 += kMergeBatch) {
            float m[kMergeBatch], l[kMergeBatch];
            float4 r[kMergeBatch];
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                const float *row = base + static_cast<size_t>(s0 + u) * GC * kPartStride;
                const bool in = s0 + u < s_end;
                m[u] = in ? __ldcg(row) : kNegBig;
                l[u] = in ? __ldcg(row + 1) : 0.0f;
                r[u] = in ? __ldcg(reinterpret_cast<const float4 *>(row + kAccOff + 4 * d4))
                          : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
            float mb = M;
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) mb = fmaxf(mb, m[u]);
            const float al = exp2f(M - mb);
            L *= al;
            A.x *= al;
            A.y *= al;
            A.z *= al;
            A.w *= al;
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                const float wgt = exp2f(m[u] - mb);
                L = fmaf(wgt, l[u], L);
                A.x = fmaf(wgt, r[u].x, A.x);
                A.y = fmaf(wgt, r[u].y, A.y);
                A.z = fmaf(wgt, r[u].z, A.z);
                A.w = fmaf(wgt, r[u].w, A.w);
            }
            M = mb;
        }
        if (d4 == 0) {
            mrow[(part * GC + h) * 2] = M;
            mrow[(part * GC + h) * 2 + 1] = L;
        }
        arow[tid] = A;
    }
    __syncthreads();
    if (tid < GC * 32) {
        const int h = tid >> 5, d4 = tid & 31;
        float M = kNegBig;
#pragma unroll
        for (int pt = 0; pt < kParts; ++pt) M = fmaxf(M, mrow[(pt * GC + h) * 2]);
        float L = 0.0f;
        float4 A = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int pt = 0; pt < kParts; ++pt) {
            const float wgt = exp2f(mrow[(pt * GC + h) * 2] - M);
            L = fmaf(wgt, mrow[(pt * GC + h) * 2 + 1], L);
            const float4 r = arow[pt * GC * 32 + tid];
            A.x = fmaf(wgt, r.x, A.x);
            A.y = fmaf(wgt, r.y, A.y);
            A.z = fmaf(wgt, r.z, A.z);
            A.w = fmaf(wgt, r.w, A.w);
        }
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
        *reinterpret_cast<float4 *>(a.out + (static_cast<size_t>(b) * a.H + h0 + h) * kHeadDim +
                                    4 * d4) = make_float4(A.x * inv, A.y * inv, A.z * inv,
                                                          A.w * inv);
    }
    if (tid == 0) {
        a.counters[prob] = 0u;  // leave the counter ready for the next call
        KVD_MARK(a.marks, 6);   // splits merged
    }
}

DecodeArgs make_decode_args(const kvd_cache &c, const Geom &g, const DecodePlan &p,
                            const float *q, float scale, const int32_t *sel_idx,
                            const int32_t *sel_cnt, float *out, float *partials,
                            uint32_t *counters, bool early_q, float sv_eps) {
    DecodeArgs a = {};
    a.sv_eps = sv_eps;
    a.early_q = early_q ? 1 : 0;
    a.k = c.k;
    a.v = c.v;
    a.k_scale = c.k_scale;
    a.v_scale = c.v_scale;
    a.q = q;
    a.out = out;
    a.sel_idx = sel_idx;
    a.sel_cnt = sel_cnt;
    a.partials = partials;
    a.counters = counters;
    a.dev_status = c.dev_status;
    a.Hkv = g.Hkv;
    a.H = g.H;
    a.G = g.G;
    a.max_seq = g.max_seq;
    a.nbmax = g.nbmax;
    a.len = g.len;
    a.NB = g.NB;
    a.seq_lens = c.seq_lens;
    a.seq_add = g.seq_add;
    a.splits = p.splits;
    a.subgroups = p.subgroups;
    a.plan_blocks = p.blocks;
    a.scale_log2 = scale * kLog2e;
    a.marks = mark_region(kMarkDecode);
    return a;
}


// ----------------------------------------------------------------------------
// The kernel and its launchers.  SV (sparse-V) kernels are instantiated by
// their own translation unit, so the plain kernels carry none of that code:
// after an L2 flush every instruction of a kernel comes from HBM again, and
// a shorter instruction stream starts sooner.
template <int DT, int GC, bool DENSE, bool SV, bool TAIL, bool WIDE>
__global__ void __launch_bounds__(TileW<DT, WIDE>::kThreads, TileW<DT, WIDE>::kMinCtas)
    decode_kernel(DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    decode_body<DT, GC, DENSE, SV, TAIL, WIDE>(a, blockIdx.x, blockIdx.y, smem);
}

template <int DT, int GC, bool DENSE, bool SV, bool TAIL, bool WIDE = false>
cudaError_t launch_decode_t(const DecodeArgs &a, int P_sub, cudaStream_t st, bool pdl) {
    using SL = SmemLayout<DT, GC, TAIL, WIDE>;
    const cudaError_t e = prepare_kernel(
        reinterpret_cast<const void *>(decode_kernel<DT, GC, DENSE, SV, TAIL, WIDE>),
        TileW<DT, WIDE>::kThreads, SL::kTotal);
    if (e != cudaSuccess) return e;
    return launch_ex(decode_kernel<DT, GC, DENSE, SV, TAIL, WIDE>, dim3(a.splits, P_sub),
                     dim3(TileW<DT, WIDE>::kThreads), SL::kTotal, st, pdl, a);
}

template <int DT, bool DENSE, bool SV, bool TAIL, bool WIDE = false>
cudaError_t launch_decode_gc(int gc, const DecodeArgs &a, int P_sub, cudaStream_t st, bool pdl) {
    switch (gc) {
        case 1: return launch_decode_t<DT, 1, DENSE, SV, TAIL, WIDE>(a, P_sub, st, pdl);
        case 2: return launch_decode_t<DT, 2, DENSE, SV, TAIL, WIDE>(a, P_sub, st, pdl);
        default: return launch_decode_t<DT, 4, DENSE, SV, TAIL, WIDE>(a, P_sub, st, pdl);
    }
}

template <bool SV>
cudaError_t launch_decode_any(const kvd_cache &c, const Geom &g, const DecodePlan &p,
                              const float *q, float scale, const int32_t *sel_idx,
                              const int32_t *sel_cnt, float *out, float *partials,
                              uint32_t *counters, cudaStream_t st, bool pdl, bool early_q,
                              float sv_eps) {
    const DecodeArgs a = make_decode_args(c, g, p, q, scale, sel_idx, sel_cnt, out, partials,
                                          counters, early_q, sv_eps);
    const int P_sub = g.B * g.Hkv * p.subgroups;
    const bool dense = sel_idx == nullptr;
    const int gc = p.heads_per_cta;
    if (p.wide) {  // quantized caches only (plan_decode)
        if (g.dtype == KVD_INT8)
            return dense ? launch_decode_gc<KVD_INT8, true, SV, false, true>(gc, a, P_sub, st, pdl)
                         : launch_decode_gc<KVD_INT8, false, SV, false, true>(gc, a, P_sub, st, pdl);
        if (g.dtype == KVD_Q8_0)
            return dense ? launch_decode_gc<KVD_Q8_0, true, SV, false, true>(gc, a, P_sub, st, pdl)
                         : launch_decode_gc<KVD_Q8_0, false, SV, false, true>(gc, a, P_sub, st, pdl);
        return dense ? launch_decode_gc<KVD_Q4_0, true, SV, false, true>(gc, a, P_sub, st, pdl)
                     : launch_decode_gc<KVD_Q4_0, false, SV, false, true>(gc, a, P_sub, st, pdl);
    }
    if (g.dtype == KVD_INT8)
        return dense ? launch_decode_gc<KVD_INT8, true, SV, false>(gc, a, P_sub, st, pdl)
                     : launch_decode_gc<KVD_INT8, false, SV, false>(gc, a, P_sub, st, pdl);
    if (g.dtype == KVD_Q8_0)
        return dense ? launch_decode_gc<KVD_Q8_0, true, SV, false>(gc, a, P_sub, st, pdl)
                     : launch_decode_gc<KVD_Q8_0, false, SV, false>(gc, a, P_sub, st, pdl);
    if (g.dtype == KVD_Q4_0)
        return dense ? launch_decode_gc<KVD_Q4_0, true, SV, false>(gc, a, P_sub, st, pdl)
                     : launch_decode_gc<KVD_Q4_0, false, SV, false>(gc, a, P_sub, st, pdl);
    return dense ? launch_decode_gc<KVD_F16, true, SV, false>(gc, a, P_sub, st, pdl)
                 : launch_decode_gc<KVD_F16, false, SV, false>(gc, a, P_sub, st, pdl);
}

}  // namespace
}  // namespace kvd
