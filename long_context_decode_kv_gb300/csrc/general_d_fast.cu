// general_d_fast.cu -- split-KV decode attention for head dims 64, 256 and
// 512 (f16 and int8 caches), the warp-specialised counterpart of the tuned
// head-dim-128 kernel.
//
// "Sparse Attention -- Quest-style block-selector for long-context decode
// (#551)", "Decode": attention of each query head over the tokens of its KV
// head's listed blocks (every block for the dense arm), split over CTAs that
// each keep an online softmax (running max m, mass l, unnormalised output),
// then merged.  "cpu-attn", Method: on the int8 cache the query is quantized
// per head like a cache row (absmax / 127), q.k is the exact int32 dot of the
// codes times both scales, and V is dequantized as code * row scale.
//
// CTA of split s of (sequence, KV head, subgroup of GC <= 4 query heads): one
// producer warp copies tiles (T tokens of a listed block: its K rows, V rows
// and on the int8 cache the two scale runs; 8-16 KiB) with 1-D bulk copies
// into a ring of shared-memory stages (12 for the shipped shapes: a multiple
// of the consumer warps, so that each stage serves one warp), each completing
// on its own mbarrier.  Each of the 12 consumer warps takes every 12th tile
// whole and keeps its own online softmax over the tiles it saw -- no CTA
// barrier inside the tile loop:
//   1. q.k: a token's row is read by D/16 lanes (16 channels each, the query
//      chunk in registers), and a reduce-scatter over those lanes leaves
//      every lane one head's score;
//   2. softmax: the tile's max and mass per head over the lanes that hold
//      that head; the weights go to the warp's shared-memory rows as (p, p)
//      pairs (int8: p times the token's V scale);
//   3. P.V: a lane owns 4 (D = 64) or D/32 (D >= 256) channels of every head
//      and every other token (D = 64) or every token (D >= 256).
// At the end the warps' states merge in shared memory in warp order, the
// CTA's (m, l, acc) go to the split partials, and the last CTA of the problem
// to arrive merges the splits in split order and writes the output.
#include "common.cuh"
#include "internal.h"

namespace kvd {
namespace {

constexpr int kFastWarps = 12;  // consumer warps; warp 12 produces
constexpr int kFastThreads = 32 * (kFastWarps + 1);
constexpr unsigned kAll = 0xffffffffu;

template <int DT, int D>
struct FastTile {
    static constexpr int kElt = DT == KVD_F16 ? 2 : 1;
    static constexpr int kRow = D * kElt;  // bytes of a token's row
    // tokens per tile: K + V of a tile within 16 KiB
    static constexpr int kT = 2 * 64 * kRow <= 16384   ? 64
                              : 2 * 32 * kRow <= 16384 ? 32
                              : 2 * 16 * kRow <= 16384 ? 16
                                                       : 8;
    static constexpr int kScaleBytes = DT == KVD_F16 ? 0 : 2 * kT * 4;
    static constexpr int kStageBytes = 2 * kT * kRow + kScaleBytes;
    // a multiple of the consumer warps: tile u goes to warp u % kFastWarps and
    // stage u % kStages, so every tile of a stage goes to one warp, which waits on
    // the stage's phases in order (warps sharing a stage could see a later
    // phase's parity as an earlier one's and read it before it lands)
    static constexpr int kStages =
        (204800 / kStageBytes < 24 ? 204800 / kStageBytes : 24) / kFastWarps * kFastWarps;
    static_assert(kStages >= kFastWarps, "a stage per consumer warp at least");
    static constexpr int kLPT = D / 16;      // q.k: lanes per token (16 channels each)
    static constexpr int kTPP = 32 / kLPT;   // tokens per q.k pass
    static constexpr int kPasses = kT / kTPP;
    static constexpr int kCPL = D >= 128 ? D / 32 : 4;  // P.V: channels per lane
    static constexpr int kLPV = D / kCPL;    // P.V: lanes per token
    static constexpr int kTPV = 32 / kLPV;   // tokens per P.V step
    static_assert(kT % kTPP == 0 && kT % kTPV == 0, "tile shape");
};

// Shared memory: the ring, the barriers and stage records, the query, and per
// consumer warp its tile's weight pairs.
template <int DT, int D, int GC>
struct FastLayout {
    using TL = FastTile<DT, D>;
    static constexpr int kRing = TL::kStages * TL::kStageBytes;
    static constexpr int kMerge = kFastWarps * GC * (D + 2) * 4;  // the warps' states, after the loop
    static constexpr int kBarOff = ((kRing > kMerge ? kRing : kMerge) + 127) / 128 * 128;
    static constexpr int kRecOff = kBarOff + 16 * TL::kStages;    // [stages] tokens in the tile
    static constexpr int kQOff = (kRecOff + 4 * TL::kStages + 15) / 16 * 16;
    static constexpr int kQBytes = GC * D * 4;                    // f32 query or int8 codes
    static constexpr int kQsOff = kQOff + kQBytes;                // [GC] query scales (int8)
    static constexpr int kFlagOff = kQsOff + 16;
    static constexpr int kPwOff = kFlagOff + 16;                  // [warp][T][GC] (p, p)
    static constexpr int kTotal = kPwOff + kFastWarps * TL::kT * GC * 8;
};

template <int DT, int D, int GC>
__global__ void __launch_bounds__(kFastThreads, 1)
    gd_fast_kernel(kvd_cache c, const float *q, int H, int G, float scale_log2,
                   const int32_t *sel_idx, const int32_t *sel_cnt, int splits, int subgroups,
                   float *part_acc, float *part_ml, float *out, uint32_t *counters) {
    using TL = FastTile<DT, D>;
    using SL = FastLayout<DT, D, GC>;
    constexpr int S = TL::kStages, T = TL::kT;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + SL::kBarOff);
    uint64_t *empty = full + S;
    int *stage_nt = reinterpret_cast<int *>(smem + SL::kRecOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SL::kFlagOff);
    int *issued_s = reinterpret_cast<int *>(smem + SL::kFlagOff + 4);
    float *qs_s = reinterpret_cast<float *>(smem + SL::kQsOff);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, prob = blockIdx.y;
    const int sub = prob % subgroups, p = prob / subgroups;  // p = b * Hkv + h
    const int b = p / c.n_kv_heads, kvh = p % c.n_kv_heads;
    const int h0 = kvh * G + sub * GC;  // first query head of the CTA

    const int len = c.len, NB = (len + kBlock - 1) / kBlock;
    const size_t nbmax = static_cast<size_t>(c.max_seq / kBlock);
    const size_t row0 = static_cast<size_t>(p) * c.max_seq;
    const bool dense = sel_idx == nullptr;
    int n_list = NB;
    if (!dense) {  // a count outside [0, NB] is reported and clamped
        n_list = sel_cnt[p];
        if (n_list < 0 || n_list > NB) {
            if (tid == 0) report_status(c.dev_status, KVD_ERR_INVALID);
            n_list = n_list < 0 ? 0 : NB;
        }
    }
    const int32_t *list = dense ? nullptr : sel_idx + p * nbmax;
    constexpr int TPB = kBlock / T;  // tiles per block
    const int i0 = static_cast<int>(static_cast<long long>(split) * n_list / splits);
    const int i1 = static_cast<int>(static_cast<long long>(split + 1) * n_list / splits);
    const int U = (i1 - i0) * TPB;  // tiles of this split

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        *abort_flag = 0;
        *issued_s = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kFastWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int u = 0;
            for (; u < U; ++u) {
                const int s = u % S;
                if (u >= S && !mbar_wait(&empty[s], ((u / S) - 1) & 1, abort_flag)) {
                    *abort_flag = 1;
                    report_status(c.dev_status, KVD_ERR_TIMEOUT);
                    break;
                }
                const int j = dense ? i0 + u / TPB : list[i0 + u / TPB];
                int nt = -1, t0 = 0;
                if (j >= 0 && j < NB) {
                    t0 = j * kBlock + (u % TPB) * T;
                    nt = len - t0 < T ? len - t0 : T;
                    if (nt < 0) nt = 0;
                } else if (u % TPB == 0) {
                    report_status(c.dev_status, KVD_ERR_INVALID);  // a bad block id: skipped
                }
                stage_nt[s] = nt;
                if (nt <= 0) {
                    mbar_arrive(&full[s]);
                    continue;
                }
                uint8_t *st = smem + s * TL::kStageBytes;
                const uint32_t rows = static_cast<uint32_t>(nt * TL::kRow);
                // a scale run rounded up to 4 floats stays inside the block
                const uint32_t sc4 = DT == KVD_F16 ? 0u : static_cast<uint32_t>((nt + 3) / 4 * 16);
                mbar_arrive_expect_tx(&full[s], 2 * rows + 2 * sc4);
                tma_load_1d(st, static_cast<const uint8_t *>(c.k) + (row0 + t0) * TL::kRow, rows,
                            &full[s], pol);
                tma_load_1d(st + T * TL::kRow,
                            static_cast<const uint8_t *>(c.v) + (row0 + t0) * TL::kRow, rows,
                            &full[s], pol);
                if constexpr (DT != KVD_F16) {
                    float *ss = reinterpret_cast<float *>(st + 2 * T * TL::kRow);
                    tma_load_1d(ss, static_cast<const float *>(c.k_scale) + row0 + t0, sc4,
                                &full[s], pol);
                    tma_load_1d(ss + T, static_cast<const float *>(c.v_scale) + row0 + t0, sc4,
                                &full[s], pol);
                }
            }
            *issued_s = u;
        }
        __syncthreads();  // (A) the consumers are done with the ring
        __syncthreads();  // (B) the warps' states are written
        return;
    }

    // ---------------------------------------------------------- consumers
    // the CTA's query heads: f32 (f16 cache) or absmax int8 codes and scales
    const float *qp = q + (static_cast<size_t>(b) * H + h0) * D;
    if constexpr (DT == KVD_F16) {
        float *q_f = reinterpret_cast<float *>(smem + SL::kQOff);
        for (int i = tid; i < GC * D; i += kFastWarps * 32) q_f[i] = qp[i];
    } else {
        int8_t *q_c = reinterpret_cast<int8_t *>(smem + SL::kQOff);
        for (int g = warp; g < GC; g += kFastWarps) {
            float a = 0.0f;
            for (int d = lane; d < D; d += 32) a = fmaxf(a, fabsf(qp[g * D + d]));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(kAll, a, o));
            const float qs = __fdiv_rn(a, 127.0f);
            for (int d = lane; d < D; d += 32) {
                int code = 0;
                if (qs != 0.0f)
                    code = max(-127, min(127, __float2int_rn(__fdiv_rn(qp[g * D + d], qs))));
                q_c[g * D + d] = static_cast<int8_t>(code);
            }
            if (lane == 0) qs_s[g] = qs;
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kFastWarps * 32) : "memory");

    // q.k lane: token slot ts (0 .. TPP-1) and channel part cp (16 channels)
    const int ts = lane / TL::kLPT, cp = lane % TL::kLPT;
    constexpr int kHeadSpan = TL::kLPT / GC;  // lanes of a token holding one head after the scatter
    const int hq = cp / kHeadSpan;            // the head this lane's scores belong to
    float qf[DT == KVD_F16 ? GC : 1][16];
    uint32_t qi[DT == KVD_F16 ? 1 : GC][4];
    float q_scale = 1.0f;
    if constexpr (DT == KVD_F16) {
        const float *q_f = reinterpret_cast<const float *>(smem + SL::kQOff);
#pragma unroll
        for (int g = 0; g < GC; ++g)
#pragma unroll
            for (int k = 0; k < 16; ++k) qf[g][k] = q_f[g * D + 16 * cp + k];
    } else {
        const int8_t *q_c = reinterpret_cast<const int8_t *>(smem + SL::kQOff);
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            const uint4 w = *reinterpret_cast<const uint4 *>(q_c + g * D + 16 * cp);
            qi[g][0] = w.x;
            qi[g][1] = w.y;
            qi[g][2] = w.z;
            qi[g][3] = w.w;
        }
        q_scale = qs_s[hq];
    }
    // P.V lane: token slot vs and channels vc .. vc + CPL - 1
    const int vs = lane / TL::kLPV, vc = (lane % TL::kLPV) * TL::kCPL;
    float2 acc[GC][TL::kCPL / 2];
#pragma unroll
    for (int g = 0; g < GC; ++g)
#pragma unroll
        for (int k = 0; k < TL::kCPL / 2; ++k) acc[g][k] = make_float2(0.0f, 0.0f);
    float m_run = -__int_as_float(0x7f800000), l_run = 0.0f;  // head hq's state
    float2 *pw = reinterpret_cast<float2 *>(smem + SL::kPwOff) + warp * T * GC;

    for (int u = warp; u < U; u += kFastWarps) {
        const int s = u % S;
        const bool ok = mbar_wait(&full[s], (u / S) & 1, abort_flag);
        if (!__all_sync(kAll, ok)) {
            if (lane == 0) {
                *abort_flag = 1;
                report_status(c.dev_status, KVD_ERR_TIMEOUT);
            }
            break;
        }
        const int nt = stage_nt[s];
        if (nt > 0) {
            const uint8_t *st = smem + s * TL::kStageBytes;
            const float *ksc = reinterpret_cast<const float *>(st + 2 * T * TL::kRow);
            // ---- 1. q.k: score of head hq for the tokens pass * TPP + ts
            float x[TL::kPasses];
            float mt = -__int_as_float(0x7f800000);
#pragma unroll
            for (int ps = 0; ps < TL::kPasses; ++ps) {
                const int t = ps * TL::kTPP + ts;
                const uint8_t *row = st + t * TL::kRow;
                float part[GC];
                if constexpr (DT == KVD_F16) {
                    const uint4 w0 = *reinterpret_cast<const uint4 *>(row + 32 * cp);
                    const uint4 w1 = *reinterpret_cast<const uint4 *>(row + 32 * cp + 16);
                    const __half2 *h2a = reinterpret_cast<const __half2 *>(&w0);
                    const __half2 *h2b = reinterpret_cast<const __half2 *>(&w1);
                    float kx[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 fa = __half22float2(h2a[i]), fb = __half22float2(h2b[i]);
                        kx[2 * i] = fa.x;
                        kx[2 * i + 1] = fa.y;
                        kx[8 + 2 * i] = fb.x;
                        kx[8 + 2 * i + 1] = fb.y;
                    }
#pragma unroll
                    for (int g = 0; g < GC; ++g) {
                        float2 a2 = make_float2(0.0f, 0.0f);
#pragma unroll
                        for (int k = 0; k < 16; k += 2)
                            a2 = __ffma2_rn(make_float2(qf[g][k], qf[g][k + 1]),
                                            make_float2(kx[k], kx[k + 1]), a2);
                        part[g] = a2.x + a2.y;
                    }
                } else {
                    const uint4 w = *reinterpret_cast<const uint4 *>(row + 16 * cp);
#pragma unroll
                    for (int g = 0; g < GC; ++g) {
                        int dd = __dp4a(static_cast<int>(w.x), static_cast<int>(qi[g][0]), 0);
                        dd = __dp4a(static_cast<int>(w.y), static_cast<int>(qi[g][1]), dd);
                        dd = __dp4a(static_cast<int>(w.z), static_cast<int>(qi[g][2]), dd);
                        dd = __dp4a(static_cast<int>(w.w), static_cast<int>(qi[g][3]), dd);
                        part[g] = __int_as_float(dd);  // an int32 carried in a float register
                    }
                }
                // reduce-scatter over the token's LPT lanes: the top bits of
                // cp pick the head, the rest sum
                float v;
                if constexpr (DT == KVD_F16) {
                    if constexpr (GC == 4) {
                        const bool up = (cp & (2 * kHeadSpan)) != 0;
                        float k0 = up ? part[2] : part[0], k1 = up ? part[3] : part[1];
                        k0 += __shfl_xor_sync(kAll, up ? part[0] : part[2], 2 * kHeadSpan);
                        k1 += __shfl_xor_sync(kAll, up ? part[1] : part[3], 2 * kHeadSpan);
                        const bool mid = (cp & kHeadSpan) != 0;
                        v = (mid ? k1 : k0) + __shfl_xor_sync(kAll, mid ? k0 : k1, kHeadSpan);
                    } else if constexpr (GC == 2) {
                        const bool up = (cp & kHeadSpan) != 0;
                        v = (up ? part[1] : part[0]) +
                            __shfl_xor_sync(kAll, up ? part[0] : part[1], kHeadSpan);
                    } else {
                        v = part[0];
                    }
#pragma unroll
                    for (int o = kHeadSpan / 2; o > 0; o >>= 1) v += __shfl_xor_sync(kAll, v, o);
                    x[ps] = t < nt ? v * scale_log2 : -__int_as_float(0x7f800000);
                } else {
                    int vi;
                    if constexpr (GC == 4) {
                        const bool up = (cp & (2 * kHeadSpan)) != 0;
                        int k0 = __float_as_int(up ? part[2] : part[0]);
                        int k1 = __float_as_int(up ? part[3] : part[1]);
                        k0 += __shfl_xor_sync(kAll, __float_as_int(up ? part[0] : part[2]),
                                              2 * kHeadSpan);
                        k1 += __shfl_xor_sync(kAll, __float_as_int(up ? part[1] : part[3]),
                                              2 * kHeadSpan);
                        const bool mid = (cp & kHeadSpan) != 0;
                        vi = (mid ? k1 : k0) + __shfl_xor_sync(kAll, mid ? k0 : k1, kHeadSpan);
                    } else if constexpr (GC == 2) {
                        const bool up = (cp & kHeadSpan) != 0;
                        vi = __float_as_int(up ? part[1] : part[0]) +
                             __shfl_xor_sync(kAll, __float_as_int(up ? part[0] : part[1]),
                                             kHeadSpan);
                    } else {
                        vi = __float_as_int(part[0]);
                    }
#pragma unroll
                    for (int o = kHeadSpan / 2; o > 0; o >>= 1) vi += __shfl_xor_sync(kAll, vi, o);
                    x[ps] = t < nt ? static_cast<float>(vi) * (q_scale * ksc[t]) * scale_log2
                                   : -__int_as_float(0x7f800000);
                }
                mt = fmaxf(mt, x[ps]);
            }
            // ---- 2. online softmax of head hq over the tile (its lanes: the
            // token slots, whose values are alike within a head's span)
#pragma unroll
            for (int o = TL::kLPT; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(kAll, mt, o));
            const float m_new = fmaxf(m_run, mt);
            const float alpha = exp2f(m_run - m_new);
            float lt = 0.0f;
            const float *vsc = ksc + T;
#pragma unroll
            for (int ps = 0; ps < TL::kPasses; ++ps) {
                const int t = ps * TL::kTPP + ts;
                const float pe = exp2f(x[ps] - m_new);  // 0 past the tile's tokens
                lt += pe;
                const float w = DT == KVD_F16 ? pe : (t < nt ? pe * vsc[t] : 0.0f);
                if (cp % kHeadSpan == 0) pw[t * GC + hq] = make_float2(w, w);
            }
#pragma unroll
            for (int o = TL::kLPT; o < 32; o <<= 1) lt += __shfl_xor_sync(kAll, lt, o);
            l_run = l_run * alpha + lt;
            m_run = m_new;
            // every lane rescales its accumulators of every head
#pragma unroll
            for (int g = 0; g < GC; ++g) {
                const float ag = __shfl_sync(kAll, alpha, g * kHeadSpan);
#pragma unroll
                for (int k = 0; k < TL::kCPL / 2; ++k) {
                    acc[g][k].x *= ag;
                    acc[g][k].y *= ag;
                }
            }
            __syncwarp();
            // ---- 3. P.V over the tile's tokens vs, vs + TPV, ...
            const uint8_t *vrow = st + T * TL::kRow + vc * TL::kElt;
            for (int t = vs; t < nt; t += TL::kTPV) {
                float2 vv[TL::kCPL / 2];
                if constexpr (DT == KVD_F16) {
                    if constexpr (TL::kCPL >= 8) {  // 16-byte pieces of 8 channels
#pragma unroll
                        for (int j = 0; j < TL::kCPL / 8; ++j) {
                            const uint4 w =
                                reinterpret_cast<const uint4 *>(vrow + t * TL::kRow)[j];
                            const __half2 *h2 = reinterpret_cast<const __half2 *>(&w);
#pragma unroll
                            for (int i = 0; i < 4; ++i) vv[4 * j + i] = __half22float2(h2[i]);
                        }
                    } else {
                        const uint2 w = *reinterpret_cast<const uint2 *>(vrow + t * TL::kRow);
                        vv[0] = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
                        vv[1] = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
                    }
                } else {  // 4-byte words of 4 codes
#pragma unroll
                    for (int j = 0; j < TL::kCPL / 4; ++j) {
                        const uint32_t w =
                            reinterpret_cast<const uint32_t *>(vrow + t * TL::kRow)[j];
                        vv[2 * j] = make_float2(
                            static_cast<float>(static_cast<int8_t>(w & 0xffu)),
                            static_cast<float>(static_cast<int8_t>((w >> 8) & 0xffu)));
                        vv[2 * j + 1] = make_float2(
                            static_cast<float>(static_cast<int8_t>((w >> 16) & 0xffu)),
                            static_cast<float>(static_cast<int8_t>(w >> 24)));
                    }
                }
#pragma unroll
                for (int g = 0; g < GC; ++g) {
                    const float2 pp = pw[t * GC + g];
#pragma unroll
                    for (int k = 0; k < TL::kCPL / 2; ++k) acc[g][k] = __ffma2_rn(vv[k], pp, acc[g][k]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    __syncthreads();  // (A) every tile consumed: the ring holds the warps' states next
    const bool aborted = *abort_flag != 0;
    // the token slots' sums of each channel (P.V lanes vs, same channels)
#pragma unroll
    for (int o = TL::kLPV; o < 32; o <<= 1)
#pragma unroll
        for (int g = 0; g < GC; ++g)
#pragma unroll
            for (int k = 0; k < TL::kCPL / 2; ++k) {
                acc[g][k].x += __shfl_xor_sync(kAll, acc[g][k].x, o);
                acc[g][k].y += __shfl_xor_sync(kAll, acc[g][k].y, o);
            }
    float *mg = reinterpret_cast<float *>(smem);  // [warp][GC][D + 2]: acc, m, l
    if (!aborted) {
        if (vs == 0) {
#pragma unroll
            for (int g = 0; g < GC; ++g)
#pragma unroll
                for (int k = 0; k < TL::kCPL / 2; ++k)
                    *reinterpret_cast<float2 *>(mg + (warp * GC + g) * (D + 2) + vc + 2 * k) =
                        acc[g][k];
        }
        if (ts == 0 && cp % kHeadSpan == 0) {
            mg[(warp * GC + hq) * (D + 2) + D] = m_run;
            mg[(warp * GC + hq) * (D + 2) + D + 1] = l_run;
        }
    }
    __syncthreads();  // (B)
    if (aborted) {
        // wind down: wait (bounded) for the copies still landing in the ring
        if (tid == 0) {
            const int issued = *issued_s;
            volatile int never = 0;
            for (int i = max(0, issued - S); i < issued; ++i)
                (void)mbar_wait(&full[i % S], (i / S) & 1, &never);
        }
        return;
    }
    // the CTA's state per head, the warps taken in order (one split: the output)
    const size_t slot = static_cast<size_t>(p) * splits + split;
    for (int i = tid; i < GC * D; i += kFastWarps * 32) {
        const int g = i / D, d = i % D;
        float M = -__int_as_float(0x7f800000);
        for (int w = 0; w < kFastWarps; ++w) M = fmaxf(M, mg[(w * GC + g) * (D + 2) + D]);
        float A = 0.0f, L = 0.0f;
        for (int w = 0; w < kFastWarps; ++w) {
            const float *r = mg + (w * GC + g) * (D + 2);
            const float wgt = r[D] == -__int_as_float(0x7f800000) ? 0.0f : exp2f(r[D] - M);
            A = fmaf(wgt, r[d], A);
            L = fmaf(wgt, r[D + 1], L);
        }
        const int gg = sub * GC + g;  // the head within the KV head's group
        if (splits == 1) {
            out[(static_cast<size_t>(b) * H + kvh * G + gg) * D + d] = L > 0.0f ? A * (1.0f / L) : 0.0f;
            continue;
        }
        part_acc[(slot * G + gg) * D + d] = A;
        if (d == 0) {
            part_ml[(slot * G + gg) * 2] = M;
            part_ml[(slot * G + gg) * 2 + 1] = L;
        }
    }
    if (splits == 1) return;
    // ---- the last CTA of this problem to arrive merges every split, in
    // split order: weights 2^(m_s - M), divided by the merged mass
    int *last_s = reinterpret_cast<int *>(smem + SL::kFlagOff + 8);
    asm volatile("bar.sync 1, %0;" ::"n"(kFastWarps * 32) : "memory");  // every partial store first
    if (tid == 0)
        *last_s = atomic_add_acq_rel_gpu(&counters[prob], 1u) == static_cast<unsigned>(splits - 1);
    asm volatile("bar.sync 1, %0;" ::"n"(kFastWarps * 32) : "memory");
    if (!*last_s) return;
    // (m, l) of every split and head into shared memory (the ring is free),
    // then a thread per (head, 4 channels) sums the splits' accumulators
    const float ninf = -__int_as_float(0x7f800000);
    const size_t s0 = static_cast<size_t>(p) * splits;
    float2 *ml = reinterpret_cast<float2 *>(smem);  // [GC][splits]
    for (int i = tid; i < GC * splits; i += kFastWarps * 32) {
        const int g = i / splits, sp = i % splits;
        const float *r = part_ml + ((s0 + sp) * G + sub * GC + g) * 2;
        ml[i] = make_float2(__ldcg(r), __ldcg(r + 1));
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kFastWarps * 32) : "memory");
    for (int i = tid; i < GC * D / 4; i += kFastWarps * 32) {
        const int g = i / (D / 4), d4 = i % (D / 4), gg = sub * GC + g;
        float M = ninf;
        for (int sp = 0; sp < splits; ++sp) M = fmaxf(M, ml[g * splits + sp].x);
        float L = 0.0f;
        float4 A = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 4
        for (int sp = 0; sp < splits; ++sp) {
            const float2 r = ml[g * splits + sp];
            const float w = r.x == ninf ? 0.0f : exp2f(r.x - M);
            L = fmaf(w, r.y, L);
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(
                part_acc + ((s0 + sp) * G + gg) * D + 4 * d4));
            A.x = fmaf(w, a.x, A.x);
            A.y = fmaf(w, a.y, A.y);
            A.z = fmaf(w, a.z, A.z);
            A.w = fmaf(w, a.w, A.w);
        }
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
        *reinterpret_cast<float4 *>(out + (static_cast<size_t>(b) * H + kvh * G + gg) * D +
                                    4 * d4) = make_float4(A.x * inv, A.y * inv, A.z * inv,
                                                          A.w * inv);
    }
    if (tid == 0) counters[prob] = 0u;  // ready for the next call
}

template <int DT, int D, int GC>
cudaError_t fast_t(const kvd_cache &c, const float *q, int H, int G, float scale_log2,
                   const int32_t *sel_idx, const int32_t *sel_cnt, int max_blocks,
                   float *out, float *partials, uint32_t *counters, cudaStream_t st) {
    using SL = FastLayout<DT, D, GC>;
    static_assert(SL::kTotal <= 227 * 1024, "shared memory");
    auto kern = gd_fast_kernel<DT, D, GC>;
    int occ = 0;
    cudaError_t e = prepare_kernel(reinterpret_cast<const void *>(kern), kFastThreads, SL::kTotal,
                                   &occ);
    if (e != cudaSuccess) return e;
    const int P = c.batch * c.n_kv_heads, subgroups = G / GC;
    const int P_sub = P * subgroups;
    // one wave of one CTA per SM, every split holding at least one listed block
    int splits = device_sm_count() * (occ > 0 ? occ : 1) / P_sub;
    if (splits > max_blocks) splits = max_blocks;
    if (splits < 1) splits = 1;
    float *part_acc = partials;
    float *part_ml = partials + static_cast<size_t>(P) * splits * G * D;
    kern<<<dim3(splits, P_sub), kFastThreads, SL::kTotal, st>>>(
        c, q, H, G, scale_log2, sel_idx, sel_cnt, splits, subgroups, part_acc, part_ml, out,
        counters);
    return cudaGetLastError();
}

template <int DT, int D>
cudaError_t fast_d(const kvd_cache &c, const float *q, int H, int G, float scale_log2,
                   const int32_t *sel_idx, const int32_t *sel_cnt, int max_blocks, float *out,
                   float *partials, uint32_t *counters, cudaStream_t st) {
    if (G == 1)
        return fast_t<DT, D, 1>(c, q, H, G, scale_log2, sel_idx, sel_cnt, max_blocks, out,
                                partials, counters, st);
    if (G == 2)
        return fast_t<DT, D, 2>(c, q, H, G, scale_log2, sel_idx, sel_cnt, max_blocks, out,
                                partials, counters, st);
    return fast_t<DT, D, 4>(c, q, H, G, scale_log2, sel_idx, sel_cnt, max_blocks, out,
                            partials, counters, st);
}

}  // namespace

bool gd_fast_supported(const kvd_cache &c, int G) {
    return (c.head_dim == 64 || c.head_dim == 256 || c.head_dim == 512) &&
           (G == 1 || G == 2 || G == 4 || G == 8 || G == 16);
}

// The decode with the splits merged by the last CTA of each problem (the
// output written directly); only for gd_fast_supported shapes.  counters:
// one per (sequence, KV head, subgroup), zero between calls.
cudaError_t launch_decode_gd_fast(const kvd_cache &c, const float *q, int n_heads,
                                  float scale_log2, const int32_t *sel_idx,
                                  const int32_t *sel_cnt, int max_blocks, float *out,
                                  float *partials, uint32_t *counters, cudaStream_t st) {
    const int G = n_heads / c.n_kv_heads;
    if (c.head_dim == 512)
        return c.dtype == KVD_F16 ? fast_d<KVD_F16, 512>(c, q, n_heads, G, scale_log2, sel_idx,
                                                          sel_cnt, max_blocks, out, partials,
                                                          counters, st)
                                  : fast_d<KVD_INT8, 512>(c, q, n_heads, G, scale_log2, sel_idx,
                                                           sel_cnt, max_blocks, out, partials,
                                                           counters, st);
    if (c.dtype == KVD_F16)
        return c.head_dim == 64
                   ? fast_d<KVD_F16, 64>(c, q, n_heads, G, scale_log2, sel_idx, sel_cnt,
                                         max_blocks, out, partials, counters, st)
                   : fast_d<KVD_F16, 256>(c, q, n_heads, G, scale_log2, sel_idx, sel_cnt,
                                          max_blocks, out, partials, counters, st);
    return c.head_dim == 64 ? fast_d<KVD_INT8, 64>(c, q, n_heads, G, scale_log2, sel_idx,
                                                    sel_cnt, max_blocks, out, partials,
                                                    counters, st)
                            : fast_d<KVD_INT8, 256>(c, q, n_heads, G, scale_log2, sel_idx,
                                                     sel_cnt, max_blocks, out, partials,
                                                     counters, st);
}

}  // namespace kvd
