// general_d_decode.cu -- split-KV decode attention for head dims other than
// 128 (any multiple of 16 up to 1024; f16 and int8 caches).
//
// "Sparse Attention -- Quest-style block-selector for long-context decode
// (#551)", "Decode": attention of each query head over the tokens of its KV
// head's listed blocks (every block for the dense arm), split over CTAs that
// each keep an online softmax (running max m, mass l, unnormalised output),
// then merged.  "cpu-attn", Method: on the int8 cache the query is quantized
// per head like a cache row (absmax / 127), q.k is the exact int32 dot of the
// codes times both scales, and V is dequantized as code * row scale.
//
// CTA (256 threads) of split s of problem p (sequence, KV head), G query
// heads at once.  The listed blocks are cut into tiles of T tokens (64, or
// fewer for large D so that K and V of a tile fit 32 KiB); every thread
// copies 16-byte pieces of the tiles two ahead into a 3-stage shared-memory
// ring (cp.async, one commit group per tile), and per tile:
//   1. q.k: a row of K is read by a group of lanes (16 bytes each), several
//      rows per warp when D is small; one score per (head, token) in shared
//      memory, pre-multiplied by softmax_scale * log2(e);
//   2. softmax: per head (a warp each) the block max, the rescale factor of
//      the running sums, and p = 2^(s - m);
//   3. P.V: thread i owns channels 4 (i % (D/4)) .. +3 of every head and the
//      tokens i / (D/4) (mod 256 / (D/4)) of the block.
// The subgroups' sums are added in a fixed order at the end, so the result
// does not depend on timing.

#include "common.cuh"
#include "internal.h"

namespace kvd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 3;  // K/V tiles in flight: the one read and two ahead


__device__ __forceinline__ void half8(const uint4 &w, float (&x)[8]) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }

// Tokens per tile: a whole block while K + V of 64 tokens fit 32 KiB, else
// the largest power-of-two share of it that does (at least 8).
__host__ __device__ constexpr int tile_tokens(int D, int elt) {
    int T = 64;
    while (T > 8 && 2 * T * D * elt > 32768) T >>= 1;
    return T;
}

__host__ __device__ constexpr int stage_bytes(int D, int elt, int T, bool scales) {
    return 2 * T * D * elt + (scales ? 2 * T * 4 : 0);
}

// DC: the head dim fixed at compile time (its loops then fold), or 0 to read
// it from the cache.
template <int DT, int G, int DC>
__global__ void __launch_bounds__(kThreads, G <= 2 ? 4 : (G <= 4 ? 3 : (G <= 8 ? 2 : 1)))
gd_decode_kernel(kvd_cache c, const float *q, int H,
                                                             float scale_log2,
                                                             const int32_t *sel_idx,
                                                             const int32_t *sel_cnt, int splits,
                                                             float *part_acc, float *part_ml) {
    constexpr int kElt = DT == KVD_F16 ? 2 : 1;
    constexpr bool kScales = DT != KVD_F16;
    extern __shared__ __align__(16) float smem[];
    const int D = DC > 0 ? DC : c.head_dim;
    const int T = tile_tokens(D, kElt), TPB = kBlock / T;
    const int SB = stage_bytes(D, kElt, T, kScales);
    float *sc = smem;               // [G][64] scores, then weights
    float *sm_m = sc + G * kBlock;  // [G] running max (log2 domain)
    float *sm_l = sm_m + G;         // [G] running mass
    float *sm_a = sm_l + G;         // [G] rescale of this tile
    float *sm_qs = sm_a + G;        // [G] query scales (int8 cache)
    float *qbuf = sm_qs + G;        // [G][D] f32 query (f16 cache) or int8 codes; at the end
                                    // the [G][D] sums of the subgroups
    unsigned char *ring = reinterpret_cast<unsigned char *>(qbuf + G * D);  // kStages x SB
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.y, s = blockIdx.x;
    const int b = p / c.n_kv_heads, h = p % c.n_kv_heads;

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
    const int i0 = static_cast<int>(static_cast<long long>(s) * n_list / splits);
    const int i1 = static_cast<int>(static_cast<long long>(s + 1) * n_list / splits);
    const int U = (i1 - i0) * TPB;  // tiles of this split

    // tile u: first token t0 and token count nt (0 past the sequence's end,
    // -1 for a caller's bad block id)
    auto tile = [&](int u, int &t0, int &nt) {
        const int j = dense ? i0 + u / TPB : list[i0 + u / TPB];
        if (j < 0 || j >= NB) {
            nt = -1;
            t0 = 0;
            return;
        }
        t0 = j * kBlock + (u % TPB) * T;
        nt = len - t0 < T ? len - t0 : T;
        if (nt < 0) nt = 0;
    };
    // tile u's K rows, V rows (and scales) into stage u % kStages; one
    // commit group per tile, empty past the end, so every thread counts alike
    auto issue = [&](int u) {
        if (u < U) {
            int t0, nt;
            tile(u, t0, nt);
            if (nt > 0) {
                unsigned char *st = ring + (u % kStages) * SB;
                const size_t rb = static_cast<size_t>(D) * kElt;
                const unsigned char *gk = static_cast<const unsigned char *>(c.k) + (row0 + t0) * rb;
                const unsigned char *gv = static_cast<const unsigned char *>(c.v) + (row0 + t0) * rb;
                const int nchunk = static_cast<int>(nt * rb / 16);
                for (int i = tid; i < nchunk; i += kThreads) {
                    cp_async16(st + 16 * i, gk + 16 * i);
                    cp_async16(st + T * rb + 16 * i, gv + 16 * i);
                }
                if (kScales && tid < nt) {
                    float *ss = reinterpret_cast<float *>(st + 2 * T * rb);
                    cp_async4(ss + tid, static_cast<const float *>(c.k_scale) + row0 + t0 + tid);
                    cp_async4(ss + T + tid, static_cast<const float *>(c.v_scale) + row0 + t0 + tid);
                }
            }
        }
        cp_async_commit();
    };
    issue(0);
    issue(1);

    const float *qp = q + (static_cast<size_t>(b) * H + static_cast<size_t>(h) * G) * D;
    if constexpr (DT == KVD_F16) {
        for (int i = tid; i < G * D; i += kThreads) qbuf[i] = qp[i];
    } else {  // a warp per head: absmax codes, as the cache rows
        int8_t *qc = reinterpret_cast<int8_t *>(qbuf);
        for (int g = warp; g < G; g += kWarps) {
            float a = 0.0f;
            for (int d = lane; d < D; d += 32) a = fmaxf(a, fabsf(qp[g * D + d]));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            const float qs = __fdiv_rn(a, 127.0f);
            for (int d = lane; d < D; d += 32) {
                int code = 0;
                if (qs != 0.0f) code = max(-127, min(127, __float2int_rn(__fdiv_rn(qp[g * D + d], qs))));
                qc[g * D + d] = static_cast<int8_t>(code);
            }
            if (lane == 0) sm_qs[g] = qs;
        }
    }
    for (int g = tid; g < G; g += kThreads) {
        sm_m[g] = -__int_as_float(0x7f800000);
        sm_l[g] = 0.0f;
    }
    __syncthreads();

    // q.k lane mapping: CPR 16-byte chunks per row, LPR lanes per row
    constexpr int kCh = DT == KVD_F16 ? 8 : 16;  // channels per 16-byte chunk
    const int CPR = D / kCh;
    int LPR = 1;
    while (LPR < CPR && LPR < 32) LPR <<= 1;
    const int RPW = 32 / LPR;  // rows per warp pass
    const int sub = lane / LPR, cl = lane % LPR;
    // a lane owns at most one chunk of each row (CPR <= 32): its query chunk
    // stays in registers (f16: 8 floats a head, int8: 16 codes a head)
    constexpr bool kQReg = DT == KVD_F16 ? G <= 8 : true;
    const bool qreg_ok = kQReg && CPR <= 32;
    float qf[kQReg && DT == KVD_F16 ? G : 1][8];
    uint4 qi[kQReg && DT != KVD_F16 ? G : 1];
    if (qreg_ok && cl < CPR) {
        if constexpr (DT == KVD_F16) {
#pragma unroll
            for (int g = 0; g < (kQReg ? G : 1); ++g)
#pragma unroll
                for (int k = 0; k < 8; ++k) qf[g][k] = qbuf[g * D + cl * 8 + k];
        } else {
#pragma unroll
            for (int g = 0; g < G; ++g)
                qi[g] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const int8_t *>(qbuf) +
                                                         g * D + cl * 16);
        }
    }
    // P.V mapping
    const int NV = D / 4, NSG = kThreads / NV;
    const int vi = tid % NV, sg = tid / NV;
    float acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[g][k] = 0.0f;

    for (int u = 0; u < U; ++u) {
        issue(u + 2);  // into the stage read two tiles ago (released by the barrier below)
        cp_async_wait_2();
        __syncthreads();
        int t0, nt;
        tile(u, t0, nt);
        if (nt < 0 && tid == 0 && u % TPB == 0) report_status(c.dev_status, KVD_ERR_INVALID);
        if (nt > 0) {
            const unsigned char *st = ring + (u % kStages) * SB;
            const size_t rb = static_cast<size_t>(D) * kElt;
            const float *sks = reinterpret_cast<const float *>(st + 2 * T * rb);
            // 1. scores
            for (int tt = warp * RPW + sub; tt - sub < nt; tt += kWarps * RPW) {
                const bool live = tt < nt;
                const uint4 *row = reinterpret_cast<const uint4 *>(st + tt * rb);
                if constexpr (DT == KVD_F16) {
                    float a[G];
#pragma unroll
                    for (int g = 0; g < G; ++g) a[g] = 0.0f;
                    if (live && qreg_ok) {
                        if (cl < CPR) {
                            float x[8];
                            half8(row[cl], x);
#pragma unroll
                            for (int g = 0; g < (kQReg ? G : 1); ++g)
#pragma unroll
                                for (int k = 0; k < 8; ++k) a[g] = fmaf(qf[g][k], x[k], a[g]);
                        }
                    } else if (live) {
                        for (int ch = cl; ch < CPR; ch += LPR) {
                            float x[8];
                            half8(row[ch], x);
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                const float4 qa = *reinterpret_cast<const float4 *>(qbuf + g * D + ch * 8);
                                const float4 qb = *reinterpret_cast<const float4 *>(qbuf + g * D + ch * 8 + 4);
                                a[g] += qa.x * x[0] + qa.y * x[1] + qa.z * x[2] + qa.w * x[3] +
                                        qb.x * x[4] + qb.y * x[5] + qb.z * x[6] + qb.w * x[7];
                            }
                        }
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float v = a[g];
                        for (int o = LPR >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                        if (live && cl == 0) sc[g * kBlock + tt] = v * scale_log2;
                    }
                } else {
                    int a[G];
#pragma unroll
                    for (int g = 0; g < G; ++g) a[g] = 0;
                    if (live && qreg_ok) {
                        if (cl < CPR) {
                            const uint4 kw = row[cl];
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                a[g] = __dp4a(static_cast<int>(kw.x), static_cast<int>(qi[g].x), a[g]);
                                a[g] = __dp4a(static_cast<int>(kw.y), static_cast<int>(qi[g].y), a[g]);
                                a[g] = __dp4a(static_cast<int>(kw.z), static_cast<int>(qi[g].z), a[g]);
                                a[g] = __dp4a(static_cast<int>(kw.w), static_cast<int>(qi[g].w), a[g]);
                            }
                        }
                    } else if (live) {
                        const int8_t *qc = reinterpret_cast<const int8_t *>(qbuf);
                        for (int ch = cl; ch < CPR; ch += LPR) {
                            const uint4 kw = row[ch];
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                const uint4 qw = *reinterpret_cast<const uint4 *>(qc + g * D + ch * 16);
                                a[g] = __dp4a(static_cast<int>(kw.x), static_cast<int>(qw.x), a[g]);
                                a[g] = __dp4a(static_cast<int>(kw.y), static_cast<int>(qw.y), a[g]);
                                a[g] = __dp4a(static_cast<int>(kw.z), static_cast<int>(qw.z), a[g]);
                                a[g] = __dp4a(static_cast<int>(kw.w), static_cast<int>(qw.w), a[g]);
                            }
                        }
                    }
                    const float ks = live ? sks[tt] : 0.0f;
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        int v = a[g];
                        for (int o = LPR >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                        if (live && cl == 0)
                            sc[g * kBlock + tt] = static_cast<float>(v) * (sm_qs[g] * ks) * scale_log2;
                    }
                }
            }
            __syncthreads();
            // 2. online softmax, a warp per head
            for (int g = warp; g < G; g += kWarps) {
                const float x0 = lane < nt ? sc[g * kBlock + lane] : -__int_as_float(0x7f800000);
                const float x1 = lane + 32 < nt ? sc[g * kBlock + lane + 32] : -__int_as_float(0x7f800000);
                float mt = fmaxf(x0, x1);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                const float m_old = sm_m[g];
                const float m_new = fmaxf(m_old, mt);
                const float p0 = exp2f(x0 - m_new), p1 = exp2f(x1 - m_new);
                sc[g * kBlock + lane] = p0;
                sc[g * kBlock + lane + 32] = p1;
                float sum = p0 + p1;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                if (lane == 0) {
                    const float alpha = exp2f(m_old - m_new);
                    sm_a[g] = alpha;
                    sm_l[g] = sm_l[g] * alpha + sum;
                    sm_m[g] = m_new;
                }
            }
            __syncthreads();
            // 3. P.V
            if (sg < NSG) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float al = sm_a[g];
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc[g][k] *= al;
                }
                const unsigned char *sv = st + T * rb;
                for (int tt = sg; tt < nt; tt += NSG) {
                    float x[4];
                    if constexpr (DT == KVD_F16) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(sv + tt * rb + 8 * vi);
                        const float2 u0 = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
                        const float2 u1 = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
                        x[0] = u0.x; x[1] = u0.y; x[2] = u1.x; x[3] = u1.y;
                    } else {
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(sv + tt * rb + 4 * vi);
                        const float vs = sks[T + tt];
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            x[k] = static_cast<float>(static_cast<int8_t>(w >> (8 * k))) * vs;
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float pw = sc[g * kBlock + tt];
#pragma unroll
                        for (int k = 0; k < 4; ++k) acc[g][k] = fmaf(pw, x[k], acc[g][k]);
                    }
                }
            }
        }
        __syncthreads();
    }
    // the subgroups' sums, added in subgroup order (the query buffer and the
    // ring are free now): all at once when [NSG][G][D] fits there, else one
    // subgroup after another
    float *red = qbuf;
    const size_t slot = static_cast<size_t>(p) * splits + s;
    if (static_cast<size_t>(NSG) * G * D * sizeof(float) <=
        static_cast<size_t>(G) * D * sizeof(float) + static_cast<size_t>(kStages) * SB) {
        if (sg < NSG) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int k = 0; k < 4; ++k) red[(sg * G + g) * D + 4 * vi + k] = acc[g][k];
        }
        __syncthreads();
        for (int i = tid; i < G * D; i += kThreads) {
            float a = red[i];
            for (int r = 1; r < NSG; ++r) a += red[r * G * D + i];
            part_acc[slot * G * D + i] = a;
        }
        for (int g = tid; g < G; g += kThreads) {
            part_ml[(slot * G + g) * 2] = sm_m[g];
            part_ml[(slot * G + g) * 2 + 1] = sm_l[g];
        }
        return;
    }
    for (int r = 0; r < NSG; ++r) {
        if (sg == r) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float *o = red + g * D + 4 * vi + k;
                    *o = r == 0 ? acc[g][k] : *o + acc[g][k];
                }
        }
        __syncthreads();
    }
    for (int i = tid; i < G * D; i += kThreads) part_acc[slot * G * D + i] = red[i];
    for (int g = tid; g < G; g += kThreads) {
        part_ml[(slot * G + g) * 2] = sm_m[g];
        part_ml[(slot * G + g) * 2 + 1] = sm_l[g];
    }
}

// One CTA per (sequence, query head): the splits' partials weighted by
// 2^(m_s - M) (M their max), divided by the merged mass; no token at all
// gives zeros.
__global__ void __launch_bounds__(128) gd_merge_kernel(const float *part_acc,
                                                       const float *part_ml, int Hkv, int G,
                                                       int D, int splits, float *out) {
    extern __shared__ float wsh[];  // [splits] weights, then [4] reduction
    __shared__ float red[4];
    const int bh = blockIdx.x, tid = threadIdx.x;
    const int H = Hkv * G;
    const int b = bh / H, hq = bh % H, p = b * Hkv + hq / G, g = hq % G;
    auto ml = [&](int s, int k) { return part_ml[((static_cast<size_t>(p) * splits + s) * G + g) * 2 + k]; };
    float m = -__int_as_float(0x7f800000);
    for (int s = tid; s < splits; s += blockDim.x) m = fmaxf(m, ml(s, 0));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    float l = 0.0f;
    for (int s = tid; s < splits; s += blockDim.x) {
        const float ms = ml(s, 0);
        const float w = ms == -__int_as_float(0x7f800000) ? 0.0f : exp2f(ms - M);
        wsh[s] = w;
        l += w * ml(s, 1);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if ((tid & 31) == 0) red[tid >> 5] = l;
    __syncthreads();
    const float L = (red[0] + red[1]) + (red[2] + red[3]);
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    for (int d = tid; d < D; d += blockDim.x) {
        float o = 0.0f;
        for (int s = 0; s < splits; ++s) {
            const float w = wsh[s];
            if (w != 0.0f) o = fmaf(w, part_acc[((static_cast<size_t>(p) * splits + s) * G + g) * D + d], o);
        }
        out[static_cast<size_t>(bh) * D + d] = o * inv;
    }
}

template <int DT, int G, int DC = 0>
cudaError_t decode_g(const kvd_cache &c, const float *q, int H, float scale_log2,
                     const int32_t *sel_idx, const int32_t *sel_cnt, int max_blocks,
                     float *partials, int *splits_out, cudaStream_t st) {
    constexpr int kElt = DT == KVD_F16 ? 2 : 1;
    const int T = tile_tokens(c.head_dim, kElt);
    const size_t smem = (static_cast<size_t>(G) * (kBlock + 4) + static_cast<size_t>(G) * c.head_dim) *
                            sizeof(float) +
                        static_cast<size_t>(kStages) * stage_bytes(c.head_dim, kElt, T, DT != KVD_F16);
    auto kern = gd_decode_kernel<DT, G, DC>;
    // one wave: the CTAs that fit on every SM at once, shared by the problems
    int occ = 0;
    cudaError_t e = prepare_kernel(reinterpret_cast<const void *>(kern), kThreads, smem, &occ);
    if (e != cudaSuccess) return e;
    const int P = c.batch * c.n_kv_heads;
    const int splits = gd_splits(P, max_blocks, device_sm_count(), occ);
    float *part_acc = partials;
    float *part_ml = partials + static_cast<size_t>(P) * splits * G * c.head_dim;
    kern<<<dim3(splits, P), kThreads, smem, st>>>(c, q, H, scale_log2, sel_idx, sel_cnt, splits,
                                                 part_acc, part_ml);
    *splits_out = splits;
    return cudaGetLastError();
}

template <int DT>
cudaError_t decode_dt(const kvd_cache &c, const float *q, int H, float scale_log2,
                      const int32_t *sel_idx, const int32_t *sel_cnt, int max_blocks,
                      float *partials, int *splits, cudaStream_t st) {
    // common head dims (64, 96, 256) of GQA groups of 4 and 8, with folded loops
    const int G = H / c.n_kv_heads;
    if (c.head_dim == 64 && G == 4) return decode_g<DT, 4, 64>(c, q, H, scale_log2, sel_idx, sel_cnt, max_blocks, partials, splits, st);
    if (c.head_dim == 64 && G == 8) return decode_g<DT, 8, 64>(c, q, H, scale_log2, sel_idx, sel_cnt, max_blocks, partials, splits, st);
    if (c.head_dim == 96 && G == 4) return decode_g<DT, 4, 96>(c, q, H, scale_log2, sel_idx, sel_cnt, max_blocks, partials, splits, st);
    if (c.head_dim == 96 && G == 8) return decode_g<DT, 8, 96>(c, q, H, scale_log2, sel_idx, sel_cnt, max_blocks, partials, splits, st);
    if (c.head_dim == 256 && G == 4) return decode_g<DT, 4, 256>(c, q, H, scale_log2, sel_idx, sel_cnt, max_blocks, partials, splits, st);
    if (c.head_dim == 256 && G == 8) return decode_g<DT, 8, 256>(c, q, H, scale_log2, sel_idx, sel_cnt, max_blocks, partials, splits, st);
    switch (G) {
        case 1: return decode_g<DT, 1>(c, q, H, scale_log2, sel_idx, sel_cnt, max_blocks, partials, splits, st);
        case 2: return decode_g<DT, 2>(c, q, H, scale_log2, sel_idx, sel_cnt, max_blocks, partials, splits, st);
        case 4: return decode_g<DT, 4>(c, q, H, scale_log2, sel_idx, sel_cnt, max_blocks, partials, splits, st);
        case 8: return decode_g<DT, 8>(c, q, H, scale_log2, sel_idx, sel_cnt, max_blocks, partials, splits, st);
        default: return decode_g<DT, 16>(c, q, H, scale_log2, sel_idx, sel_cnt, max_blocks, partials, splits, st);
    }
}

}  // namespace

// Splits per problem: the problems share one wave of the decode kernel,
// per_sm (at most 4) CTAs on every SM -- several CTAs per SM hide the tile
// loop's barriers -- and a split has at least one listed block.  Rounded
// down, so no second wave starts with a few CTAs; per_sm = 0 gives the
// upper bound the workspace is sized for.
int gd_splits(int problems, int max_blocks, int sm_count, int per_sm) {
    const int slots = (per_sm < 1 || per_sm > 4 ? 4 : per_sm) * sm_count;
    int s = per_sm < 1 ? (slots + problems - 1) / problems : slots / problems;
    if (s > max_blocks) s = max_blocks;
    return s < 1 ? 1 : s;
}

size_t gd_partials_bytes(int problems, int G, int D, int splits) {
    return static_cast<size_t>(problems) * splits * G * (static_cast<size_t>(D) + 2) * sizeof(float);
}

cudaError_t launch_decode_gd(const kvd_cache &c, const float *q, int n_heads, float scale,
                             const int32_t *sel_idx, const int32_t *sel_cnt, int max_blocks,
                             float *out, float *partials, uint32_t *counters, cudaStream_t st) {
    const int P = c.batch * c.n_kv_heads, G = n_heads / c.n_kv_heads, D = c.head_dim;
    const float scale_log2 = scale * kLog2e;
    if (gd_fast_supported(c, G))  // its splits merge inside the launch
        return launch_decode_gd_fast(c, q, n_heads, scale_log2, sel_idx, sel_cnt, max_blocks,
                                     out, partials, counters, st);
    int splits = 1;
    cudaError_t e = c.dtype == KVD_F16
                        ? decode_dt<KVD_F16>(c, q, n_heads, scale_log2, sel_idx, sel_cnt,
                                             max_blocks, partials, &splits, st)
                        : decode_dt<KVD_INT8>(c, q, n_heads, scale_log2, sel_idx, sel_cnt,
                                              max_blocks, partials, &splits, st);
    if (e != cudaSuccess) return e;
    float *part_acc = partials;
    float *part_ml = partials + static_cast<size_t>(P) * splits * G * D;
    gd_merge_kernel<<<c.batch * n_heads, 128, splits * sizeof(float), st>>>(
        part_acc, part_ml, c.n_kv_heads, G, D, splits, out);
    return cudaGetLastError();
}

}  // namespace kvd
