// append_dev.cuh -- one warp appends the new tokens of one (sequence, KV head)
// that fall in one cache block, and updates that block's key envelope.
//
// "Sparse Attention -- Quest-style block-selector for long-context decode
// (#551)", S2/S3 "Fill op" and "All-KV-types composition (bug-747)": for every
// block the new tokens touch, reduce the channel-wise min and max of the new
// f16 keys; merge (min/max) into a block that already held tokens, overwrite
// a block that starts in the new range.  Bounds always come from the f16 keys
// before quantization.  "cpu-attn", Method: K and V are quantized per token
// per head (absmax int8) at append time; the q8_0 type quantizes each group
// of 32 channels with its own f16 scale instead, and q4_0 to 4-bit codes.
//
// Lane l owns channels 4l..4l+3, so every row is read as one coalesced
// 256-byte line.
#pragma once

#include "common.cuh"

namespace kvd {

__device__ __forceinline__ void load_half4(const __half *p, float (&x)[4]) {
    const uint2 w = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}

__device__ __forceinline__ void load_in4(const __half *p, float (&x)[4]) { load_half4(p, x); }

__device__ __forceinline__ void load_in4(const float *p, float (&x)[4]) {
    const float4 w = *reinterpret_cast<const float4 *>(p);
    x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
}

// Channels 4 lane .. 4 lane + 3 of stored row r of K (is_v false) or V, as
// the decode reads them: f16 as is, int8 code * row scale, q8_0 code * group
// scale, q4_0 (code - 8) * group scale, each product one f32 rounding.
template <int DT>
__device__ __forceinline__ void load_row4(const kvd_cache &c, bool is_v, size_t r, int lane,
                                          float (&x)[4]) {
    const void *base = is_v ? c.v : c.k;
    const void *scl = is_v ? c.v_scale : c.k_scale;
    if constexpr (DT == KVD_F16) {
        load_half4(static_cast<const __half *>(base) + r * kHeadDim + 4 * lane, x);
    } else if constexpr (DT == KVD_Q4_0) {
        const uint32_t b = *reinterpret_cast<const uint16_t *>(
            static_cast<const uint8_t *>(base) + r * (kHeadDim / 2) + 2 * lane);
        const float d = __half2float(static_cast<const __half *>(scl)[r * (kHeadDim / 32) +
                                                                      (lane >> 3)]);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            x[j] = static_cast<float>(static_cast<int>((b >> (4 * j)) & 15u) - 8) * d;
    } else {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(static_cast<const int8_t *>(base) +
                                                               r * kHeadDim + 4 * lane);
        const float s = DT == KVD_INT8
                            ? static_cast<const float *>(scl)[r]
                            : __half2float(static_cast<const __half *>(scl)[r * (kHeadDim / 32) +
                                                                            (lane >> 3)]);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            x[j] = static_cast<float>(static_cast<int8_t>(w >> (8 * j))) * s;
    }
}

// "SCSA: Self-Calibrating Subquadratic Attention", "2. Mechanism": a group
// of keys read only through its moments keeps its member count, key centroid
// and value mean.  Here the group is a cache block: its f16 key and value
// means over the stored rows [lo, hi) (the rows' f32 sum in token order over
// the count, rounded once), recomputed from the rows whenever the block
// grows, so they never depend on how the rows were appended.
template <int DT>
__device__ __forceinline__ void block_means_warp(const kvd_cache &c, size_t row0, int blk,
                                                 long lo, long hi, int lane) {
    float sk[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    constexpr int kBatch = 8;  // rows whose loads are in flight together
    for (long t0 = lo; t0 < hi; t0 += kBatch) {
        float xk[kBatch][4], xv[kBatch][4];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (t0 + u < hi) {
                load_row4<DT>(c, false, row0 + t0 + u, lane, xk[u]);
                load_row4<DT>(c, true, row0 + t0 + u, lane, xv[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (t0 + u < hi) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    sk[j] += xk[u][j];
                    sv[j] += xv[u][j];
                }
            }
        }
    }
    const float n = static_cast<float>(hi - lo);
    uint2 mk, mv;
    __half *k4 = reinterpret_cast<__half *>(&mk);
    __half *v4 = reinterpret_cast<__half *>(&mv);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        k4[j] = __float2half_rn(__fdiv_rn(sk[j], n));
        v4[j] = __float2half_rn(__fdiv_rn(sv[j], n));
    }
    const size_t nbmax = static_cast<size_t>(c.max_seq / kBlock);
    __half *rec = static_cast<__half *>(c.moments) +
                  ((row0 / c.max_seq) * nbmax + blk) * (2 * kHeadDim);
    *reinterpret_cast<uint2 *>(rec + 4 * lane) = mk;
    *reinterpret_cast<uint2 *>(rec + kHeadDim + 4 * lane) = mv;
}

// Tokens [max(lo, len0), min(lo + 64, len0 + n_new)) of cache block blk of
// (sequence b, KV head h), taken from k_new / v_new [B, n_new, Hkv, 128] of
// IN (f16, or f32 as "cpu-attn" Usage feeds its cache).  f32 input: the f16
// cache stores each value's nearest f16 (and bounds those); the quantized
// caches quantize the f32 values, and round the keys' envelope outward to f16
// so that the bounds still hold every key.
// MEANS: also the block's means when the cache keeps them (callers that
// never see such a cache leave that code out).
template <int DT, bool MEANS = true, typename IN = __half>
__device__ __forceinline__ void append_block_warp(const kvd_cache &c, const IN *k_new,
                                                  const IN *v_new, int n_new, int len0,
                                                  int blk, int b, int h, int lane) {
    constexpr bool kF32In = sizeof(IN) == 4;
    const long lo = static_cast<long>(blk) * kBlock;
    const long nlo = lo > len0 ? lo : len0;
    const long nhi = (lo + kBlock) < (static_cast<long>(len0) + n_new) ? (lo + kBlock)
                                                                      : (static_cast<long>(len0) + n_new);
    const bool merge = lo < len0;
    const size_t row0 = (static_cast<size_t>(b) * c.n_kv_heads + h) * c.max_seq;

    float mn[4], mx[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) { mn[j] = __int_as_float(0x7f800000); mx[j] = -mn[j]; }

    for (long t = nlo; t < nhi; ++t) {
        const size_t src = ((static_cast<size_t>(b) * n_new + (t - len0)) * c.n_kv_heads + h) *
                               kHeadDim + 4 * lane;
        float kx[4], vx[4];
        load_in4(k_new + src, kx);
        load_in4(v_new + src, vx);
        if (kF32In && DT == KVD_F16) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // the f16 cache holds the nearest f16
                kx[j] = __half2float(__float2half_rn(kx[j]));
                vx[j] = __half2float(__float2half_rn(vx[j]));
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) { mn[j] = fminf(mn[j], kx[j]); mx[j] = fmaxf(mx[j], kx[j]); }
        const size_t dst = (row0 + t) * kHeadDim + 4 * lane;
        if (DT == KVD_F16) {
            if constexpr (kF32In) {  // the rounded values (exact in f16)
                uint2 kw, vw;
                *reinterpret_cast<__half2 *>(&kw.x) = __floats2half2_rn(kx[0], kx[1]);
                *reinterpret_cast<__half2 *>(&kw.y) = __floats2half2_rn(kx[2], kx[3]);
                *reinterpret_cast<__half2 *>(&vw.x) = __floats2half2_rn(vx[0], vx[1]);
                *reinterpret_cast<__half2 *>(&vw.y) = __floats2half2_rn(vx[2], vx[3]);
                *reinterpret_cast<uint2 *>(static_cast<__half *>(c.k) + dst) = kw;
                *reinterpret_cast<uint2 *>(static_cast<__half *>(c.v) + dst) = vw;
            } else {  // verbatim copy of the f16 bits
                *reinterpret_cast<uint2 *>(static_cast<__half *>(c.k) + dst) =
                    *reinterpret_cast<const uint2 *>(k_new + src);
                *reinterpret_cast<uint2 *>(static_cast<__half *>(c.v) + dst) =
                    *reinterpret_cast<const uint2 *>(v_new + src);
            }
        } else if (DT == KVD_Q4_0) {
            __half kd, vd;
            const uint32_t kc = quantize_q4_0_warp(kx, &kd, lane);
            const uint32_t vc = quantize_q4_0_warp(vx, &vd, lane);
            const size_t dst4 = (row0 + t) * (kHeadDim / 2) + 2 * lane;  // 2 bytes per lane
            *reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(c.k) + dst4) =
                static_cast<uint16_t>(kc);
            *reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(c.v) + dst4) =
                static_cast<uint16_t>(vc);
            if ((lane & 7) == 0) {  // one lane per 32-channel group
                const size_t si = (row0 + t) * (kHeadDim / 32) + (lane >> 3);
                static_cast<__half *>(c.k_scale)[si] = kd;
                static_cast<__half *>(c.v_scale)[si] = vd;
            }
        } else if (DT == KVD_Q8_0) {
            __half kd, vd;
            const uint32_t kc = quantize_group32_warp(kx, &kd);
            const uint32_t vc = quantize_group32_warp(vx, &vd);
            *reinterpret_cast<uint32_t *>(static_cast<int8_t *>(c.k) + dst) = kc;
            *reinterpret_cast<uint32_t *>(static_cast<int8_t *>(c.v) + dst) = vc;
            if ((lane & 7) == 0) {  // one lane per 32-channel group
                const size_t si = (row0 + t) * (kHeadDim / 32) + (lane >> 3);
                static_cast<__half *>(c.k_scale)[si] = kd;
                static_cast<__half *>(c.v_scale)[si] = vd;
            }
        } else {
            float ks, vs;
            const uint32_t kc = quantize_row_warp(kx, &ks);
            const uint32_t vc = quantize_row_warp(vx, &vs);
            *reinterpret_cast<uint32_t *>(static_cast<int8_t *>(c.k) + dst) = kc;
            *reinterpret_cast<uint32_t *>(static_cast<int8_t *>(c.v) + dst) = vc;
            if (lane == 0) {
                static_cast<float *>(c.k_scale)[row0 + t] = ks;
                static_cast<float *>(c.v_scale)[row0 + t] = vs;
            }
        }
    }
    // bounds row of the block: (kmin, kmax) pairs of channels 4*lane .. 4*lane+3
    const size_t nbmax = static_cast<size_t>(c.max_seq / kBlock);
    const size_t bidx = (((static_cast<size_t>(b) * c.n_kv_heads + h) * nbmax + blk) * kHeadDim +
                         4 * lane) * 2;
    __half2 *bounds = reinterpret_cast<__half2 *>(static_cast<__half *>(c.kbounds) + bidx);
    if (merge) {
        const uint4 old = *reinterpret_cast<const uint4 *>(bounds);
        const __half2 *o2 = reinterpret_cast<const __half2 *>(&old);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(o2[j]);
            mn[j] = fminf(mn[j], f.x);
            mx[j] = fmaxf(mx[j], f.y);
        }
    }
    uint4 w;
    __half2 *w2 = reinterpret_cast<__half2 *>(&w);
    if (kF32In && DT != KVD_F16) {
        // f32 keys: the envelope rounded outward (exact for the old f16 bounds)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w2[j] = __halves2half2(__float2half_rd(mn[j]), __float2half_ru(mx[j]));
    } else {
        // every value is an f16 already, so the conversions back are exact
#pragma unroll
        for (int j = 0; j < 4; ++j) w2[j] = __floats2half2_rn(mn[j], mx[j]);
    }
    *reinterpret_cast<uint4 *>(bounds) = w;
    if (MEANS && c.moments) {
        __syncwarp();  // the group scales written by other lanes are visible
        block_means_warp<DT>(c, row0, blk, lo, nhi, lane);
    }
}

}  // namespace kvd
