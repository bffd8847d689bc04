/*
 * oracle.c -- plain, slow, fp64 CPU oracle for Quest-style sparse decode
 * attention over an f16, absmax-int8, q8_0 or q4_0 KV cache, with the
 * sparse-V (eps mode) and moment-tail variants.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library; the two meet only at the seeded input tensors.
 *
 * Sources (the pages this restates, by title and section):
 *  [QUEST]  "Sparse Attention -- Quest-style block-selector for long-context
 *           decode (#551)", sections "Method: Quest-style min/max block
 *           bounds", "S2/S3 engineering design" (fill op, selector op,
 *           FA-VEC block-skip), "Gate ladder", and "All-KV-types composition
 *           (bug-747)" (pre-quant envelope, merge-vs-overwrite fill).
 *  [CPUATT] "cpu-attn" (Hugging Face kernels card), sections "Method",
 *           "Usage", "Correctness", "Requirements and limits".
 *  [SCSA]   "SCSA: Self-Calibrating Subquadratic Attention", section
 *           "2. Mechanism" (sink / recent suffix always attended exactly;
 *           the moment tail of the groups not read exactly).
 *  The sparse-V (eps mode) functions follow [QUEST] "Adaptive tau (the eps
 *  mode)" and "Compose" item 3.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes with its reason):
 *  R1  int8 code = round-half-to-even of the IEEE f32 quotient x/s, clamped
 *      to [-127, 127]; s = fl32(absmax/127) stored as f32.
 *  R2  a row whose f32 scale is 0 stores scale 0 and all-zero codes.
 *  R3  the top-K budget counts non-forced blocks only; the sink and recent
 *      blocks are added on top; ties in the bound go to the lower index.
 *  R4  sink blocks are those meeting [0, sink_tokens); recent blocks are
 *      those meeting [L - recent_tokens, L).
 *  R5  the bound uses the raw f32 query (no softmax scale: a positive factor
 *      does not change the ranking) on both cache types.
 *  R6  attention over an empty token set returns the zero vector.
 *  R7  sparse-V (eps mode): the mean weight a position is compared with is
 *      taken over its 16-token chunk of the attended positions.
 *  R8  q8_0 (named, not defined, by the pages): per 32-channel group an f16
 *      scale fl16(fl32(amax/127)) and codes round-half-even(fl32(x/d))
 *      clamped to +-127; the query is quantized per row as for int8, and the
 *      logit sums the exact per-group dots times the group scales.
 *  R9  q4_0 (named, not defined, by the pages): per 32-channel group the
 *      f16 scale fl16(fl32(m/-8)) of the largest-magnitude value m, codes
 *      clamp(round-half-even(fl32(x/d)) + 8, 0, 15), two per byte.
 *  R10 moment tail on Quest blocks: every block of [0, L) that the
 *      selection leaves out contributes m_j exp(scale q . c_K) at c_V, with
 *      c_K, c_V the means of the block's stored (dequantized) keys and
 *      values rounded to f16 and q the unquantized f32 query.
 *  R11 f32 append input: the f16 cache stores the nearest f16 of each
 *      value; the quantized caches quantize the f32 values and round the
 *      f32 keys' block envelope outward to f16.
 *
 * Every floating-point step runs in IEEE binary64 unless a step of the
 * method fixes f32 (the quantizer's scale and quotient, R1).  Build with
 * -ffp-contract=off so no fused multiply-add changes a rounding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F16 0
#define ORC_INT8 1
#define ORC_Q8_0 2
#define ORC_Q4_0 3
#define ORC_QGROUP 32

/* ------------------------------------------------------------------ */
/* binary16 -> binary64, exact.  Written from the IEEE 754 binary16     */
/* layout: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.    */
/* ------------------------------------------------------------------ */
double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);             /* subnormal: f * 2^-24 */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(f + 1024), e - 25); /* (1024+f) * 2^(e-15-10) */
    return sign ? -mag : mag;
}

/* ------------------------------------------------------------------ */
/* binary64 -> binary16, rounded to nearest, ties to even, from the      */
/* same layout: a normal half holds (1024 + f) * 2^(e-25) for e = 1..30, */
/* a subnormal f * 2^-24; magnitudes from 65520 up round to infinity.   */
/* Scaling by a power of two is exact in binary64, so rounding the       */
/* scaled value to an integer rounds the value itself.                  */
/* ------------------------------------------------------------------ */
uint16_t orc_double_to_half(double x)
{
    uint16_t sign = (uint16_t)(signbit(x) ? 0x8000 : 0);
    double a = fabs(x);
    if (isnan(x)) return 0x7e00;
    if (a == 0.0) return sign;
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    int k;
    (void)frexp(a, &k);              /* a = m * 2^k, m in [0.5, 1): a in [2^(k-1), 2^k) */
    int e = k - 1;                   /* a in [2^e, 2^(e+1)) */
    if (e < -14) {                   /* subnormal range: units of 2^-24 */
        double n = nearbyint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)n);  /* n == 1024 is the smallest normal */
    }
    double n = nearbyint(ldexp(a, 10 - e));      /* in [1024, 2048] */
    if (n == 2048.0) {
        n = 1024.0;
        ++e;
    }
    if (e > 15) return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(n - 1024.0));
}

/* ------------------------------------------------------------------ */
/* Absmax int8 quantization of one row  [CPUATT Method; R1, R2].        */
/* The scale is the f32 value nearest absmax/127.  Each code is the     */
/* f32 quotient x/s rounded half-to-even and clamped to +-127.          */
/* A binary64 quotient of two f32 values rounded once to f32 equals the */
/* correctly rounded f32 quotient (53 >= 2*24+2), so this reproduces    */
/* IEEE f32 division exactly.                                            */
/* ------------------------------------------------------------------ */
void orc_quantize_row(const float *x, int n, int8_t *code, float *scale)
{
    double amax = 0.0;
    for (int i = 0; i < n; ++i) {
        double a = fabs((double)x[i]);
        if (a > amax) amax = a;
    }
    float s = (float)(amax / 127.0);
    *scale = s;
    for (int i = 0; i < n; ++i) {
        if (s == 0.0f) { code[i] = 0; continue; }
        float quot = (float)((double)x[i] / (double)s);
        double r = nearbyint((double)quot);  /* default mode: ties to even */
        if (r > 127.0) r = 127.0;
        if (r < -127.0) r = -127.0;
        code[i] = (int8_t)r;
    }
}

/* ------------------------------------------------------------------ */
/* q8_0: absmax int8 per group of 32 channels with a binary16 scale     */
/* (the llama.cpp cache type of [QUEST] "All-KV-types composition" and  */
/* "The decode win lives on quantized KV"; R8):                          */
/*   d_g = fl16(fl32(amax_g / 127)),                                     */
/*   code = round-half-even(fl32(x / d_g)) clamped to +-127 (0 if d_g=0) */
/* d: n / 32 binary16 bits.                                               */
/* ------------------------------------------------------------------ */
void orc_quantize_group32(const float *x, int n, int8_t *code, uint16_t *d)
{
    for (int g = 0; g < n / ORC_QGROUP; ++g) {
        const float *xg = x + g * ORC_QGROUP;
        double amax = 0.0;
        for (int i = 0; i < ORC_QGROUP; ++i) {
            double a = fabs((double)xg[i]);
            if (a > amax) amax = a;
        }
        float s32 = (float)(amax / 127.0);
        d[g] = orc_double_to_half((double)s32);
        double dg = orc_half_to_double(d[g]);
        for (int i = 0; i < ORC_QGROUP; ++i) {
            if (dg == 0.0) { code[g * ORC_QGROUP + i] = 0; continue; }
            float qg = (float)((double)xg[i] / dg);
            double rq = nearbyint((double)qg);  /* ties to even */
            rq = rq > 127.0 ? 127.0 : (rq < -127.0 ? -127.0 : rq);
            code[g * ORC_QGROUP + i] = (int8_t)rq;
        }
    }
}

/* ------------------------------------------------------------------ */
/* q4_0: 4-bit codes per group of 32 channels with a binary16 scale     */
/* (the llama.cpp cache type named by [QUEST] "All-KV-types            */
/* composition"; R9).  m is the group's value of largest magnitude (the */
/* first one in channel order); d = fl16(fl32(m / -8)), so m maps to    */
/* -8; code = clamp(round-half-even(fl32(x / d)) + 8, 0, 15) (all 8 if  */
/* d = 0); the value is d * (code - 8).  Byte i of a group holds         */
/* channels 2i (low nibble) and 2i+1 (high nibble).                      */
/* packed: n / 2 bytes; d: n / 32 binary16 bits.                          */
/* ------------------------------------------------------------------ */
void orc_quantize_q4_0(const float *x, int n, uint8_t *packed, uint16_t *d)
{
    for (int g = 0; g < n / ORC_QGROUP; ++g) {
        const float *xg = x + g * ORC_QGROUP;
        double amax = 0.0, m = 0.0;
        for (int i = 0; i < ORC_QGROUP; ++i) {
            double mag = fabs((double)xg[i]);
            if (mag > amax) {
                amax = mag;
                m = (double)xg[i];
            }
        }
        float s32 = (float)(m / -8.0);
        d[g] = orc_double_to_half((double)s32);
        double dq = orc_half_to_double(d[g]);
        int c4[ORC_QGROUP];
        for (int i = 0; i < ORC_QGROUP; ++i) {
            if (dq == 0.0) { c4[i] = 8; continue; }
            float qt = (float)((double)xg[i] / dq);
            double r4 = nearbyint((double)qt) + 8.0;   /* ties to even */
            c4[i] = (int)(r4 < 0.0 ? 0.0 : (r4 > 15.0 ? 15.0 : r4));
        }
        for (int i = 0; i < ORC_QGROUP / 2; ++i)
            packed[g * (ORC_QGROUP / 2) + i] = (uint8_t)(c4[2 * i] | (c4[2 * i + 1] << 4));
    }
}

/* The 4-bit code of channel c of a packed row. */
static int q4_code(const uint8_t *row, int c)
{
    return (row[c / 2] >> (4 * (c & 1))) & 15;
}

/* ------------------------------------------------------------------ */
/* Cache description (layouts of the head-major cache).                */
/*   K, V     [B, Hkv, max_seq, D]   f16 bits or int8 codes            */
/*   ks, vs   [B, Hkv, max_seq]      f32 (int8 cache only)             */
/*   kd, vd   [B, Hkv, max_seq, D/32] f16 bits (q8_0, q4_0 caches)      */
/*   K, V of a q4_0 cache: [B, Hkv, max_seq, D/2] packed 4-bit codes     */
/*   kmin/kmax[B, Hkv, max_seq/blk, D] f16 bits                        */
/* ------------------------------------------------------------------ */
typedef struct {
    int dtype, B, Hkv, D, max_seq, blk, len;
    void *K, *V;
    float *ks, *vs;
    uint16_t *kmin, *kmax;
    uint16_t *kd, *vd;
} orc_cache;

static size_t row_index(const orc_cache *c, int b, int h, long t)
{
    return ((size_t)b * c->Hkv + h) * (size_t)c->max_seq + (size_t)t;
}

static size_t bound_index(const orc_cache *c, int b, int h, int blk_id)
{
    size_t nbmax = (size_t)(c->max_seq / c->blk);
    return (((size_t)b * c->Hkv + h) * nbmax + (size_t)blk_id) * (size_t)c->D;
}

/* ------------------------------------------------------------------ */
/* Append n_new tokens  [QUEST S2/S3 "Fill op", All-KV-types            */
/* composition; CPUATT Method "quantize per token per head at append"]. */
/* k_new, v_new: [B, n_new, Hkv, D] f16 bits.                           */
/* Cache rows: f16 stored verbatim, or int8 codes + f32 scale per row.  */
/* Bounds: per (seq, KV head, block) channel-wise min and max of the     */
/* f16 keys (the pre-quantization envelope).  A block that already       */
/* holds tokens is merged (min with old min, max with old max); a block  */
/* that starts inside the new range is overwritten.                      */
/* Returns 0, or -1 if the append would pass max_seq.                    */
/* ------------------------------------------------------------------ */
int orc_append(orc_cache *c, const uint16_t *k_new, const uint16_t *v_new, int n_new)
{
    if (n_new < 0 || (long)c->len + n_new > c->max_seq) return -1;
    const int D = c->D;
    float *row = (float *)malloc(sizeof(float) * (size_t)D);
    for (int b = 0; b < c->B; ++b)
        for (int h = 0; h < c->Hkv; ++h) {
            /* rows */
            for (int i = 0; i < n_new; ++i) {
                long t = (long)c->len + i;
                const uint16_t *kin = k_new + (((size_t)b * n_new + i) * c->Hkv + h) * D;
                const uint16_t *vin = v_new + (((size_t)b * n_new + i) * c->Hkv + h) * D;
                size_t r = row_index(c, b, h, t);
                if (c->dtype == ORC_F16) {
                    memcpy((uint16_t *)c->K + r * D, kin, sizeof(uint16_t) * D);
                    memcpy((uint16_t *)c->V + r * D, vin, sizeof(uint16_t) * D);
                } else if (c->dtype == ORC_Q4_0) {
                    const int ng = D / ORC_QGROUP;
                    for (int d = 0; d < D; ++d) row[d] = (float)orc_half_to_double(kin[d]);
                    orc_quantize_q4_0(row, D, (uint8_t *)c->K + r * (D / 2), c->kd + r * ng);
                    for (int d = 0; d < D; ++d) row[d] = (float)orc_half_to_double(vin[d]);
                    orc_quantize_q4_0(row, D, (uint8_t *)c->V + r * (D / 2), c->vd + r * ng);
                } else if (c->dtype == ORC_Q8_0) {
                    const int ng = D / ORC_QGROUP;
                    for (int d = 0; d < D; ++d) row[d] = (float)orc_half_to_double(kin[d]);
                    orc_quantize_group32(row, D, (int8_t *)c->K + r * D, c->kd + r * ng);
                    for (int d = 0; d < D; ++d) row[d] = (float)orc_half_to_double(vin[d]);
                    orc_quantize_group32(row, D, (int8_t *)c->V + r * D, c->vd + r * ng);
                } else {
                    for (int d = 0; d < D; ++d) row[d] = (float)orc_half_to_double(kin[d]);
                    orc_quantize_row(row, D, (int8_t *)c->K + r * D, &c->ks[r]);
                    for (int d = 0; d < D; ++d) row[d] = (float)orc_half_to_double(vin[d]);
                    orc_quantize_row(row, D, (int8_t *)c->V + r * D, &c->vs[r]);
                }
            }
            /* bounds of every block meeting [len, len+n_new) */
            if (n_new == 0) continue;
            int b0 = c->len / c->blk;
            int b1 = (c->len + n_new - 1) / c->blk;
            for (int q = b0; q <= b1; ++q) {
                long lo = (long)q * c->blk, hi = lo + c->blk;
                long nlo = lo > c->len ? lo : c->len;
                long nhi = hi < (long)c->len + n_new ? hi : (long)c->len + n_new;
                int merge = lo < c->len;         /* block held tokens already */
                uint16_t *mn = c->kmin + bound_index(c, b, h, q);
                uint16_t *mx = c->kmax + bound_index(c, b, h, q);
                for (int d = 0; d < D; ++d) {
                    uint16_t bmin = 0, bmax = 0;
                    double vmin = INFINITY, vmax = -INFINITY;
                    if (merge) {
                        bmin = mn[d]; vmin = orc_half_to_double(bmin);
                        bmax = mx[d]; vmax = orc_half_to_double(bmax);
                    }
                    for (long t = nlo; t < nhi; ++t) {
                        int i = (int)(t - c->len);
                        uint16_t kb = k_new[(((size_t)b * n_new + i) * c->Hkv + h) * D + d];
                        double kv = orc_half_to_double(kb);
                        if (kv < vmin) { vmin = kv; bmin = kb; }
                        if (kv > vmax) { vmax = kv; bmax = kb; }
                    }
                    mn[d] = bmin;
                    mx[d] = bmax;
                }
            }
        }
    free(row);
    c->len += n_new;
    return 0;
}

/* ------------------------------------------------------------------ */
/* Binary16 rounding toward -inf (dir < 0) or +inf (dir > 0): the f16   */
/* nearest below or above x, x itself when it is an f16.  From the      */
/* nearest f16 (orc_double_to_half) stepped once to its neighbour when  */
/* it lies on the wrong side of x.                                       */
/* ------------------------------------------------------------------ */
uint16_t orc_double_to_half_dir(double x, int dir)
{
    uint16_t h = orc_double_to_half(x);
    double y = orc_half_to_double(h);
    int toward_pos;
    if (dir < 0 && y > x) toward_pos = 0;
    else if (dir > 0 && y < x) toward_pos = 1;
    else return h;
    int neg = (h & 0x8000) != 0;
    if ((h & 0x7fff) == 0)                       /* +-0: the smallest subnormal */
        return toward_pos ? 0x0001 : 0x8001;
    if (neg == toward_pos) return (uint16_t)(h - 1);  /* magnitude shrinks */
    return (uint16_t)(h + 1);                         /* magnitude grows */
}

/* ------------------------------------------------------------------ */
/* Append with f32 input  [CPUATT Usage: the cache takes f32 K/V per    */
/* token; QUEST All-KV-types composition: bounds from the keys before   */
/* quantization].  Reading R11:                                          */
/*  - the f16 cache stores each value's nearest f16, so it is exactly   */
/*    orc_append of those f16 values;                                    */
/*  - the quantized caches quantize the f32 values themselves, and a    */
/*    block's bounds are the f32 keys' envelope rounded outward to f16   */
/*    (kmin toward -inf, kmax toward +inf), merged as usual, so they    */
/*    still bound every key.                                             */
/* k_new, v_new: [B, n_new, Hkv, D] f32.  Returns 0, or -1 past max_seq. */
/* ------------------------------------------------------------------ */
int orc_append_f32(orc_cache *c, const float *k_new, const float *v_new, int n_new)
{
    if (n_new < 0 || (long)c->len + n_new > c->max_seq) return -1;
    const int D = c->D;
    const size_t n_all = (size_t)c->B * (size_t)n_new * c->Hkv * D;
    if (c->dtype == ORC_F16) {
        uint16_t *kh = (uint16_t *)malloc(sizeof(uint16_t) * (n_all ? n_all : 1));
        uint16_t *vh = (uint16_t *)malloc(sizeof(uint16_t) * (n_all ? n_all : 1));
        for (size_t i = 0; i < n_all; ++i) {
            kh[i] = orc_double_to_half((double)k_new[i]);
            vh[i] = orc_double_to_half((double)v_new[i]);
        }
        int rc = orc_append(c, kh, vh, n_new);
        free(vh);
        free(kh);
        return rc;
    }
    const int ng = D / ORC_QGROUP;
    for (int b = 0; b < c->B; ++b)
        for (int h = 0; h < c->Hkv; ++h) {
            for (int i = 0; i < n_new; ++i) {
                const float *kx = k_new + (((size_t)b * n_new + i) * c->Hkv + h) * D;
                const float *vx = v_new + (((size_t)b * n_new + i) * c->Hkv + h) * D;
                size_t r = row_index(c, b, h, (long)c->len + i);
                if (c->dtype == ORC_Q4_0) {
                    orc_quantize_q4_0(kx, D, (uint8_t *)c->K + r * (D / 2), c->kd + r * ng);
                    orc_quantize_q4_0(vx, D, (uint8_t *)c->V + r * (D / 2), c->vd + r * ng);
                } else if (c->dtype == ORC_Q8_0) {
                    orc_quantize_group32(kx, D, (int8_t *)c->K + r * D, c->kd + r * ng);
                    orc_quantize_group32(vx, D, (int8_t *)c->V + r * D, c->vd + r * ng);
                } else {
                    orc_quantize_row(kx, D, (int8_t *)c->K + r * D, &c->ks[r]);
                    orc_quantize_row(vx, D, (int8_t *)c->V + r * D, &c->vs[r]);
                }
            }
            if (n_new == 0) continue;
            int q0 = c->len / c->blk, q1 = (c->len + n_new - 1) / c->blk;
            for (int q = q0; q <= q1; ++q) {
                long first = (long)q * c->blk;
                long t0 = first > c->len ? first : c->len;
                long t1 = first + c->blk < (long)c->len + n_new ? first + c->blk
                                                                 : (long)c->len + n_new;
                int held = first < c->len;       /* block held tokens already */
                uint16_t *lo16 = c->kmin + bound_index(c, b, h, q);
                uint16_t *hi16 = c->kmax + bound_index(c, b, h, q);
                for (int d = 0; d < D; ++d) {
                    double xmin = INFINITY, xmax = -INFINITY;
                    for (long t = t0; t < t1; ++t) {
                        double x = (double)k_new[(((size_t)b * n_new + (t - c->len)) * c->Hkv
                                                  + h) * D + d];
                        if (x < xmin) xmin = x;
                        if (x > xmax) xmax = x;
                    }
                    uint16_t dn = orc_double_to_half_dir(xmin, -1);
                    uint16_t up = orc_double_to_half_dir(xmax, +1);
                    if (held) {
                        if (orc_half_to_double(lo16[d]) < orc_half_to_double(dn)) dn = lo16[d];
                        if (orc_half_to_double(hi16[d]) > orc_half_to_double(up)) up = hi16[d];
                    }
                    lo16[d] = dn;
                    hi16[d] = up;
                }
            }
        }
    c->len += n_new;
    return 0;
}

/* ------------------------------------------------------------------ */
/* Block upper bounds  [QUEST Method "Per-query upper bound"; S2        */
/* selector op "GQA -> max UB over the query group"].                    */
/*   UB_h(j) = sum_d max(q_h[d]*kmin_j[d], q_h[d]*kmax_j[d])             */
/*   UB(j)   = max over the G query heads h of the group of UB_h(j)      */
/* q: [G, D] f32 (R5).  kmin, kmax: [NB, D] f16 bits of one KV head.     */
/* ub_heads ([G, NB]) and mag ([NB]) may be NULL.  mag(j) is             */
/* max_h sum_d |max(q_h[d]*kmin_j[d], q_h[d]*kmax_j[d])|, the size of    */
/* the terms, which sets the scale of rounding in the sum.               */
/* ------------------------------------------------------------------ */
void orc_block_scores(int G, int D, int NB, const float *q,
                      const uint16_t *kmin, const uint16_t *kmax,
                      double *ub_heads, double *ub, double *mag)
{
    for (int j = 0; j < NB; ++j) {
        double best = -INFINITY, best_mag = 0.0;
        for (int h = 0; h < G; ++h) {
            double s = 0.0, m = 0.0;
            for (int d = 0; d < D; ++d) {
                double qd = (double)q[(size_t)h * D + d];
                double a = qd * orc_half_to_double(kmin[(size_t)j * D + d]);
                double bb = qd * orc_half_to_double(kmax[(size_t)j * D + d]);
                double t = a > bb ? a : bb;
                s += t;
                m += fabs(t);
            }
            if (ub_heads) ub_heads[(size_t)h * NB + j] = s;
            if (s > best) best = s;
            if (m > best_mag) best_mag = m;
        }
        ub[j] = best;
        if (mag) mag[j] = best_mag;
    }
}

/* Forced blocks  [QUEST Method "Top-K block selection ... PLUS the     */
/* recent window + attention-sink block"; SCSA Mechanism; R4].          */
/* Sink blocks: [0, sink_end).  Recent blocks: [recent_begin, NB).      */
void orc_forced_range(int L, int blk, int sink_tokens, int recent_tokens,
                      int *sink_end, int *recent_begin)
{
    int NB = (L + blk - 1) / blk;
    int se = (sink_tokens + blk - 1) / blk;
    if (se > NB) se = NB;
    int rb = NB;
    if (recent_tokens > 0) {
        long start = (long)L - recent_tokens;
        if (start < 0) start = 0;
        rb = (int)(start / blk);
    }
    *sink_end = se;
    *recent_begin = rb;
}

typedef struct { double ub; int idx; } orc_cand;

static int cand_cmp(const void *pa, const void *pb)
{
    const orc_cand *a = (const orc_cand *)pa, *b = (const orc_cand *)pb;
    if (a->ub > b->ub) return -1;           /* larger bound first */
    if (a->ub < b->ub) return 1;
    return (a->idx > b->idx) - (a->idx < b->idx); /* then lower index */
}

/* ------------------------------------------------------------------ */
/* Block selection  [QUEST Method "Top-K block selection"; S2 selector  */
/* op; R3, R4].  ub: [NB] group bounds.  Writes the selected block ids   */
/* ascending into sel and returns their count.  If kth_ub is not NULL it */
/* receives the bound of the last block taken by the top-K step (NAN if  */
/* that step took none).                                                  */
/* ------------------------------------------------------------------ */
int orc_select(int L, int blk, const double *ub, int k_sel, int sink_tokens,
               int recent_tokens, int *sel, double *kth_ub)
{
    int NB = (L + blk - 1) / blk;
    int se, rb;
    orc_forced_range(L, blk, sink_tokens, recent_tokens, &se, &rb);
    char *take = (char *)calloc((size_t)(NB > 0 ? NB : 1), 1);
    orc_cand *cand = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)(NB > 0 ? NB : 1));
    int nc = 0;
    for (int j = 0; j < NB; ++j) {
        if (j < se || j >= rb) take[j] = 1;
        else { cand[nc].ub = ub[j]; cand[nc].idx = j; ++nc; }
    }
    int keff = k_sel < nc ? k_sel : nc;
    if (keff < 0) keff = 0;
    qsort(cand, (size_t)nc, sizeof(orc_cand), cand_cmp);
    for (int i = 0; i < keff; ++i) take[cand[i].idx] = 1;
    if (kth_ub) *kth_ub = keff > 0 ? cand[keff - 1].ub : NAN;
    int n = 0;
    for (int j = 0; j < NB; ++j)
        if (take[j]) sel[n++] = j;
    free(cand);
    free(take);
    return n;
}

/* Softmax-weighted sum over n rows given their logits:                 */
/*   out = sum_i exp(l_i - M) v_i / sum_i exp(l_i - M),  M = max_i l_i  */
/* Values come from a callback-free row reader: vrow(i, d).             */
/* The two attention routines below fill logits and read values.        */

/* ------------------------------------------------------------------ */
/* f16 attention of one query head over a token set  [QUEST S3 block    */
/* skip: unselected blocks contribute nothing; CPUATT Method with       */
/* f16 rows in place of int8].                                          */
/*   logit_t = scale * sum_d q[d] * k_t[d];  p = softmax(logit);        */
/*   out[d] = sum_t p_t v_t[d]                                          */
/* K, V: [max_seq, D] rows of one (seq, KV head).  sel: ascending block */
/* ids (n_sel >= 0), or n_sel < 0 for every token in [0, L).             */
/* ------------------------------------------------------------------ */
static long token_list(int L, int blk, const int *sel, int n_sel, long *tok)
{
    long n = 0;
    if (n_sel < 0) {
        for (long t = 0; t < L; ++t) tok[n++] = t;
        return n;
    }
    for (int i = 0; i < n_sel; ++i)
        for (long t = (long)sel[i] * blk; t < (long)(sel[i] + 1) * blk && t < L; ++t)
            tok[n++] = t;
    return n;
}

void orc_attend_f16(int D, int L, int blk, const float *q, double scale,
                    const uint16_t *K, const uint16_t *V,
                    const int *sel, int n_sel, double *out)
{
    long cap = (long)L + 1;
    long *tok = (long *)malloc(sizeof(long) * (size_t)cap);
    long n = token_list(L, blk, sel, n_sel, tok);
    double *lg = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double M = -INFINITY;
    for (long i = 0; i < n; ++i) {
        const uint16_t *k = K + (size_t)tok[i] * D;
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += (double)q[d] * orc_half_to_double(k[d]);
        lg[i] = scale * s;
        if (lg[i] > M) M = lg[i];
    }
    double Z = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (long i = 0; i < n; ++i) {
        double w = exp(lg[i] - M);
        Z += w;
        const uint16_t *v = V + (size_t)tok[i] * D;
        for (int d = 0; d < D; ++d) out[d] += w * orc_half_to_double(v[d]);
    }
    if (n > 0)
        for (int d = 0; d < D; ++d) out[d] /= Z;   /* R6: empty set -> 0 */
    free(lg);
    free(tok);
}

/* ------------------------------------------------------------------ */
/* Sparse-V, eps mode  ["Sparse Attention -- Quest-style block-selector */
/* ...", section "Adaptive tau (the eps mode)" and "Compose" item 3]:   */
/* inside the attended blocks, the V term of a position is dropped when */
/* its weight is below eps times the mean weight around it, so that the */
/* dropped share of the softmax mass stays below eps.  The positions    */
/* stay in the softmax denominator.                                      */
/* Reading R7 (the page leaves the extent of its running sums to the    */
/* kernel): the mean is taken over the position's chunk, the attended   */
/* positions t with the same t / ORC_SV_CHUNK:                          */
/*   m_c = max_{t in c} s_t,  p_t = exp(s_t - m_c),                     */
/*   keep V_t  iff  not (p_t < eps * (sum_{u in c} p_u) / |c|).         */
/* keep[i] is set for the i-th position of the list tok[0..n).          */
/* ------------------------------------------------------------------ */
#define ORC_SV_CHUNK 16

void orc_sparse_v_keep(long n, const long *tok, const double *lg, double eps, int *keep)
{
    long i = 0;
    while (i < n) {
        long j = i;
        while (j < n && tok[j] / ORC_SV_CHUNK == tok[i] / ORC_SV_CHUNK) ++j;
        double m = -INFINITY;
        for (long u = i; u < j; ++u)
            if (lg[u] > m) m = lg[u];
        double sum = 0.0;
        for (long u = i; u < j; ++u) sum += exp(lg[u] - m);
        double thr = eps * sum / (double)(j - i);
        for (long u = i; u < j; ++u) keep[u] = !(exp(lg[u] - m) < thr);
        i = j;
    }
}

/* Attention of one head with sparse-V (eps mode) over an f16 cache: as */
/* orc_attend_f16, the numerator summing only the kept positions.       */
/* dropped (optional): the dropped share of the softmax mass.           */
void orc_attend_f16_sv(int D, int L, int blk, const float *q, double scale,
                       const uint16_t *K, const uint16_t *V, const int *sel, int n_sel,
                       double eps, double *out, double *dropped)
{
    long cap = (long)L + 1;
    long *tok = (long *)malloc(sizeof(long) * (size_t)cap);
    long n = token_list(L, blk, sel, n_sel, tok);
    double *lg = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
    int *keep = (int *)calloc((size_t)(n > 0 ? n : 1), sizeof(int));
    double M = -INFINITY;
    for (long i = 0; i < n; ++i) {
        const uint16_t *k = K + (size_t)tok[i] * D;
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += (double)q[d] * orc_half_to_double(k[d]);
        lg[i] = scale * s;
        if (lg[i] > M) M = lg[i];
    }
    orc_sparse_v_keep(n, tok, lg, eps, keep);
    double Z = 0.0, Zd = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (long i = 0; i < n; ++i) {
        double w = exp(lg[i] - M);
        Z += w;
        if (!keep[i]) {
            Zd += w;
            continue;
        }
        const uint16_t *vr = V + (size_t)tok[i] * D;
        for (int d = 0; d < D; ++d) out[d] += w * orc_half_to_double(vr[d]);
    }
    if (n > 0)
        for (int d = 0; d < D; ++d) out[d] /= Z;
    if (dropped) *dropped = n > 0 ? Zd / Z : 0.0;
    free(keep);
    free(lg);
    free(tok);
}

/* The same over an absmax-int8 cache (logits as orc_attend_int8).      */
void orc_attend_int8_sv(int D, int L, int blk, const int8_t *qc, float q_scale, double scale,
                        const int8_t *K, const int8_t *V, const float *ks, const float *vs,
                        const int *sel, int n_sel, double eps, double *out, double *dropped)
{
    long cap = (long)L + 1;
    long *tok = (long *)malloc(sizeof(long) * (size_t)cap);
    long n = token_list(L, blk, sel, n_sel, tok);
    double *lg = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
    int *keep = (int *)calloc((size_t)(n > 0 ? n : 1), sizeof(int));
    double M = -INFINITY;
    for (long i = 0; i < n; ++i) {
        int64_t dot = 0;
        const int8_t *k = K + (size_t)tok[i] * D;
        for (int d = 0; d < D; ++d) dot += (int64_t)qc[d] * (int64_t)k[d];
        lg[i] = scale * ((double)dot * (double)q_scale * (double)ks[tok[i]]);
        if (lg[i] > M) M = lg[i];
    }
    orc_sparse_v_keep(n, tok, lg, eps, keep);
    double Z = 0.0, Zd = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (long i = 0; i < n; ++i) {
        double w = exp(lg[i] - M);
        Z += w;
        if (!keep[i]) {
            Zd += w;
            continue;
        }
        double vsc = (double)vs[tok[i]];
        const int8_t *vr = V + (size_t)tok[i] * D;
        for (int d = 0; d < D; ++d) out[d] += w * vsc * (double)vr[d];
    }
    if (n > 0)
        for (int d = 0; d < D; ++d) out[d] /= Z;
    if (dropped) *dropped = n > 0 ? Zd / Z : 0.0;
    free(keep);
    free(lg);
    free(tok);
}

/* ------------------------------------------------------------------ */
/* q8_0 attention of one query head (R8), with sparse-V at eps (eps = 0 */
/* keeps every V term):                                                  */
/*   logit_t = softmax_scale * q_scale * sum_g d_g(k_t) * dot_g(t),      */
/*   dot_g(t) = sum_{d in group g} q_code[d] * k_code_t[d]  (exact)      */
/*   out[d]  = sum_t softmax(logit)_t * d_g(v_t) * v_code_t[d]           */
/* qc/q_scale: the head's query quantized per row (orc_quantize_row).   */
/* kd, vd: [max_seq, D/32] binary16 bits of one (seq, KV head).          */
/* ------------------------------------------------------------------ */
void orc_attend_q8_0(int D, int L, int blk, const int8_t *qc, float q_scale, double scale,
                     const int8_t *K, const int8_t *V, const uint16_t *kd, const uint16_t *vd,
                     const int *sel, int n_sel, double eps, double *out, double *dropped)
{
    const int ng = D / ORC_QGROUP;
    long cap = (long)L + 1;
    long *tok = (long *)malloc(sizeof(long) * (size_t)cap);
    long n = token_list(L, blk, sel, n_sel, tok);
    double *lg = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
    int *keep = (int *)calloc((size_t)(n > 0 ? n : 1), sizeof(int));
    double M = -INFINITY;
    for (long i = 0; i < n; ++i) {
        const int8_t *k = K + (size_t)tok[i] * D;
        double acc = 0.0;
        for (int g = 0; g < ng; ++g) {
            int64_t dot = 0;
            for (int d = g * ORC_QGROUP; d < (g + 1) * ORC_QGROUP; ++d)
                dot += (int64_t)qc[d] * (int64_t)k[d];
            acc += orc_half_to_double(kd[(size_t)tok[i] * ng + g]) * (double)dot;
        }
        lg[i] = scale * (double)q_scale * acc;
        if (lg[i] > M) M = lg[i];
    }
    orc_sparse_v_keep(n, tok, lg, eps, keep);
    double Z = 0.0, Zd = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (long i = 0; i < n; ++i) {
        double w = exp(lg[i] - M);
        Z += w;
        if (!keep[i]) {
            Zd += w;
            continue;
        }
        const int8_t *vq = V + (size_t)tok[i] * D;
        for (int d = 0; d < D; ++d)
            out[d] += w * orc_half_to_double(vd[(size_t)tok[i] * ng + d / ORC_QGROUP]) *
                      (double)vq[d];
    }
    if (n > 0)
        for (int d = 0; d < D; ++d) out[d] /= Z;
    if (dropped) *dropped = n > 0 ? Zd / Z : 0.0;
    free(keep);
    free(lg);
    free(tok);
}

/* ------------------------------------------------------------------ */
/* q4_0 attention of one query head (R9), with sparse-V at eps:         */
/*   logit_t = softmax_scale * q_scale * sum_g d_g(k_t) * dot_g(t),      */
/*   dot_g(t) = sum_{c in g} q_code[c] * (k_code_t[c] - 8)   (exact)     */
/*   out[c]  = sum_t softmax(logit)_t * d_g(v_t) * (v_code_t[c] - 8)     */
/* K, V: [max_seq, D/2] packed rows; kd, vd: [max_seq, D/32] binary16.  */
/* ------------------------------------------------------------------ */
void orc_attend_q4_0(int D, int L, int blk, const int8_t *qc, float q_scale, double scale,
                     const uint8_t *K, const uint8_t *V, const uint16_t *kd,
                     const uint16_t *vd, const int *sel, int n_sel, double eps, double *out,
                     double *dropped)
{
    const int ng = D / ORC_QGROUP;
    long cap = (long)L + 1;
    long *tok = (long *)malloc(sizeof(long) * (size_t)cap);
    long n = token_list(L, blk, sel, n_sel, tok);
    double *lg = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
    int *keep = (int *)calloc((size_t)(n > 0 ? n : 1), sizeof(int));
    double M = -INFINITY;
    for (long i = 0; i < n; ++i) {
        const uint8_t *k = K + (size_t)tok[i] * (D / 2);
        double sum = 0.0;
        for (int g = 0; g < ng; ++g) {
            int64_t dot = 0;
            for (int c = g * ORC_QGROUP; c < (g + 1) * ORC_QGROUP; ++c)
                dot += (int64_t)qc[c] * (int64_t)(q4_code(k, c) - 8);
            sum += orc_half_to_double(kd[(size_t)tok[i] * ng + g]) * (double)dot;
        }
        lg[i] = scale * (double)q_scale * sum;
        if (lg[i] > M) M = lg[i];
    }
    orc_sparse_v_keep(n, tok, lg, eps, keep);
    double Z = 0.0, Zd = 0.0;
    for (int c = 0; c < D; ++c) out[c] = 0.0;
    for (long i = 0; i < n; ++i) {
        double w = exp(lg[i] - M);
        Z += w;
        if (!keep[i]) {
            Zd += w;
            continue;
        }
        const uint8_t *v4 = V + (size_t)tok[i] * (D / 2);
        for (int c = 0; c < D; ++c)
            out[c] += w * orc_half_to_double(vd[(size_t)tok[i] * ng + c / ORC_QGROUP]) *
                      (double)(q4_code(v4, c) - 8);
    }
    if (n > 0)
        for (int c = 0; c < D; ++c) out[c] /= Z;
    if (dropped) *dropped = n > 0 ? Zd / Z : 0.0;
    free(keep);
    free(lg);
    free(tok);
}

/* ------------------------------------------------------------------ */
/* Exact integer q.k dots  [CPUATT Method: integer logit dots, exact].     */
/*   dot_t = sum_d q_code[d] * k_code_t[d]   (|dot| <= D*127*127)       */
/* ------------------------------------------------------------------ */
void orc_qk_int8(int D, long n, const int8_t *qc, const int8_t *K, int64_t *dots)
{
    for (long t = 0; t < n; ++t) {
        int64_t s = 0;
        for (int d = 0; d < D; ++d) s += (int64_t)qc[d] * (int64_t)K[(size_t)t * D + d];
        dots[t] = s;
    }
}

/* ------------------------------------------------------------------ */
/* int8 attention of one query head  [CPUATT Method]:                   */
/*   logit_t = dot_t * q_scale * k_scale_t * softmax_scale              */
/*   out[d]  = sum_t softmax(logit)_t * v_scale_t * v_code_t[d]         */
/* qc/q_scale: the head's query quantized by orc_quantize_row.          */
/* ------------------------------------------------------------------ */
void orc_attend_int8(int D, int L, int blk, const int8_t *qc, float q_scale, double scale,
                     const int8_t *K, const int8_t *V, const float *ks, const float *vs,
                     const int *sel, int n_sel, double *out)
{
    long cap = (long)L + 1;
    long *tok = (long *)malloc(sizeof(long) * (size_t)cap);
    long n = token_list(L, blk, sel, n_sel, tok);
    double *lg = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double M = -INFINITY;
    for (long i = 0; i < n; ++i) {
        int64_t dot = 0;
        orc_qk_int8(D, 1, qc, K + (size_t)tok[i] * D, &dot);
        lg[i] = (double)dot * (double)q_scale * (double)ks[tok[i]] * scale;
        if (lg[i] > M) M = lg[i];
    }
    double Z = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (long i = 0; i < n; ++i) {
        double w = exp(lg[i] - M);
        Z += w;
        double sv = (double)vs[tok[i]];
        const int8_t *v = V + (size_t)tok[i] * D;
        for (int d = 0; d < D; ++d) out[d] += w * sv * (double)v[d];
    }
    if (n > 0)
        for (int d = 0; d < D; ++d) out[d] /= Z;
    free(lg);
    free(tok);
}

/* ------------------------------------------------------------------ */
/* Attention over float rows (dequantized cache)  [CPUATT Correctness:  */
/* the reference is float attention over the dequantized rows].  q: [D] */
/* f32; K, V: the int8 rows times their scales, formed here in binary64. */
/* With q_code != NULL the query is the dequantized int8 query          */
/* (q_scale * q_code) instead of q.                                      */
/* ------------------------------------------------------------------ */
void orc_attend_dequant(int D, int L, int blk, const float *q, const int8_t *q_code,
                        float q_scale, double scale, const int8_t *K, const int8_t *V,
                        const float *ks, const float *vs, const int *sel, int n_sel,
                        double *out)
{
    long cap = (long)L + 1;
    long *tok = (long *)malloc(sizeof(long) * (size_t)cap);
    long n = token_list(L, blk, sel, n_sel, tok);
    double *lg = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double M = -INFINITY;
    for (long i = 0; i < n; ++i) {
        double s = 0.0;
        for (int d = 0; d < D; ++d) {
            double qd = q_code ? (double)q_scale * (double)q_code[d] : (double)q[d];
            double kd = (double)ks[tok[i]] * (double)K[(size_t)tok[i] * D + d];
            s += qd * kd;
        }
        lg[i] = scale * s;
        if (lg[i] > M) M = lg[i];
    }
    double Z = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (long i = 0; i < n; ++i) {
        double w = exp(lg[i] - M);
        Z += w;
        for (int d = 0; d < D; ++d)
            out[d] += w * ((double)vs[tok[i]] * (double)V[(size_t)tok[i] * D + d]);
    }
    if (n > 0)
        for (int d = 0; d < D; ++d) out[d] /= Z;
    free(lg);
    free(tok);
}

/* ------------------------------------------------------------------ */
/* Moment tail  [SCSA "2. Mechanism", per-query steps "Moment tail" and */
/* "Output"; applied to Quest blocks as reading R10]: a group of keys   */
/* that is not read exactly still contributes, through its member count */
/* m, key centroid c_K and value mean c_V, the term m * exp(a) at c_V   */
/* inside the shared softmax normalizer, a = scale * q . c_K.           */
/* ------------------------------------------------------------------ */

/* The per-block means of rows X [L][D] (binary64; the cache's stored    */
/* rows, dequantized), each rounded once to binary16: block j holds the  */
/* m_j = min(blk, L - j * blk) rows j * blk .. j * blk + m_j - 1.        */
/* mean: [ceil(L / blk)][D] binary16 bit patterns.                       */
void orc_block_moments(int D, int L, int blk, const double *X, uint16_t *mean)
{
    int nb = (L + blk - 1) / blk;
    for (int j = 0; j < nb; ++j) {
        int lo = j * blk;
        int m = L - lo < blk ? L - lo : blk;
        for (int d = 0; d < D; ++d) {
            double sum = 0.0;
            for (int t = lo; t < lo + m; ++t) sum += X[(size_t)t * D + d];
            mean[(size_t)j * D + d] = orc_double_to_half(sum / (double)m);
        }
    }
}

/* Attention of one query head over the tokens of the listed blocks,     */
/* exactly, plus the moment tail of every other block of [0, L).         */
/* q_exact: the query the exact logits use (the f32 query, or for the    */
/* quantized cache types its dequantized int8 codes); q_tail: the f32    */
/* query (R10).  K, V: [L][D] the cache's rows in binary64 (dequantized). */
/* mK, mV: [ceil(L / blk)][D] binary16 block means (orc_block_moments).  */
/* Terms:                                                                */
/*   listed token t:   x_t = scale * q_exact . K_t,           value V_t  */
/*   unlisted block j: x_j = scale * q_tail . mK_j + ln m_j,  value mV_j */
/*   out = sum_i exp(x_i - M) value_i / sum_i exp(x_i - M),  M = max x.  */
/* ------------------------------------------------------------------ */
void orc_attend_tail(int D, int L, int blk, const double *q_exact, const double *q_tail,
                     double scale, const double *K, const double *V, const int *sel,
                     int n_sel, const uint16_t *mK, const uint16_t *mV, double *out)
{
    int nb = (L + blk - 1) / blk;
    char *listed = (char *)calloc((size_t)(nb > 0 ? nb : 1), 1);
    for (int i = 0; i < n_sel; ++i)
        if (sel[i] >= 0 && sel[i] < nb) listed[sel[i]] = 1;
    long n_terms = (long)L + nb;
    double *x = (double *)malloc(sizeof(double) * (size_t)(n_terms > 0 ? n_terms : 1));
    const double **val = (const double **)malloc(sizeof(double *) * (size_t)(n_terms > 0 ? n_terms : 1));
    double *tail_val = (double *)malloc(sizeof(double) * (size_t)(nb > 0 ? nb : 1) * D);
    long n = 0;
    for (int j = 0; j < nb; ++j) {
        int lo = j * blk;
        int mj = L - lo < blk ? L - lo : blk;
        if (listed[j]) {
            for (int t = lo; t < lo + mj; ++t) {
                double s = 0.0;
                for (int d = 0; d < D; ++d) s += q_exact[d] * K[(size_t)t * D + d];
                x[n] = scale * s;
                val[n++] = V + (size_t)t * D;
            }
        } else {
            double s = 0.0;
            for (int d = 0; d < D; ++d)
                s += q_tail[d] * orc_half_to_double(mK[(size_t)j * D + d]);
            for (int d = 0; d < D; ++d)
                tail_val[(size_t)j * D + d] = orc_half_to_double(mV[(size_t)j * D + d]);
            x[n] = scale * s + log((double)mj);
            val[n++] = tail_val + (size_t)j * D;
        }
    }
    double M = -INFINITY;
    for (long i = 0; i < n; ++i)
        if (x[i] > M) M = x[i];
    double Z = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (long i = 0; i < n; ++i) {
        double w = exp(x[i] - M);
        Z += w;
        for (int d = 0; d < D; ++d) out[d] += w * val[i][d];
    }
    if (n > 0)
        for (int d = 0; d < D; ++d) out[d] /= Z;
    free(tail_val);
    free(val);
    free(x);
    free(listed);
}

/* ------------------------------------------------------------------ */
/* One decode step for every (seq, KV head) of a cache                   */
/* [QUEST S2/S3: selector then block-skipping attention; CPUATT Usage:  */
/* query head h reads KV head h / (H / Hkv)].                            */
/* q: [B, H, D] f32.  out: [B, H, D].  With dense != 0 every token is    */
/* attended and no selection is made.  sel_idx ([B, Hkv, NB]) and        */
/* sel_cnt ([B, Hkv]) receive the selection when not NULL.  For the      */
/* int8 cache each query head is quantized once (CPUATT Method).         */
/* Problems (seq, KV head) are independent, and so are the query heads   */
/* once their problem's selection is made; n_threads > 1 spreads the      */
/* selections, then the (problem, query head) attentions, over OpenMP     */
/* threads.  Each head's arithmetic is the same on any thread count.      */
/* Returns 0, or -1 on bad arguments.                                     */
/* ------------------------------------------------------------------ */
int orc_decode(const orc_cache *c, int H, const float *q, double scale, int k_sel,
               int sink_tokens, int recent_tokens, int dense, int *sel_idx, int *sel_cnt,
               double *out, int n_threads)
{
    if (H % c->Hkv != 0 || c->len <= 0) return -1;
    const int G = H / c->Hkv, D = c->D, L = c->len;
    const int NB = (L + c->blk - 1) / c->blk;
    const int nbmax = c->max_seq / c->blk;
    const int P = c->B * c->Hkv;
    int *sel_all = (int *)malloc(sizeof(int) * (size_t)NB * (size_t)P);
    int *n_all = (int *)malloc(sizeof(int) * (size_t)P);
#ifdef _OPENMP
    if (n_threads < 1) n_threads = 1;
#endif
    /* the selection of every problem (its group's shared block set) */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
    for (int p = 0; p < P; ++p) {
        int b = p / c->Hkv, g = p % c->Hkv;
        const float *qg = q + ((size_t)b * H + (size_t)g * G) * D;
        int *sel = sel_all + (size_t)p * NB;
        n_all[p] = -1;
        if (!dense) {
            double *ub = (double *)malloc(sizeof(double) * (size_t)NB);
            orc_block_scores(G, D, NB, qg, c->kmin + bound_index(c, b, g, 0),
                             c->kmax + bound_index(c, b, g, 0), NULL, ub, NULL);
            n_all[p] = orc_select(L, c->blk, ub, k_sel, sink_tokens, recent_tokens, sel, NULL);
            free(ub);
            if (sel_idx) memcpy(sel_idx + (size_t)p * nbmax, sel, sizeof(int) * (size_t)n_all[p]);
            if (sel_cnt) sel_cnt[p] = n_all[p];
        }
    }
    /* each query head over its problem's selection (or every token) */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
    for (int u = 0; u < P * G; ++u) {
        const int p = u / G, hh = u % G;
        const int b = p / c->Hkv, g = p % c->Hkv;
        const int *sel = sel_all + (size_t)p * NB;
        const int n_sel = n_all[p];
        const size_t r0 = row_index(c, b, g, 0);
        const float *qh = q + ((size_t)b * H + (size_t)g * G + hh) * D;
        double *o = out + ((size_t)b * H + (size_t)g * G + hh) * D;
        if (c->dtype == ORC_F16) {
            orc_attend_f16(D, L, c->blk, qh, scale, (const uint16_t *)c->K + r0 * D,
                           (const uint16_t *)c->V + r0 * D, sel, n_sel, o);
        } else if (c->dtype == ORC_Q4_0) {
            int8_t *qc = (int8_t *)malloc((size_t)D);
            float qs;
            orc_quantize_row(qh, D, qc, &qs);
            orc_attend_q4_0(D, L, c->blk, qc, qs, scale, (const uint8_t *)c->K + r0 * (D / 2),
                            (const uint8_t *)c->V + r0 * (D / 2), c->kd + r0 * (D / ORC_QGROUP),
                            c->vd + r0 * (D / ORC_QGROUP), sel, n_sel, 0.0, o, NULL);
            free(qc);
        } else if (c->dtype == ORC_Q8_0) {
            int8_t *qc = (int8_t *)malloc((size_t)D);
            float qs;
            orc_quantize_row(qh, D, qc, &qs);
            orc_attend_q8_0(D, L, c->blk, qc, qs, scale, (const int8_t *)c->K + r0 * D,
                            (const int8_t *)c->V + r0 * D, c->kd + r0 * (D / ORC_QGROUP),
                            c->vd + r0 * (D / ORC_QGROUP), sel, n_sel, 0.0, o, NULL);
            free(qc);
        } else {
            int8_t *qc = (int8_t *)malloc((size_t)D);
            float qs;
            orc_quantize_row(qh, D, qc, &qs);
            orc_attend_int8(D, L, c->blk, qc, qs, scale, (const int8_t *)c->K + r0 * D,
                            (const int8_t *)c->V + r0 * D, c->ks + r0, c->vs + r0,
                            sel, n_sel, o);
            free(qc);
        }
    }
    free(sel_all);
    free(n_all);
    return 0;
}

int orc_num_threads_available(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
