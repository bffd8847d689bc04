// common.cuh -- device helpers shared by the kvdecode kernels (sm_103a).
//
// Inline PTX for the Blackwell data-movement path: mbarrier phases, 1-D TMA
// bulk copies global->shared (cp.async.bulk ... complete_tx), L2 cache
// policies, and programmatic dependent launch (griddepcontrol).  Every wait
// on an mbarrier is bounded in time; when the bound runs out the kernel
// records KVD_ERR_TIMEOUT in the cache's status word and winds down instead
// of trapping.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvdecode.h"

namespace kvd {

constexpr int kHeadDim = 128;     // D
constexpr int kBlock = 64;        // B_SEL
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -1.0e30f;  // finite "minus infinity" for running maxima
// Device waits give up after this many nanoseconds of wall time.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------- PTX ---
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Stage marks (builds with -DKVD_MARKS only; kvd_debug_stage_marks): the
// calling thread writes the global timer to slot `slot` of this CTA's row of
// `marks` (kMarkSlots words per CTA, CTAs numbered x-fastest; rows past
// kMarkCtas are not recorded).  Without the flag the macro is empty.
constexpr int kMarkSlots = 16;
constexpr int kMarkCtas = 4096;
#ifdef KVD_MARKS
#define KVD_MARK(marks, slot)                                                              \
    do {                                                                                   \
        const unsigned kvd_cta_ = blockIdx.y * gridDim.x + blockIdx.x;                     \
        if ((marks) != nullptr && kvd_cta_ < static_cast<unsigned>(kMarkCtas))             \
            (marks)[static_cast<size_t>(kvd_cta_) * kMarkSlots + (slot)] = global_timer_ns(); \
    } while (0)
// The latest of the callers' timer values (every caller writes; the
// maximum stays): when the last of several warps reached the mark.
#define KVD_MARK_LAST(marks, slot)                                                         \
    do {                                                                                   \
        const unsigned kvd_cta_ = blockIdx.y * gridDim.x + blockIdx.x;                     \
        if ((marks) != nullptr && kvd_cta_ < static_cast<unsigned>(kMarkCtas))             \
            atomicMax((marks) + static_cast<size_t>(kvd_cta_) * kMarkSlots + (slot),       \
                      global_timer_ns());                                                  \
    } while (0)
#else
#define KVD_MARK(marks, slot) \
    do {                      \
    } while (0)
#define KVD_MARK_LAST(marks, slot) \
    do {                           \
    } while (0)
#endif

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Both arrive forms return the barrier state token (unused by callers).
__device__ __forceinline__ uint64_t mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    uint64_t state;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
                 : "=l"(state)
                 : "r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
    return state;
}

__device__ __forceinline__ uint64_t mbar_arrive(uint64_t *bar) {
    uint64_t state;
    asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];"
                 : "=l"(state)
                 : "r"(smem_addr(bar))
                 : "memory");
    return state;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits until the phase with the given parity has completed.  Returns false
// when `abort_flag` (shared memory) becomes non-zero or limit_ns of wall time
// pass.
__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity,
                                                volatile int *abort_flag, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > limit_ns) return false;
        }
    }
}

// mbar_wait_limit with the kernels' limit, kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          volatile int *abort_flag) {
    return mbar_wait_limit(bar, parity, abort_flag, kWaitLimitNs);
}

// L2 policy for data read once per step (K/V blocks): evict first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D TMA bulk copy global -> shared; completes `bytes` transactions on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void tma_load_1d(void *dst, const void *src, uint32_t bytes,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch: wait for the upstream grid's memory, and
// allow the downstream grid to start its prologue.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Arrival on a GPU-scope counter by one thread right after a CTA barrier.
// The release covers every store the CTA made before the barrier, and the
// acquire every store that earlier arrivals released; a barrier after the
// call extends the acquire to the whole CTA.
__device__ __forceinline__ unsigned atomic_add_acq_rel_gpu(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void report_status(int32_t *dev_status, int code) {
    if (dev_status) atomicCAS(reinterpret_cast<int *>(dev_status), 0, code);
}

// Sequence b's own length when the cache carries per-sequence lengths (one
// outside [0, len] is reported and clamped), else the cache's len.
__device__ __forceinline__ int seq_len_of(const int32_t *seq_lens, int b, int len,
                                          int32_t *dev_status) {
    if (!seq_lens) return len;
    int l = seq_lens[b];
    if (l < 0 || l > len) {
        report_status(dev_status, KVD_ERR_INVALID);
        l = l < 0 ? 0 : len;
    }
    return l;
}

// Quest forced blocks and candidates of a sequence of L tokens: sink blocks
// [0, se), recent blocks [rb, NB), candidates [se, rb).
struct ForcedRange {
    int NB, se, rb;
};
__device__ __host__ __forceinline__ ForcedRange forced_range(int L, int sink_tokens,
                                                             int recent_tokens) {
    ForcedRange f;
    f.NB = (L + kBlock - 1) / kBlock;
    f.se = (sink_tokens + kBlock - 1) / kBlock;
    if (f.se > f.NB) f.se = f.NB;
    f.rb = f.NB;
    if (recent_tokens > 0) {
        long start = static_cast<long>(L) - recent_tokens;
        if (start < 0) start = 0;
        f.rb = static_cast<int>(start / kBlock);
    }
    if (f.rb < f.se) f.rb = f.se;
    return f;
}

// ------------------------------------------------------------ numerics ---
// Order-preserving map f32 -> u32 (larger float, larger key); -0 maps as +0.
__device__ __forceinline__ uint32_t float_to_key(float f) {
    if (f == 0.0f) f = 0.0f;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// q8_0 quantization of one 128-wide row held 4 values per lane by a full
// warp: the 8 lanes 8g..8g+7 hold group g (channels 32g..32g+31).  The
// group's scale is d = fl16(absmax/127) (the IEEE f32 quotient rounded to
// f16), code = round-half-even(x/d) in f32, clamped to +-127, and a zero
// scale gives zero codes.  Returns the packed codes of the lane's 4 values
// and writes the group's scale to *d (all lanes of the group).
__device__ __forceinline__ uint32_t quantize_group32_warp(const float (&x)[4], __half *d) {
    float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const __half dh = __float2half_rn(__fdiv_rn(a, 127.0f));
    *d = dh;
    const float s = __half2float(dh);
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        int c = 0;
        if (s != 0.0f) {
            const float r = rintf(__fdiv_rn(x[j], s));
            c = static_cast<int>(fminf(fmaxf(r, -127.0f), 127.0f));
        }
        packed |= (static_cast<uint32_t>(c) & 0xffu) << (8 * j);
    }
    return packed;
}

// q4_0 quantization of one 128-wide row held 4 values per lane by a full
// warp (group g = lanes 8g..8g+7).  m is the group's value of largest
// magnitude, the first one in channel order; the scale is d = fl16(m/-8)
// (the IEEE f32 quotient rounded to f16); code = round-half-even(x/d) + 8 in
// f32, clamped to [0, 15] (8 when d is 0).  Returns the lane's two bytes:
// channel 4l in the low nibble of the first, 4l+1 in its high nibble, and
// so on; writes the group's scale to *d.
__device__ __forceinline__ uint32_t quantize_q4_0_warp(const float (&x)[4], __half *d,
                                                       int lane) {
    float mag = -1.0f, m = 0.0f;
    int idx = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (fabsf(x[j]) > mag) {
            mag = fabsf(x[j]);
            m = x[j];
            idx = 4 * lane + j;
        }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mag, o);
        const float ov = __shfl_xor_sync(0xffffffffu, m, o);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        if (om > mag || (om == mag && oi < idx)) {
            mag = om;
            m = ov;
            idx = oi;
        }
    }
    const __half dh = __float2half_rn(__fdiv_rn(m, -8.0f));
    *d = dh;
    const float s = __half2float(dh);
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        int c = 8;
        if (s != 0.0f) {
            const float r = rintf(__fdiv_rn(x[j], s)) + 8.0f;
            c = static_cast<int>(fminf(fmaxf(r, 0.0f), 15.0f));
        }
        packed |= static_cast<uint32_t>(c) << (4 * j);
    }
    return packed;  // 16 bits: channels 4l .. 4l+3, low nibble first
}

// Absmax int8 quantization of one 128-wide row held 4 values per lane by a
// full warp (lane l holds x[4l..4l+3]).  scale = absmax/127 (IEEE f32
// division), code = round-half-even(x/scale) clamped to +-127, and a zero
// scale gives zero codes.  Returns the packed codes of the lane's 4 values
// (value 4l in the low byte) and writes the scale to *scale (all lanes).
__device__ __forceinline__ uint32_t quantize_row_warp(const float (&x)[4], float *scale) {
    float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float s = __fdiv_rn(a, 127.0f);
    *scale = s;
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        int c = 0;
        if (s != 0.0f) {
            c = __float2int_rn(__fdiv_rn(x[j], s));
            c = max(-127, min(127, c));
        }
        packed |= (static_cast<uint32_t>(c) & 0xffu) << (8 * j);
    }
    return packed;
}

}  // namespace kvd
