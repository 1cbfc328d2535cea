// device_utils.cuh -- sm_103a building blocks for the verify kernels:
// mbarrier + 1-D bulk-copy (TMA engine) staging, bounded waits, the MUFU
// base-2 exponential, and element traits for fp32 / bf16 logit rows.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "spec_verify.h"

namespace specv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr double kLog2eD = 1.4426950408889634073599246810019;
constexpr double kLn2D = 0.69314718055994530941723212145818;
constexpr int kMaxK = SPEC_MAX_K;

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity to complete, giving up
// after ~2 s of wall time.  Returns false on time-out.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// 1-D bulk copy global -> shared (TMA engine, no tensor map), completing
// `bytes` of transaction count on `bar`.  dst, src 16-B aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// The same copy with an L2 cache policy (from l2_policy_evict_first): the
// copied lines are the first the L2 replaces.
__device__ __forceinline__ void bulk_g2s_hint(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
        "[%3], %4;" ::"r"(smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// An L2 policy that marks the accessed lines evict-first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Bulk prefetch of [src, src + bytes) into L2 by the TMA engine, without
// registers or shared memory (src and bytes multiples of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Atomic add with acquire-release semantics at GPU scope: the caller's
// earlier writes are visible to whoever later acquires the counter, and
// the caller sees the writes released by earlier adders.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Release-add and release-store at GPU scope, acquire-load at GPU scope.
__device__ __forceinline__ void red_add_release_gpu(int *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_gpu(int *p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Hardware base-2 exponential (MUFU.EX2): ~2 ulp, subnormal results flushed
// to zero, ex2(-inf) = 0, ex2(NaN) = NaN.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pair arithmetic (two IEEE fp32 operations per instruction,
// each rounded to nearest like the scalar forms).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// NaN-propagating max.
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void set_status(int *status, int code) {
    atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- elements
template <int DT>
struct Elem;

template <>
struct Elem<SPEC_F32> {
    static constexpr int kBytes = 4;
    static constexpr int kPerVec = 4;  // elements per 16-byte vector
    static constexpr int kPairs = 2;   // element pairs per vector
    __device__ static __forceinline__ void unpack(const uint4 &v, float (&x)[4]) {
        x[0] = __uint_as_float(v.x);
        x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z);
        x[3] = __uint_as_float(v.w);
    }
    __device__ static __forceinline__ float vmax_nan(const uint4 &v) {
        return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                        fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
    __device__ static __forceinline__ float load1(const void *base, int64_t idx) {
        return __ldg(reinterpret_cast<const float *>(base) + idx);
    }
    // element pairs of a 16-byte vector
    __device__ static __forceinline__ float2 pair(const uint4 &v, int p) {
        return p == 0 ? make_float2(__uint_as_float(v.x), __uint_as_float(v.y))
                      : make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    }
    static constexpr uint32_t kNegInfWord = 0xff800000u;
    // NaN-propagating max over four vectors
    __device__ static __forceinline__ float vmax4_nan(const uint4 (&v)[4]) {
        float m = vmax_nan(v[0]);
        m = fmax_nan(m, vmax_nan(v[1]));
        m = fmax_nan(m, vmax_nan(v[2]));
        return fmax_nan(m, vmax_nan(v[3]));
    }
};

template <>
struct Elem<SPEC_BF16> {
    static constexpr int kBytes = 2;
    static constexpr int kPerVec = 8;
    static constexpr int kPairs = 4;  // element pairs per vector
    __device__ static __forceinline__ void unpack(const uint4 &v, float (&x)[8]) {
        x[0] = __uint_as_float(v.x << 16);
        x[1] = __uint_as_float(v.x & 0xffff0000u);
        x[2] = __uint_as_float(v.y << 16);
        x[3] = __uint_as_float(v.y & 0xffff0000u);
        x[4] = __uint_as_float(v.z << 16);
        x[5] = __uint_as_float(v.z & 0xffff0000u);
        x[6] = __uint_as_float(v.w << 16);
        x[7] = __uint_as_float(v.w & 0xffff0000u);
    }
    __device__ static __forceinline__ float vmax_nan(const uint4 &v) {
        // packed bf16x2 NaN-propagating max, then the two halves
        __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&v.x);
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&v.y);
        __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162 *>(&v.z);
        __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162 *>(&v.w);
        __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
        uint32_t u = *reinterpret_cast<uint32_t *>(&m);
        return fmax_nan(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    }
    __device__ static __forceinline__ float load1(const void *base, int64_t idx) {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(base) + idx);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    __device__ static __forceinline__ float2 word_pair(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    // element pairs of a 16-byte vector (p = 0..3: one 32-bit word each)
    __device__ static __forceinline__ float2 pair(const uint4 &v, int p) {
        return word_pair(p == 0 ? v.x : p == 1 ? v.y : p == 2 ? v.z : v.w);
    }
    static constexpr uint32_t kNegInfWord = 0xff80ff80u;
    // NaN-propagating max over four vectors: one packed bf16x2 tree over the
    // 16 words, then the two halves
    __device__ static __forceinline__ float vmax4_nan(const uint4 (&v)[4]) {
        __nv_bfloat162 m[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&v[j].x);
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&v[j].y);
            const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162 *>(&v[j].z);
            const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162 *>(&v[j].w);
            m[j] = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
        }
        const __nv_bfloat162 t = __hmax2_nan(__hmax2_nan(m[0], m[1]), __hmax2_nan(m[2], m[3]));
        const uint32_t u = *reinterpret_cast<const uint32_t *>(&t);
        return fmax_nan(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    }
};

// ---------------------------------------------------------------- partials
// Arg-max partial: largest value, lowest index among equals; idx = -1 marks
// a NaN; idx = INT_MAX marks "no element".
struct ArgPart {
    float v;
    int i;
};

__device__ __forceinline__ ArgPart arg_merge(ArgPart a, ArgPart b) {
    if (a.i == -1 || b.i == -1) return ArgPart{a.v, -1};
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}

__device__ __forceinline__ ArgPart shfl_arg(ArgPart p, int off) {
    return ArgPart{__shfl_xor_sync(0xffffffffu, p.v, off), __shfl_xor_sync(0xffffffffu, p.i, off)};
}

__device__ __forceinline__ ArgPart warp_arg(ArgPart p) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) p = arg_merge(p, shfl_arg(p, off));
    return p;
}

// c = log2(e) / T as the fp32 quotient of fp32(log2 e) and T, rounded to
// nearest (an IEEE division: within an ulp or so of log2(e) / T); 0 for
// greedy (T == 0); NaN for an invalid temperature.  Every kernel derives the
// scale the same way.  It is computed in fp32: a stats_kernel CTA derives it
// for every sequence of the batch in its prologue, and an fp64 division per
// sequence there took several microseconds per call on GB300's fp64 pipe.
__device__ __forceinline__ float temp_scale(float T) {
    if (T == 0.0f) return 0.0f;
    if (!(T > 0.0f) || !isfinite(T)) return __int_as_float(0x7fc00000);
    const float c = __fdiv_rn(kLog2e, T);
    return isfinite(c) ? c : __int_as_float(0x7fc00000);
}

// Residual weight max(0, p_v - q_v) with p_v = 2^(z_t*c - Lt), q_v likewise;
// L is passed as an fp32 hi/lo pair.  Operations are pinned (no contraction
// choices left to the compiler) so that every kernel computes identical
// bits for the same inputs.
__device__ __forceinline__ float resid_weight(float zt, float zd, float c, float lth, float ltl,
                                              float ldh, float ldl) {
    const float at = __fsub_rn(__fmaf_rn(zt, c, -lth), ltl);
    const float ad = __fsub_rn(__fmaf_rn(zd, c, -ldh), ldl);
    return fmaxf(__fsub_rn(ex2(at), ex2(ad)), 0.0f);
}

// Two residual weights at once in packed fp32.  Lane for lane these are the
// operations of resid_weight (x - y is rounded exactly as x + (-y)), so the
// bits are the same; nl* are the negated hi/lo parts of L.
__device__ __forceinline__ float2 resid_weight2(float2 zt, float2 zd, float2 c2, float2 nlth2, float2 nltl2,
                                                float2 nldh2, float2 nldl2) {
    const float2 at = fadd2(ffma2(zt, c2, nlth2), nltl2);
    const float2 ad = fadd2(ffma2(zd, c2, nldh2), nldl2);
    const float2 d = fadd2(make_float2(ex2(at.x), ex2(at.y)), make_float2(-ex2(ad.x), -ex2(ad.y)));
    return make_float2(fmaxf(d.x, 0.0f), fmaxf(d.y, 0.0f));
}

// Target/draft probability weight 2^(z*c - M) relative to the row max M.
__device__ __forceinline__ float prob_weight(float z, float c, float M) {
    return ex2(__fmaf_rn(z, c, -M));
}

}  // namespace specv
