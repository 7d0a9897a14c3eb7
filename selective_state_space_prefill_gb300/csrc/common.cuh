// common.cuh -- device helpers shared by the libssm kernels (sm_103a).
//
// Hand-written PTX for the pieces with no CUDA C++ spelling: the mbarrier
// wait/arrive protocol, TMA tensor copies, the hardware base-2 exponential and
// the global nanosecond timer.  Nothing here is derived from compiled code.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------------ scalars
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// 2^x with the MUFU.EX2 unit (ex2.approx.ftz.f32: relative error ~2^-22).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// x * sigmoid(x) = x / (1 + e^-x), e^-x through ex2, division by the MUFU reciprocal.
__device__ __forceinline__ float silu(float x) {
    return __fdividef(x, 1.0f + ex2(-x * kLog2e));
}

// log2(x) with the MUFU.LG2 unit (lg2.approx.ftz.f32).
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(v) = log(1 + e^v), with e = e^v from MUFU.EX2:
//   v > 20       -> v: the correction log1p(e^-v) < 2.1e-9 is below the fp32 resolution of v;
//   e < 1/16     -> log1p(e) by its alternating Taylor series e - e^2/2 + e^3/3 - e^4/4 + e^5/5
//                   (Horner form); the first dropped term bounds the relative error by
//                   e^5/6 < 1.6e-7, and there is no cancellation however small e is;
//   otherwise    -> log2(1 + e) * ln 2 through MUFU.LG2; 1 + e carries at most 2^-24 absolute
//                   rounding and the result is at least log(17/16) = 0.06, so the relative
//                   error stays near 1e-6.
__device__ __forceinline__ float softplus(float v) {
    const float e = ex2(v * kLog2e);
    float s = fmaf(e, 0.2f, -0.25f);
    s = fmaf(e, s, 1.0f / 3.0f);
    s = fmaf(e, s, -0.5f);
    s = fmaf(e, s, 1.0f);
    const float series = e * s;
    const float viaLog = lg2(1.0f + e) * kLn2;
    return v > 20.0f ? v : (e < 0.0625f ? series : viaLog);
}

// The per-token activations, chosen by the precision of the token inputs.
//   bf16 inputs: the MUFU forms above; their few-ulp error is far below the resolution of
//                a bf16 input.
//   fp32 inputs: CUDA's expf and log1pf with IEEE division.  Outputs of the mixer reach
//                tens of times their RMS and carry the relative error of u and delta
//                through the state sum, so the fp32 path keeps these to a few ulp.
template <typename Tin> __device__ __forceinline__ float silu_in(float x) { return silu(x); }
template <> __device__ __forceinline__ float silu_in<float>(float x) { return __fdiv_rn(x, 1.0f + expf(-x)); }
template <typename Tin> __device__ __forceinline__ float softplus_in(float v) { return softplus(v); }
template <> __device__ __forceinline__ float softplus_in<float>(float v) { return v > 20.0f ? v : log1pf(expf(v)); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once (no transaction bytes).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive once and add `bytes` to the transaction count the phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// Bounded wait for phase `parity` of `bar`.  Returns false if it did not
// complete within `limit_ns` nanoseconds of wall time (the caller then reports
// SSM_DEV_WAIT_TIMEOUT and leaves); never spins forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 255u) == 255u && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ------------------------------------------------------------------ TMA
// 3-D tiled tensor copy global -> shared, completing on `bar` (transaction bytes).
// The innermost coordinate c0 times the element size must be a multiple of 16
// bytes; callers pass channel offsets that are multiples of 32 elements and
// state offsets of 0.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

}  // namespace ssm
