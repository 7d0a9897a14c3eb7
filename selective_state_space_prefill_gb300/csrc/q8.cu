// q8.cu -- local 8-bit quantized reduction of P partial buffers on sm_103a.
//
// The arithmetic of the quantized all-reduce in "Scaling State-Space Models on
// Multiple GPUs with Tensor Parallelism" (Methodology 4: quantize partials to
// 8 bits, sum, dequantize), done over P buffers already in this GPU's HBM.
// Per block of 128 elements, one scale shared by the P partials:
//   amax = max |x_p[i]|;  inv = 127/amax;  scale = amax/127     (IEEE fp32 division)
//   q_p[i] = rne(x_p[i] * inv) in [-127, 127];  S[i] = sum_p q_p[i];  out[i] = S[i] * scale
// Every fp32 step is a correctly rounded operation (__fdiv_rn, __fmul_rn,
// __float2int_rn, __int2float_rn), so S and scale are bit-identical to any
// IEEE-fp32 evaluation of the same steps.
//
// One warp per block: lane l owns elements 4l .. 4l+3 of every partial, loaded
// as one 8-byte (bf16) or 16-byte (fp32) vector; the block maximum is a 5-step
// shuffle reduction.  Pure streaming: read P*2 bytes, write 2-4 bytes per element.
#include "common.cuh"
#include "kernels.h"

namespace ssm {
namespace {

constexpr int kBlock = 128;
constexpr int kThreads = 256;   // 8 blocks of 128 elements per CTA

__device__ __forceinline__ void load4(const float* p, int64_t i, int64_t n, float v[4]) {
    if (i + 3 < n) {
        const float4 t = *reinterpret_cast<const float4*>(p + i);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = i + e < n ? p[i + e] : 0.f;
    }
}

__device__ __forceinline__ void load4(const __nv_bfloat16* p, int64_t i, int64_t n, float v[4]) {
    if (i + 3 < n) {
        const uint2 raw = *reinterpret_cast<const uint2*>(p + i);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = i + e < n ? __bfloat162float(p[i + e]) : 0.f;
    }
}

__device__ __forceinline__ void store4(float* p, int64_t i, int64_t n, const float o[4]) {
    if (i + 3 < n) {
        *reinterpret_cast<float4*>(p + i) = make_float4(o[0], o[1], o[2], o[3]);
    } else {
        for (int e = 0; e < 4; ++e)
            if (i + e < n) p[i + e] = o[e];
    }
}

__device__ __forceinline__ void store4(__nv_bfloat16* p, int64_t i, int64_t n, const float o[4]) {
    if (i + 3 < n) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(o[0], o[1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(o[2], o[3]);
        uint2 raw;
        raw.x = *reinterpret_cast<uint32_t*>(&lo);
        raw.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(p + i) = raw;
    } else {
        for (int e = 0; e < 4; ++e)
            if (i + e < n) p[i + e] = __float2bfloat16_rn(o[e]);
    }
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads)
k_q8(const Q8Args a) {
    const int64_t blk = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (blk * kBlock >= a.n) return;
    const int64_t i0 = blk * kBlock + 4 * lane;

    float v[kMaxPartials][4];
    float amax = 0.f;
#pragma unroll
    for (int p = 0; p < kMaxPartials; ++p) {
        if (p < a.P) {
            load4(reinterpret_cast<const Tin*>(a.partials[p]), i0, a.n, v[p]);
#pragma unroll
            for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(v[p][e]));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));

    float inv = 0.f, scale = 0.f;
    if (amax > 0.f) {
        inv = __fdiv_rn(127.0f, amax);
        scale = __fdiv_rn(amax, 127.0f);
    }
    int s[4] = {0, 0, 0, 0};
    if (amax > 0.f) {
#pragma unroll
        for (int p = 0; p < kMaxPartials; ++p) {
            if (p < a.P) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int qv = __float2int_rn(__fmul_rn(v[p][e], inv));
                    qv = qv > 127 ? 127 : (qv < -127 ? -127 : qv);
                    s[e] += qv;
                }
            }
        }
    }
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = __fmul_rn(__int2float_rn(s[e]), scale);
    store4(reinterpret_cast<Tout*>(a.out), i0, a.n, o);
    if (a.sums) {
        if (i0 + 3 < a.n) {
            *reinterpret_cast<int4*>(a.sums + i0) = make_int4(s[0], s[1], s[2], s[3]);
        } else {
            for (int e = 0; e < 4; ++e)
                if (i0 + e < a.n) a.sums[i0 + e] = s[e];
        }
    }
    if (a.scales && lane == 0) a.scales[blk] = scale;
}

}  // namespace

int launch_q8(const Q8Args& a, bool in_bf16, bool out_bf16, cudaStream_t stream, const char** why) {
    const int64_t nblk = (a.n + kBlock - 1) / kBlock;
    const int64_t ctas = (nblk + kThreads / 32 - 1) / (kThreads / 32);
    if (ctas > 0x7fffffff) {
        *why = "n too large for one launch";
        return -1;
    }
    dim3 grid((unsigned)ctas);
    if (in_bf16) {
        if (out_bf16) k_q8<__nv_bfloat16, __nv_bfloat16><<<grid, kThreads, 0, stream>>>(a);
        else k_q8<__nv_bfloat16, float><<<grid, kThreads, 0, stream>>>(a);
    } else {
        if (out_bf16) k_q8<float, __nv_bfloat16><<<grid, kThreads, 0, stream>>>(a);
        else k_q8<float, float><<<grid, kThreads, 0, stream>>>(a);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return -1;
    }
    return 0;
}

}  // namespace ssm
