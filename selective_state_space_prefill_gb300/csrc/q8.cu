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
// Layout: 16 lanes per 128-element block, each lane owning 8 consecutive
// elements of every partial (one 16-byte load per bf16 partial, two per fp32
// partial), so a warp covers two blocks and keeps P x 16 bytes per lane in
// flight; the block maximum is a 4-step shuffle reduction inside the half-warp.
// Pure streaming: read P*2 bytes, write 2-4 (+4 for the sums) bytes per element.
#include "common.cuh"
#include "kernels.h"

namespace ssm {
namespace {

constexpr int kBlock = 128;
constexpr int kVec = 8;                     // elements per lane
constexpr int kLanesPerBlock = kBlock / kVec;   // 16
constexpr int kThreads = 256;               // 16 blocks of 128 elements per CTA

__device__ __forceinline__ void load8(const float* p, int64_t i, int64_t n, float v[kVec]) {
    if (i + kVec - 1 < n) {
        const float4 a = *reinterpret_cast<const float4*>(p + i);
        const float4 b = *reinterpret_cast<const float4*>(p + i + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e) v[e] = i + e < n ? p[i + e] : 0.f;
    }
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, int64_t i, int64_t n, float v[kVec]) {
    if (i + kVec - 1 < n) {
        const uint4 raw = *reinterpret_cast<const uint4*>(p + i);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
            v[2 * k] = f.x;
            v[2 * k + 1] = f.y;
        }
    } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e) v[e] = i + e < n ? __bfloat162float(p[i + e]) : 0.f;
    }
}

__device__ __forceinline__ void store8(float* p, int64_t i, int64_t n, const float o[kVec]) {
    if (i + kVec - 1 < n) {
        *reinterpret_cast<float4*>(p + i) = make_float4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<float4*>(p + i + 4) = make_float4(o[4], o[5], o[6], o[7]);
    } else {
        for (int e = 0; e < kVec; ++e)
            if (i + e < n) p[i + e] = o[e];
    }
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, int64_t i, int64_t n, const float o[kVec]) {
    if (i + kVec - 1 < n) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * k], o[2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(p + i) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        for (int e = 0; e < kVec; ++e)
            if (i + e < n) p[i + e] = __float2bfloat16_rn(o[e]);
    }
}

template <typename Tin, typename Tout, int P>
__global__ void __launch_bounds__(kThreads)
k_q8(const Q8Args a) {
    const int64_t blk = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / kLanesPerBlock;
    const int sub = threadIdx.x % kLanesPerBlock;
    // Every lane takes part in the shuffles; lanes of a block past n just see zeros.
    const int64_t i0 = blk * kBlock + kVec * sub;

    float v[P][kVec];
    float amax = 0.f;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        load8(reinterpret_cast<const Tin*>(a.partials[p]), i0, a.n, v[p]);
#pragma unroll
        for (int e = 0; e < kVec; ++e) amax = fmaxf(amax, fabsf(v[p][e]));
    }
#pragma unroll
    for (int off = kLanesPerBlock / 2; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (i0 >= a.n) return;

    float inv = 0.f, scale = 0.f;
    if (amax > 0.f) {
        inv = __fdiv_rn(127.0f, amax);
        scale = __fdiv_rn(amax, 127.0f);
    }
    int s[kVec];
#pragma unroll
    for (int e = 0; e < kVec; ++e) s[e] = 0;
    if (amax > 0.f) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
#pragma unroll
            for (int e = 0; e < kVec; ++e) {
                int qv = __float2int_rn(__fmul_rn(v[p][e], inv));
                qv = qv > 127 ? 127 : (qv < -127 ? -127 : qv);
                s[e] += qv;
            }
        }
    }
    float o[kVec];
#pragma unroll
    for (int e = 0; e < kVec; ++e) o[e] = __fmul_rn(__int2float_rn(s[e]), scale);
    store8(reinterpret_cast<Tout*>(a.out), i0, a.n, o);
    if (a.sums) {
        if (i0 + kVec - 1 < a.n) {
            *reinterpret_cast<int4*>(a.sums + i0) = make_int4(s[0], s[1], s[2], s[3]);
            *reinterpret_cast<int4*>(a.sums + i0 + 4) = make_int4(s[4], s[5], s[6], s[7]);
        } else {
            for (int e = 0; e < kVec; ++e)
                if (i0 + e < a.n) a.sums[i0 + e] = s[e];
        }
    }
    if (a.scales && sub == 0) a.scales[blk] = scale;
}

}  // namespace

int launch_q8(const Q8Args& a, bool in_bf16, bool out_bf16, cudaStream_t stream, const char** why) {
    const int64_t nblk = (a.n + kBlock - 1) / kBlock;
    const int64_t blocks_per_cta = kThreads / kLanesPerBlock;
    const int64_t ctas = (nblk + blocks_per_cta - 1) / blocks_per_cta;
    if (ctas > 0x7fffffff) {
        *why = "n too large for one launch";
        return -1;
    }
    dim3 grid((unsigned)ctas);
    // one instantiation per partial count, so the value registers match P exactly
    switch (a.P) {
#define SSM_Q8_CASE(PP)                                                                              \
        case PP:                                                                                   \
            if (in_bf16) {                                                                         \
                if (out_bf16) k_q8<__nv_bfloat16, __nv_bfloat16, PP><<<grid, kThreads, 0, stream>>>(a); \
                else k_q8<__nv_bfloat16, float, PP><<<grid, kThreads, 0, stream>>>(a);              \
            } else {                                                                               \
                if (out_bf16) k_q8<float, __nv_bfloat16, PP><<<grid, kThreads, 0, stream>>>(a);     \
                else k_q8<float, float, PP><<<grid, kThreads, 0, stream>>>(a);                      \
            }                                                                                      \
            break;
        SSM_Q8_CASE(1) SSM_Q8_CASE(2) SSM_Q8_CASE(3) SSM_Q8_CASE(4)
        SSM_Q8_CASE(5) SSM_Q8_CASE(6) SSM_Q8_CASE(7) SSM_Q8_CASE(8)
#undef SSM_Q8_CASE
        default:
            *why = "P out of range";
            return -1;
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return -1;
    }
    return 0;
}

}  // namespace ssm
