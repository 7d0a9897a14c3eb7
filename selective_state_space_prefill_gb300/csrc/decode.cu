// decode.cu -- selective-SSM decode on sm_103a: T >= 1 tokens per request, in place on the
// cached states ("Scaling State-Space Models on Multiple GPUs with Tensor
// Parallelism", Methodology 3: the state cached at prefill is reused token by
// token without recomputing the prompt).
//
// Per request r and channel d (slot s = state_slot ? state_slot[r] : r):
//   xc = conv_b + w0 cs[s][0] + w1 cs[s][1] + w2 cs[s][2] + w3 x     (cs: last 3 raw inputs)
//   u = SiLU(xc), delta = softplus(dt + dt_bias)
//   h[n] = exp(delta A[n]) h[n] + delta B[n] u,  y = sum_n C[n] h[n] + D u
//   out = y SiLU(z);  cs[s] <- (cs[s][1], cs[s][2], x)
// for each of the request's T tokens in order (T = 1 is the classic decode step;
// T = 2..16 serves speculative / verification blocks).
//
// The step moves ~164 bytes per (request, channel) and needs ~110 instructions
// on them, so it is bound by HBM (and by launch latency at small batch).  One
// thread owns one (request, channel) and all 16 of its states: the per-token work
// is done once, the 64-byte state row moves as four 16-byte vectors, and a warp
// covers 32 consecutive channels (2 KB of contiguous state).  Channel parameters
// are re-read per request from L2; the grid walks requests in its y dimension.
#include "common.cuh"
#include "kernels.h"

namespace ssm {
namespace {

constexpr int kThreads = 128;           // channels per CTA

template <typename T> struct Vec4;
template <> struct Vec4<float> {
    static __device__ __forceinline__ float4 load(const float* p) { return *reinterpret_cast<const float4*>(p); }
};
template <> struct Vec4<__nv_bfloat16> {
    static __device__ __forceinline__ float4 load(const __nv_bfloat16* p) {
        const uint2 raw = *reinterpret_cast<const uint2*>(p);
        const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
        const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
        const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
        return make_float4(a.x, a.y, b.x, b.y);
    }
};

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads)
k_decode(const DecodeArgs p) {
    const int d = blockIdx.x * kThreads + threadIdx.x;
    const int r = blockIdx.y;
    if (d >= p.d_inner) return;
    const int slot = p.state_slot ? p.state_slot[r] : r;
    if (slot < 0 || slot >= p.n_slots) {
        atomicOr(p.status, 2u);
        return;
    }
    float* cs = p.conv_state + (int64_t)slot * 3 * p.conv_state_ld + d;
    float c0 = cs[0], c1 = cs[p.conv_state_ld], c2 = cs[2 * p.conv_state_ld];
    float4* hp = reinterpret_cast<float4*>(p.ssm_state + (int64_t)slot * p.ssm_state_stride_b + (int64_t)d * 16);
    float4 h[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) h[q] = hp[q];
    float4 A2[4];
    const float4* Ar = reinterpret_cast<const float4*>(p.A + (int64_t)d * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 a = Ar[q];
        A2[q] = make_float4(a.x * kLog2e, a.y * kLog2e, a.z * kLog2e, a.w * kLog2e);
    }
    const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (int64_t)d * 4);
    const float cb = p.conv_b[d], Dd = p.Dskip[d], bias = p.dt_bias[d];

    // the next token's x, z, dt are loaded while the current one is computed
    const Tin* xg = reinterpret_cast<const Tin*>(p.x) + (int64_t)r * p.in_stride_b + d;
    const Tin* zg = reinterpret_cast<const Tin*>(p.z) + (int64_t)r * p.in_stride_b + d;
    const Tin* dg = reinterpret_cast<const Tin*>(p.dt) + (int64_t)r * p.in_stride_b + d;
    Tin xn = xg[0], zn = zg[0], dn = dg[0];
    for (int t = 0; t < p.n_tokens; ++t) {
        const float xt = to_f32(xn), zt = to_f32(zn), dtt = to_f32(dn);
        if (t + 1 < p.n_tokens) {
            const int64_t o = (int64_t)(t + 1) * p.in_stride_t;
            xn = xg[o];
            zn = zg[o];
            dn = dg[o];
        }
        const Tin* Bm = reinterpret_cast<const Tin*>(p.Bm) + ((int64_t)r * p.n_tokens + t) * 16;
        const Tin* Cm = reinterpret_cast<const Tin*>(p.Cm) + ((int64_t)r * p.n_tokens + t) * 16;

        float xc = fmaf(w.x, c0, cb);
        xc = fmaf(w.y, c1, xc);
        xc = fmaf(w.z, c2, xc);
        xc = fmaf(w.w, xt, xc);
        c0 = c1;
        c1 = c2;
        c2 = xt;
        const float u = silu_in<Tin>(xc);
        const float delta = softplus_in<Tin>(dtt + bias);
        const float du = delta * u;
        float y = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 Bq = Vec4<Tin>::load(Bm + 4 * q);
            const float4 Cq = Vec4<Tin>::load(Cm + 4 * q);
            float4 hv = h[q];
            hv.x = fmaf(ex2(delta * A2[q].x), hv.x, du * Bq.x);
            hv.y = fmaf(ex2(delta * A2[q].y), hv.y, du * Bq.y);
            hv.z = fmaf(ex2(delta * A2[q].z), hv.z, du * Bq.z);
            hv.w = fmaf(ex2(delta * A2[q].w), hv.w, du * Bq.w);
            h[q] = hv;
            y = fmaf(Cq.x, hv.x, y);
            y = fmaf(Cq.y, hv.y, y);
            y = fmaf(Cq.z, hv.z, y);
            y = fmaf(Cq.w, hv.w, y);
        }
        y = fmaf(Dd, u, y);
        reinterpret_cast<Tout*>(p.out)[(int64_t)r * p.out_stride_b + (int64_t)t * p.out_stride_t + d] =
            from_f32<Tout>(y * silu_in<Tin>(zt));
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) hp[q] = h[q];
    cs[0] = c0;
    cs[p.conv_state_ld] = c1;
    cs[2 * p.conv_state_ld] = c2;
}

}  // namespace

int launch_decode(const DecodeArgs& a, bool in_bf16, bool out_bf16, cudaStream_t stream, const char** why) {
    if (a.batch > 65535) {
        *why = "batch above 65535";
        return -1;
    }
    dim3 grid((a.d_inner + kThreads - 1) / kThreads, a.batch);
    if (in_bf16) {
        if (out_bf16) k_decode<__nv_bfloat16, __nv_bfloat16><<<grid, kThreads, 0, stream>>>(a);
        else k_decode<__nv_bfloat16, float><<<grid, kThreads, 0, stream>>>(a);
    } else {
        if (out_bf16) k_decode<float, __nv_bfloat16><<<grid, kThreads, 0, stream>>>(a);
        else k_decode<float, float><<<grid, kThreads, 0, stream>>>(a);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return -1;
    }
    return 0;
}

}  // namespace ssm
