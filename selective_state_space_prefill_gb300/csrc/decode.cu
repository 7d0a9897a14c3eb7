// decode.cu -- one-token selective-SSM decode step on sm_103a, in place on the
// cached states ("Scaling State-Space Models on Multiple GPUs with Tensor
// Parallelism", Methodology 3: the state cached at prefill is reused token by
// token without recomputing the prompt).
//
// Per request r and channel d (slot s = state_slot ? state_slot[r] : r):
//   xc = conv_b + w0 cs[s][0] + w1 cs[s][1] + w2 cs[s][2] + w3 x     (cs: last 3 raw inputs)
//   u = SiLU(xc), delta = softplus(dt + dt_bias)
//   h[n] = exp(delta A[n]) h[n] + delta B[n] u,  y = sum_n C[n] h[n] + D u
//   out = y SiLU(z);  cs[s] <- (cs[s][1], cs[s][2], x)
//
// The step moves ~160 bytes per (request, channel) and does ~100 flops on
// them, so it is bound by HBM (and by launch latency at small batch).  Four
// lanes share a channel, each owning four of the 16 states, so the state row
// (64 B) is read and written as one 16-byte vector per lane and a warp touches
// 512 contiguous bytes; the partial readouts meet through two shuffles.
#include "common.cuh"
#include "kernels.h"

namespace ssm {
namespace {

constexpr int kThreads = 128;           // 32 channels x 4 lanes
constexpr int kChanPerCta = kThreads / 4;
constexpr int kReqPerCta = 4;           // requests walked by each CTA (parameters stay in registers)

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
    const int lane = threadIdx.x & 31;
    const int q = threadIdx.x & 3;                         // state quad: states 4q .. 4q+3
    const int d = blockIdx.x * kChanPerCta + (threadIdx.x >> 2);
    if (d >= p.d_inner) return;                            // whole 4-lane groups leave together
    const unsigned gmask = 0xFu << (lane & ~3);

    const float4 Aq = *reinterpret_cast<const float4*>(p.A + (int64_t)d * 16 + 4 * q);
    const float A2[4] = {Aq.x * kLog2e, Aq.y * kLog2e, Aq.z * kLog2e, Aq.w * kLog2e};
    const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (int64_t)d * 4);
    const float cb = p.conv_b[d], Dd = p.Dskip[d], bias = p.dt_bias[d];

    const int r0 = blockIdx.y * kReqPerCta;
#pragma unroll
    for (int rr = 0; rr < kReqPerCta; ++rr) {
        const int r = r0 + rr;
        if (r >= p.batch) break;
        const int slot = p.state_slot ? p.state_slot[r] : r;
        if (slot < 0 || slot >= p.n_slots) {
            if (q == 0) atomicOr(p.status, 2u);
            continue;
        }
        const Tin* xr = reinterpret_cast<const Tin*>(p.x) + (int64_t)r * p.in_stride_b + d;
        const float xt = to_f32(*xr);
        const float zt = to_f32(*(reinterpret_cast<const Tin*>(p.z) + (int64_t)r * p.in_stride_b + d));
        const float dtt = to_f32(*(reinterpret_cast<const Tin*>(p.dt) + (int64_t)r * p.in_stride_b + d));

        // conv window: lanes 0..2 of the group each hold one of the three cached inputs
        float* cs = p.conv_state + (int64_t)slot * 3 * p.conv_state_ld + d;
        const float mine = q < 3 ? cs[(int64_t)q * p.conv_state_ld] : 0.f;
        const int base = lane & ~3;
        const float c0 = __shfl_sync(gmask, mine, base + 0);
        const float c1 = __shfl_sync(gmask, mine, base + 1);
        const float c2 = __shfl_sync(gmask, mine, base + 2);
        float xc = fmaf(w.x, c0, cb);
        xc = fmaf(w.y, c1, xc);
        xc = fmaf(w.z, c2, xc);
        xc = fmaf(w.w, xt, xc);
        const float u = silu(xc);
        const float delta = softplus(dtt + bias);
        const float du = delta * u;

        const float4 Bq = Vec4<Tin>::load(reinterpret_cast<const Tin*>(p.Bm) + (int64_t)r * 16 + 4 * q);
        const float4 Cq = Vec4<Tin>::load(reinterpret_cast<const Tin*>(p.Cm) + (int64_t)r * 16 + 4 * q);
        float4* hp = reinterpret_cast<float4*>(p.ssm_state + (int64_t)slot * p.ssm_state_stride_b +
                                               (int64_t)d * 16 + 4 * q);
        float4 h = *hp;
        h.x = fmaf(ex2(delta * A2[0]), h.x, du * Bq.x);
        h.y = fmaf(ex2(delta * A2[1]), h.y, du * Bq.y);
        h.z = fmaf(ex2(delta * A2[2]), h.z, du * Bq.z);
        h.w = fmaf(ex2(delta * A2[3]), h.w, du * Bq.w);
        *hp = h;
        float y = Cq.x * h.x;
        y = fmaf(Cq.y, h.y, y);
        y = fmaf(Cq.z, h.z, y);
        y = fmaf(Cq.w, h.w, y);
        y += __shfl_xor_sync(gmask, y, 1);
        y += __shfl_xor_sync(gmask, y, 2);

        if (q == 0) {
            y = fmaf(Dd, u, y);
            Tout* o = reinterpret_cast<Tout*>(p.out) + (int64_t)r * p.out_stride_b + d;
            *o = from_f32<Tout>(y * silu(zt));
        }
        if (q < 3) cs[(int64_t)q * p.conv_state_ld] = q == 0 ? c1 : (q == 1 ? c2 : xt);
    }
}

}  // namespace

int launch_decode(const DecodeArgs& a, bool in_bf16, bool out_bf16, cudaStream_t stream, const char** why) {
    dim3 grid((a.d_inner + kChanPerCta - 1) / kChanPerCta, (a.batch + kReqPerCta - 1) / kReqPerCta);
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
