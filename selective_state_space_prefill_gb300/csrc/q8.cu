// q8.cu -- local 8-bit quantized reduction of P partial buffers on sm_103a.
//
// The arithmetic of the quantized all-reduce in "Scaling State-Space Models on
// Multiple GPUs with Tensor Parallelism" (Methodology 4: quantize partials to
// 8 bits, sum, dequantize), done over P buffers already in this GPU's HBM.
// Per block of 128 elements, one scale shared by the P partials:
//   amax = max |x_p[i]|;  inv = 127/amax;  scale = amax/127     (IEEE fp32 division)
//   q_p[i] = rne(x_p[i] * inv) in [-127, 127];  S[i] = sum_p q_p[i];  out[i] = S[i] * scale
// Every fp32 step is a correctly rounded operation, so S and scale are
// bit-identical to any IEEE-fp32 evaluation of the same steps.
//
// Layout: 16 lanes per 128-element block, each lane owning 8 consecutive
// elements of every partial (one 16-byte load per bf16 partial, two per fp32
// partial), so a warp covers two blocks.  The partials stay in registers as the
// raw 32-bit words they were loaded as (two bf16 per word), which keeps the
// register count low enough for 6 CTAs of 256 threads per SM and so more bytes
// in flight: the kernel is bound by HBM latency x bytes in flight.
//
// Rounding: for a block of finite values, fl(x * inv) lies within 127.5 in
// magnitude (|x| <= amax, so x * inv <= 127 (1 + 2^-24)), and adding 1.5 * 2^23
// to it in fp32 rounds it to an integer, ties to even, in the low mantissa bits
// of the sum; the bits of the P sums are added as integers.  The clamp to
// [-127, 127] is therefore never active for finite blocks.  The multiply and the
// add are the scalar __fmul_rn / __fadd_rn, which are never contracted into a
// fused multiply-add (that would round the unrounded product and break ties).
// A block holding an Inf or NaN (detected by a NaN-propagating maximum) takes
// the plain path: NaN-ignoring maximum, round-to-nearest-even conversion and
// clamp.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace ssm {
namespace {

constexpr int kBlock = 128;
constexpr int kVec = 8;                         // elements per lane
constexpr int kLanesPerBlock = kBlock / kVec;   // 16
constexpr int kThreads = 256;                   // 16 blocks of 128 elements per CTA
constexpr uint32_t kMagicBits = 0x4B400000u;    // bits of 1.5 * 2^23
constexpr float kMagic = 12582912.0f;           // 1.5 * 2^23

// |a| and the NaN-propagating maximum of two bf16 pairs, exact.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t m, uint32_t w) {
    uint32_t a, r;
    asm("abs.bf16x2 %0, %1;" : "=r"(a) : "r"(w));
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(a));
    return r;
}
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float lo_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// kVec elements starting at i as raw 32-bit words; elements at or past n read as 0.
template <typename Tin>
__device__ __forceinline__ void load_words(const Tin* p, int64_t i, int64_t n, uint32_t* w) {
    constexpr int NW = kVec * (int)sizeof(Tin) / 4;
    if (i + kVec <= n) {
#pragma unroll
        for (int k = 0; k < NW / 4; ++k) {
            const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p + i) + k);
            w[4 * k] = u.x;
            w[4 * k + 1] = u.y;
            w[4 * k + 2] = u.z;
            w[4 * k + 3] = u.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            if constexpr (sizeof(Tin) == 2) {
                const uint16_t* h = reinterpret_cast<const uint16_t*>(p);
                const uint32_t lo = i + 2 * k < n ? h[i + 2 * k] : 0u;
                const uint32_t hi = i + 2 * k + 1 < n ? h[i + 2 * k + 1] : 0u;
                w[k] = lo | (hi << 16);
            } else {
                const uint32_t* f = reinterpret_cast<const uint32_t*>(p);
                w[k] = i + k < n ? f[i + k] : 0u;
            }
        }
    }
}

// Element e of the lane's words, widened to fp32 (exact).
template <typename Tin>
__device__ __forceinline__ float elem(const uint32_t* w, int e) {
    if constexpr (sizeof(Tin) == 2) return (e & 1) ? hi_f32(w[e >> 1]) : lo_f32(w[e >> 1]);
    else return __uint_as_float(w[e]);
}

__device__ __forceinline__ void store8(float* p, int64_t i, int64_t n, const float o[kVec]) {
    if (i + kVec <= n) {
        __stcs(reinterpret_cast<float4*>(p + i), make_float4(o[0], o[1], o[2], o[3]));
        __stcs(reinterpret_cast<float4*>(p + i) + 1, make_float4(o[4], o[5], o[6], o[7]));
    } else {
        for (int e = 0; e < kVec; ++e)
            if (i + e < n) p[i + e] = o[e];
    }
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, int64_t i, int64_t n, const float o[kVec]) {
    if (i + kVec <= n) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * k], o[2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        __stcs(reinterpret_cast<uint4*>(p + i), make_uint4(w[0], w[1], w[2], w[3]));
    } else {
        for (int e = 0; e < kVec; ++e)
            if (i + e < n) p[i + e] = __float2bfloat16_rn(o[e]);
    }
}

template <typename Tin, typename Tout, int P>
__global__ void __launch_bounds__(kThreads)
k_q8(const Q8Args a) {
    constexpr int NW = kVec * (int)sizeof(Tin) / 4;     // words per lane per partial
    const int64_t blk = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / kLanesPerBlock;
    const int lane = threadIdx.x & 31;
    const int sub = lane % kLanesPerBlock;
    // Every lane takes part in the shuffles; lanes of a block past n just see zeros.
    const int64_t i0 = blk * kBlock + kVec * sub;

    uint32_t w[P][NW];
#pragma unroll
    for (int p = 0; p < P; ++p) load_words<Tin>(reinterpret_cast<const Tin*>(a.partials[p]), i0, a.n, w[p]);

    // block maximum of |x|, NaN-propagating so that a non-finite value shows
    float amax;
    if constexpr (sizeof(Tin) == 2) {
        uint32_t m = 0;
#pragma unroll
        for (int p = 0; p < P; ++p)
#pragma unroll
            for (int k = 0; k < NW; ++k) m = absmax_bf16x2(m, w[p][k]);
        amax = max_nan(lo_f32(m), hi_f32(m));
    } else {
        amax = 0.f;
#pragma unroll
        for (int p = 0; p < P; ++p)
#pragma unroll
            for (int k = 0; k < NW; ++k) amax = max_nan(amax, fabsf(__uint_as_float(w[p][k])));
    }
#pragma unroll
    for (int off = kLanesPerBlock / 2; off > 0; off >>= 1)
        amax = max_nan(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const bool finite = amax <= FLT_MAX;          // the same in every lane of the block
    if (!finite) {
        // Inf or NaN in the block: the NaN-ignoring maximum, over this block's lanes only
        const unsigned gmask = 0xffffu << (lane & ~(kLanesPerBlock - 1));
        amax = 0.f;
#pragma unroll
        for (int p = 0; p < P; ++p)
#pragma unroll
            for (int e = 0; e < kVec; ++e) amax = fmaxf(amax, fabsf(elem<Tin>(w[p], e)));
#pragma unroll
        for (int off = kLanesPerBlock / 2; off > 0; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, off));
    }
    if (i0 >= a.n) return;

    float inv = 0.f, scale = 0.f;
    if (amax > 0.f) {
        inv = __fdiv_rn(127.0f, amax);
        scale = __fdiv_rn(amax, 127.0f);
    }
    int s[kVec];
    float o[kVec];
    if (finite) {
        // bits(fl(fl(x * inv) + 1.5 * 2^23)) = kMagicBits + q; an all-zero block has inv = 0, q = 0
        uint32_t acc[kVec];
#pragma unroll
        for (int e = 0; e < kVec; ++e) acc[e] = 0u;
#pragma unroll
        for (int p = 0; p < P; ++p)
#pragma unroll
            for (int e = 0; e < kVec; ++e)
                acc[e] += __float_as_uint(__fadd_rn(__fmul_rn(elem<Tin>(w[p], e), inv), kMagic));
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            const uint32_t bits = acc[e] - (uint32_t)(P - 1) * kMagicBits;   // kMagicBits + S, |S| <= 1016
            s[e] = (int)(bits - kMagicBits);
            o[e] = __fmul_rn(__fadd_rn(__uint_as_float(bits), -kMagic), scale);   // float(S) is exact
        }
    } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e) s[e] = 0;
        if (amax > 0.f) {
#pragma unroll
            for (int p = 0; p < P; ++p)
#pragma unroll
                for (int e = 0; e < kVec; ++e) {
                    int qv = __float2int_rn(__fmul_rn(elem<Tin>(w[p], e), inv));
                    qv = qv > 127 ? 127 : (qv < -127 ? -127 : qv);
                    s[e] += qv;
                }
        }
#pragma unroll
        for (int e = 0; e < kVec; ++e) o[e] = __fmul_rn(__int2float_rn(s[e]), scale);
    }
    store8(reinterpret_cast<Tout*>(a.out), i0, a.n, o);
    if (a.sums) {
        if (i0 + kVec <= a.n) {
            __stcs(reinterpret_cast<int4*>(a.sums + i0), make_int4(s[0], s[1], s[2], s[3]));
            __stcs(reinterpret_cast<int4*>(a.sums + i0) + 1, make_int4(s[4], s[5], s[6], s[7]));
        } else {
            for (int e = 0; e < kVec; ++e)
                if (i0 + e < a.n) a.sums[i0 + e] = s[e];
        }
    }
    if (a.scales && sub == 0) a.scales[blk] = scale;
}

// ------------------------------------------------------------------ rank-local halves
// A tensor-parallel rank cannot run k_q8 on the other ranks' partials: it sees only its own.
// The same arithmetic then splits into (1) the rank's block maxima (k_q8_absmax; the
// out_proj kernel emits them too), (2) after a MAX all-reduce of those maxima, the rank's
// int8 codes with the shared per-block scale (k_q8_quantize), and (3) after the ranks'
// codes are gathered, the int32 sums and the dequantized output (k_q8_sum).  Every step is
// the same correctly rounded fp32 operation as in k_q8, so (3) o (2) o max(1) reproduces
// k_q8's sums, scales and outputs bit for bit.

// Blocks per 16-lane group in the two single-partial kernels: one lane then has kGroupBlocks
// independent 16-byte loads in flight, as the P-partial kernels have P.
constexpr int kGroupBlocks = 4;

// amax[j] = max |x_i| over block j (a NaN is ignored, an infinity kept).
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
k_q8_absmax(const void* x, int64_t n, float* amax) {
    constexpr int NW = kVec * (int)sizeof(Tin) / 4;
    const int64_t grp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / kLanesPerBlock;
    const int sub = (threadIdx.x & 31) % kLanesPerBlock;
    uint32_t w[kGroupBlocks][NW];
#pragma unroll
    for (int j = 0; j < kGroupBlocks; ++j)
        load_words<Tin>(reinterpret_cast<const Tin*>(x), (grp * kGroupBlocks + j) * kBlock + kVec * sub, n, w[j]);
#pragma unroll
    for (int j = 0; j < kGroupBlocks; ++j) {
        const int64_t blk = grp * kGroupBlocks + j;
        float m = 0.f;
#pragma unroll
        for (int e = 0; e < kVec; ++e) m = fmaxf(m, fabsf(elem<Tin>(w[j], e)));
#pragma unroll
        for (int off = kLanesPerBlock / 2; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (sub == 0 && blk * kBlock < n) amax[blk] = m;
    }
}

// codes[i] = clamp(rne(x_i * inv_j), -127, 127), inv_j = 127 / amax[j] (0 when amax[j] is 0 or
// not a number); scales[j] = amax[j] / 127 (0 likewise).
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
k_q8_quantize(const void* x, int64_t n, const float* amax_in, int8_t* codes, float* scales) {
    constexpr int NW = kVec * (int)sizeof(Tin) / 4;
    const int64_t grp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / kLanesPerBlock;
    const int sub = (threadIdx.x & 31) % kLanesPerBlock;
    uint32_t w[kGroupBlocks][NW];
    float am[kGroupBlocks];
#pragma unroll
    for (int j = 0; j < kGroupBlocks; ++j) {
        const int64_t blk = grp * kGroupBlocks + j;
        load_words<Tin>(reinterpret_cast<const Tin*>(x), blk * kBlock + kVec * sub, n, w[j]);
        am[j] = blk * kBlock < n ? __ldg(amax_in + blk) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kGroupBlocks; ++j) {
        const int64_t blk = grp * kGroupBlocks + j;
        const int64_t i0 = blk * kBlock + kVec * sub;
        if (i0 >= n) break;
        float inv = 0.f, scale = 0.f;
        if (am[j] > 0.f) {
            inv = __fdiv_rn(127.0f, am[j]);
            scale = __fdiv_rn(am[j], 127.0f);
        }
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            int qv = __float2int_rn(__fmul_rn(elem<Tin>(w[j], e), inv));   // a NaN converts to 0
            qv = qv > 127 ? 127 : (qv < -127 ? -127 : qv);
            packed[e >> 2] |= ((uint32_t)qv & 0xffu) << (8 * (e & 3));
        }
        if (i0 + kVec <= n) {
            __stcs(reinterpret_cast<uint2*>(codes + i0), make_uint2(packed[0], packed[1]));
        } else {
            for (int e = 0; e < kVec; ++e)
                if (i0 + e < n) codes[i0 + e] = (int8_t)((packed[e >> 2] >> (8 * (e & 3))) & 0xffu);
        }
        if (scales && sub == 0) scales[blk] = scale;
    }
}

struct Q8SumArgs {
    const int8_t* codes[kMaxPartials];
    const float* scales;
    int64_t n;
    void* out;
    int32_t* sums;
};

// S[i] = sum_p codes_p[i] (int32), out[i] = float(S[i]) * scale_j.
template <typename Tout, int P>
__global__ void __launch_bounds__(kThreads)
k_q8_sum(const Q8SumArgs a) {
    const int64_t blk = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / kLanesPerBlock;
    const int sub = (threadIdx.x & 31) % kLanesPerBlock;
    const int64_t i0 = blk * kBlock + kVec * sub;
    if (i0 >= a.n) return;
    int s[kVec];
#pragma unroll
    for (int e = 0; e < kVec; ++e) s[e] = 0;
    const bool whole = i0 + kVec <= a.n;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        uint32_t w0 = 0u, w1 = 0u;
        if (whole) {
            const uint2 u = __ldcs(reinterpret_cast<const uint2*>(a.codes[p] + i0));
            w0 = u.x;
            w1 = u.y;
        } else {
            for (int e = 0; e < kVec; ++e)
                if (i0 + e < a.n) {
                    const uint32_t byte = (uint32_t)(uint8_t)a.codes[p][i0 + e];
                    if (e < 4) w0 |= byte << (8 * e);
                    else w1 |= byte << (8 * (e - 4));
                }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            s[e] += (int)(w0 << (24 - 8 * e)) >> 24;                 // sign-extended byte e
            s[4 + e] += (int)(w1 << (24 - 8 * e)) >> 24;
        }
    }
    const float scale = __ldg(a.scales + blk);
    float o[kVec];
#pragma unroll
    for (int e = 0; e < kVec; ++e) o[e] = __fmul_rn(__int2float_rn(s[e]), scale);   // float(S) is exact
    store8(reinterpret_cast<Tout*>(a.out), i0, a.n, o);
    if (a.sums) {
        if (whole) {
            __stcs(reinterpret_cast<int4*>(a.sums + i0), make_int4(s[0], s[1], s[2], s[3]));
            __stcs(reinterpret_cast<int4*>(a.sums + i0) + 1, make_int4(s[4], s[5], s[6], s[7]));
        } else {
            for (int e = 0; e < kVec; ++e)
                if (i0 + e < a.n) a.sums[i0 + e] = s[e];
        }
    }
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
    // one instantiation per partial count, so the word registers match P exactly
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

// One launch covers ceil(n / 128) blocks of 128 elements, 16 blocks per CTA.
static bool q8_grid(int64_t n, dim3* grid, const char** why) {
    const int64_t nblk = (n + kBlock - 1) / kBlock;
    const int64_t ctas = (nblk + kThreads / kLanesPerBlock - 1) / (kThreads / kLanesPerBlock);
    if (ctas > 0x7fffffff) {
        *why = "n too large for one launch";
        return false;
    }
    *grid = dim3((unsigned)ctas);
    return true;
}

static int q8_launched(const char** why) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return -1;
    }
    return 0;
}

int launch_q8_absmax(const void* x, bool in_bf16, int64_t n, float* amax, cudaStream_t stream, const char** why) {
    dim3 grid;
    if (!q8_grid((n + kGroupBlocks - 1) / kGroupBlocks, &grid, why)) return -1;
    if (in_bf16) k_q8_absmax<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(x, n, amax);
    else k_q8_absmax<float><<<grid, kThreads, 0, stream>>>(x, n, amax);
    return q8_launched(why);
}

int launch_q8_quantize(const void* x, bool in_bf16, int64_t n, const float* amax, int8_t* codes, float* scales,
                       cudaStream_t stream, const char** why) {
    dim3 grid;
    if (!q8_grid((n + kGroupBlocks - 1) / kGroupBlocks, &grid, why)) return -1;
    if (in_bf16) k_q8_quantize<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(x, n, amax, codes, scales);
    else k_q8_quantize<float><<<grid, kThreads, 0, stream>>>(x, n, amax, codes, scales);
    return q8_launched(why);
}

int launch_q8_sum(int P, const int8_t* const* codes, const float* scales, int64_t n, void* out, bool out_bf16,
                  int32_t* sums, cudaStream_t stream, const char** why) {
    dim3 grid;
    if (!q8_grid(n, &grid, why)) return -1;
    Q8SumArgs a{};
    for (int p = 0; p < P; ++p) a.codes[p] = codes[p];
    a.scales = scales;
    a.n = n;
    a.out = out;
    a.sums = sums;
    switch (P) {
#define SSM_Q8S_CASE(PP)                                                                          \
        case PP:                                                                                \
            if (out_bf16) k_q8_sum<__nv_bfloat16, PP><<<grid, kThreads, 0, stream>>>(a);        \
            else k_q8_sum<float, PP><<<grid, kThreads, 0, stream>>>(a);                         \
            break;
        SSM_Q8S_CASE(1) SSM_Q8S_CASE(2) SSM_Q8S_CASE(3) SSM_Q8S_CASE(4)
        SSM_Q8S_CASE(5) SSM_Q8S_CASE(6) SSM_Q8S_CASE(7) SSM_Q8S_CASE(8)
#undef SSM_Q8S_CASE
        default:
            *why = "P out of range";
            return -1;
    }
    return q8_launched(why);
}

}  // namespace ssm
