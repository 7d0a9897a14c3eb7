// prefill.cu -- selective-SSM prefill on sm_103a.
//
// Computes, for every batch row b, channel d and token t (N = 16 states, conv width 4),
//   u_t = SiLU(conv_b + sum_k conv_w[k] x_{t-3+k}),  delta_t = softplus(dt_t + dt_bias),
//   h_t[n] = exp(delta_t A[n]) h_{t-1}[n] + delta_t B_t[n] u_t,
//   out_t = (sum_n C_t[n] h_t[n] + D u_t) * SiLU(z_t),
// and the final conv and SSM states.  The recurrence never leaves its channel
// ("Scaling State-Space Models on Multiple GPUs with Tensor Parallelism",
// Methodology 2, local recurrence) and the final states are the cache that
// decode continues from (Methodology 3).
//
// Design (one GB300; the path is bound by the FP32/MUFU pipes and instruction
// issue, with HBM next; no tensor cores: the recurrence is diagonal, not a
// contraction):
//   * One CTA owns 16 channels of one batch row for the WHOLE sequence, so the
//     carry between time chunks stays in registers: no scratch memory, no
//     inter-CTA waits, one launch.
//   * Lane l of a warp works on channel l % 16 and on half g = l / 16 of the 16
//     states (states 8g .. 8g+7, as four f32x2 pairs).  The two halves of a
//     channel share the per-token work: each computes conv/SiLU/softplus for half
//     of the tokens and the results meet through shuffles; their partial
//     readouts C.h meet the same way.
//   * Time advances in chunks of TC = S*K tokens.  Warp j of the S warps owns the
//     K consecutive tokens [j*K, j*K + K) of the chunk.
//   * Staging: a 3-stage ring of TMA tile copies (x with a 3-token conv halo,
//     z, dt as [TC x 16] boxes; B, C as [TC x 16] boxes) completing on mbarriers,
//     issued two chunks ahead by one thread.  Out-of-range rows/channels arrive
//     as zeros.  B and C are widened to fp32 once per chunk by the whole CTA.
//   * The scan is a chunked associative scan of (a, b) pairs, two states at a
//     time in packed f32x2 arithmetic:
//       1. per lane, a_i = 2^(delta_i A'[n]), b_i = delta_i u_i B_i[n] for its K
//          tokens and the sub-chunk aggregate (prod a, folded b) -- the product
//          of the a_i is taken as 2^(A'[n] * sum delta_i);
//       2. the S sub-chunk aggregates meet in shared memory; each warp folds the
//          ones before it onto the carried-in chunk state to get its start state,
//          and every warp folds all S to get the next chunk's carry;
//       3. each lane replays its K tokens from the start state and accumulates
//          y_i += C_i[n] h_i[n].
//   * The split of the work depends only on the compile-time S and K, never on
//     d_inner, the grid or occupancy, so a channel's result is bit-identical
//     whatever channel slice it is computed in.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace ssm {

namespace {

constexpr int kCD = 16;      // channels per CTA
constexpr int kN = 16;       // d_state
constexpr int kStages = 3;   // TMA ring depth

constexpr int align128(int v) { return (v + 127) / 128 * 128; }

template <int S, int K, typename Tin>
struct Layout {
    static constexpr int TC = S * K;
    static constexpr int XROWS = TC + 3;
    static constexpr int ES = (int)sizeof(Tin);
    static constexpr int X_BYTES = XROWS * kCD * ES;
    static constexpr int Z_BYTES = TC * kCD * ES;
    static constexpr int BC_BYTES = TC * kN * ES;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_Z = align128(OFF_X + X_BYTES);
    static constexpr int OFF_DT = align128(OFF_Z + Z_BYTES);
    static constexpr int OFF_B = align128(OFF_DT + Z_BYTES);
    static constexpr int OFF_C = align128(OFF_B + BC_BYTES);
    static constexpr int STAGE = align128(OFF_C + BC_BYTES);
    static constexpr int TX = X_BYTES + 2 * Z_BYTES + 2 * BC_BYTES;   // bytes per stage fill
    // after the ring: fp32 B and C of the chunk (two parities), the exchange slots, barriers
    static constexpr int BCF = TC * kN * 4;
    static constexpr int OFF_BF = kStages * STAGE;       // [2][TC][16]
    static constexpr int OFF_CF = OFF_BF + 2 * BCF;      // [2][TC][16]
    static constexpr int OFF_XCH = OFF_CF + 2 * BCF;     // [2 slots][S][32] float4
    static constexpr int XCH_BYTES = 2 * S * 32 * 16;
    static constexpr int OFF_OUT = align128(OFF_XCH + XCH_BYTES);   // [2 parities][TC][16] output tiles
    static constexpr int OUT_BYTES = 2 * TC * kCD * 4;
    static constexpr int OFF_BAR = OFF_OUT + OUT_BYTES;
    static constexpr int TOTAL = OFF_BAR + kStages * 8;
};

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Two consecutive bf16 / fp32 elements widened to float2.
__device__ __forceinline__ float2 load_pair(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ float2 load_pair(const float* p) { return *reinterpret_cast<const float2*>(p); }

// kSeg: the launch covers several sequence segments (blockIdx.z); without it the CTA owns
// the whole row and none of the segment bookkeeping is compiled in.
template <int S, int K, typename Tin, typename Tout, bool kSeg>
__global__ void __launch_bounds__(S * 32, 3)
k_prefill(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
          const __grid_constant__ CUtensorMap tm_dt, const __grid_constant__ CUtensorMap tm_B,
          const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_out,
          const PrefillArgs p) {
    using Lay = Layout<S, K, Tin>;
    constexpr int TC = Lay::TC;
    constexpr int KH = K / 2;            // tokens whose per-token work this lane does
    static_assert(K % 2 == 0, "K must be even");
    extern __shared__ __align__(128) unsigned char smem[];
    float* Bf0 = reinterpret_cast<float*>(smem + Lay::OFF_BF);
    float* Cf0 = reinterpret_cast<float*>(smem + Lay::OFF_CF);
    float4* xch = reinterpret_cast<float4*>(smem + Lay::OFF_XCH);
    Tout* out_s = reinterpret_cast<Tout*>(smem + Lay::OFF_OUT);          // [2][TC][16]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::OFF_BAR);

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int c = lane & 15;             // channel within the CTA
    const int g = lane >> 4;             // state half: states 8g .. 8g+7
    const int d0 = blockIdx.x * kCD;
    const int b = blockIdx.y;
    const int d = d0 + c;
    const bool dvalid = d < p.d_inner;
    const int L = p.seqlen;
    // sequence segment blockIdx.z: tokens [blockIdx.z * seg_len, min(L, (blockIdx.z + 1) * seg_len))
    auto seg_first_token = [&]() { return kSeg ? (int)blockIdx.z * p.seg_len : 0; };
    const int n_iter = kSeg ? (min(L - seg_first_token(), p.seg_len) + TC - 1) / TC : (L + TC - 1) / TC;

    // TMA destinations need 128-byte alignment; refuse (and report) rather than fault.
    if (smem_u32(smem) & 127u) {
        if (threadIdx.x == 0) atomicOr(p.status, 4u);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_z);
        prefetch_tmap(&tm_dt);
        prefetch_tmap(&tm_B);
        prefetch_tmap(&tm_C);
    }
    __syncthreads();

    auto issue = [&](int it) {
        const int s = it % kStages;
        unsigned char* st = smem + s * Lay::STAGE;
        const int t0 = seg_first_token() + it * TC;
        mbar_arrive_expect_tx(&full[s], Lay::TX);
        tma_load_3d(st + Lay::OFF_X, &tm_x, &full[s], d0, t0 - 3, b);
        tma_load_3d(st + Lay::OFF_Z, &tm_z, &full[s], d0, t0, b);
        tma_load_3d(st + Lay::OFF_DT, &tm_dt, &full[s], d0, t0, b);
        tma_load_3d(st + Lay::OFF_B, &tm_B, &full[s], 0, t0, b);
        tma_load_3d(st + Lay::OFF_C, &tm_C, &full[s], 0, t0, b);
    };
    if (threadIdx.x == 0) {
        for (int it = 0; it < kStages - 1 && it < n_iter; ++it) issue(it);
    }

    // ---- per-channel parameters (zeros for channels past d_inner)
    float A2[8];    // A[d][8g + m] * log2(e): exp(delta A) = 2^(delta A2)
    float Dd = 0.f, bias = 0.f, w0 = 0.f, w1 = 0.f, w2 = 0.f, w3 = 0.f, cb = 0.f;
    float2 carry[4];
#pragma unroll
    for (int m = 0; m < 8; ++m) A2[m] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) carry[q] = f2(0.f, 0.f);
    if (dvalid) {
        const float4* Ar = reinterpret_cast<const float4*>(p.A + (int64_t)d * kN + 8 * g);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float4 v = __ldg(Ar + q);
            A2[4 * q + 0] = v.x * kLog2e;
            A2[4 * q + 1] = v.y * kLog2e;
            A2[4 * q + 2] = v.z * kLog2e;
            A2[4 * q + 3] = v.w * kLog2e;
        }
        const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w + (int64_t)d * 4));
        w0 = w.x; w1 = w.y; w2 = w.z; w3 = w.w;
        cb = __ldg(p.conv_b + d);
        Dd = __ldg(p.Dskip + d);
        bias = __ldg(p.dt_bias + d);
        if (kSeg && blockIdx.z > 0) {
            // the start state of this segment, left in the workspace by the carry pass
            const float2* hs = reinterpret_cast<const float2*>(
                p.ws + (((int64_t)(blockIdx.z - 1) * gridDim.y + b) * p.d_inner + d) * 32 + 8 * g);
#pragma unroll
            for (int q = 0; q < 4; ++q) carry[q] = hs[q];
        } else if (p.ssm_state_in) {
            const float2* hs = reinterpret_cast<const float2*>(
                p.ssm_state_in + (int64_t)b * p.ssm_state_stride_b + (int64_t)d * kN + 8 * g);
#pragma unroll
            for (int q = 0; q < 4; ++q) carry[q] = hs[q];
        }
    }

    for (int it = 0; it < n_iter; ++it) {
        const int s = it % kStages;
        const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((it / kStages) & 1));
        const unsigned char* st = smem + s * Lay::STAGE;
        const Tin* xs = reinterpret_cast<const Tin*>(st + Lay::OFF_X);
        const Tin* zs = reinterpret_cast<const Tin*>(st + Lay::OFF_Z);
        const Tin* dts = reinterpret_cast<const Tin*>(st + Lay::OFF_DT);
        float* Bf = Bf0 + (it & 1) * TC * kN;
        float* Cf = Cf0 + (it & 1) * TC * kN;
        if (ok) {
            // ---- B and C of the chunk widened to fp32 once, by the whole CTA.  The
            // parity buffer written here was last read in chunk it-2, which every
            // warp finished before the barriers of chunk it-1.
            const Tin* Bs = reinterpret_cast<const Tin*>(st + Lay::OFF_B);
            const Tin* Cs = reinterpret_cast<const Tin*>(st + Lay::OFF_C);
#pragma unroll
            for (int e = 2 * threadIdx.x; e < TC * kN; e += 2 * S * 32) {
                *reinterpret_cast<float2*>(Bf + e) = load_pair(Bs + e);
                *reinterpret_cast<float2*>(Cf + e) = load_pair(Cs + e);
            }
        }
        if (__syncthreads_or(!ok)) {
            // A copy never completed: record it, let every issued copy land (bounded) and stop.
            if (threadIdx.x == 0) {
                atomicOr(p.status, 1u);
                for (int j = it; j < n_iter && j < it + kStages - 1; ++j)
                    (void)mbar_wait_bounded(&full[j % kStages], (uint32_t)((j / kStages) & 1),
                                            100000000ull);
                bulk_wait_all();
            }
            return;
        }
        if (p.out_tma && it > 0 && threadIdx.x == 0) {
            // the previous chunk's output tile (staged and fenced before this barrier) leaves by TMA;
            // rows past L and channels past d_inner are outside the map and not written.  The tile
            // written two chunks ago, in the buffer this chunk reuses, has then been read.
            tma_store_3d(&tm_out, out_s + ((it - 1) & 1) * TC * kCD, d0, seg_first_token() + (it - 1) * TC, b);
            bulk_commit();
            bulk_wait_read_all_but_last();
        }

        // ---- per-token work for this lane's half of the warp's K tokens:
        //      conv + SiLU, softplus step, skip term
        const int row0 = warp * K;            // first token of this warp in the chunk
        const int tbase = seg_first_token() + it * TC + row0;   // its absolute index
        const int r0 = row0 + KH * g;         // first token this lane computes
        float xm3 = to_f32(xs[(r0 + 0) * kCD + c]);   // x[t-3] (tile row 0 = chunk start - 3)
        float xm2 = to_f32(xs[(r0 + 1) * kCD + c]);
        float xm1 = to_f32(xs[(r0 + 2) * kCD + c]);
        if (it == 0 && (!kSeg || blockIdx.z == 0) && warp == 0 && g == 0 && p.conv_state_in != nullptr && dvalid) {
            const float* cs = p.conv_state_in + (int64_t)b * 3 * p.conv_state_ld + d;
            xm3 = cs[0];
            xm2 = cs[p.conv_state_ld];
            xm1 = cs[2 * p.conv_state_ld];
        }
        float dl_own[KH], du_own[KH], ud[KH];
        float dsum = 0.f;
#pragma unroll
        for (int k = 0; k < KH; ++k) {
            const float xt = to_f32(xs[(r0 + k + 3) * kCD + c]);
            float xc = fmaf(w0, xm3, cb);
            xc = fmaf(w1, xm2, xc);
            xc = fmaf(w2, xm1, xc);
            xc = fmaf(w3, xt, xc);
            xm3 = xm2; xm2 = xm1; xm1 = xt;
            const float u = silu_in<Tin>(xc);
            float delta = softplus_in<Tin>(to_f32(dts[(r0 + k) * kCD + c]) + bias);
            if (tbase + KH * g + k >= L) delta = 0.f;   // padding rows: a = 1, b = 0 (identity)
            dl_own[k] = delta;
            du_own[k] = delta * u;
            ud[k] = Dd * u;
            dsum += delta;
        }
        // the two halves of the channel trade their tokens' delta and delta*u
        float dl[K], du[K];
#pragma unroll
        for (int k = 0; k < KH; ++k) {
            dl[k] = __shfl_sync(0xffffffffu, dl_own[k], c);
            dl[KH + k] = __shfl_sync(0xffffffffu, dl_own[k], c + 16);
            du[k] = __shfl_sync(0xffffffffu, du_own[k], c);
            du[KH + k] = __shfl_sync(0xffffffffu, du_own[k], c + 16);
        }
        dsum += __shfl_xor_sync(0xffffffffu, dsum, 16);

        // ---- the scan, two states at a time (pairs 4g .. 4g+3 of this lane)
        float ylane[K];
#pragma unroll
        for (int i = 0; i < K; ++i) ylane[i] = 0.f;
        const float* bw = Bf + row0 * kN + 8 * g;
        const float* cw = Cf + row0 * kN + 8 * g;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float2 Ap = f2(A2[2 * r], A2[2 * r + 1]);
            float2 a[K], bb[K];
            float2 agg = f2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const float2 e = __fmul2_rn(f2(dl[i], dl[i]), Ap);
                a[i] = f2(ex2(e.x), ex2(e.y));
                const float2 Bi = *reinterpret_cast<const float2*>(bw + i * kN + 2 * r);
                bb[i] = __fmul2_rn(f2(du[i], du[i]), Bi);
                agg = __ffma2_rn(a[i], agg, bb[i]);
            }
            const float2 ea = __fmul2_rn(f2(dsum, dsum), Ap);
            xch[((r & 1) * S + warp) * 32 + lane] = make_float4(ex2(ea.x), ex2(ea.y), agg.x, agg.y);
            __syncthreads();
            if (r == 0 && threadIdx.x == 0 && it + kStages - 1 < n_iter) {
                // every warp has finished chunk it-1, so its stage can be refilled
                issue(it + kStages - 1);
            }
            float2 h = carry[r], hs = h;
#pragma unroll
            for (int j = 0; j < S; ++j) {
                const float4 e = xch[((r & 1) * S + j) * 32 + lane];
                if (j == warp) hs = h;
                h = __ffma2_rn(f2(e.x, e.y), h, f2(e.z, e.w));
            }
            carry[r] = h;
            h = hs;
#pragma unroll
            for (int i = 0; i < K; ++i) {
                h = __ffma2_rn(a[i], h, bb[i]);
                const float2 Ci = *reinterpret_cast<const float2*>(cw + i * kN + 2 * r);
                ylane[i] = fmaf(Ci.x, h.x, fmaf(Ci.y, h.y, ylane[i]));
            }
        }

        // ---- the two halves' readouts meet; each lane gates and stores its own tokens
        const int t_own = tbase + KH * g;
#pragma unroll
        for (int k = 0; k < KH; ++k) {
            // each half sends the other the partial readout of the other's token: one shuffle
            const float mine = g ? ylane[KH + k] : ylane[k];
            const float other = __shfl_xor_sync(0xffffffffu, g ? ylane[k] : ylane[KH + k], 16);
            const int t = t_own + k;
            if (dvalid && t < L) {
                const float yv = (mine + other) + ud[k];
                const float gz = silu_in<Tin>(to_f32(zs[(r0 + k) * kCD + c]));
                if (p.out_tma)
                    out_s[((it & 1) * TC + r0 + k) * kCD + c] = from_f32<Tout>(yv * gz);
                else
                    reinterpret_cast<Tout*>(p.out)[(int64_t)b * p.out_stride_b + (int64_t)t * p.out_stride_t + d] =
                        from_f32<Tout>(yv * gz);
            }
        }
        if (p.out_tma) fence_proxy_async_smem();         // the tile is read by the next chunk's store
    }
    if (p.out_tma) {
        __syncthreads();
        if (threadIdx.x == 0) {
            if (n_iter > 0) {
                tma_store_3d(&tm_out, out_s + ((n_iter - 1) & 1) * TC * kCD, d0,
                             seg_first_token() + (n_iter - 1) * TC, b);
                bulk_commit();
            }
            bulk_wait_all();
        }
    }

    // ---- final states (last segment): h_L and the last three raw inputs
    if ((!kSeg || (int)blockIdx.z == p.n_seg - 1) && warp == 0 && dvalid) {
        float2* hs = reinterpret_cast<float2*>(p.ssm_state_out + (int64_t)b * p.ssm_state_stride_b +
                                               (int64_t)d * kN + 8 * g);
#pragma unroll
        for (int q = 0; q < 4; ++q) hs[q] = carry[q];
        if (g == 0) {
            const Tin* xg = reinterpret_cast<const Tin*>(p.x) + (int64_t)b * p.in_stride_b + d;
            float* co = p.conv_state_out + (int64_t)b * 3 * p.conv_state_ld + d;
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const int t = L - 3 + k;
                float v = 0.f;
                if (t >= 0) {
                    v = to_f32(xg[(int64_t)t * p.in_stride_t]);
                } else if (p.conv_state_in != nullptr) {
                    v = p.conv_state_in[(int64_t)b * 3 * p.conv_state_ld + (int64_t)(t + 3) * p.conv_state_ld + d];
                }
                co[(int64_t)k * p.conv_state_ld] = v;
            }
        }
    }
}

// ------------------------------------------------------------------ segmented prefill
// Long rows with few (batch x channel-group) CTAs leave most SMs idle, so the sequence
// can be cut into segments that run in parallel: the recurrence composes, and the
// pair (prod_t a_t, state from zero) of a segment carries it from its start state to
// its end state.  Pass A computes that pair for every segment but the last; pass B
// walks the segments of each (b, d, n) in order and turns the pairs into start
// states; pass C is k_prefill, each segment starting from its start state.

template <int S, int K, typename Tin>
struct AggLayout {
    static constexpr int TC = S * K;
    static constexpr int ES = (int)sizeof(Tin);
    static constexpr int X_BYTES = (TC + 3) * kCD * ES;
    static constexpr int DT_BYTES = TC * kCD * ES;
    static constexpr int B_BYTES = TC * kN * ES;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_DT = align128(OFF_X + X_BYTES);
    static constexpr int OFF_B = align128(OFF_DT + DT_BYTES);
    static constexpr int STAGE = align128(OFF_B + B_BYTES);
    static constexpr int TX = X_BYTES + DT_BYTES + B_BYTES;
    static constexpr int OFF_BF = kStages * STAGE;           // fp32 B of the chunk, [TC][16]
    static constexpr int OFF_XCH = OFF_BF + TC * kN * 4;     // [4 pairs][S][32] float4
    static constexpr int OFF_BAR = OFF_XCH + 4 * S * 32 * 16;
    static constexpr int TOTAL = OFF_BAR + kStages * 8;
};

// Pass A: segment sg (< n_seg - 1, always a whole number of chunks) of 16 channels of
// row b: the state reached from zero and the product of the decays, into ws.
template <int S, int K, typename Tin>
__global__ void __launch_bounds__(S * 32, 3)
k_prefill_agg(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dt,
              const __grid_constant__ CUtensorMap tm_B, const PrefillArgs p) {
    using Lay = AggLayout<S, K, Tin>;
    constexpr int TC = Lay::TC;
    constexpr int KH = K / 2;
    extern __shared__ __align__(128) unsigned char smem[];
    float* Bf = reinterpret_cast<float*>(smem + Lay::OFF_BF);
    float4* xch = reinterpret_cast<float4*>(smem + Lay::OFF_XCH);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::OFF_BAR);

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int c = lane & 15;
    const int g = lane >> 4;
    const int d0 = blockIdx.x * kCD;
    const int b = blockIdx.y;
    const int sg = blockIdx.z;
    const int d = d0 + c;
    const bool dvalid = d < p.d_inner;
    const int T0 = sg * p.seg_len;
    const int n_iter = p.seg_len / TC;

    if (smem_u32(smem) & 127u) {
        if (threadIdx.x == 0) atomicOr(p.status, 4u);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_dt);
        prefetch_tmap(&tm_B);
    }
    __syncthreads();

    auto issue = [&](int it) {
        const int s = it % kStages;
        unsigned char* st = smem + s * Lay::STAGE;
        const int t0 = T0 + it * TC;
        mbar_arrive_expect_tx(&full[s], Lay::TX);
        tma_load_3d(st + Lay::OFF_X, &tm_x, &full[s], d0, t0 - 3, b);
        tma_load_3d(st + Lay::OFF_DT, &tm_dt, &full[s], d0, t0, b);
        tma_load_3d(st + Lay::OFF_B, &tm_B, &full[s], 0, t0, b);
    };
    if (threadIdx.x == 0) {
        for (int it = 0; it < kStages - 1 && it < n_iter; ++it) issue(it);
    }

    float A2[8];
    float bias = 0.f, w0 = 0.f, w1 = 0.f, w2 = 0.f, w3 = 0.f, cb = 0.f;
    float2 carry[4], decay[4];
#pragma unroll
    for (int m = 0; m < 8; ++m) A2[m] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        carry[q] = f2(0.f, 0.f);
        decay[q] = f2(1.f, 1.f);
    }
    if (dvalid) {
        const float4* Ar = reinterpret_cast<const float4*>(p.A + (int64_t)d * kN + 8 * g);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float4 v = __ldg(Ar + q);
            A2[4 * q + 0] = v.x * kLog2e;
            A2[4 * q + 1] = v.y * kLog2e;
            A2[4 * q + 2] = v.z * kLog2e;
            A2[4 * q + 3] = v.w * kLog2e;
        }
        const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w + (int64_t)d * 4));
        w0 = w.x; w1 = w.y; w2 = w.z; w3 = w.w;
        cb = __ldg(p.conv_b + d);
        bias = __ldg(p.dt_bias + d);
    }

    for (int it = 0; it < n_iter; ++it) {
        const int s = it % kStages;
        const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((it / kStages) & 1));
        const unsigned char* st = smem + s * Lay::STAGE;
        const Tin* xs = reinterpret_cast<const Tin*>(st + Lay::OFF_X);
        const Tin* dts = reinterpret_cast<const Tin*>(st + Lay::OFF_DT);
        if (ok) {
            // the previous chunk's readers of Bf all passed its exchange barrier
            const Tin* Bs = reinterpret_cast<const Tin*>(st + Lay::OFF_B);
#pragma unroll
            for (int e = 2 * threadIdx.x; e < TC * kN; e += 2 * S * 32)
                *reinterpret_cast<float2*>(Bf + e) = load_pair(Bs + e);
        }
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) {
                atomicOr(p.status, 1u);
                for (int j = it; j < n_iter && j < it + kStages - 1; ++j)
                    (void)mbar_wait_bounded(&full[j % kStages], (uint32_t)((j / kStages) & 1), 100000000ull);
            }
            return;
        }
        // every warp has finished chunk it-1, so its stage can be refilled
        if (threadIdx.x == 0 && it + kStages - 1 < n_iter) issue(it + kStages - 1);

        const int row0 = warp * K;
        const int r0 = row0 + KH * g;
        float xm3 = to_f32(xs[(r0 + 0) * kCD + c]);
        float xm2 = to_f32(xs[(r0 + 1) * kCD + c]);
        float xm1 = to_f32(xs[(r0 + 2) * kCD + c]);
        if (it == 0 && sg == 0 && warp == 0 && g == 0 && p.conv_state_in != nullptr && dvalid) {
            const float* cs = p.conv_state_in + (int64_t)b * 3 * p.conv_state_ld + d;
            xm3 = cs[0];
            xm2 = cs[p.conv_state_ld];
            xm1 = cs[2 * p.conv_state_ld];
        }
        float dl_own[KH], du_own[KH];
        float dsum = 0.f;
#pragma unroll
        for (int k = 0; k < KH; ++k) {
            const float xt = to_f32(xs[(r0 + k + 3) * kCD + c]);
            float xc = fmaf(w0, xm3, cb);
            xc = fmaf(w1, xm2, xc);
            xc = fmaf(w2, xm1, xc);
            xc = fmaf(w3, xt, xc);
            xm3 = xm2; xm2 = xm1; xm1 = xt;
            const float u = silu_in<Tin>(xc);
            const float delta = softplus_in<Tin>(to_f32(dts[(r0 + k) * kCD + c]) + bias);
            dl_own[k] = delta;
            du_own[k] = delta * u;
            dsum += delta;
        }
        float dl[K], du[K];
#pragma unroll
        for (int k = 0; k < KH; ++k) {
            dl[k] = __shfl_sync(0xffffffffu, dl_own[k], c);
            dl[KH + k] = __shfl_sync(0xffffffffu, dl_own[k], c + 16);
            du[k] = __shfl_sync(0xffffffffu, du_own[k], c);
            du[KH + k] = __shfl_sync(0xffffffffu, du_own[k], c + 16);
        }
        dsum += __shfl_xor_sync(0xffffffffu, dsum, 16);

        // sub-chunk aggregates of all four state pairs, then one exchange
        const float* bw = Bf + row0 * kN + 8 * g;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float2 Ap = f2(A2[2 * r], A2[2 * r + 1]);
            float2 agg = f2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const float2 e = __fmul2_rn(f2(dl[i], dl[i]), Ap);
                const float2 a = f2(ex2(e.x), ex2(e.y));
                const float2 Bi = *reinterpret_cast<const float2*>(bw + i * kN + 2 * r);
                agg = __ffma2_rn(a, agg, __fmul2_rn(f2(du[i], du[i]), Bi));
            }
            const float2 ea = __fmul2_rn(f2(dsum, dsum), Ap);
            xch[(r * S + warp) * 32 + lane] = make_float4(ex2(ea.x), ex2(ea.y), agg.x, agg.y);
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float2 h = carry[r], dec = decay[r];
#pragma unroll
            for (int j = 0; j < S; ++j) {
                const float4 e = xch[(r * S + j) * 32 + lane];
                h = __ffma2_rn(f2(e.x, e.y), h, f2(e.z, e.w));
                dec = __fmul2_rn(dec, f2(e.x, e.y));
            }
            carry[r] = h;
            decay[r] = dec;
        }
    }
    if (dvalid) {
        float2* w = reinterpret_cast<float2*>(p.ws + (((int64_t)sg * gridDim.y + b) * p.d_inner + d) * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            w[4 * g + q] = carry[q];          // states 8g .. 8g+7
            w[8 + 4 * g + q] = decay[q];      // their decay products
        }
    }
}

// Pass B: one thread per (b, d, n) folds the segments in order; entry sg of ws then holds the
// start state of segment sg + 1 in place of segment sg's state from zero.
__global__ void __launch_bounds__(256)
k_prefill_carry(const PrefillArgs p, int batch) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;      // (b, d, n)
    const int64_t per_row = (int64_t)p.d_inner * kN;
    if (i >= batch * per_row) return;
    const int64_t b = i / per_row;
    const int64_t dn = i - b * per_row;
    const int64_t d = dn / kN, n = dn - d * kN;
    float h = p.ssm_state_in ? p.ssm_state_in[b * p.ssm_state_stride_b + dn] : 0.f;
    for (int sg = 0; sg < p.n_seg - 1; ++sg) {
        float* w = p.ws + (((int64_t)sg * batch + b) * p.d_inner + d) * 32;
        h = fmaf(w[16 + n], h, w[n]);
        w[n] = h;
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 3-D map over [dim2][dim1][dim0] elements with byte strides s1 (dim1) and s2 (dim2).
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t dim0, uint64_t dim1,
              uint64_t dim2, uint64_t s1, uint64_t s2, uint32_t box0, uint32_t box1) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {dim0, dim1, dim2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int S, int K, typename Tin, typename Tout>
int launch_t(const PrefillLaunch& q, cudaStream_t stream, const char** why) {
    using Lay = Layout<S, K, Tin>;
    constexpr int TC = Lay::TC;
    const int es = (int)sizeof(Tin);
    const CUtensorMapDataType dt =
        sizeof(Tin) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const PrefillArgs& a = q.args;
    const uint64_t sb = (uint64_t)(q.batch > 1 ? a.in_stride_b : (int64_t)a.seqlen * a.in_stride_t) * es;
    const uint64_t st = (uint64_t)a.in_stride_t * es;
    const uint64_t bc_t = (uint64_t)kN * es, bc_b = (uint64_t)a.seqlen * kN * es;
    CUtensorMap mx, mz, mdt, mB, mC, mo;
    if (!make_map(&mx, a.x, dt, a.d_inner, a.seqlen, q.batch, st, sb, kCD, TC + 3) ||
        !make_map(&mz, q.z, dt, a.d_inner, a.seqlen, q.batch, st, sb, kCD, TC) ||
        !make_map(&mdt, q.dt, dt, a.d_inner, a.seqlen, q.batch, st, sb, kCD, TC) ||
        !make_map(&mB, q.Bm, dt, kN, a.seqlen, q.batch, bc_t, bc_b, kN, TC) ||
        !make_map(&mC, q.Cm, dt, kN, a.seqlen, q.batch, bc_t, bc_b, kN, TC)) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point missing or layout rejected)";
        return -1;
    }
    // the output leaves by TMA stores when its base and strides are 16-byte multiples
    PrefillArgs ak = a;
    const uint64_t eo = sizeof(Tout);
    const uint64_t ot = (uint64_t)a.out_stride_t * eo;
    const uint64_t ob = q.batch > 1 ? (uint64_t)a.out_stride_b * eo : (uint64_t)a.seqlen * ot;
    ak.out_tma = (reinterpret_cast<uintptr_t>(a.out) % 16 == 0 && ot % 16 == 0 && ob % 16 == 0) ? 1 : 0;
    if (ak.out_tma &&
        !make_map(&mo, a.out, sizeof(Tout) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  a.d_inner, a.seqlen, q.batch, ot, ob, kCD, TC))
        ak.out_tma = 0;
    if (!ak.out_tma) mo = mx;                        // not read
    const unsigned gx = (unsigned)((a.d_inner + kCD - 1) / kCD);
    if (a.n_seg > 1) {
        // pass A (segments 0 .. n_seg-2), then pass B
        using ALay = AggLayout<S, K, Tin>;
        static ContextMemo agg_attr;
        auto kagg = k_prefill_agg<S, K, Tin>;
        if (!opt_in_dynamic_smem(agg_attr, kagg, ALay::TOTAL, why)) return -1;
        kagg<<<dim3(gx, q.batch, a.n_seg - 1), S * 32, ALay::TOTAL, stream>>>(mx, mdt, mB, a);
        const int64_t n = (int64_t)q.batch * a.d_inner * kN;
        k_prefill_carry<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(a, q.batch);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) {
            *why = cudaGetErrorString(e);
            return -1;
        }
    }
    static ContextMemo attr_row, attr_seg;
    auto kern = a.n_seg > 1 ? k_prefill<S, K, Tin, Tout, true> : k_prefill<S, K, Tin, Tout, false>;
    if (!opt_in_dynamic_smem(a.n_seg > 1 ? attr_seg : attr_row, kern, Lay::TOTAL, why)) return -1;
    kern<<<dim3(gx, q.batch, a.n_seg), S * 32, Lay::TOTAL, stream>>>(mx, mz, mdt, mB, mC, mo, ak);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return -1;
    }
    return 0;
}

}  // namespace

// Compile-time split of a chunk: S warps x K tokens.
constexpr int kS = 4;
constexpr int kK = 16;
static_assert(kS * kK == kPrefillChunk, "segments are whole chunks");

int launch_prefill(const PrefillLaunch& q, cudaStream_t stream, const char** why) {
    if (q.in_bf16) {
        return q.out_bf16 ? launch_t<kS, kK, __nv_bfloat16, __nv_bfloat16>(q, stream, why)
                          : launch_t<kS, kK, __nv_bfloat16, float>(q, stream, why);
    }
    return q.out_bf16 ? launch_t<kS, kK, float, __nv_bfloat16>(q, stream, why)
                      : launch_t<kS, kK, float, float>(q, stream, why);
}

}  // namespace ssm
