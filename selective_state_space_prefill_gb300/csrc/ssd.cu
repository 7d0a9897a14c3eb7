// ssd.cu -- the SSD (Mamba-2-style) variant of the selective-SSM mixer on sm_103a: prefill on the
// tcgen05 tensor cores and a one-token decode step.
//
// The mixer of "Scaling State-Space Models on Multiple GPUs with Tensor Parallelism" keeps every
// channel's recurrence local (Methodology 2) and caches the state between prefill and decode
// (Methodology 3); the pages name Mamba, Falcon-Mamba and Zamba as the model families it serves.
// This file computes the Mamba-2 form of that mixer (Dao and Gu, "Transformers are SSMs", 2024):
// per batch row b, head h (group g = h / (H / G)), position p < 64 and state n < 64,
//   x, B, C = SiLU(causal width-4 depthwise conv of the channels [x | B | C]),
//   delta_t = softplus(dt_t + dt_bias[h]),
//   S_t[p][n] = exp(delta_t A[h]) S_{t-1}[p][n] + delta_t x_t[p] B_t[n],
//   y_t[p] = sum_n C_t[n] S_t[p][n] + D[h] x_t[p],   out_t = y_t SiLU(z_t).
//
// The decay is a scalar per head, so inside a chunk of Q = 128 tokens the recurrence is a
// sequence of dense contractions (the SSD "dual" form).  With s_i = sum_{r<=i} delta_r A[h]:
//   G = C B^T                                   [Q x Q]
//   M[i][j] = G[i][j] exp(s_i - s_j) delta_j    (j <= i, else 0)
//   Y = M X + exp(s)_i (C S_prev^T) + D X        (X = the chunk's x, [Q x 64])
//   S = exp(s_Q) S_prev + sum_j exp(s_Q - s_j) delta_j x_j (x) B_j
// Those four products run on the 5th-generation tensor cores (tcgen05, kind::f16, M = 128,
// fp32 accumulators in TMEM).  bf16 operands alone would round x, B, C, M and S by 2^-9 each,
// far above the mixer's error budget, so every operand is carried as a bf16 pair hi + lo
// (hi = bf16(v), lo = bf16(v - hi), |v - hi - lo| <= 2^-17 |v|) and each product is the sum
// hi*hi + hi*lo + lo*hi.
//
// Kernels:
//   k_ssd_bc      (pre-pass) conv + SiLU of every group's B and C channels, written as hi/lo
//                 planes [t][n] (the K-major operands of C B^T and C S^T) and, for B, also as
//                 token-major planes [n][t] (the K-major operand of the state update).
//   k_ssd_chunk   one CTA per (batch row, head) walks the row's chunks in order, so the fp32
//                 state stays on chip: TMA brings the raw x (with a 3-token conv halo), z and the
//                 B/C tiles; the CTA's threads compute the x conv, the decays and the operands
//                 they own (X, the state-update weights, M, S) into 128-byte-swizzled shared
//                 memory; one thread issues the MMAs; the threads read the accumulators back
//                 with tcgen05.ld.
//   k_ssd_decode  one CTA per (request, head): the one-token recurrence on the cached state
//                 [64 x 64] in place, then k_ssd_decode_shift moves the conv windows of the B
//                 and C channels (shared by the heads of a group, so they move after every head
//                 has read them).
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace ssm {
namespace {

using Tin_bf16 = __nv_bfloat16;  // the prefill's token inputs (x, B, C, z, dt) are bf16

constexpr int kQ = 128;        // tokens per chunk (the MMA's M)
constexpr int kP = 64;         // head dim
constexpr int kNs = 64;        // d_state
constexpr int kTh = 256;       // threads of k_ssd_chunk: warp w reads TMEM lanes 32 (w % 4).., column half w / 4

// tcgen05.mma kind::f16 instruction descriptors: fp32 accumulator, bf16 A and B, both K-major,
// M = 128, N = 128 or 64.
constexpr uint32_t kIdescN128 = (1u << 4) | (1u << 7) | (1u << 10) | (16u << 17) | (8u << 24);
constexpr uint32_t kIdescN64 = (1u << 4) | (1u << 7) | (1u << 10) | (8u << 17) | (8u << 24);

// Shared memory of k_ssd_chunk (byte offsets from a 1024-aligned base).  Operand tiles are
// K-major rows of 64 bf16 (128 bytes) in 128-byte-swizzle atoms; a K extent of 128 is two such
// regions ("r0", "r1").
struct Smem {
    static constexpr int CHI = 0, CLO = 16384, BHI = 32768, BLO = 49152;  // [128 t][64 n] (TMA)
    static constexpr int MHI = 0, MLO = 32768;       // M hi / lo, r0 and r1 [128 i][64 j] each (over C, B)
    static constexpr int BTHI = 65536, BTLO = 81920; // B^T hi / lo, r0 and r1 [64 n][64 t] each (TMA)
    static constexpr int XHI = 98304, XLO = 114688;  // X^T hi / lo, r0 and r1 [64 p][64 t] each
    static constexpr int XW = 131072;                // weighted X^T, hi rows 0-63 / lo rows 64-127,
                                                     // r0 and r1 [128][64 t] each; later fp32 scratch
    static constexpr int SHI = 163840, SLO = 172032; // S hi / lo [64 p][64 n]
    static constexpr int XR = 180224;                // raw x [131 t][64 p] bf16 (TMA, unswizzled)
    static constexpr int ZT = 197632;                // z [128 t][64 p] bf16 (TMA, unswizzled)
    static constexpr int DL = 214016;                // delta [128] f32
    static constexpr int CS = DL + 512;              // s (chunk-local cumulative delta*A) [128] f32
    static constexpr int CW = CS + 512;              // conv weights of the head's x channels [64][4]
    static constexpr int CB = CW + 1024;             // conv bias [64]
    static constexpr int WS = CB + 256;              // per-warp scan totals [4]
    static constexpr int BAR = WS + 64;              // bar_a, bar_b, bar_mma
    static constexpr int SLOT = BAR + 32;            // TMEM base address
    static constexpr int TOTAL = SLOT + 16;
    static constexpr int ALLOC = TOTAL + 1024;       // + slack to align the base to 1024
    static constexpr int XR_BYTES = (kQ + 3) * kP * 2;
    static constexpr int TX_A = XR_BYTES + 4 * 8192;     // raw x + B^T hi/lo
    static constexpr int TX_B = 4 * 16384 + kQ * kP * 2; // C hi/lo, B hi/lo + z
    static constexpr int SCR_LD = 68;                    // fp32 scratch row stride (floats)
};
static_assert(Smem::XR + Smem::XR_BYTES <= Smem::ZT, "raw x tile overlaps z");
static_assert(Smem::ALLOC <= 232448, "shared memory above the 227 KB per-CTA limit");
static_assert(64 * Smem::SCR_LD * 4 <= 32768, "scratch larger than the weighted-X region");

// Byte offset of element (row, col) in a 128-byte-swizzled K-major region of 64-element rows.
__device__ __forceinline__ uint32_t sw128(int row, int col) {
    return (uint32_t)(row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1)));
}

__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(v);
    lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b) {
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

__device__ __forceinline__ void st_u16(unsigned char* base, uint32_t off, __nv_bfloat16 v) {
    *reinterpret_cast<__nv_bfloat16*>(base + off) = v;
}

// Four K-steps (K = 64) of D (+)= A B^T for K-major operands at shared addresses a, b.
__device__ __forceinline__ void mma_k64(uint32_t d, uint32_t a, uint32_t b, uint32_t idesc, bool first) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_bf16(d, smem_desc_sw128(a + 32 * kk), smem_desc_sw128(b + 32 * kk), idesc, (first && kk == 0) ? 0u : 1u);
}

// ------------------------------------------------------------------ pre-pass: B and C
// grid (ceil(L / 64), G, batch), 256 threads: 64 tokens x 64 states of group g.
template <typename Tin>
__global__ void __launch_bounds__(256)
k_ssd_bc(const SsdArgs p) {
    __shared__ __nv_bfloat16 tr[2][kNs][64 + 8];     // B hi / lo of the block, state-major
    const int t0 = blockIdx.x * 64, g = blockIdx.y, b = blockIdx.z;
    const int G = p.n_groups, BG = p.batch * G, bg = b * G + g, L = p.seqlen;
    const int64_t HP = (int64_t)p.n_heads * kP, Cx = HP + 2 * (int64_t)G * kNs;
    const Tin* xb = reinterpret_cast<const Tin*>(p.xBC) + (int64_t)b * p.xbc_stride_b;
    __nv_bfloat16* bc = reinterpret_cast<__nv_bfloat16*>(p.workspace);
    __nv_bfloat16* bt = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<unsigned char*>(p.workspace) + p.ws_bt_off);
    auto raw = [&](int t, int64_t c) -> float {
        if (t >= 0) return to_f32(xb[(int64_t)t * p.xbc_stride_t + c]);
        return p.conv_state_in ? p.conv_state_in[((int64_t)b * 3 + 3 + t) * Cx + c] : 0.f;
    };
    for (int e = threadIdx.x; e < 64 * kNs; e += 256) {
        const int tl = e / kNs, n = e % kNs, t = t0 + tl;
        if (t >= L) continue;
#pragma unroll
        for (int which = 0; which < 2; ++which) {          // 0: C (planes 0, 1), 1: B (planes 2, 3)
            const int64_t c = HP + (which ? 0 : (int64_t)G * kNs) + (int64_t)g * kNs + n;
            const float4 w = *reinterpret_cast<const float4*>(p.conv_w + c * 4);
            float xc = fmaf(w.x, raw(t - 3, c), p.conv_b[c]);
            xc = fmaf(w.y, raw(t - 2, c), xc);
            xc = fmaf(w.z, raw(t - 1, c), xc);
            xc = fmaf(w.w, raw(t, c), xc);
            __nv_bfloat16 hi, lo;
            split_bf16(silu_in<Tin>(xc), hi, lo);
            const int kind = which ? 2 : 0;
            bc[(((int64_t)kind * BG + bg) * L + t) * kNs + n] = hi;
            bc[(((int64_t)(kind + 1) * BG + bg) * L + t) * kNs + n] = lo;
            if (which) {
                tr[0][n][tl] = hi;
                tr[1][n][tl] = lo;
            }
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 2 * kNs * 64; e += 256) {
        const int k = e / (kNs * 64), n = (e / 64) % kNs, tl = e % 64, t = t0 + tl;
        if (t < L) bt[(((int64_t)k * BG + bg) * kNs + n) * p.ws_lp + t] = tr[k][n][tl];
    }
    // the conv window of the B and C channels after the last token
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x < 2 * kNs) {
        const int which = threadIdx.x / kNs, n = threadIdx.x % kNs;
        const int64_t c = HP + (which ? 0 : (int64_t)G * kNs) + (int64_t)g * kNs + n;
#pragma unroll
        for (int k = 0; k < 3; ++k) p.conv_state_out[((int64_t)b * 3 + k) * Cx + c] = raw(L - 3 + k, c);
    }
}

// ------------------------------------------------------------------ prefill chunks
template <typename Tout>
__global__ void __launch_bounds__(kTh, 1)
k_ssd_chunk(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
            const __grid_constant__ CUtensorMap tm_bc, const __grid_constant__ CUtensorMap tm_bt,
            const SsdArgs p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float* s_dl = reinterpret_cast<float*>(sm + Smem::DL);
    float* s_cs = reinterpret_cast<float*>(sm + Smem::CS);
    float* s_cw = reinterpret_cast<float*>(sm + Smem::CW);
    float* s_cb = reinterpret_cast<float*>(sm + Smem::CB);
    float* s_ws = reinterpret_cast<float*>(sm + Smem::WS);
    uint64_t* bar_a = reinterpret_cast<uint64_t*>(sm + Smem::BAR);   // raw x + B^T of a chunk
    uint64_t* bar_b = bar_a + 1;                                     // C, B tiles + z of a chunk
    uint64_t* bar_m = bar_a + 2;                                     // MMA completion
    uint32_t* slot = reinterpret_cast<uint32_t*>(sm + Smem::SLOT);
    const uint32_t sb = smem_u32(sm);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, hf = warp >> 2;
    const int i = 32 * q + lane;                     // this thread's token row of the chunk
    const int h = blockIdx.x, b = blockIdx.y;
    const int H = p.n_heads, G = p.n_groups, L = p.seqlen;
    const int g = h / (H / G), BG = p.batch * G, bg = b * G + g;
    const int64_t HP = (int64_t)H * kP, Cx = HP + 2 * (int64_t)G * kNs;
    const int nch = (L + kQ - 1) / kQ;
    const float A2 = p.A[h] * kLog2e, bias = p.dt_bias[h], Dh = p.Dskip[h];
    const Tin_bf16* dtp = reinterpret_cast<const Tin_bf16*>(p.dt) + (int64_t)b * p.dt_stride_b + h;

    if (tid == 0) {
        mbar_init(bar_a, 1);
        mbar_init(bar_b, 1);
        mbar_init(bar_m, 1);
        fence_barrier_init();
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_z);
        prefetch_tmap(&tm_bc);
        prefetch_tmap(&tm_bt);
    }
    if (warp == 0) tmem_alloc(slot, 512);
    if (tid < kP) {
        const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (h * (int64_t)kP + tid) * 4);
        s_cw[4 * tid + 0] = w.x;
        s_cw[4 * tid + 1] = w.y;
        s_cw[4 * tid + 2] = w.z;
        s_cw[4 * tid + 3] = w.w;
        s_cb[tid] = p.conv_b[h * (int64_t)kP + tid];
    }
    // the state S[p][n] for p = i (q < 2), n in [32 hf, 32 hf + 32): fp32 in registers
    float S[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) S[k] = 0.f;
    if (q < 2 && p.ssm_state_in) {
        const float4* src = reinterpret_cast<const float4*>(
            p.ssm_state_in + (((int64_t)b * H + h) * kP + i) * kNs + 32 * hf);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 v = src[k];
            S[4 * k] = v.x; S[4 * k + 1] = v.y; S[4 * k + 2] = v.z; S[4 * k + 3] = v.w;
        }
    }
    // write S as the hi/lo operand tiles [p][n] the first chunk's C S^T reads
    auto store_state = [&]() {
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
            uint32_t whi[4], wlo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                __nv_bfloat16 h0, l0, h1, l1;
                split_bf16(S[8 * c8 + 2 * k], h0, l0);
                split_bf16(S[8 * c8 + 2 * k + 1], h1, l1);
                whi[k] = pack2(h0, h1);
                wlo[k] = pack2(l0, l1);
            }
            const uint32_t off = sw128(i, 32 * hf + 8 * c8);
            *reinterpret_cast<uint4*>(sm + Smem::SHI + off) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
            *reinterpret_cast<uint4*>(sm + Smem::SLO + off) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
        }
    };
    if (q < 2) store_state();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t tG = tmem, tYi = tmem + 128, tYe = tmem + 192, tDS = tmem + 256;

    auto issue_a = [&](int c) {
        const int t0 = c * kQ;
        mbar_arrive_expect_tx(bar_a, Smem::TX_A);
        tma_load_3d(sm + Smem::XR, &tm_x, bar_a, h * kP, t0 - 3, b);
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int r = 0; r < 2; ++r)
                tma_load_3d(sm + (k ? Smem::BTLO : Smem::BTHI) + r * 8192, &tm_bt, bar_a, t0 + 64 * r, 0,
                            k * BG + bg);
    };
    auto issue_b_tiles = [&](int c) {
        const int t0 = c * kQ;
        mbar_arrive_expect_tx(bar_b, Smem::TX_B);
#pragma unroll
        for (int k = 0; k < 4; ++k) tma_load_3d(sm + 16384 * k, &tm_bc, bar_b, 0, t0, k * BG + bg);
    };
    auto issue_b_z = [&](int c) { tma_load_3d(sm + Smem::ZT, &tm_z, bar_b, h * kP, c * kQ, b); };
    if (tid == 0) {
        issue_a(0);
        issue_b_tiles(0);
        issue_b_z(0);
    }

    int waited_a = 0, waited_b = 0, issued_a = 1, issued_b = 1, mma_wait = 0;
    bool bad = false;
    float xv[32];                                    // x of (token i, positions 32 hf ..), fp32
    for (int c = 0; c < nch && !bad; ++c) {
        const int t0 = c * kQ;
        // ---- raw x and B^T of the chunk
        bool ok = mbar_wait_bounded(bar_a, (uint32_t)(waited_a & 1));
        ++waited_a;
        if (__syncthreads_or(!ok)) { bad = true; break; }

        // ---- delta and the chunk-local cumulative decay exponent s (in log2 units)
        if (hf == 0) {
            const int t = t0 + i;
            float dl = 0.f;
            if (t < L) dl = softplus_in<Tin_bf16>(to_f32(dtp[(int64_t)t * p.dt_stride_t]) + bias);
            float v = dl * A2;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (lane == 31) s_ws[q] = v;
            s_dl[i] = dl;
            s_cs[i] = v;
        }
        __syncthreads();
        if (hf == 0) {
            float off = 0.f;
            for (int k = 0; k < q; ++k) off += s_ws[k];
            s_cs[i] += off;
        }
        __syncthreads();
        const float s_i = s_cs[i], s_Q = s_cs[kQ - 1], dl_i = s_dl[i];

        // ---- conv + SiLU of x (token i, positions 32 hf ..), written as X^T hi/lo and the
        //      state-update operand w_i x_i (w_i = 2^(s_Q - s_i) delta_i), hi rows / lo rows
        {
            float r[4][32];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int row = i + k;                    // tile row of token t0 + i - 3 + k
                if (c == 0 && row < 3 && p.conv_state_in) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        r[k][e] = p.conv_state_in[((int64_t)b * 3 + row) * Cx + h * (int64_t)kP + 32 * hf + e];
                } else {
                    const uint4* src = reinterpret_cast<const uint4*>(sm + Smem::XR + row * 128 + 64 * hf);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint4 u = src[e];
                        const uint32_t ws4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            r[k][8 * e + 2 * f] = __uint_as_float(ws4[f] << 16);
                            r[k][8 * e + 2 * f + 1] = __uint_as_float(ws4[f] & 0xffff0000u);
                        }
                    }
                }
            }
            const float wi = ex2(s_Q - s_i) * dl_i;
            const int reg = i >> 6, col = i & 63;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int pp = 32 * hf + e;
                const float* w = s_cw + 4 * pp;
                float xc = fmaf(w[0], r[0][e], s_cb[pp]);
                xc = fmaf(w[1], r[1][e], xc);
                xc = fmaf(w[2], r[2][e], xc);
                xc = fmaf(w[3], r[3][e], xc);
                const float u = silu_in<Tin_bf16>(xc);
                xv[e] = u;
                __nv_bfloat16 hi, lo;
                split_bf16(u, hi, lo);
                st_u16(sm, Smem::XHI + reg * 8192 + sw128(pp, col), hi);
                st_u16(sm, Smem::XLO + reg * 8192 + sw128(pp, col), lo);
                split_bf16(wi * u, hi, lo);
                st_u16(sm, Smem::XW + reg * 16384 + sw128(pp, col), hi);
                st_u16(sm, Smem::XW + reg * 16384 + sw128(64 + pp, col), lo);
            }
        }
        fence_proxy_async_smem();

        // ---- C, B tiles and z of the chunk
        ok = mbar_wait_bounded(bar_b, (uint32_t)(waited_b & 1));
        ++waited_b;
        tc_fence_before();
        if (__syncthreads_or(!ok)) { bad = true; break; }
        if (tid == 0) {
            tc_fence_after();
            // G = C B^T
            mma_k64(tG, sb + Smem::CHI, sb + Smem::BHI, kIdescN128, true);
            mma_k64(tG, sb + Smem::CHI, sb + Smem::BLO, kIdescN128, false);
            mma_k64(tG, sb + Smem::CLO, sb + Smem::BHI, kIdescN128, false);
            // Y_inter = C S_prev^T
            mma_k64(tYe, sb + Smem::CHI, sb + Smem::SHI, kIdescN64, true);
            mma_k64(tYe, sb + Smem::CHI, sb + Smem::SLO, kIdescN64, false);
            mma_k64(tYe, sb + Smem::CLO, sb + Smem::SHI, kIdescN64, false);
            // dS^T = (w x)^T B over the chunk's 128 tokens: rows 0-63 from the hi part of w x,
            // rows 64-127 from its lo part, each times B hi + B lo
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    mma_k64(tDS, sb + Smem::XW + r * 16384, sb + (k ? Smem::BTLO : Smem::BTHI) + r * 8192, kIdescN64,
                            k == 0 && r == 0);
            mma_commit(bar_m);
        }
        ok = mbar_wait_bounded(bar_m, (uint32_t)(mma_wait & 1));
        ++mma_wait;
        if (__syncthreads_or(!ok)) { bad = true; break; }
        tc_fence_after();
        if (tid == 0 && c + 1 < nch) {               // raw x and B^T of the chunk are consumed
            issue_a(c + 1);
            ++issued_a;
        }

        // ---- M = G exp(s_i - s_j) delta_j (j <= i) as hi/lo, over the C and B tiles
        {
            const int j0 = 64 * hf;
            const uint32_t mh = Smem::MHI + hf * 16384, ml = Smem::MLO + hf * 16384;
            if (j0 > 32 * q + 31) {
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint32_t off = (uint32_t)(i * 128 + ((c8 ^ (i & 7)) << 4));
                    *reinterpret_cast<uint4*>(sm + mh + off) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(sm + ml + off) = make_uint4(0, 0, 0, 0);
                }
            } else {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float v[32];
                    tmem_ld32(tG + ((uint32_t)(32 * q) << 16) + (uint32_t)(j0 + 32 * half), v);
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        uint32_t whi[4], wlo[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            __nv_bfloat16 hh[2], ll[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int jl = 8 * c8 + 2 * k + e, j = j0 + 32 * half + jl;
                                const float m = j <= i ? v[jl] * ex2(s_i - s_cs[j]) * s_dl[j] : 0.f;
                                split_bf16(m, hh[e], ll[e]);
                            }
                            whi[k] = pack2(hh[0], hh[1]);
                            wlo[k] = pack2(ll[0], ll[1]);
                        }
                        const int ch = 4 * half + c8;
                        const uint32_t off = (uint32_t)(i * 128 + ((ch ^ (i & 7)) << 4));
                        *reinterpret_cast<uint4*>(sm + mh + off) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
                        *reinterpret_cast<uint4*>(sm + ml + off) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
                    }
                }
            }
        }

        // ---- state: S = 2^(s_Q) S + dS (hi part rows + lo part rows of the accumulator)
        {
            float v[32];
            tmem_ld32(tDS + ((uint32_t)(32 * q) << 16) + (uint32_t)(32 * hf), v);
            float* scr = reinterpret_cast<float*>(sm + Smem::XW);
            if (q >= 2) {
                float4* dst = reinterpret_cast<float4*>(scr + (i - 64) * Smem::SCR_LD + 32 * hf);
#pragma unroll
                for (int k = 0; k < 8; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            }
            tc_fence_before();
            __syncthreads();
            if (q < 2) {
                const float eQ = ex2(s_Q);
                const float4* src = reinterpret_cast<const float4*>(scr + i * Smem::SCR_LD + 32 * hf);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float4 o = src[k];
                    S[4 * k] = fmaf(eQ, S[4 * k], v[4 * k] + o.x);
                    S[4 * k + 1] = fmaf(eQ, S[4 * k + 1], v[4 * k + 1] + o.y);
                    S[4 * k + 2] = fmaf(eQ, S[4 * k + 2], v[4 * k + 2] + o.z);
                    S[4 * k + 3] = fmaf(eQ, S[4 * k + 3], v[4 * k + 3] + o.w);
                }
                store_state();
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- Y_intra = M X
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int r = 0; r < 2; ++r)
                mma_k64(tYi, sb + Smem::MHI + r * 16384, sb + Smem::XHI + r * 8192, kIdescN64, r == 0);
#pragma unroll
            for (int r = 0; r < 2; ++r)
                mma_k64(tYi, sb + Smem::MHI + r * 16384, sb + Smem::XLO + r * 8192, kIdescN64, false);
#pragma unroll
            for (int r = 0; r < 2; ++r)
                mma_k64(tYi, sb + Smem::MLO + r * 16384, sb + Smem::XHI + r * 8192, kIdescN64, false);
            mma_commit(bar_m);
        }
        ok = mbar_wait_bounded(bar_m, (uint32_t)(mma_wait & 1));
        ++mma_wait;
        if (__syncthreads_or(!ok)) { bad = true; break; }
        tc_fence_after();
        if (tid == 0 && c + 1 < nch) issue_b_tiles(c + 1);   // M (over C and B) is consumed

        // ---- out = (Y_intra + 2^(s_i) Y_inter + D x) SiLU(z)
        {
            float yi[32], ye[32];
            tmem_ld32(tYi + ((uint32_t)(32 * q) << 16) + (uint32_t)(32 * hf), yi);
            tmem_ld32(tYe + ((uint32_t)(32 * q) << 16) + (uint32_t)(32 * hf), ye);
            const float ei = ex2(s_i);
            const int t = t0 + i;
            float o[32];
            const uint4* zs = reinterpret_cast<const uint4*>(sm + Smem::ZT + i * 128 + 64 * hf);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint4 u = zs[e];
                const uint32_t ws4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    const int k = 8 * e + 2 * f;
                    const float z0 = __uint_as_float(ws4[f] << 16), z1 = __uint_as_float(ws4[f] & 0xffff0000u);
                    o[k] = fmaf(ei, ye[k], yi[k] + Dh * xv[k]) * silu_in<Tin_bf16>(z0);
                    o[k + 1] = fmaf(ei, ye[k + 1], yi[k + 1] + Dh * xv[k + 1]) * silu_in<Tin_bf16>(z1);
                }
            }
            if (t < L) {
                Tout* dst = reinterpret_cast<Tout*>(p.out) + (int64_t)b * p.out_stride_b + (int64_t)t * p.out_stride_t +
                            (int64_t)h * kP + 32 * hf;
                if constexpr (sizeof(Tout) == 4) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        reinterpret_cast<float4*>(dst)[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t w4[4];
#pragma unroll
                        for (int f = 0; f < 4; ++f)
                            w4[f] = pack2(__float2bfloat16_rn(o[8 * k + 2 * f]), __float2bfloat16_rn(o[8 * k + 2 * f + 1]));
                        reinterpret_cast<uint4*>(dst)[k] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && c + 1 < nch) {               // z of the chunk is consumed
            issue_b_z(c + 1);
            ++issued_b;
        }
    }

    if (bad) {
        if (tid == 0) {
            atomicOr(p.status, 1u);
            // let every copy still in flight land before the CTA's shared memory goes away
            if (issued_a > waited_a) (void)mbar_wait_bounded(bar_a, (uint32_t)(waited_a & 1), 100000000ull);
            if (issued_b > waited_b) (void)mbar_wait_bounded(bar_b, (uint32_t)(waited_b & 1), 100000000ull);
            (void)mbar_wait_bounded(bar_m, (uint32_t)(mma_wait & 1), 100000000ull);
        }
    } else {
        // final SSM state and the x channels' conv window
        if (q < 2) {
            float4* dst = reinterpret_cast<float4*>(p.ssm_state_out + (((int64_t)b * H + h) * kP + i) * kNs + 32 * hf);
#pragma unroll
            for (int k = 0; k < 8; ++k) dst[k] = make_float4(S[4 * k], S[4 * k + 1], S[4 * k + 2], S[4 * k + 3]);
        }
        if (tid < 3 * kP) {
            const int k = tid / kP, pp = tid % kP, t = L - 3 + k;
            const int64_t ch = h * (int64_t)kP + pp;
            float v = 0.f;
            if (t >= 0)
                v = to_f32(reinterpret_cast<const Tin_bf16*>(p.xBC)[(int64_t)b * p.xbc_stride_b + (int64_t)t * p.xbc_stride_t + ch]);
            else if (p.conv_state_in)
                v = p.conv_state_in[((int64_t)b * 3 + 3 + t) * Cx + ch];
            p.conv_state_out[((int64_t)b * 3 + k) * Cx + ch] = v;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ decode
// grid (H, batch), 256 threads: thread (p = tid / 4, quarter tid % 4) owns states n in
// [16 quarter, 16 quarter + 16) of position p.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256)
k_ssd_decode(const SsdDecodeArgs a) {
    __shared__ float u[3 * 64];                     // x of the head, B and C of its group
    const int h = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
    const int H = a.n_heads, G = a.n_groups, g = h / (H / G);
    const int64_t HP = (int64_t)H * kP, Cx = HP + 2 * (int64_t)G * kNs;
    const int slot = a.state_slot ? a.state_slot[r] : r;
    if (slot < 0 || slot >= a.n_slots) {
        if (tid == 0) atomicOr(a.status, 2u);
        return;
    }
    if (tid < 192) {
        const int seg = tid / 64, k = tid % 64;
        const int64_t c = seg == 0 ? h * (int64_t)kP + k : HP + (seg == 2 ? (int64_t)G * kNs : 0) + (int64_t)g * kNs + k;
        float* cs = a.conv_state + (int64_t)slot * 3 * Cx + c;
        const float c0 = cs[0], c1 = cs[Cx], c2 = cs[2 * Cx];
        const float xt = to_f32(reinterpret_cast<const Tin*>(a.xBC)[(int64_t)r * Cx + c]);
        const float4 w = *reinterpret_cast<const float4*>(a.conv_w + c * 4);
        float xc = fmaf(w.x, c0, a.conv_b[c]);
        xc = fmaf(w.y, c1, xc);
        xc = fmaf(w.z, c2, xc);
        xc = fmaf(w.w, xt, xc);
        u[tid] = silu_in<Tin>(xc);
        if (seg == 0) {                              // the head's own x channels move now
            cs[0] = c1;
            cs[Cx] = c2;
            cs[2 * Cx] = xt;
        }
    }
    __syncthreads();
    const float dl = softplus_in<Tin>(to_f32(reinterpret_cast<const Tin*>(a.dt)[(int64_t)r * H + h]) + a.dt_bias[h]);
    const float dA = ex2(dl * a.A[h] * kLog2e);
    const int pp = tid >> 2, n0 = 16 * (tid & 3);
    float4* sp = reinterpret_cast<float4*>(a.ssm_state + (((int64_t)slot * H + h) * kP + pp) * kNs + n0);
    const float dx = dl * u[pp];
    float y = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float4 s = sp[k];
        const float* Bn = u + 64 + n0 + 4 * k;
        const float* Cn = u + 128 + n0 + 4 * k;
        s.x = fmaf(dA, s.x, dx * Bn[0]);
        s.y = fmaf(dA, s.y, dx * Bn[1]);
        s.z = fmaf(dA, s.z, dx * Bn[2]);
        s.w = fmaf(dA, s.w, dx * Bn[3]);
        y = fmaf(Cn[0], s.x, y);
        y = fmaf(Cn[1], s.y, y);
        y = fmaf(Cn[2], s.z, y);
        y = fmaf(Cn[3], s.w, y);
        sp[k] = s;
    }
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    y += __shfl_xor_sync(0xffffffffu, y, 2);
    if ((tid & 3) == 0) {
        const int64_t o = (int64_t)r * HP + h * (int64_t)kP + pp;
        const float zt = to_f32(reinterpret_cast<const Tin*>(a.z)[o]);
        reinterpret_cast<Tout*>(a.out)[o] = from_f32<Tout>(fmaf(a.Dskip[h], u[pp], y) * silu_in<Tin>(zt));
    }
}

// The conv windows of the B and C channels move after every head has read them.
// grid (batch), 256 threads over the 2 G 64 channels.
template <typename Tin>
__global__ void __launch_bounds__(256)
k_ssd_decode_shift(const SsdDecodeArgs a) {
    const int r = blockIdx.x;
    const int slot = a.state_slot ? a.state_slot[r] : r;
    if (slot < 0 || slot >= a.n_slots) return;       // reported by k_ssd_decode
    const int64_t HP = (int64_t)a.n_heads * kP, Cx = HP + 2 * (int64_t)a.n_groups * kNs;
    for (int64_t c = HP + threadIdx.x; c < Cx; c += 256) {
        float* cs = a.conv_state + (int64_t)slot * 3 * Cx + c;
        const float c1 = cs[Cx], c2 = cs[2 * Cx];
        cs[0] = c1;
        cs[Cx] = c2;
        cs[2 * Cx] = to_f32(reinterpret_cast<const Tin*>(a.xBC)[(int64_t)r * Cx + c]);
    }
}

// 3-D bf16 tensor map: dims {d0, d1, d2} (d0 innermost), byte strides {s1, s2}, box {b0, b1, 1}.
bool make_map3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
               uint32_t b0, uint32_t b1, bool swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

}  // namespace

SsdWorkspace ssd_workspace_layout(int batch, int seqlen, int n_groups) {
    SsdWorkspace w{};
    const int64_t BG = (int64_t)batch * n_groups;
    w.lp = round_up(seqlen, kQ);
    w.bt_off = round_up(4 * BG * seqlen * kNs * 2, 256);
    w.bytes = (size_t)(w.bt_off + 2 * BG * kNs * w.lp * 2);
    return w;
}

int launch_ssd_prefill(const SsdArgs& a0, bool out_bf16, cudaStream_t stream, const char** why) {
    SsdArgs a = a0;
    const SsdWorkspace w = ssd_workspace_layout(a.batch, a.seqlen, a.n_groups);
    a.ws_bt_off = w.bt_off;
    a.ws_lp = w.lp;
    const int64_t HP = (int64_t)a.n_heads * kP, Cx = HP + 2 * (int64_t)a.n_groups * kNs;
    const int64_t BG = (int64_t)a.batch * a.n_groups;
    const int L = a.seqlen;

    k_ssd_bc<Tin_bf16><<<dim3((unsigned)((L + 63) / 64), (unsigned)a.n_groups, (unsigned)a.batch), 256, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return -1;
    }

    CUtensorMap mx, mz, mbc, mbt;
    const uint64_t xs_b = a.batch > 1 ? (uint64_t)a.xbc_stride_b * 2 : (uint64_t)L * a.xbc_stride_t * 2;
    const uint64_t zs_b = a.batch > 1 ? (uint64_t)a.z_stride_b * 2 : (uint64_t)L * a.z_stride_t * 2;
    const unsigned char* ws = static_cast<const unsigned char*>(a.workspace);
    if (!make_map3(&mx, a.xBC, (uint64_t)Cx, (uint64_t)L, (uint64_t)a.batch, (uint64_t)a.xbc_stride_t * 2, xs_b, kP,
                   kQ + 3, false) ||
        !make_map3(&mz, a.z, (uint64_t)HP, (uint64_t)L, (uint64_t)a.batch, (uint64_t)a.z_stride_t * 2, zs_b, kP, kQ,
                   false) ||
        !make_map3(&mbc, ws, kNs, (uint64_t)L, (uint64_t)(4 * BG), kNs * 2, (uint64_t)L * kNs * 2, kNs, kQ, true) ||
        !make_map3(&mbt, ws + w.bt_off, (uint64_t)L, kNs, (uint64_t)(2 * BG), (uint64_t)w.lp * 2,
                   (uint64_t)w.lp * kNs * 2, 64, kNs, true)) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point missing or layout rejected)";
        return -1;
    }
    auto kern = out_bf16 ? k_ssd_chunk<__nv_bfloat16> : k_ssd_chunk<float>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        *why = "cudaGetDevice failed";
        return -1;
    }
    static unsigned long long done[2] = {0, 0};
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&done[out_bf16], __ATOMIC_ACQUIRE) & bit)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::ALLOC) != cudaSuccess) {
            *why = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize) failed";
            return -1;
        }
        __atomic_fetch_or(&done[out_bf16], bit, __ATOMIC_ACQ_REL);
    }
    kern<<<dim3((unsigned)a.n_heads, (unsigned)a.batch), kTh, Smem::ALLOC, stream>>>(mx, mz, mbc, mbt, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return -1;
    }
    return 0;
}

int launch_ssd_decode(const SsdDecodeArgs& a, bool in_bf16, bool out_bf16, cudaStream_t stream, const char** why) {
    const dim3 grid((unsigned)a.n_heads, (unsigned)a.batch);
    if (in_bf16) {
        if (out_bf16) k_ssd_decode<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, stream>>>(a);
        else k_ssd_decode<__nv_bfloat16, float><<<grid, 256, 0, stream>>>(a);
        k_ssd_decode_shift<__nv_bfloat16><<<a.batch, 256, 0, stream>>>(a);
    } else {
        if (out_bf16) k_ssd_decode<float, __nv_bfloat16><<<grid, 256, 0, stream>>>(a);
        else k_ssd_decode<float, float><<<grid, 256, 0, stream>>>(a);
        k_ssd_decode_shift<float><<<a.batch, 256, 0, stream>>>(a);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return -1;
    }
    return 0;
}

}  // namespace ssm
