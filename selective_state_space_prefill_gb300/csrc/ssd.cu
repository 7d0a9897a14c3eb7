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
//   M[i][j] = G[i][j] exp(s_i - s_j) delta_j    (j < i, else 0),  M[i][i] = G[i][i] delta_i + D
//   Y = M X + exp(s)_i (C S_prev^T)              (X = the chunk's x, [Q x 64]; D x rides on M's diagonal)
//   S = exp(s_Q) S_prev + sum_j exp(s_Q - s_j) delta_j x_j (x) B_j
// Those four products run on the 5th-generation tensor cores (tcgen05, kind::f16, M = 128,
// fp32 accumulators in TMEM).  bf16 operands alone would round x, B, C, M and S by 2^-9 each,
// far above the mixer's error budget, so every operand is carried as a bf16 pair hi + lo
// (hi = bf16(v), lo = bf16(v - hi), |v - hi - lo| <= 2^-17 |v|) and each product is the sum
// hi*hi + hi*lo + lo*hi.
//
// Kernels:
//   k_ssd_pre     (pre-pass) conv + SiLU of every group's B and C channels, written as hi/lo
//                 planes [t][n] (the K-major operands of C B^T and C S^T) and, for B, also as
//                 token-major planes [n][t] (the K-major operand of the state update); and, in
//                 the same launch, delta and the chunk-local decay sums of every head.
//   k_ssd_chunk   a CTA walks chunks of (batch row, head) pairs in order, so the fp32 state
//                 stays on chip: a producer warp brings the raw x (with a 3-token conv halo), z,
//                 the B/C tiles and the chunk's delta and decay sums by TMA and issues the MMAs;
//                 16 worker warps compute the x conv and the operands they own (X, the
//                 state-update weights, M, S) into 128-byte-swizzled shared memory, read the
//                 accumulators back with tcgen05.ld, and send the output tile out by TMA stores.
//                 With no more rows than resident CTAs there is one CTA per row; with more, one
//                 CTA per SM takes an equal span of all rows' chunks (no partly filled last
//                 wave), and a row cut between two CTAs passes its state through the workspace.
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
constexpr int kTh = 512;       // threads of k_ssd_chunk: warp w reads TMEM lanes 32 (w % 4) .. + 31
constexpr int kWG = kTh / 128; // column groups: warp w works on column group w / 4 of its rows
constexpr int kCW = kP / kWG;  // columns of x, y, S per thread (16)
constexpr int kMJ = kQ / kWG;  // columns of M per thread (32)
static_assert(kCW % 8 == 0 && kMJ % 32 == 0, "column split");

// tcgen05.mma kind::f16 instruction descriptors: fp32 accumulator, bf16 A and B, both K-major,
// M = 128, N = 128 or 64.
constexpr uint32_t kIdescN128 = (1u << 4) | (1u << 7) | (1u << 10) | (16u << 17) | (8u << 24);
constexpr uint32_t kIdescN64 = (1u << 4) | (1u << 7) | (1u << 10) | (8u << 17) | (8u << 24);
// ... with A (bit 15) or B (bit 16) MN-major: the operand's rows run along K, its M or N
// elements contiguous in each 128-byte row
constexpr uint32_t kIdescN64_AMN = kIdescN64 | (1u << 15);
constexpr uint32_t kIdescN64_BMN = kIdescN64 | (1u << 16);
constexpr uint32_t kIdescN128_BMN = kIdescN128 | (1u << 16);

// Shared memory of k_ssd_chunk (byte offsets from a 1024-aligned base).  Operand tiles are
// K-major rows of 64 bf16 (128 bytes) in 128-byte-swizzle atoms; a K extent of 128 is two such
// regions ("r0", "r1").
struct Smem {
    static constexpr int CHI = 0, CLO = 16384, BHI = 32768, BLO = 49152;  // [128 t][64 n] (TMA)
    static constexpr int MHI = 0, MLO = 32768;       // M hi / lo, r0 and r1 [128 i][64 j] each (over C, B)
    static constexpr int BTHI = 65536, BTLO = 81920; // B^T hi / lo, r0 and r1 [64 n][64 t] each (TMA)
    static constexpr int XHI = 98304, XLO = 114688;  // X hi / lo [128 t][64 p] (MN-major operand); once
                                                     // Y_intra has run, the output tile for the TMA store
    static constexpr int XW = 131072;                // w x hi [128 t][64 p], then w x lo at XW + 16384
                                                     // (MN-major operand); later fp32 scratch
    static constexpr int SHI = 163840, SLO = 172032; // S hi / lo [64 p][64 n]
    static constexpr int XR = 180224;                // raw x [131 t][64 p] bf16 (TMA, 128-byte swizzle)
    static constexpr int ZT = 197632;                // z [128 t][64 p] bf16 (TMA, 128-byte swizzle)
    static constexpr int DL = 214016;                // delta [2][128] f32 (by chunk parity, TMA)
    static constexpr int CS = DL + 1024;             // s (chunk-local cumulative delta*A) [2][128] f32 (TMA)
    static constexpr int CW = CS + 1024;             // conv weights of the head's x channels [64][4]
    static constexpr int CB = CW + 1024;             // conv bias [64]
    static constexpr int BAR = CB + 256;             // nine mbarriers (TMA, MMA groups, hand-offs)
    static constexpr int SLOT = BAR + 80;            // TMEM base address, error flag
    static constexpr int SPAN = SLOT + 16;           // the CTA's span of chunks (SsdSpan, 64 bytes), the
    static constexpr int ITEM = SPAN + 64;           // current item (b, h, c0, c1)
    static constexpr int DH = ITEM + 16;             // and D of its head
    static constexpr int EC = DH + 16;               // column factors 2^(s_last - s_j) delta_j of the
                                                     // three 32-column blocks that can lie wholly
                                                     // below a warp's rows [96] f32
    static constexpr int TOTAL = EC + 512;
    static constexpr int ALLOC = TOTAL + 1024;       // + slack to align the base to 1024
    static constexpr int XR_BYTES = (kQ + 3) * kP * 2;
    static constexpr int TX_A = XR_BYTES + 4 * 8192 + 2 * 512;   // raw x + B^T hi/lo + delta, s
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

// Four K-steps (K = 64) of D (+)= A B^T for K-major operands at shared addresses a, b.
// Descriptor of an MN-major tile with 128-byte swizzling: rows of 128 bytes run along K, groups of
// 8 rows are 1024 bytes apart (stride byte offset) and a second block of 64 M or N elements starts
// `lbo` bytes after the first (leading byte offset).  A K-step of 16 rows advances it 2048 bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// The descriptor's address field counts 16-byte units, so a 32-byte K-step adds 2 to it.
__device__ __forceinline__ void mma_k64(uint32_t d, uint32_t a, uint32_t b, uint32_t idesc, bool first) {
    const uint64_t da = smem_desc_sw128(a), db = smem_desc_sw128(b);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_bf16(d, da + 2 * kk, db + 2 * kk, idesc, (first && kk == 0) ? 0u : 1u);
}

// ------------------------------------------------------------------ pre-pass: B and C
// One block of 256 threads: kBcT tokens (block bx of nbx) x 64 states of group g of row b.  The
// raw B and C channels of the block's tokens and their 3-token halo are staged in shared memory
// with 16-byte loads first; the conv then reads them from there.
constexpr int kBcT = 32;
template <typename Tin>
__device__ __forceinline__ void ssd_bc_block(const SsdArgs& p, int bx, int nbx, int g, int b) {
    __shared__ __align__(16) __nv_bfloat16 raw_s[kBcT + 3][2][kNs];  // token row x (C, B) x state
    __shared__ float hist[3][2][kNs];                                 // conv_state_in rows (first block)
    __shared__ __nv_bfloat16 tr[2][kNs][kBcT + 8];                    // B hi / lo of the block, state-major
    const int t0 = bx * kBcT;
    const int G = p.n_groups, BG = p.batch * G, bg = b * G + g, L = p.seqlen;
    const int64_t HP = (int64_t)p.n_heads * kP, Cx = HP + 2 * (int64_t)G * kNs;
    const Tin* xb = reinterpret_cast<const Tin*>(p.xBC) + (int64_t)b * p.xbc_stride_b;
    __nv_bfloat16* bc = reinterpret_cast<__nv_bfloat16*>(p.workspace);
    __nv_bfloat16* bt = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<unsigned char*>(p.workspace) + p.ws_bt_off);
    auto chan = [&](int which, int n) -> int64_t {                    // 0: C, 1: B
        return HP + (which ? 0 : (int64_t)G * kNs) + (int64_t)g * kNs + n;
    };
    // rows r = 0 .. kBcT + 2 hold tokens t0 - 3 + r; 8 bf16 per 16-byte vector, 8 vectors per 64
    // states.  Every load of a thread is issued before the first store, so their latencies overlap.
    constexpr int kVec = (kBcT + 3) * 2 * 8, kPer = (kVec + 255) / 256;
    uint4 val[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = threadIdx.x + 256 * j;
        const int r = e / 16, which = (e / 8) & 1, v = e & 7, t = t0 - 3 + r;
        val[j] = make_uint4(0, 0, 0, 0);
        if (e < kVec && t >= 0 && t < L)
            val[j] = *reinterpret_cast<const uint4*>(xb + (int64_t)t * p.xbc_stride_t + chan(which, 8 * v));
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = threadIdx.x + 256 * j;
        if (e < kVec) *reinterpret_cast<uint4*>(&raw_s[e / 16][(e / 8) & 1][8 * (e & 7)]) = val[j];
    }
    if (t0 == 0 && threadIdx.x < 2 * kNs) {
        const int which = threadIdx.x / kNs, n = threadIdx.x % kNs;
#pragma unroll
        for (int k = 0; k < 3; ++k)
            hist[k][which][n] = p.conv_state_in ? p.conv_state_in[((int64_t)b * 3 + k) * Cx + chan(which, n)] : 0.f;
    }
    __syncthreads();
    auto rawv = [&](int r, int which, int n) -> float {               // token t0 - 3 + r
        return (t0 == 0 && r < 3) ? hist[r][which][n] : __bfloat162float(raw_s[r][which][n]);
    };
    {
        // thread: channel n of C (which 0) or B (which 1), the half of the block's tokens `half`;
        // the conv window moves along in registers and the plane pointers by one row
        constexpr int kHalf = kBcT / 2;
        const int n = threadIdx.x & 63, which = (threadIdx.x >> 6) & 1, half = threadIdx.x >> 7;
        const int64_t c = chan(which, n);
        const float4 w = *reinterpret_cast<const float4*>(p.conv_w + c * 4);
        const float cb = p.conv_b[c];
        const int kind = which ? 2 : 0;
        const int tl0 = kHalf * half;
        __nv_bfloat16* hi_p = bc + (((int64_t)kind * BG + bg) * L + t0 + tl0) * kNs + n;
        __nv_bfloat16* lo_p = bc + (((int64_t)(kind + 1) * BG + bg) * L + t0 + tl0) * kNs + n;
        float x0 = rawv(tl0, which, n), x1 = rawv(tl0 + 1, which, n), x2 = rawv(tl0 + 2, which, n);
        const int n_tok = min(kHalf, L - t0 - tl0);
#pragma unroll 4
        for (int k = 0; k < n_tok; ++k) {
            const float x3 = rawv(tl0 + k + 3, which, n);
            float xc = fmaf(w.x, x0, cb);
            xc = fmaf(w.y, x1, xc);
            xc = fmaf(w.z, x2, xc);
            xc = fmaf(w.w, x3, xc);
            __nv_bfloat16 hi, lo;
            split_bf16(silu_in<Tin>(xc), hi, lo);
            hi_p[(int64_t)k * kNs] = hi;
            lo_p[(int64_t)k * kNs] = lo;
            if (which) {
                tr[0][n][tl0 + k] = hi;
                tr[1][n][tl0 + k] = lo;
            }
            x0 = x1;
            x1 = x2;
            x2 = x3;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 2 * kNs * kBcT; e += 256) {
        const int k = e / (kNs * kBcT), n = (e / kBcT) % kNs, tl = e % kBcT, t = t0 + tl;
        if (t < L) bt[(((int64_t)k * BG + bg) * kNs + n) * p.ws_lp + t] = tr[k][n][tl];
    }
    // the conv window of the B and C channels after the last token
    if (bx == nbx - 1 && threadIdx.x < 2 * kNs) {
        const int which = threadIdx.x / kNs, n = threadIdx.x % kNs;
        const int64_t c = chan(which, n);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int t = L - 3 + k;
            p.conv_state_out[((int64_t)b * 3 + k) * Cx + c] =
                t >= 0 ? to_f32(xb[(int64_t)t * p.xbc_stride_t + c])
                       : (p.conv_state_in ? p.conv_state_in[((int64_t)b * 3 + 3 + t) * Cx + c] : 0.f);
        }
    }
}

// ------------------------------------------------------------------ pre-pass: delta and s
// One warp per (batch row b, head h, 128-token chunk cx); lane l takes tokens [4 l, 4 l + 4) of
// the chunk: delta = softplus(dt + dt_bias) (0 past L) and s, the running sum of delta A log2(e)
// from the chunk's start (constant past L).  The lanes' partial sums meet in a warp scan, and
// each plane's chunk row leaves as one contiguous 512-byte store of the warp.
__device__ __forceinline__ void ssd_dt_warp(const SsdArgs& p, int cx, int b, int h) {
    const int lane = threadIdx.x & 31, L = p.seqlen;
    const int t0 = cx * kQ + 4 * lane;
    const uint16_t* dtp = reinterpret_cast<const uint16_t*>(p.dt) + (int64_t)b * p.dt_stride_b + h;
    const float bias = p.dt_bias[h], A2 = p.A[h] * kLog2e;
    uint16_t raw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) raw[k] = t0 + k < L ? dtp[(int64_t)(t0 + k) * p.dt_stride_t] : (uint16_t)0;
    float d[4], s[4], run = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        d[k] = t0 + k < L ? softplus_in<Tin_bf16>(__uint_as_float((uint32_t)raw[k] << 16) + bias) : 0.f;
        run = fmaf(d[k], A2, run);
        s[k] = run;
    }
    // exclusive sum of the earlier lanes' totals
    float inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
    }
    const float off = inc - run;
    float* dl = reinterpret_cast<float*>(static_cast<unsigned char*>(p.workspace) + p.ws_ds_off) +
                ((int64_t)b * p.n_heads + h) * p.ws_lp + t0;
    float* sc = dl + (int64_t)p.batch * p.n_heads * p.ws_lp;
    *reinterpret_cast<float4*>(dl) = make_float4(d[0], d[1], d[2], d[3]);
    *reinterpret_cast<float4*>(sc) = make_float4(s[0] + off, s[1] + off, s[2] + off, s[3] + off);
}

// Both pre-passes in one launch, so that they run side by side: blocks [0, n_bc) convolve B and C
// (grid ceil(L / kBcT) x G x batch, flattened); the rest hold eight delta-and-s warps each, warp w
// on head w % H of row (w / H) % batch, chunk w / (H batch): a block's warps are neighbouring
// heads, whose dt values share each token's row.
__global__ void __launch_bounds__(256)
k_ssd_pre(const SsdArgs p, int nbx, int n_bc, int ncx) {
    const int blk = blockIdx.x;
    if (blk == 0) {                                  // the chunk kernel's hand-off flags start clear
        unsigned int* flags = reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(p.workspace) + p.ws_flag_off);
        for (int e = threadIdx.x; e < p.n_slots; e += 256) flags[e] = 0u;
    }
    if (blk < n_bc) {
        const int bx = blk % nbx, g = (blk / nbx) % p.n_groups, b = blk / (nbx * p.n_groups);
        ssd_bc_block<Tin_bf16>(p, bx, nbx, g, b);
    } else {
        const int64_t w = (int64_t)(blk - n_bc) * 8 + (threadIdx.x >> 5);
        const int64_t HB = (int64_t)p.n_heads * p.batch;
        if (w < (int64_t)ncx * HB) ssd_dt_warp(p, (int)(w / HB), (int)((w / p.n_heads) % p.batch), (int)(w % p.n_heads));
    }
}

// ------------------------------------------------------------------ prefill chunks
// Warps 0-15 ("workers") own the arithmetic on the threads; warp 16 ("producer", one elected
// lane) issues every TMA copy and tcgen05.mma.  A chunk runs in phases; the tensor cores work on
// one group of products while the workers work on the next:
//   workers                                         producer
//   2. (raw x, delta, s) conv + SiLU -> X, w x       1. (C, B tiles; previous chunk done)
//      -> "X ready"                                     G = C B^T, Y_inter = C S_prev^T; z
//   3. (G) M -> over the C, B tiles -> "M ready"     2. (X ready) dS^T = (w x)^T B
//   4. (dS) S = 2^(s_Q) S + dS -> S tiles            3. (M ready) Y_intra = M X
//   5. (Y_intra, z) out = (Y_intra + 2^(s_i) Y_inter) 4. (dS) refill raw x, B^T, delta, s
//      SiLU(z) -> over X -> TMA store -> "chunk done" 5. (Y_intra) refill C, B
// Each TMA group, MMA group and hand-off completes its own mbarrier once per chunk.  Every wait
// is bounded; a worker whose wait expires keeps walking the chunk without waiting and the error
// is OR-reduced at the next worker barrier, so no warp is ever left waiting at a barrier.
constexpr int kWorkers = kTh;                        // 512 worker threads
constexpr int kThAll = kTh + 32;                     // + the producer warp

__device__ __forceinline__ void workers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kWorkers) : "memory"); }
__device__ __forceinline__ bool workers_any(bool v) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((uint32_t)v), "n"(kWorkers) : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ work split
// The chunks of all (batch row, head) pairs, flattened row-major (unit u = row * nch + c, row =
// b H + h), are cut into gridDim.x contiguous spans of near-equal length, one per CTA.  A CTA
// walks the pieces of rows ("items") its span covers; the state stays on chip within an item.
// With more rows than CTAs every span holds at least nch units, so a row is cut at most once:
// its head (chunks [0, c)) ends CTA i's span and its tail starts CTA i+1's.  CTA i walks that
// head first and CTA i+1 the tail last, and the state at the cut passes through hand-off slot i
// of the workspace behind a release/acquire flag; the tail's wait is then normally over before
// it starts.  With no more rows than CTAs the launch has one CTA per row and nothing is cut.
struct SsdItem {
    int b, h, c0, c1;                                // chunks [c0, c1) of row (b, h)
};

struct SsdSpan {
    int64_t u0, u1;                                  // units [u0, u1)
    int nch, H, rf, rl;                              // chunks per row, heads, first and last row
    bool head, tail;                                 // the span ends inside row rl / starts inside row rf

    __device__ SsdSpan(int64_t rows, int nch_, int H_, int cta, int n_cta) : nch(nch_), H(H_) {
        const int64_t total = rows * nch_;
        const int64_t q = total / n_cta, r = total % n_cta;   // floor(i total / n) without overflow
        u0 = q * cta + r * cta / n_cta;
        u1 = q * (cta + 1) + r * (cta + 1) / n_cta;
        if (u1 <= u0) {
            rf = 0;
            rl = -1;
            head = tail = false;
            return;
        }
        rf = (int)(u0 / nch_);
        rl = (int)((u1 - 1) / nch_);
        head = u1 < (int64_t)(rl + 1) * nch_;
        tail = u0 > (int64_t)rf * nch_;
    }
    __device__ int n_items() const { return rl - rf + 1; }
    // items in walking order: the head of a row the next CTA continues first, then whole rows,
    // then the tail of a row the previous CTA began
    __device__ SsdItem item(int j) const {
        const int n = rl - rf + 1;
        int r;
        if (head && j == 0) r = rl;
        else if (tail && j == n - 1) r = rf;
        else r = rf + (tail ? 1 : 0) + (j - (head ? 1 : 0));
        const int64_t base = (int64_t)r * nch;
        SsdItem it;
        it.b = r / H;
        it.h = r % H;
        it.c0 = (int)(u0 > base ? u0 - base : 0);
        it.c1 = (int)(u1 - base < nch ? u1 - base : nch);
        return it;
    }
};

static_assert(sizeof(SsdSpan) <= Smem::ITEM - Smem::SPAN, "the span overlaps the item");
static_assert(Smem::ITEM % 16 == 0 && Smem::SPAN % 8 == 0, "span and item alignment");

__device__ __forceinline__ void st_release_gpu(unsigned int* p, unsigned int v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Bounded wait for a hand-off flag to turn non-zero; returns the flag (0 if the wait ran out).
__device__ __forceinline__ unsigned int flag_wait_bounded(const unsigned int* f, uint64_t limit_ns = 2000000000ull) {
    unsigned int v = ld_acquire_gpu(f);
    if (v) return v;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(256);
        v = ld_acquire_gpu(f);
        if (v) return v;
        if (globaltimer_ns() - t0 > limit_ns) return 0u;
    }
}

// hi/lo bf16 pairs of two floats, packed as (lo element in the low half)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

template <typename Tout>
__global__ void __launch_bounds__(kThAll, 1)
k_ssd_chunk(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
            const __grid_constant__ CUtensorMap tm_bc, const __grid_constant__ CUtensorMap tm_bt,
            const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_ds,
            const SsdArgs p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float* s_cw = reinterpret_cast<float*>(sm + Smem::CW);
    float* s_cb = reinterpret_cast<float*>(sm + Smem::CB);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Smem::BAR);
    // TMA groups (raw x + B^T, C/B tiles, z), MMA groups (G + Y_inter, dS, Y_intra), hand-offs
    enum { kBarA = 0, kBarB, kBarZ, kBarG, kBarD, kBarY, kXReady, kMReady, kDone, NBAR };
    uint32_t* slot = reinterpret_cast<uint32_t*>(sm + Smem::SLOT);
    int* s_err = reinterpret_cast<int*>(sm + Smem::SLOT + 4);
    const uint32_t sb = smem_u32(sm);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool producer = warp == kWorkers / 32;
    const int q = warp & 3, cg = (warp >> 2) & (kWG - 1);
    const int i = 32 * q + lane;                     // a worker's token row of the chunk
    const int H = p.n_heads, G = p.n_groups, L = p.seqlen;
    const int BG = p.batch * G, HG = H / G;
    const int64_t HP = (int64_t)H * kP, Cx = HP + 2 * (int64_t)G * kNs;
    const int nch = (L + kQ - 1) / kQ;
    // the span lives in shared memory and each item's (b, h, c0, c1) beside it, so that the
    // workers keep only the step and chunk counters in registers across the chunk loop
    SsdSpan* s_span = reinterpret_cast<SsdSpan*>(sm + Smem::SPAN);
    int* s_item = reinterpret_cast<int*>(sm + Smem::ITEM);        // b, h, c0, c1
    float* s_Dh = reinterpret_cast<float*>(sm + Smem::DH);
    // the hand-off slots [n_slots][64][64] and their flags [n_slots] in the workspace
    auto slot_state = [&](int k) {
        return reinterpret_cast<float*>(static_cast<unsigned char*>(p.workspace) + p.ws_ho_off) + (int64_t)k * kP * kNs;
    };
    auto slot_flag = [&](int k) {
        return reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(p.workspace) + p.ws_flag_off) + k;
    };

    if (tid == 0) {
        for (int k = 0; k < NBAR; ++k) mbar_init(&bars[k], k >= kXReady ? kWorkers / 32 : 1);
        *s_span = SsdSpan((int64_t)p.batch * H, nch, H, (int)blockIdx.x, (int)gridDim.x);
        *s_err = 0;
        fence_barrier_init();
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_z);
        prefetch_tmap(&tm_bc);
        prefetch_tmap(&tm_bt);
    }
    if (warp == 0) tmem_alloc(slot, 512);
    __syncthreads();                                 // the span is in shared memory
    const int n_items = s_span->n_items();
    const int n_steps = (int)(s_span->u1 - s_span->u0);   // chunks this CTA walks
    // the state S[p][n] for p = i (workers with q < 2), n in [kCW cg, kCW cg + kCW): fp32 registers
    float S[kCW];
#pragma unroll
    for (int k = 0; k < kCW; ++k) S[k] = 0.f;
    bool bad = false;                                // (workers) a wait of this worker ran out
    // S as the hi/lo operand tiles [p][n] that C S^T reads
    auto store_state = [&]() {
#pragma unroll
        for (int c8 = 0; c8 < kCW / 8; ++c8) {
            uint32_t whi[4], wlo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) split2(S[8 * c8 + 2 * k], S[8 * c8 + 2 * k + 1], whi[k], wlo[k]);
            const uint32_t off = sw128(i, kCW * cg + 8 * c8);
            *reinterpret_cast<uint4*>(sm + Smem::SHI + off) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
            *reinterpret_cast<uint4*>(sm + Smem::SLO + off) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
        }
    };
    // (workers) an item's per-head parameters and start state: the conv weights of the head's x
    // channels, D, and S -- from ssm_state_in (or zeros) at a row's start, else from the hand-off
    // slot of the CTA that walked the row's head.  Ends with a worker barrier.
    auto begin_item = [&](int jt) {
        const SsdItem it = s_span->item(jt);
        if (tid == 0) {
            s_item[0] = it.b;
            s_item[1] = it.h;
            s_item[2] = it.c0;
            s_item[3] = it.c1;
            *s_Dh = p.Dskip[it.h];
        }
        if (tid < kP) {
            const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (it.h * (int64_t)kP + tid) * 4);
            s_cw[4 * tid + 0] = w.x;
            s_cw[4 * tid + 1] = w.y;
            s_cw[4 * tid + 2] = w.z;
            s_cw[4 * tid + 3] = w.w;
            s_cb[tid] = p.conv_b[it.h * (int64_t)kP + tid];
        }
        const float* src = nullptr;
        if (it.c0 == 0) {
            if (p.ssm_state_in) src = p.ssm_state_in + ((int64_t)it.b * H + it.h) * kP * kNs;
        } else {
            unsigned int f = 1u;
            if (tid == 0) {
                f = flag_wait_bounded(slot_flag(blockIdx.x - 1));
                if (f == 0u) atomicOr(p.status, 1u);
            }
            if (workers_any(f != 1u)) bad = true;
            __threadfence();
            src = slot_state(blockIdx.x - 1);
        }
        if (q < 2) {
            if (src) {
                const float4* s4 = reinterpret_cast<const float4*>(src + (int64_t)i * kNs + kCW * cg);
#pragma unroll
                for (int k = 0; k < kCW / 4; ++k) {
                    const float4 v = __ldcg(s4 + k);
                    S[4 * k] = v.x; S[4 * k + 1] = v.y; S[4 * k + 2] = v.z; S[4 * k + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int k = 0; k < kCW; ++k) S[k] = 0.f;
            }
            store_state();
        }
        fence_proxy_async_smem();
        workers_sync();
    };
    // (workers) an item's end: at a row's end the final SSM state and the conv window of the head's
    // x channels; else the state into this CTA's hand-off slot and its flag raised (2: an error).
    auto end_item = [&]() {
        const SsdItem it = {s_item[0], s_item[1], s_item[2], s_item[3]};
        if (it.c1 == nch) {
            if (bad) {
                atomicOr(p.status, 1u);
                return;
            }
            if (q < 2) {
                float4* dst = reinterpret_cast<float4*>(p.ssm_state_out + (((int64_t)it.b * H + it.h) * kP + i) * kNs +
                                                        kCW * cg);
#pragma unroll
                for (int k = 0; k < kCW / 4; ++k) dst[k] = make_float4(S[4 * k], S[4 * k + 1], S[4 * k + 2], S[4 * k + 3]);
            }
            if (tid < 3 * kP) {
                const int k = tid / kP, pp = tid % kP, t = L - 3 + k;
                const int64_t ch = it.h * (int64_t)kP + pp;
                float v = 0.f;
                if (t >= 0)
                    v = to_f32(reinterpret_cast<const Tin_bf16*>(p.xBC)[(int64_t)it.b * p.xbc_stride_b + (int64_t)t * p.xbc_stride_t + ch]);
                else if (p.conv_state_in)
                    v = p.conv_state_in[((int64_t)it.b * 3 + 3 + t) * Cx + ch];
                p.conv_state_out[((int64_t)it.b * 3 + k) * Cx + ch] = v;
            }
        } else {
            if (q < 2) {
                float4* dst = reinterpret_cast<float4*>(slot_state(blockIdx.x) + (int64_t)i * kNs + kCW * cg);
#pragma unroll
                for (int k = 0; k < kCW / 4; ++k) __stcg(dst + k, make_float4(S[4 * k], S[4 * k + 1], S[4 * k + 2], S[4 * k + 3]));
            }
            __threadfence();
            const bool any_bad = workers_any(bad);
            if (tid == 0) st_release_gpu(slot_flag(blockIdx.x), any_bad ? 2u : 1u);
        }
    };
    if (!producer && n_items > 0) begin_item(0);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    // accumulators: G (128 columns), Y_intra and Y_inter (128 each: the hi*hi (+ lo*hi) products in
    // columns 0-63, the hi*lo products in 64-127), dS^T (64)
    const uint32_t tG = tmem, tYi = tmem + 128, tYe = tmem + 256, tDS = tmem + 384;

    if (producer) {
        if (lane == 0) {
            // the copies of chunk c of item `it`, the kk-th chunk this CTA walks
            auto issue_a = [&](const SsdItem& it, int c, int kk) {   // raw x (3-token halo), B^T hi/lo
                const int t0 = c * kQ, bg = it.b * G + it.h / HG;
                mbar_arrive_expect_tx(&bars[kBarA], Smem::TX_A);
                tma_load_3d(sm + Smem::XR, &tm_x, &bars[kBarA], it.h * kP, t0 - 3, it.b);
                // delta and s of the chunk into the parity buffers
                tma_load_3d(sm + Smem::DL + (kk & 1) * 512, &tm_ds, &bars[kBarA], t0, it.b * H + it.h, 0);
                tma_load_3d(sm + Smem::CS + (kk & 1) * 512, &tm_ds, &bars[kBarA], t0, p.batch * H + it.b * H + it.h, 0);
                for (int k = 0; k < 2; ++k)
                    for (int r = 0; r < 2; ++r)
                        tma_load_3d(sm + (k ? Smem::BTLO : Smem::BTHI) + r * 8192, &tm_bt, &bars[kBarA],
                                    t0 + 64 * r, 0, k * BG + bg);
            };
            auto issue_b = [&](const SsdItem& it, int c) {           // C hi, C lo, B hi, B lo
                const int bg = it.b * G + it.h / HG;
                mbar_arrive_expect_tx(&bars[kBarB], 4 * 16384);
                for (int k = 0; k < 4; ++k) tma_load_3d(sm + 16384 * k, &tm_bc, &bars[kBarB], 0, c * kQ, k * BG + bg);
            };
            auto issue_z = [&](const SsdItem& it, int c) {
                mbar_arrive_expect_tx(&bars[kBarZ], kQ * kP * 2);
                tma_load_3d(sm + Smem::ZT, &tm_z, &bars[kBarZ], it.h * kP, c * kQ, it.b);
            };
            // phase parity of the c-th completion of a once-per-chunk barrier
            auto wait = [&](int k, int c) -> bool {
                if (mbar_wait_bounded(&bars[k], (uint32_t)(c & 1))) return true;
                *reinterpret_cast<volatile int*>(s_err) = 1;
                atomicOr(p.status, 1u);
                return false;
            };
            int ia = 0, ib = 0, iz = 0;              // copies issued per group
            int ng = 0, nd = 0, ny = 0;              // MMA groups committed
            SsdItem it = n_items > 0 ? s_span->item(0) : SsdItem{0, 0, 0, 0};
            int jt = 0, c = it.c0;                   // item and chunk of step ks
            if (n_steps > 0) {
                issue_b(it, c);
                issue_a(it, c, 0);
                issue_z(it, c);
                ia = ib = iz = 1;
            }
            int ks = 0;
            for (; ks < n_steps; ++ks) {
                if (!wait(kBarB, ks)) break;
                if (ks > 0) {
                    if (!wait(kDone, ks - 1)) break; // every worker is past step ks-1
                    issue_z(it, c);
                    ++iz;
                }
                tc_fence_after();
                mma_k64(tG, sb + Smem::CHI, sb + Smem::BHI, kIdescN128, true);
                mma_k64(tG, sb + Smem::CHI, sb + Smem::BLO, kIdescN128, false);
                mma_k64(tG, sb + Smem::CLO, sb + Smem::BHI, kIdescN128, false);
                // Y_inter: C hi against S hi and S lo stacked along N (the two tiles are adjacent),
                // then C lo against S hi into the first half
                mma_k64(tYe, sb + Smem::CHI, sb + Smem::SHI, kIdescN128, true);
                mma_k64(tYe, sb + Smem::CLO, sb + Smem::SHI, kIdescN64, false);
                mma_commit(&bars[kBarG]);
                ++ng;
                if (!wait(kXReady, ks)) break;
                tc_fence_after();
                // dS^T = (w x)^T B: rows 0-63 from the hi part of w x, rows 64-127 from its lo part
                // (the MN-major A operand's two 64-row blocks), each times B hi + B lo
                {
                    const uint64_t da = smem_desc_sw128_mn(sb + Smem::XW, 16384);
#pragma unroll
                    for (int k = 0; k < 2; ++k)
#pragma unroll
                        for (int k16 = 0; k16 < kQ / 16; ++k16) {
                            const uint64_t db = smem_desc_sw128(sb + (k ? Smem::BTLO : Smem::BTHI) + (k16 >> 2) * 8192 +
                                                                32 * (k16 & 3));
                            mma_bf16(tDS, da + (uint64_t)(2048 >> 4) * k16, db, kIdescN64_AMN, (k | k16) != 0);
                        }
                }
                mma_commit(&bars[kBarD]);
                ++nd;
                if (!wait(kMReady, ks)) break;
                tc_fence_after();
                // Y_intra = M X: A = M (K-major, two 64-column regions); B = X (MN-major [t][p]).
                // M hi runs against X hi and X lo stacked along N (the X lo tile is the second
                // 64-wide MN block, 16 KB on), M lo against X hi into the first half.
                {
                    const uint64_t dxx = smem_desc_sw128_mn(sb + Smem::XHI, 16384);
                    const uint64_t dmh = smem_desc_sw128(sb + Smem::MHI), dml = smem_desc_sw128(sb + Smem::MLO);
#pragma unroll
                    for (int k16 = 0; k16 < kQ / 16; ++k16) {
                        const uint64_t ka = (uint64_t)((k16 >> 2) * (16384 >> 4) + 2 * (k16 & 3));
                        mma_bf16(tYi, dmh + ka, dxx + (uint64_t)(2048 >> 4) * k16, kIdescN128_BMN, k16 != 0);
                    }
#pragma unroll
                    for (int k16 = 0; k16 < kQ / 16; ++k16) {
                        const uint64_t ka = (uint64_t)((k16 >> 2) * (16384 >> 4) + 2 * (k16 & 3));
                        mma_bf16(tYi, dml + ka, dxx + (uint64_t)(2048 >> 4) * k16, kIdescN64_BMN, true);
                    }
                }
                mma_commit(&bars[kBarY]);
                ++ny;
                // the next step's chunk: the next of this item, else the first of the next item
                SsdItem nx = it;
                int nc = c + 1, nj = jt;
                if (nc == it.c1 && jt + 1 < n_items) {
                    nj = jt + 1;
                    nx = s_span->item(nj);
                    nc = nx.c0;
                }
                if (ks + 1 < n_steps) {
                    if (!wait(kBarD, ks)) break;     // raw x (conv done) and B^T (dS done) are free
                    issue_a(nx, nc, ks + 1);
                    ++ia;
                    if (!wait(kBarY, ks)) break;     // M over C, B (and G, Y_inter) are consumed
                    issue_b(nx, nc);
                    ++ib;
                }
                it = nx;
                c = nc;
                jt = nj;
            }
            if (ks < n_steps) {
                // stopped early: let every copy and MMA group still in flight finish (its last
                // completion) before shared memory and TMEM go away
                const int last[6] = {ia, ib, iz, ng, nd, ny};
                for (int k = 0; k < 6; ++k)
                    if (last[k] > 0) (void)mbar_wait_bounded(&bars[k], (uint32_t)((last[k] - 1) & 1), 100000000ull);
            }
        }
    } else {
        float* s_dl2 = reinterpret_cast<float*>(sm + Smem::DL);   // [2][128]: delta by chunk parity
        float* s_cs2 = reinterpret_cast<float*>(sm + Smem::CS);   // [2][128]: s by chunk parity
        auto wait = [&](int k, int c) {
            if (!bad && !mbar_wait_bounded(&bars[k], (uint32_t)(c & 1))) {
                bad = true;
                atomicOr(p.status, 1u);
            }
        };
        auto arrive = [&](int k) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[k]);
        };
        int ks = 0;                                  // chunks walked so far
        for (int jt = 0; jt < n_items; ++jt) {
          const int c1 = s_item[3];
          for (int c = s_item[2]; c < c1; ++c, ++ks) {
            const int t0 = c * kQ;
            float* s_dl = s_dl2 + (ks & 1) * kQ;
            float* s_cs = s_cs2 + (ks & 1) * kQ;

            // ---- 2. conv + SiLU of x (raw x, B^T, delta and s of the chunk landed together)
            wait(kBarA, ks);
            const float s_i = s_cs[i], s_Q = s_cs[kQ - 1], dl_i = s_dl[i];
            if (tid < 3 * 32) {
                // for a block of M wholly below a warp's rows: 2^(s_i - s_j) = 2^(s_i - s_last)
                // 2^(s_last - s_j), both exponents <= 0 (s falls along the chunk), s_last the
                // block's last column; read after this step's worker barrier
                float* s_ec = reinterpret_cast<float*>(sm + Smem::EC);
                s_ec[tid] = ex2(s_cs[(tid & ~31) + 31] - s_cs[tid]) * s_dl[tid];
            }
            {
                // x of token i, positions kCW cg .., written as X hi/lo and as the state-update
                // operand w_i x_i (w_i = 2^(s_Q - s_i) delta_i), hi and lo tiles
                float r[4][kCW];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int row = i + k;                    // tile row of token t0 + i - 3 + k
                    if (c == 0 && row < 3 && p.conv_state_in) {
                        const int b = s_item[0], h = s_item[1];
#pragma unroll
                        for (int e = 0; e < kCW; ++e)
                            r[k][e] = p.conv_state_in[((int64_t)b * 3 + row) * Cx + h * (int64_t)kP + kCW * cg + e];
                    } else {
#pragma unroll
                        for (int e = 0; e < kCW / 8; ++e) {
                            const uint4 u = *reinterpret_cast<const uint4*>(
                                sm + Smem::XR + row * 128 + (((((kCW / 8) * cg + e) ^ (row & 7))) << 4));
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
                float u[kCW];
#pragma unroll
                for (int e = 0; e < kCW; ++e) {
                    const int pp = kCW * cg + e;
                    const float* w = s_cw + 4 * pp;
                    float xc = fmaf(w[0], r[0][e], s_cb[pp]);
                    xc = fmaf(w[1], r[1][e], xc);
                    xc = fmaf(w[2], r[2][e], xc);
                    xc = fmaf(w[3], r[3][e], xc);
                    u[e] = silu_in<Tin_bf16>(xc);
                }
                // X is free once the previous chunk's output tile, staged there, has been read by its
                // store; this barrier also tells every worker whether any of them has seen an error
                if (tid == 0) bulk_wait_read();
                if (workers_any(bad)) bad = true;
                // row i (token) of X and of w x, positions kCW cg .. as 16-byte swizzled chunks
#pragma unroll
                for (int c8 = 0; c8 < kCW / 8; ++c8) {
                    uint32_t xh[4], xl[4], wh[4], wl[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float a0 = u[8 * c8 + 2 * k], a1 = u[8 * c8 + 2 * k + 1];
                        split2(a0, a1, xh[k], xl[k]);
                        split2(wi * a0, wi * a1, wh[k], wl[k]);
                    }
                    const uint32_t off = sw128(i, kCW * cg + 8 * c8);
                    *reinterpret_cast<uint4*>(sm + Smem::XHI + off) = make_uint4(xh[0], xh[1], xh[2], xh[3]);
                    *reinterpret_cast<uint4*>(sm + Smem::XLO + off) = make_uint4(xl[0], xl[1], xl[2], xl[3]);
                    *reinterpret_cast<uint4*>(sm + Smem::XW + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                    *reinterpret_cast<uint4*>(sm + Smem::XW + 16384 + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                }
            }
            fence_proxy_async_smem();
            arrive(kXReady);

            // ---- 3. M = G 2^(s_i - s_j) delta_j (j < i), M[i][i] = G[i][i] delta_i + D, as hi/lo
            //      over the C and B tiles: columns [kMJ cg, kMJ cg + kMJ) of row i
            wait(kBarG, ks);
            tc_fence_after();
            {
                const float Dh = *s_Dh;
                const int j0 = kMJ * cg;
                static_assert(kMJ == 32, "one 32-column block of M per thread");
                if (j0 > 32 * q + 31) {                  // entirely above the diagonal
#pragma unroll
                    for (int c8 = 0; c8 < kMJ / 8; ++c8) {
                        const int jj = j0 + 8 * c8;
                        const uint32_t off = (uint32_t)((jj >> 6) * 16384 + i * 128 + ((((jj & 63) >> 3) ^ (i & 7)) << 4));
                        *reinterpret_cast<uint4*>(sm + Smem::MHI + off) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4*>(sm + Smem::MLO + off) = make_uint4(0, 0, 0, 0);
                    }
                } else if (j0 + 31 < 32 * q) {           // entirely below: the factored decay
                    const float* s_ec = reinterpret_cast<const float*>(sm + Smem::EC);
                    const float er = ex2(s_i - s_cs[j0 + 31]);
                    float v[32];
                    tmem_ld32(tG + ((uint32_t)(32 * q) << 16) + (uint32_t)j0, v);
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        const float4 ea = *reinterpret_cast<const float4*>(s_ec + j0 + 8 * c8);
                        const float4 eb = *reinterpret_cast<const float4*>(s_ec + j0 + 8 * c8 + 4);
                        const float ej[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
                        float m[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) m[e] = v[8 * c8 + e] * (ej[e] * er);
                        uint32_t whi[4], wlo[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) split2(m[2 * k], m[2 * k + 1], whi[k], wlo[k]);
                        const int jj = j0 + 8 * c8;
                        const uint32_t off = (uint32_t)((jj >> 6) * 16384 + i * 128 + ((((jj & 63) >> 3) ^ (i & 7)) << 4));
                        *reinterpret_cast<uint4*>(sm + Smem::MHI + off) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
                        *reinterpret_cast<uint4*>(sm + Smem::MLO + off) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
                    }
                } else {
#pragma unroll
                    for (int half = 0; half < kMJ / 32; ++half) {
                        const int jb = j0 + 32 * half;
                        float v[32];
                        tmem_ld32(tG + ((uint32_t)(32 * q) << 16) + (uint32_t)jb, v);
#pragma unroll
                        for (int c8 = 0; c8 < 4; ++c8) {
                            const float4 sa = *reinterpret_cast<const float4*>(s_cs + jb + 8 * c8);
                            const float4 sb4 = *reinterpret_cast<const float4*>(s_cs + jb + 8 * c8 + 4);
                            const float4 da = *reinterpret_cast<const float4*>(s_dl + jb + 8 * c8);
                            const float4 db4 = *reinterpret_cast<const float4*>(s_dl + jb + 8 * c8 + 4);
                            const float sj[8] = {sa.x, sa.y, sa.z, sa.w, sb4.x, sb4.y, sb4.z, sb4.w};
                            const float dj[8] = {da.x, da.y, da.z, da.w, db4.x, db4.y, db4.z, db4.w};
                            float m[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int jl = 8 * c8 + e, j = jb + jl;
                                // the skip term D x_i rides on the diagonal: Y = M X then includes it
                                m[e] = j < i ? v[jl] * ex2(s_i - sj[e]) * dj[e] : (j == i ? fmaf(v[jl], dl_i, Dh) : 0.f);
                            }
                            uint32_t whi[4], wlo[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) split2(m[2 * k], m[2 * k + 1], whi[k], wlo[k]);
                            const int jj = jb + 8 * c8;
                            const uint32_t off = (uint32_t)((jj >> 6) * 16384 + i * 128 + ((((jj & 63) >> 3) ^ (i & 7)) << 4));
                            *reinterpret_cast<uint4*>(sm + Smem::MHI + off) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
                            *reinterpret_cast<uint4*>(sm + Smem::MLO + off) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            arrive(kMReady);

            // ---- 4. state: S = 2^(s_Q) S + dS (the accumulator's hi-part rows + lo-part rows)
            wait(kBarD, ks);
            tc_fence_after();
            {
                float v[kCW];
                tmem_ld16(tDS + ((uint32_t)(32 * q) << 16) + (uint32_t)(kCW * cg), v);
                float* scr = reinterpret_cast<float*>(sm + Smem::XW);   // w x is consumed by dS
                if (q >= 2) {
                    float4* dst = reinterpret_cast<float4*>(scr + (i - 64) * Smem::SCR_LD + kCW * cg);
#pragma unroll
                    for (int k = 0; k < kCW / 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                }
                tc_fence_before();
                workers_sync();
                if (q < 2) {
                    const float eQ = ex2(s_Q);
                    const float4* src = reinterpret_cast<const float4*>(scr + i * Smem::SCR_LD + kCW * cg);
#pragma unroll
                    for (int k = 0; k < kCW / 4; ++k) {
                        const float4 o = src[k];
                        S[4 * k] = fmaf(eQ, S[4 * k], v[4 * k] + o.x);
                        S[4 * k + 1] = fmaf(eQ, S[4 * k + 1], v[4 * k + 1] + o.y);
                        S[4 * k + 2] = fmaf(eQ, S[4 * k + 2], v[4 * k + 2] + o.z);
                        S[4 * k + 3] = fmaf(eQ, S[4 * k + 3], v[4 * k + 3] + o.w);
                    }
                    store_state();                       // Y_inter, its reader, completed with G
                }
            }
            fence_proxy_async_smem();

            // ---- 5. out = (Y_intra + 2^(s_i) Y_inter) SiLU(z)   (Y_intra holds D x through M's diagonal)
            wait(kBarY, ks);
            wait(kBarZ, ks);
            tc_fence_after();
            {
                float yi[kCW], ye[kCW], y2[kCW];
                const uint32_t lanes = (uint32_t)(32 * q) << 16;
                tmem_ld16(tYi + lanes + (uint32_t)(kCW * cg), yi);
                tmem_ld16(tYi + lanes + (uint32_t)(64 + kCW * cg), y2);
#pragma unroll
                for (int k = 0; k < kCW; ++k) yi[k] += y2[k];
                tmem_ld16(tYe + lanes + (uint32_t)(kCW * cg), ye);
                tmem_ld16(tYe + lanes + (uint32_t)(64 + kCW * cg), y2);
#pragma unroll
                for (int k = 0; k < kCW; ++k) ye[k] += y2[k];
                const float ei = ex2(s_i);
                float o[kCW];
#pragma unroll
                for (int e = 0; e < kCW / 8; ++e) {
                    const uint4 u = *reinterpret_cast<const uint4*>(sm + Smem::ZT + i * 128 + ((((kCW / 8) * cg + e) ^ (i & 7)) << 4));
                    const uint32_t ws4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        const int k = 8 * e + 2 * f;
                        const float z0 = __uint_as_float(ws4[f] << 16), z1 = __uint_as_float(ws4[f] & 0xffff0000u);
                        o[k] = fmaf(ei, ye[k], yi[k]) * silu_in<Tin_bf16>(z0);
                        o[k + 1] = fmaf(ei, ye[k + 1], yi[k + 1]) * silu_in<Tin_bf16>(z1);
                    }
                }
                // the tile row goes to shared memory over X (consumed by Y_intra), 128-byte swizzled,
                // and leaves by one TMA store per 128-byte column block (rows past L are not written)
                if constexpr (sizeof(Tout) == 4) {
                    unsigned char* row = sm + Smem::XHI + (cg >> 1) * 16384 + i * 128;
#pragma unroll
                    for (int k = 0; k < kCW / 4; ++k)
                        *reinterpret_cast<float4*>(row + ((((cg & 1) * (kCW / 4) + k) ^ (i & 7)) << 4)) =
                            make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
                } else {
                    unsigned char* row = sm + Smem::XHI + i * 128;
#pragma unroll
                    for (int k = 0; k < kCW / 8; ++k) {
                        uint32_t w4[4];
#pragma unroll
                        for (int f = 0; f < 4; ++f)
                            w4[f] = pack2(__float2bfloat16_rn(o[8 * k + 2 * f]), __float2bfloat16_rn(o[8 * k + 2 * f + 1]));
                        *reinterpret_cast<uint4*>(row + ((((kCW / 8) * cg + k) ^ (i & 7)) << 4)) =
                            make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
            fence_proxy_async_smem();
            workers_sync();
            if (tid == 0 && !bad) {
                constexpr int kBoxes = sizeof(Tout) == 4 ? 2 : 1;
                const int b = s_item[0], h = s_item[1];
#pragma unroll
                for (int k = 0; k < kBoxes; ++k)
                    tma_store_3d(&tm_out, sm + Smem::XHI + k * 16384, h * kP + k * (kP / kBoxes), t0, b);
                bulk_commit();
            }
            if (c + 1 < c1) {
                tc_fence_before();
                arrive(kDone);
            }
          }
          // the item ends: its state goes out (or on to the next CTA), and the next item's
          // parameters and start state come in before its last chunk is reported done, so before
          // the producer may issue the next item's products
          end_item();
          if (jt + 1 < n_items) {
              workers_sync();                        // every worker is done with the ended item
              begin_item(jt + 1);
          }
          tc_fence_before();
          arrive(kDone);
        }
        if (tid == 0) bulk_wait_read();              // the last output tile has left shared memory
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
    // the 16 KB state of (slot, head) is requested first, so its latency overlaps the conv below
    const int pp = tid >> 2, n0 = 16 * (tid & 3);
    float4* sp = reinterpret_cast<float4*>(a.ssm_state + (((int64_t)slot * H + h) * kP + pp) * kNs + n0);
    float4 st[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) st[k] = sp[k];
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
    const float dx = dl * u[pp];
    float y = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float4 s = st[k];
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

// 3-D tensor map (bf16 unless f32): dims {d0, d1, d2} (d0 innermost), byte strides {s1, s2}, box {b0, b1, 1}.
// promote256: L2 fetches in 256-byte units (for boxes whose rows are contiguous beyond 128 bytes);
// else 128-byte units, for boxes that take one head's 128-byte slice of each token row, whose
// neighbouring slice another CTA reads at another time.
bool make_map3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
               uint32_t b0, uint32_t b1, bool swizzle, bool f32 = false, bool promote256 = true) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
               dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               promote256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

}  // namespace

SsdWorkspace ssd_workspace_layout(int batch, int seqlen, int n_heads, int n_groups) {
    SsdWorkspace w{};
    const int64_t BG = (int64_t)batch * n_groups, BH = (int64_t)batch * n_heads;
    w.lp = round_up(seqlen, kQ);
    w.bt_off = round_up(4 * BG * seqlen * kNs * 2, 256);
    w.ds_off = round_up(w.bt_off + 2 * BG * kNs * w.lp * 2, 256);
    w.n_slots = (int)(BH < kSsdMaxCtas ? BH : kSsdMaxCtas);
    w.ho_off = round_up(w.ds_off + 2 * BH * w.lp * 4, 256);
    w.flag_off = w.ho_off + (int64_t)w.n_slots * kP * kNs * 4;
    w.bytes = (size_t)round_up(w.flag_off + (int64_t)w.n_slots * 4, 16);
    return w;
}

int launch_ssd_prefill(const SsdArgs& a0, bool out_bf16, cudaStream_t stream, const char** why) {
    SsdArgs a = a0;
    const SsdWorkspace w = ssd_workspace_layout(a.batch, a.seqlen, a.n_heads, a.n_groups);
    a.ws_bt_off = w.bt_off;
    a.ws_ds_off = w.ds_off;
    a.ws_lp = w.lp;
    a.ws_ho_off = w.ho_off;
    a.ws_flag_off = w.flag_off;
    a.n_slots = w.n_slots;
    const int64_t HP = (int64_t)a.n_heads * kP, Cx = HP + 2 * (int64_t)a.n_groups * kNs;
    const int64_t BG = (int64_t)a.batch * a.n_groups;
    const int L = a.seqlen;

    {
        const int nbx = (L + kBcT - 1) / kBcT, ncx = (int)(w.lp / kQ);
        const int64_t n_bc = (int64_t)nbx * a.n_groups * a.batch;
        const int64_t n_dt = ((int64_t)ncx * a.batch * a.n_heads + 7) / 8;
        if (n_bc + n_dt > 0x7fffffffLL) {
            *why = "too many pre-pass blocks";
            return -1;
        }
        k_ssd_pre<<<(unsigned)(n_bc + n_dt), 256, 0, stream>>>(a, nbx, (int)n_bc, ncx);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return -1;
    }

    CUtensorMap mx, mz, mbc, mbt, mo, mds;
    const int64_t BH = (int64_t)a.batch * a.n_heads;
    const uint64_t xs_b = a.batch > 1 ? (uint64_t)a.xbc_stride_b * 2 : (uint64_t)L * a.xbc_stride_t * 2;
    const uint64_t zs_b = a.batch > 1 ? (uint64_t)a.z_stride_b * 2 : (uint64_t)L * a.z_stride_t * 2;
    const unsigned char* ws = static_cast<const unsigned char*>(a.workspace);
    // raw x and z arrive 128-byte swizzled, so that a lane reading its own token row of 128 bytes
    // hits all 32 banks across a warp
    if (!make_map3(&mx, a.xBC, (uint64_t)Cx, (uint64_t)L, (uint64_t)a.batch, (uint64_t)a.xbc_stride_t * 2, xs_b, kP,
                   kQ + 3, true, false, false) ||
        !make_map3(&mz, a.z, (uint64_t)HP, (uint64_t)L, (uint64_t)a.batch, (uint64_t)a.z_stride_t * 2, zs_b, kP, kQ,
                   true, false, false) ||
        !make_map3(&mbc, ws, kNs, (uint64_t)L, (uint64_t)(4 * BG), kNs * 2, (uint64_t)L * kNs * 2, kNs, kQ, true) ||
        !make_map3(&mbt, ws + w.bt_off, (uint64_t)L, kNs, (uint64_t)(2 * BG), (uint64_t)w.lp * 2,
                   (uint64_t)w.lp * kNs * 2, 64, kNs, true) ||
        // the output leaves through TMA stores of 128-byte-wide boxes: 32 fp32 or 64 bf16 columns
        !make_map3(&mo, a.out, (uint64_t)HP, (uint64_t)L, (uint64_t)a.batch, (uint64_t)a.out_stride_t * (out_bf16 ? 2 : 4),
                   a.batch > 1 ? (uint64_t)a.out_stride_b * (out_bf16 ? 2 : 4)
                               : (uint64_t)L * a.out_stride_t * (out_bf16 ? 2 : 4),
                   out_bf16 ? 64 : 32, kQ, true, !out_bf16) ||
        // delta and s planes [2 B H][lp] fp32, 128-token rows
        !make_map3(&mds, ws + w.ds_off, (uint64_t)w.lp, (uint64_t)(2 * BH), 1, (uint64_t)w.lp * 4,
                   (uint64_t)w.lp * 4 * 2 * BH, kQ, 1, false, true)) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point missing or layout rejected)";
        return -1;
    }
    auto kern = out_bf16 ? k_ssd_chunk<__nv_bfloat16> : k_ssd_chunk<float>;
    static ContextMemo attr[2], occ[2];
    if (!opt_in_dynamic_smem(attr[out_bf16 ? 1 : 0], kern, Smem::ALLOC, why)) return -1;
    // One CTA per (row, head) while they fit on the GPU at once; beyond that one CTA per resident
    // slot, each on an equal span of the chunks, the rows cut between CTAs handing their state on.
    // Those CTAs wait on one another, so they go out as a cooperative launch (all resident).
    void* per_sm_v = nullptr;
    if (!occ[out_bf16 ? 1 : 0].get(&per_sm_v, [&](void** out) {
            int dev = 0, n_sm = 0, per_sm = 0;
            if (cudaGetDevice(&dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThAll, Smem::ALLOC) != cudaSuccess)
                return false;
            *out = reinterpret_cast<void*>((intptr_t)per_sm * n_sm);
            return true;
        })) {
        *why = "occupancy query failed";
        return -1;
    }
    const int64_t resident = (int64_t)reinterpret_cast<intptr_t>(per_sm_v);
    const int64_t cap = resident < kSsdMaxCtas ? resident : kSsdMaxCtas;
    if (cap < 1) {
        *why = "k_ssd_chunk cannot be resident on this device";
        return -1;
    }
    const int64_t rows = (int64_t)a.batch * a.n_heads;
    const bool cut = rows > cap;
    const unsigned n_cta = (unsigned)(cut ? cap : rows);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_cta);
    cfg.blockDim = dim3(kThAll);
    cfg.dynamicSmemBytes = Smem::ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeCooperative;
    la[0].val.cooperative = cut ? 1 : 0;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mx, mz, mbc, mbt, mo, mds, a);
    if (e == cudaSuccess) e = cudaGetLastError();
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
