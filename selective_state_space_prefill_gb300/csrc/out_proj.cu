// out_proj.cu -- one tensor-parallel rank's partial of the mixer's output projection on the
// sm_103a tensor cores (tcgen05), with the per-block maxima the 8-bit all-reduce needs.
//
// "Scaling State-Space Models on Multiple GPUs with Tensor Parallelism", Methodology 1 and 4:
// the layer is split along the feature dimension, so a rank holds the mixer output of its
// channel slice, y [M][K] (M = batch * tokens), and the matching columns of the projection
// weight, W [N][K]; its partial P = y W^T [M][N] is what the ranks quantize to 8 bits and sum.
// The shared-scale codec needs max |P| over every block of 128 consecutive elements of the
// row-major partial, across ranks; this kernel emits the rank's block maxima with the partial
// (over the values it stores), so the cross-rank maximum is one small all-reduce.
//
// Design (a dense contraction, so the 5th-generation tensor cores):
//   * persistent: one CTA per SM walks 128 x 256 output tiles; K in blocks of 64 (one 128-byte
//     swizzle row of bf16);
//   * warp 0, one thread: TMA producer over a 4-stage ring of (A 128x64, B 256x64) bf16 tiles,
//     128-byte swizzled, completing on mbarriers;
//   * warp 1: allocates 512 TMEM columns, two fp32 accumulators of 128 lanes x 256 columns; one
//     thread issues tcgen05.mma kind::f16 (M 128, N 256, K 16) four times per stage, commits each
//     stage to its "empty" mbarrier and each finished tile to its buffer's "full" mbarrier, so
//     the epilogue of one tile overlaps the MMAs of the next;
//   * warps 2-5: epilogue; warp w reads TMEM lanes 32 (w % 4) .. +31 (its rows) with
//     tcgen05.ld, rounds to the output type, stores, and takes |.|-maxima of each 128-column
//     half of its row over the stored values;
//   * every wait is bounded; on a timeout the status word gets SSM_DEV_WAIT_TIMEOUT, the
//     epilogue stores nothing and TMEM is still released.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace ssm {
namespace {

constexpr int kBM = 128, kBK = 64;
constexpr int kThreads = 192;                       // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kABytes = kBM * kBK * 2;              // 16 KB

// Tile geometry for an output tile of 128 x BN (BN = 256, or 128 for problems with few tiles).
template <int BN>
struct Geo {
    static constexpr int kStages = BN == 256 ? 4 : 6;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;    // a multiple of 1024
    static constexpr int kOffBar = kStages * kStageBytes;    // full[S], empty[S], acc_full[2], acc_empty[2], TMEM address
    static constexpr int kSmemBytes = kOffBar + (2 * kStages + 4) * 8 + 16 + 1024;   // + slack to align to 1024
    static constexpr uint32_t kTmemCols = 2 * BN;            // two fp32 accumulators of 128 lanes x BN columns
    // tcgen05.mma kind::f16 instruction descriptor: fp32 accumulator (bits 4-5 = 1), bf16 A and B
    // (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
    // M >> 4 at bits 24-28.
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                       ((uint32_t)(kBM >> 4) << 24);
};

template <typename Tout, int kBN>
__global__ void __launch_bounds__(kThreads, 1)
k_out_proj(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
           const OutProjArgs p) {
    using G = Geo<kBN>;
    constexpr int kStages = G::kStages, kStageBytes = G::kStageBytes, kOffBar = G::kOffBar;
    constexpr uint32_t kTmemCols = G::kTmemCols;
    extern __shared__ unsigned char smem_raw[];
    // TMA 128-byte swizzling and the descriptors' base offset 0 want 1024-byte aligned tiles
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;           // [2]: accumulator buffer b holds a finished tile
    uint64_t* acc_empty = acc_full + 2;             // [2]: the epilogue has read buffer b
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    __shared__ int s_err;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (int)((p.N + kBN - 1) / kBN);
    const int m_tiles = (int)((p.M + kBM - 1) / kBM);
    const int nk = (int)((p.K + kBK - 1) / kBK);
    // this CTA's i-th tile: false when there is none; *m0, *n0 its origin
    auto tile = [&](int i, int* m0, int* n0) -> bool {
        const int t = (int)blockIdx.x + i * (int)gridDim.x;
        if (t >= n_tiles * m_tiles) return false;
        *m0 = (t / n_tiles) * kBM;
        *n0 = (t % n_tiles) * kBN;
        return true;
    };

    if (threadIdx.x == 0) {
        s_err = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);            // one arrival per epilogue warp
        }
        fence_barrier_init();
        prefetch_tmap(&tm_a);
        prefetch_tmap(&tm_b);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer, running ahead across tile boundaries
        int it = 0, m0, n0;
        for (int i = 0; !s_err && tile(i, &m0, &n0); ++i) {
            for (int kb = 0; kb < nk; ++kb, ++it) {
                const int s = it % kStages;
                if (it >= kStages && !mbar_wait_bounded(&empty[s], (uint32_t)(((it / kStages) + 1) & 1))) {
                    s_err = 1;
                    atomicOr(p.status, 1u);
                    break;
                }
                unsigned char* st = smem + s * kStageBytes;
                mbar_arrive_expect_tx(&full[s], kStageBytes);
                tma_load_2d(st, &tm_a, &full[s], kb * kBK, m0);
                tma_load_2d(st + kABytes, &tm_b, &full[s], kb * kBK, n0);
            }
        }
        // tail: every stage's last use has been released by the MMAs, so no arrival is still on
        // its way to this CTA's barriers when it exits
        for (int u = it - 1; u >= 0 && u >= it - kStages && !s_err; --u)
            if (!mbar_wait_bounded(&empty[u % kStages], (uint32_t)((u / kStages) & 1))) atomicOr(p.status, 1u);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer: tile i accumulates into TMEM buffer i % 2
        int it = 0, m0, n0;
        for (int tl = 0; !s_err && tile(tl, &m0, &n0); ++tl) {
            const int buf = tl & 1;
            if (tl >= 2 && !mbar_wait_bounded(&acc_empty[buf], (uint32_t)(((tl / 2) + 1) & 1))) {
                s_err = 1;
                atomicOr(p.status, 1u);
                break;
            }
            tc_fence_after();
            const uint32_t dt = tmem + (uint32_t)(buf * kBN);
            for (int kb = 0; kb < nk; ++kb, ++it) {
                const int s = it % kStages;
                if (!mbar_wait_bounded(&full[s], (uint32_t)((it / kStages) & 1))) {
                    s_err = 1;
                    atomicOr(p.status, 1u);
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(smem + s * kStageBytes);
                const uint32_t b0 = a0 + kABytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)      // 16 bf16 = 32 bytes along K per MMA
                    mma_bf16(dt, smem_desc_sw128(a0 + 32 * kk), smem_desc_sw128(b0 + 32 * kk), G::kIdesc,
                             (kb | kk) != 0);
                mma_commit(&empty[s]);                      // the stage may be refilled
            }
            mma_commit(&acc_full[buf]);                     // the tile is complete in buffer buf
        }
    } else if (warp >= 2) {
        // ---- epilogue: rows m0 + 32 q + lane of each tile, q = warp % 4
        const int q = warp & 3;
        int m0, n0;
        for (int tl = 0; tile(tl, &m0, &n0); ++tl) {
            const int buf = tl & 1;
            if (!mbar_wait_bounded(&acc_full[buf], (uint32_t)((tl / 2) & 1))) {
                atomicOr(p.status, 1u);
                break;
            }
            tc_fence_after();
            const int m = m0 + 32 * q + lane;
            const bool store = s_err == 0 && m < p.M;
            const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * kBN);
#pragma unroll 1
            for (int half = 0; half < kBN / 128; ++half) {
                const int64_t nb = n0 + 128 * half;
                float amax = 0.f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    float v[32];
                    tmem_ld32(trow + (uint32_t)(128 * half + 32 * c), v);
                    if (half == kBN / 128 - 1 && c == 3) {
                        // every TMEM read of this buffer is done: hand it back to the MMA issuer
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&acc_empty[buf]);
                    }
                    if (store && nb < p.N) {
                        Tout* o = reinterpret_cast<Tout*>(p.out) + (int64_t)m * p.ldo + nb + 32 * c;
                        if constexpr (sizeof(Tout) == 2) {
                            uint32_t w[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                                amax = fmaxf(amax, fmaxf(fabsf(__low2float(h)), fabsf(__high2float(h))));
                                w[i] = *reinterpret_cast<uint32_t*>(&h);
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                reinterpret_cast<uint4*>(o)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                reinterpret_cast<float4*>(o)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                        }
                    }
                }
                if (store && nb < p.N && p.amax) p.amax[((int64_t)m * p.N + nb) / 128] = amax;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// 2-D bf16 map over rows x K (row stride ld elements), box of `rows` x 64, 128-byte swizzle.
bool make_map_kmajor(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint64_t ld, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Tout, int BN>
int launch_bn(const OutProjArgs& a, const void* y, const void* W, int64_t ldy, int64_t ldw, int dev, int n_sm,
              cudaStream_t stream, const char** why) {
    using G = Geo<BN>;
    CUtensorMap ma, mb;
    if (!make_map_kmajor(&ma, y, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)ldy, kBM) ||
        !make_map_kmajor(&mb, W, (uint64_t)a.K, (uint64_t)a.N, (uint64_t)ldw, BN)) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point missing or layout rejected)";
        return -1;
    }
    auto kern = k_out_proj<Tout, BN>;
    static ContextMemo attr;
    if (!opt_in_dynamic_smem(attr, kern, G::kSmemBytes, why)) return -1;
    // persistent: one CTA per SM (the shared memory allows no second one, which also leaves the
    // SM's TMEM columns to this CTA), looping over the output tiles
    const int64_t tiles = ((a.M + kBM - 1) / kBM) * ((a.N + BN - 1) / BN);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = G::kSmemBytes;
    cfg.stream = stream;
    cfg.gridDim = dim3((unsigned)(tiles < n_sm ? tiles : n_sm));
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return -1;
    }
    return 0;
}

}  // namespace

int launch_out_proj(const OutProjArgs& a, const void* y, const void* W, int64_t ldy, int64_t ldw, bool out_bf16,
                    cudaStream_t stream, const char** why) {
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm < 1) {
        *why = "cudaGetDevice / multiprocessor count failed";
        return -1;
    }
    // 256-column tiles unless that leaves fewer than two tiles per SM; then 128 columns
    const int64_t tiles256 = ((a.N + 255) / 256) * ((a.M + kBM - 1) / kBM);
    const bool narrow = tiles256 < 2 * (int64_t)n_sm;
    if (out_bf16)
        return narrow ? launch_bn<__nv_bfloat16, 128>(a, y, W, ldy, ldw, dev, n_sm, stream, why)
                      : launch_bn<__nv_bfloat16, 256>(a, y, W, ldy, ldw, dev, n_sm, stream, why);
    return narrow ? launch_bn<float, 128>(a, y, W, ldy, ldw, dev, n_sm, stream, why)
                  : launch_bn<float, 256>(a, y, W, ldy, ldw, dev, n_sm, stream, why);
}

}  // namespace ssm
