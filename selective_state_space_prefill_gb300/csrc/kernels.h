// kernels.h -- internal interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; the public interface is include/ssm.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace ssm {

// ------------------------------------------------------------------ host-side memo
// Id of the calling thread's current CUDA context (cuCtxGetId), or 0 when no context is
// current or the driver entry points are missing.
uint64_t current_context_id();

// Facts that hold for the life of one CUDA context -- a __device__ symbol's address, a
// kernel's dynamic shared-memory opt-in -- remembered per device together with the id of the
// context they were taken in.  When the device's current context is a different one (after
// cudaDeviceReset, or once a new primary context has been made) they are taken again, so a
// kernel is never handed an address from a context that no longer exists.
class ContextMemo {
 public:
    // *value for the current device and context; compute(&v) runs (and must return true) when
    // nothing is remembered for that context.
    template <typename F>
    bool get(void** value, F&& compute) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return false;
        uint64_t id = current_context_id();
        if (id != 0) {
            std::lock_guard<std::mutex> g(mu_);
            if (ctx_[dev] == id) {
                *value = val_[dev];
                return true;
            }
        }
        void* v = nullptr;
        if (!compute(&v)) return false;
        id = current_context_id();     // compute's runtime call has made the context current
        std::lock_guard<std::mutex> g(mu_);
        ctx_[dev] = id;                // an id of 0 is never matched: nothing is kept without one
        val_[dev] = v;
        *value = v;
        return true;
    }

 private:
    static constexpr int kDevices = 64;
    std::mutex mu_;
    uint64_t ctx_[kDevices] = {};
    void* val_[kDevices] = {};
};

// cudaFuncSetAttribute(kern, MaxDynamicSharedMemorySize, bytes) once per device and context.
template <typename K>
bool opt_in_dynamic_smem(ContextMemo& memo, K* kern, int bytes, const char** why) {
    void* v = nullptr;
    if (!memo.get(&v, [&](void** out) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
                return false;
            *out = reinterpret_cast<void*>(1);
            return true;
        })) {
        *why = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize) failed";
        return false;
    }
    return true;
}

// Kernel-side arguments of the prefill (everything except the TMA maps).
struct PrefillArgs {
    int seqlen, d_inner;
    const void* x;                  // raw x, for the final conv state
    int64_t in_stride_b, in_stride_t;
    const float *A, *Dskip, *dt_bias, *conv_w, *conv_b;
    const float *conv_state_in, *ssm_state_in;
    int64_t conv_state_ld, ssm_state_stride_b;
    void* out;
    int64_t out_stride_b, out_stride_t;
    float *conv_state_out, *ssm_state_out;
    unsigned int* status;
    // Sequence segments: tokens [g*seg_len, min(L, (g+1)*seg_len)) of every row form segment g
    // (seg_len = seqlen and n_seg = 1 when unsegmented).  ws holds, per earlier segment g < n_seg-1
    // and (b, d), 32 floats: the segment's state from zero (then the next segment's start state)
    // and the product of its decays.
    int seg_len, n_seg;
    float* ws;
    // 1: the output leaves through TMA stores of [chunk x 16 channels] tiles staged in shared
    // memory (needs a 16-byte-aligned output with 16-byte strides); 0: per-lane stores
    int out_tma;
};

struct PrefillLaunch {
    int batch;
    bool in_bf16, out_bf16;
    const void *z, *dt, *Bm, *Cm;
    PrefillArgs args;
};

struct DecodeArgs {
    int batch, n_tokens, d_inner, n_slots;
    const void *x, *z, *dt;
    int64_t in_stride_b, in_stride_t;
    const void *Bm, *Cm;
    const float *A, *Dskip, *dt_bias, *conv_w, *conv_b;
    float *conv_state, *ssm_state;
    int64_t conv_state_ld, ssm_state_stride_b;
    const int32_t* state_slot;
    void* out;
    int64_t out_stride_b, out_stride_t;
    unsigned int* status;
};

// Tokens per prefill chunk; a sequence segment is a whole number of chunks.
constexpr int kPrefillChunk = 64;

constexpr int kMaxPartials = 8;

struct Q8Args {
    const void* partials[kMaxPartials];
    int P;
    int64_t n;
    void* out;
    int32_t* sums;
    float* scales;
};

// Output projection partial: out [M][N] (row stride ldo) = y [M][K] W[N][K]^T, and
// amax[j] = max |out| over the 128-element block j of the row-major [M][N] partial.
struct OutProjArgs {
    int64_t M, N, K;
    void* out;
    int64_t ldo;
    float* amax;
    unsigned int* status;
};

// SSD (Mamba-2-style) mixer: head dim 64, d_state 64, conv width 4, bf16 token inputs.
//   xBC [batch][L][H*64 + 2*G*64] (x of every head, then B and C of every group), z [batch][L][H*64],
//   dt [batch][L][H]; strides in elements; conv_state [batch][3][Cx], ssm_state [batch][H][64][64].
struct SsdArgs {
    int batch, seqlen, n_heads, n_groups;
    const void* xBC;
    int64_t xbc_stride_b, xbc_stride_t;
    const void* z;
    int64_t z_stride_b, z_stride_t;
    const void* dt;
    int64_t dt_stride_b, dt_stride_t;
    const float *conv_w, *conv_b, *A, *Dskip, *dt_bias;
    const float *conv_state_in, *ssm_state_in;
    void* out;
    int64_t out_stride_b, out_stride_t;
    float *conv_state_out, *ssm_state_out;
    void* workspace;                // B and C of every group after conv + SiLU, as bf16 hi/lo planes,
                                    // then delta and the chunk-local decay sums per head, then the
                                    // state hand-off slots and their flags
    int64_t ws_bt_off, ws_ds_off, ws_lp;   // filled in by launch_ssd_prefill
    int64_t ws_ho_off, ws_flag_off;
    int n_slots;
    unsigned int* status;
};

// Workspace of an SSD prefill: 4 planes [batch*G][L][64] (C hi, C lo, B hi, B lo), then at
// bt_off 2 planes [batch*G][64][lp] (B hi, B lo, token-major), then at ds_off 2 fp32 planes
// [batch*H][lp] (delta; s, the decay exponent summed from each 128-token chunk's start, in log2
// units), lp = L rounded up to 128; then at ho_off n_slots fp32 states [64][64] (a row cut
// between two CTAs passes its state there) and at flag_off their n_slots uint32 ready flags.
struct SsdWorkspace {
    size_t bytes;
    int64_t bt_off, ds_off, lp, ho_off, flag_off;
    int n_slots;
};
// Most CTAs an SSD prefill launch uses (and hand-off slots a workspace holds).
constexpr int kSsdMaxCtas = 256;
SsdWorkspace ssd_workspace_layout(int batch, int seqlen, int n_heads, int n_groups);

// One-token SSD decode for a batch of requests, in place on the cached states of their slots.
//   xBC [batch][Cx], z [batch][H*64], dt [batch][H] contiguous; conv_state [n_slots][3][Cx],
//   ssm_state [n_slots][H][64][64]; out [batch][H*64].
struct SsdDecodeArgs {
    int batch, n_heads, n_groups, n_slots;
    const void *xBC, *z, *dt;
    const float *conv_w, *conv_b, *A, *Dskip, *dt_bias;
    float *conv_state, *ssm_state;
    const int32_t* state_slot;
    void* out;
    unsigned int* status;
};

// Each returns 0 on success, or -1 with *why set to a static message.
int launch_ssd_prefill(const SsdArgs& a, bool out_bf16, cudaStream_t stream, const char** why);
int launch_ssd_decode(const SsdDecodeArgs& a, bool in_bf16, bool out_bf16, cudaStream_t stream, const char** why);
int launch_prefill(const PrefillLaunch& q, cudaStream_t stream, const char** why);
int launch_decode(const DecodeArgs& a, bool in_bf16, bool out_bf16, cudaStream_t stream, const char** why);
int launch_q8(const Q8Args& a, bool in_bf16, bool out_bf16, cudaStream_t stream, const char** why);
// the rank-local halves of the 8-bit all-reduce (block maxima; codes with the shared scale;
// sums of P ranks' codes and the dequantized output)
int launch_q8_absmax(const void* x, bool in_bf16, int64_t n, float* amax, cudaStream_t stream, const char** why);
int launch_q8_quantize(const void* x, bool in_bf16, int64_t n, const float* amax, int8_t* codes, float* scales,
                       cudaStream_t stream, const char** why);
int launch_q8_sum(int P, const int8_t* const* codes, const float* scales, int64_t n, void* out, bool out_bf16,
                  int32_t* sums, cudaStream_t stream, const char** why);
int launch_expire_wait(unsigned int* status, uint64_t limit_ns, cudaStream_t stream, const char** why);
int launch_out_proj(const OutProjArgs& a, const void* y, const void* W, int64_t ldy, int64_t ldw, bool out_bf16,
                    cudaStream_t stream, const char** why);

}  // namespace ssm
