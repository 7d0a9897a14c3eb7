// kernels.h -- internal interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; the public interface is include/ssm.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

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

// Each returns 0 on success, or -1 with *why set to a static message.
int launch_prefill(const PrefillLaunch& q, cudaStream_t stream, const char** why);
int launch_decode(const DecodeArgs& a, bool in_bf16, bool out_bf16, cudaStream_t stream, const char** why);
int launch_q8(const Q8Args& a, bool in_bf16, bool out_bf16, cudaStream_t stream, const char** why);
int launch_expire_wait(unsigned int* status, uint64_t limit_ns, cudaStream_t stream, const char** why);
int launch_out_proj(const OutProjArgs& a, const void* y, const void* W, int64_t ldy, int64_t ldw, bool out_bf16,
                    cudaStream_t stream, const char** why);

}  // namespace ssm
