// api.cu -- the extern "C" boundary of libssm (declared in include/ssm.h).
//
// Every entry point validates its arguments on the host, returns a negative
// status (with a message for ssm_last_error) before launching anything when they
// are wrong, and otherwise enqueues its kernels on the caller's stream (one
// kernel; three for a prefill cut into several sequence segments; two for the
// SSD prefill and decode).
// No entry point allocates memory or keeps per-call state.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cuda.h>

#include "ssm.h"
#include "kernels.h"

namespace ssm {

uint64_t current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static const GetCurrent get_current = []() -> GetCurrent {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                       q == cudaDriverEntryPointSuccess
                   ? reinterpret_cast<GetCurrent>(f)
                   : nullptr;
    }();
    static const GetId get_id = []() -> GetId {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                       q == cudaDriverEntryPointSuccess
                   ? reinterpret_cast<GetId>(f)
                   : nullptr;
    }();
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || c == nullptr ||
        get_id(c, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

}  // namespace ssm

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

// Device status word: SSM_DEV_* bits OR-ed in by kernels.
__device__ unsigned int g_status_word;

ssm::ContextMemo g_status_memo;

// Device address of the status word in the current device's context: a __device__ symbol's
// name in host code is not a device address, so it is asked of the runtime
// (cudaGetSymbolAddress) once per device and context.
unsigned int* status_ptr(int* err) {
    void* p = nullptr;
    if (!g_status_memo.get(&p, [](void** out) {
            return cudaGetSymbolAddress(out, g_status_word) == cudaSuccess && *out != nullptr;
        })) {
        *err = 1;
        return nullptr;
    }
    return static_cast<unsigned int*>(p);
}

}  // namespace

// Scratch of ssm_prefill_segmented_noalloc: a fixed array in the library's own device
// memory, present on every GPU that loads the library until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSM_NOALLOC_SCRATCH_BYTES];

namespace {

ssm::ContextMemo g_noalloc_memo;

// Device address of g_noalloc_scratch in the current device's context.  In host code the
// array's name stands for a host-side shadow, not a device address, so the address is asked of
// the runtime (cudaGetSymbolAddress) with that device current, once per device and context.
void* noalloc_scratch_ptr(int* err) {
    void* p = nullptr;
    if (!g_noalloc_memo.get(&p, [](void** out) {
            return cudaGetSymbolAddress(out, g_noalloc_scratch) == cudaSuccess && *out != nullptr;
        })) {
        *err = 1;
        return nullptr;
    }
    return p;
}

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool dtype_ok(int t) { return t == SSM_F32 || t == SSM_BF16; }
int esize(int t) { return t == SSM_BF16 ? 2 : 4; }

}  // namespace

namespace {

// Shared by ssm_prefill (one segment) and ssm_prefill_segmented.
int prefill_impl(const char* fn, int batch, int seqlen, int d_inner, int d_state, int d_conv,
                 ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                 const void* x, const void* z, const void* dt,
                 int64_t in_stride_b, int64_t in_stride_t,
                 const void* Bmat, const void* Cmat,
                 const float* A, const float* Dskip, const float* dt_bias,
                 const float* conv_w, const float* conv_b,
                 const float* conv_state_in, const float* ssm_state_in,
                 int64_t conv_state_ld, int64_t ssm_state_stride_b,
                 void* out, int64_t out_stride_b, int64_t out_stride_t,
                 float* conv_state_out, float* ssm_state_out,
                 int seg_len, void* workspace, size_t workspace_bytes,
                 void* cuda_stream, bool fixed_scratch = false) {
    g_err[0] = 0;
    if (batch < 1 || batch > 65535) return fail(SSM_ERR_INVALID_ARG, "%s: batch %lld not in [1, 65535]", fn, (long long)(batch));
    if (seqlen < 1 || seqlen > (1 << 30)) return fail(SSM_ERR_INVALID_ARG, "%s: seqlen %lld not in [1, 2^30]", fn, (long long)(seqlen));
    if (d_inner < 1) return fail(SSM_ERR_INVALID_ARG, "%s: d_inner %lld < 1", fn, (long long)(d_inner));
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return fail(SSM_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    if (d_state != 16) return fail(SSM_ERR_UNSUPPORTED, "%s: d_state %lld unsupported (16 only)", fn, (long long)(d_state));
    if (d_conv != 4) return fail(SSM_ERR_UNSUPPORTED, "%s: d_conv %lld unsupported (4 only)", fn, (long long)(d_conv));
    if (d_inner % 8 != 0) return fail(SSM_ERR_UNSUPPORTED, "%s: d_inner %lld is not a multiple of 8", fn, (long long)(d_inner));
    if (!x || !z || !dt || !Bmat || !Cmat || !A || !Dskip || !dt_bias || !conv_w || !conv_b || !out ||
        !conv_state_out || !ssm_state_out)
        return fail(SSM_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (in_stride_t < d_inner) return fail(SSM_ERR_INVALID_ARG, "%s: in_stride_t %lld < d_inner", fn, (long long)(in_stride_t));
    if (batch > 1 && in_stride_b < 1) return fail(SSM_ERR_INVALID_ARG, "%s: in_stride_b %lld < 1", fn, (long long)(in_stride_b));
    if (out_stride_t < d_inner) return fail(SSM_ERR_INVALID_ARG, "%s: out_stride_t %lld < d_inner", fn, (long long)(out_stride_t));
    if (batch > 1 && out_stride_b < (int64_t)(seqlen - 1) * out_stride_t + d_inner)
        return fail(SSM_ERR_INVALID_ARG, "%s: out_stride_b %lld lets batch rows overlap", fn, (long long)(out_stride_b));
    if (conv_state_ld < d_inner) return fail(SSM_ERR_INVALID_ARG, "%s: conv_state_ld %lld < d_inner", fn, (long long)(conv_state_ld));
    if (ssm_state_stride_b < 16LL * d_inner)
        return fail(SSM_ERR_INVALID_ARG, "%s: ssm_state_stride_b %lld < 16*d_inner", fn, (long long)(ssm_state_stride_b));
    const int es = esize(in_dtype);
    if (!aligned(x, 16) || !aligned(z, 16) || !aligned(dt, 16) || !aligned(Bmat, 16) || !aligned(Cmat, 16))
        return fail(SSM_ERR_MISALIGNED, "%s: x, z, dt, B and C must be 16-byte aligned", fn);
    if ((in_stride_t * es) % 16 != 0 || (batch > 1 && (in_stride_b * es) % 16 != 0))
        return fail(SSM_ERR_MISALIGNED, "%s: input strides must be multiples of 16 bytes", fn);
    if (!aligned(A, 16) || !aligned(conv_w, 16)) return fail(SSM_ERR_MISALIGNED, "%s: A and conv_w must be 16-byte aligned", fn);
    if (!aligned(ssm_state_out, 8) || (ssm_state_in && !aligned(ssm_state_in, 8)) || ssm_state_stride_b % 2 != 0)
        return fail(SSM_ERR_MISALIGNED, "%s: ssm states must be 8-byte aligned with an even batch stride", fn);
    if (!aligned(out, esize(out_dtype))) return fail(SSM_ERR_MISALIGNED, "%s: out is not element aligned", fn);
    if (seg_len < ssm::kPrefillChunk || seg_len % ssm::kPrefillChunk != 0)
        return fail(SSM_ERR_INVALID_ARG, "%s: seg_len %lld is not a positive multiple of %d", fn, (long long)seg_len,
                    ssm::kPrefillChunk);
    const int64_t n_seg = ((int64_t)seqlen + seg_len - 1) / seg_len;
    if (n_seg > 65535) return fail(SSM_ERR_INVALID_ARG, "%s: %lld segments (at most 65535)", fn, (long long)n_seg);
    if (n_seg > 1 && fixed_scratch) {
        // the library's own array stands in for the workspace; every other argument is valid
        const size_t need = ssm_prefill_workspace_bytes(batch, seqlen, d_inner, seg_len);
        if (need > (size_t)SSM_NOALLOC_SCRATCH_BYTES)
            return fail(SSM_ERR_INVALID_ARG,
                        "%s: these sizes need %zu bytes of scratch and the fixed array holds %zu "
                        "(use a longer seg_len, or ssm_prefill_segmented with a workspace)",
                        fn, need, (size_t)SSM_NOALLOC_SCRATCH_BYTES);
        int err = 0;
        workspace = noalloc_scratch_ptr(&err);
        workspace_bytes = (size_t)SSM_NOALLOC_SCRATCH_BYTES;
        if (err) return fail(SSM_ERR_CUDA, "%s: the scratch array's device address is unavailable", fn);
    }
    if (n_seg > 1) {
        const size_t need = ssm_prefill_workspace_bytes(batch, seqlen, d_inner, seg_len);
        if (!workspace || workspace_bytes < need)
            return fail(SSM_ERR_INVALID_ARG, "%s: workspace of %zu bytes given, %zu needed", fn,
                        workspace ? workspace_bytes : (size_t)0, need);
        if (!aligned(workspace, 16)) return fail(SSM_ERR_MISALIGNED, "%s: workspace must be 16-byte aligned", fn);
    }

    int serr = 0;
    unsigned int* status = status_ptr(&serr);
    if (serr) return fail(SSM_ERR_CUDA, "%s: no usable CUDA device", fn);

    ssm::PrefillLaunch q{};
    q.batch = batch;
    q.in_bf16 = in_dtype == SSM_BF16;
    q.out_bf16 = out_dtype == SSM_BF16;
    q.z = z;
    q.dt = dt;
    q.Bm = Bmat;
    q.Cm = Cmat;
    ssm::PrefillArgs& a = q.args;
    a.seqlen = seqlen;
    a.d_inner = d_inner;
    a.x = x;
    a.in_stride_b = in_stride_b;
    a.in_stride_t = in_stride_t;
    a.A = A;
    a.Dskip = Dskip;
    a.dt_bias = dt_bias;
    a.conv_w = conv_w;
    a.conv_b = conv_b;
    a.conv_state_in = conv_state_in;
    a.ssm_state_in = ssm_state_in;
    a.conv_state_ld = conv_state_ld;
    a.ssm_state_stride_b = ssm_state_stride_b;
    a.out = out;
    a.out_stride_b = out_stride_b;
    a.out_stride_t = out_stride_t;
    a.conv_state_out = conv_state_out;
    a.ssm_state_out = ssm_state_out;
    a.status = status;
    a.seg_len = n_seg > 1 ? seg_len : seqlen;
    a.n_seg = (int)n_seg;
    a.ws = n_seg > 1 ? static_cast<float*>(workspace) : nullptr;
    const char* why = "";
    if (ssm::launch_prefill(q, static_cast<cudaStream_t>(cuda_stream), &why) != 0)
        return fail(SSM_ERR_CUDA, "%s: %s", fn, why);
    return SSM_OK;
}


}  // namespace

extern "C" {

int ssm_abi_version(void) { return 108; }

const char* ssm_last_error(void) { return g_err; }

int ssm_prefill(int batch, int seqlen, int d_inner, int d_state, int d_conv,
                ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                const void* x, const void* z, const void* dt,
                int64_t in_stride_b, int64_t in_stride_t,
                const void* Bmat, const void* Cmat,
                const float* A, const float* Dskip, const float* dt_bias,
                const float* conv_w, const float* conv_b,
                const float* conv_state_in, const float* ssm_state_in,
                int64_t conv_state_ld, int64_t ssm_state_stride_b,
                void* out, int64_t out_stride_b, int64_t out_stride_t,
                float* conv_state_out, float* ssm_state_out,
                void* cuda_stream) {
    // one segment covering the whole row (seg_len rounded up to whole chunks)
    const int one = seqlen > 0 && seqlen <= (1 << 30)
                        ? (seqlen + ssm::kPrefillChunk - 1) / ssm::kPrefillChunk * ssm::kPrefillChunk
                        : ssm::kPrefillChunk;
    return prefill_impl("ssm_prefill", batch, seqlen, d_inner, d_state, d_conv, in_dtype, out_dtype, x, z, dt,
                        in_stride_b, in_stride_t, Bmat, Cmat, A, Dskip, dt_bias, conv_w, conv_b, conv_state_in,
                        ssm_state_in, conv_state_ld, ssm_state_stride_b, out, out_stride_b, out_stride_t,
                        conv_state_out, ssm_state_out, one, nullptr, 0, cuda_stream);
}

int ssm_prefill_segmented_noalloc(int batch, int seqlen, int d_inner, int d_state, int d_conv,
                                  ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                                  const void* x, const void* z, const void* dt,
                                  int64_t in_stride_b, int64_t in_stride_t,
                                  const void* Bmat, const void* Cmat,
                                  const float* A, const float* Dskip, const float* dt_bias,
                                  const float* conv_w, const float* conv_b,
                                  const float* conv_state_in, const float* ssm_state_in,
                                  int64_t conv_state_ld, int64_t ssm_state_stride_b,
                                  void* out, int64_t out_stride_b, int64_t out_stride_t,
                                  float* conv_state_out, float* ssm_state_out,
                                  int seg_len, void* cuda_stream) {
    // Nothing in the array has to start at zero: pass A writes every entry that passes B and C read.
    return prefill_impl("ssm_prefill_segmented_noalloc", batch, seqlen, d_inner, d_state, d_conv, in_dtype,
                        out_dtype, x, z, dt, in_stride_b, in_stride_t, Bmat, Cmat, A, Dskip, dt_bias, conv_w,
                        conv_b, conv_state_in, ssm_state_in, conv_state_ld, ssm_state_stride_b, out, out_stride_b,
                        out_stride_t, conv_state_out, ssm_state_out, seg_len, nullptr, 0, cuda_stream,
                        /*fixed_scratch=*/true);
}

int ssm_out_proj_partial(int64_t M, int64_t N, int64_t K, const void* y, int64_t ldy, const void* W, int64_t ldw,
                         ssm_dtype_t out_dtype, void* out, int64_t ldo, float* block_amax, void* cuda_stream) {
    static const char* fn = "ssm_out_proj_partial";
    g_err[0] = 0;
    if (M < 1 || M > 65535LL * 128) return fail(SSM_ERR_INVALID_ARG, "%s: M %lld not in [1, 65535*128]", fn, (long long)M);
    if (N < 1 || N > 65535LL * 256) return fail(SSM_ERR_INVALID_ARG, "%s: N %lld not in [1, 65535*256]", fn, (long long)N);
    if (K < 1 || K > (1LL << 31)) return fail(SSM_ERR_INVALID_ARG, "%s: K %lld out of range", fn, (long long)K);
    if (!dtype_ok(out_dtype)) return fail(SSM_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    if (!y || !W || !out) return fail(SSM_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (N % 128 != 0) return fail(SSM_ERR_UNSUPPORTED, "%s: N %lld is not a multiple of 128", fn, (long long)N);
    if (K % 8 != 0) return fail(SSM_ERR_UNSUPPORTED, "%s: K %lld is not a multiple of 8", fn, (long long)K);
    if (ldy < K || ldw < K || ldo < N) return fail(SSM_ERR_INVALID_ARG, "%s: a row stride is below the row length", fn);
    if (ldy % 8 != 0 || ldw % 8 != 0 || ldo % 8 != 0)
        return fail(SSM_ERR_MISALIGNED, "%s: row strides must be multiples of 8 elements", fn);
    if (!aligned(y, 16) || !aligned(W, 16) || !aligned(out, 16) || (block_amax && !aligned(block_amax, 4)))
        return fail(SSM_ERR_MISALIGNED, "%s: y, W and out must be 16-byte aligned", fn);
    // the kernel counts 128-row tiles and 64-wide K steps in 32 bits
    const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
    if (tiles * ((K + 63) / 64) >= (1LL << 31))
        return fail(SSM_ERR_UNSUPPORTED, "%s: %lld tiles x %lld K steps exceed 2^31", fn, (long long)tiles,
                    (long long)((K + 63) / 64));

    int serr = 0;
    unsigned int* status = status_ptr(&serr);
    if (serr) return fail(SSM_ERR_CUDA, "%s: no usable CUDA device", fn);
    ssm::OutProjArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.out = out;
    a.ldo = ldo;
    a.amax = block_amax;
    a.status = status;
    const char* why = "";
    if (ssm::launch_out_proj(a, y, W, ldy, ldw, out_dtype == SSM_BF16, static_cast<cudaStream_t>(cuda_stream), &why) != 0)
        return fail(SSM_ERR_CUDA, "%s: %s", fn, why);
    return SSM_OK;
}

size_t ssd_prefill_workspace_bytes(int batch, int seqlen, int n_heads, int n_groups) {
    if (batch < 1 || batch > 65535 || seqlen < 1 || seqlen > (1 << 30) || n_heads < 1 || n_heads > 65535 ||
        n_groups < 1 || n_heads % n_groups != 0)
        return 0;
    return ssm::ssd_workspace_layout(batch, seqlen, n_heads, n_groups).bytes;
}

int ssd_prefill(int batch, int seqlen, int n_heads, int head_dim, int n_groups, int d_state, int d_conv,
                ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                const void* xBC, int64_t xbc_stride_b, int64_t xbc_stride_t,
                const void* z, int64_t z_stride_b, int64_t z_stride_t,
                const void* dt, int64_t dt_stride_b, int64_t dt_stride_t,
                const float* conv_w, const float* conv_b,
                const float* A, const float* Dskip, const float* dt_bias,
                const float* conv_state_in, const float* ssm_state_in,
                void* out, int64_t out_stride_b, int64_t out_stride_t,
                float* conv_state_out, float* ssm_state_out,
                void* workspace, size_t workspace_bytes, void* cuda_stream) {
    static const char* fn = "ssd_prefill";
    g_err[0] = 0;
    if (batch < 1 || batch > 65535) return fail(SSM_ERR_INVALID_ARG, "%s: batch %d not in [1, 65535]", fn, batch);
    if (seqlen < 1 || seqlen > (1 << 30)) return fail(SSM_ERR_INVALID_ARG, "%s: seqlen %d not in [1, 2^30]", fn, seqlen);
    if (n_heads < 1 || n_heads > 65535) return fail(SSM_ERR_INVALID_ARG, "%s: n_heads %d not in [1, 65535]", fn, n_heads);
    if (n_groups < 1 || n_heads % n_groups != 0)
        return fail(SSM_ERR_INVALID_ARG, "%s: n_groups %d does not divide n_heads %d", fn, n_groups, n_heads);
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return fail(SSM_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    if (head_dim != 64 || d_state != 64 || d_conv != 4)
        return fail(SSM_ERR_UNSUPPORTED, "%s: head_dim %d, d_state %d, d_conv %d unsupported (64, 64, 4 only)", fn,
                    head_dim, d_state, d_conv);
    if (in_dtype != SSM_BF16) return fail(SSM_ERR_UNSUPPORTED, "%s: token inputs must be bf16", fn);
    if (!xBC || !z || !dt || !conv_w || !conv_b || !A || !Dskip || !dt_bias || !out || !conv_state_out ||
        !ssm_state_out || !workspace)
        return fail(SSM_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    const int64_t HP = 64LL * n_heads, Cx = HP + 128LL * n_groups;
    if (xbc_stride_t < Cx || z_stride_t < HP || dt_stride_t < n_heads || out_stride_t < HP)
        return fail(SSM_ERR_INVALID_ARG, "%s: a token stride is below the row width", fn);
    if (batch > 1 && (xbc_stride_b < (int64_t)(seqlen - 1) * xbc_stride_t + Cx ||
                      z_stride_b < (int64_t)(seqlen - 1) * z_stride_t + HP ||
                      dt_stride_b < (int64_t)(seqlen - 1) * dt_stride_t + n_heads))
        return fail(SSM_ERR_INVALID_ARG, "%s: a batch stride lets rows overlap", fn);
    if (batch > 1 && out_stride_b < (int64_t)(seqlen - 1) * out_stride_t + HP)
        return fail(SSM_ERR_INVALID_ARG, "%s: out_stride_b %lld lets batch rows overlap", fn, (long long)out_stride_b);
    const size_t need = ssm::ssd_workspace_layout(batch, seqlen, n_heads, n_groups).bytes;
    if (workspace_bytes < need)
        return fail(SSM_ERR_INVALID_ARG, "%s: workspace of %zu bytes given, %zu needed", fn, workspace_bytes, need);
    const int oe = esize(out_dtype);
    if (!aligned(xBC, 16) || !aligned(z, 16) || xbc_stride_t % 8 || xbc_stride_b % 8 || z_stride_t % 8 || z_stride_b % 8)
        return fail(SSM_ERR_MISALIGNED, "%s: xBC and z must be 16-byte aligned with strides of 16 bytes", fn);
    if (!aligned(out, 16) || (out_stride_t * oe) % 16 || (out_stride_b * oe) % 16)
        return fail(SSM_ERR_MISALIGNED, "%s: out must be 16-byte aligned with strides of 16 bytes", fn);
    if (!aligned(conv_w, 16) || !aligned(ssm_state_out, 16) || (ssm_state_in && !aligned(ssm_state_in, 16)) ||
        !aligned(workspace, 16) || !aligned(dt, 2))
        return fail(SSM_ERR_MISALIGNED, "%s: conv_w, the ssm states and the workspace need 16-byte alignment", fn);

    int serr = 0;
    unsigned int* status = status_ptr(&serr);
    if (serr) return fail(SSM_ERR_CUDA, "%s: no usable CUDA device", fn);
    ssm::SsdArgs a{};
    a.batch = batch;
    a.seqlen = seqlen;
    a.n_heads = n_heads;
    a.n_groups = n_groups;
    a.xBC = xBC;
    a.xbc_stride_b = xbc_stride_b;
    a.xbc_stride_t = xbc_stride_t;
    a.z = z;
    a.z_stride_b = z_stride_b;
    a.z_stride_t = z_stride_t;
    a.dt = dt;
    a.dt_stride_b = dt_stride_b;
    a.dt_stride_t = dt_stride_t;
    a.conv_w = conv_w;
    a.conv_b = conv_b;
    a.A = A;
    a.Dskip = Dskip;
    a.dt_bias = dt_bias;
    a.conv_state_in = conv_state_in;
    a.ssm_state_in = ssm_state_in;
    a.out = out;
    a.out_stride_b = out_stride_b;
    a.out_stride_t = out_stride_t;
    a.conv_state_out = conv_state_out;
    a.ssm_state_out = ssm_state_out;
    a.workspace = workspace;
    a.status = status;
    const char* why = "";
    if (ssm::launch_ssd_prefill(a, out_dtype == SSM_BF16, static_cast<cudaStream_t>(cuda_stream), &why) != 0)
        return fail(SSM_ERR_CUDA, "%s: %s", fn, why);
    return SSM_OK;
}

int ssd_decode_step(int batch, int n_heads, int head_dim, int n_groups, int d_state, int d_conv,
                    ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                    const void* xBC, const void* z, const void* dt,
                    const float* conv_w, const float* conv_b,
                    const float* A, const float* Dskip, const float* dt_bias,
                    float* conv_state, float* ssm_state, int n_slots, const int32_t* state_slot,
                    void* out, void* cuda_stream) {
    static const char* fn = "ssd_decode_step";
    g_err[0] = 0;
    if (batch < 1 || batch > 65535) return fail(SSM_ERR_INVALID_ARG, "%s: batch %d not in [1, 65535]", fn, batch);
    if (n_heads < 1 || n_heads > 65535) return fail(SSM_ERR_INVALID_ARG, "%s: n_heads %d not in [1, 65535]", fn, n_heads);
    if (n_groups < 1 || n_heads % n_groups != 0)
        return fail(SSM_ERR_INVALID_ARG, "%s: n_groups %d does not divide n_heads %d", fn, n_groups, n_heads);
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return fail(SSM_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    if (head_dim != 64 || d_state != 64 || d_conv != 4)
        return fail(SSM_ERR_UNSUPPORTED, "%s: head_dim %d, d_state %d, d_conv %d unsupported (64, 64, 4 only)", fn,
                    head_dim, d_state, d_conv);
    if (!xBC || !z || !dt || !conv_w || !conv_b || !A || !Dskip || !dt_bias || !conv_state || !ssm_state || !out)
        return fail(SSM_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (n_slots < 1 || (!state_slot && n_slots < batch))
        return fail(SSM_ERR_INVALID_ARG, "%s: n_slots %d too small", fn, n_slots);
    const int es = esize(in_dtype);
    if (!aligned(conv_w, 16) || !aligned(ssm_state, 16))
        return fail(SSM_ERR_MISALIGNED, "%s: conv_w and ssm_state need 16-byte alignment", fn);
    if (!aligned(xBC, es) || !aligned(z, es) || !aligned(dt, es) || !aligned(out, esize(out_dtype)) ||
        !aligned(conv_state, 4) || (state_slot && !aligned(state_slot, 4)))
        return fail(SSM_ERR_MISALIGNED, "%s: a pointer is not element aligned", fn);
    int serr = 0;
    unsigned int* status = status_ptr(&serr);
    if (serr) return fail(SSM_ERR_CUDA, "%s: no usable CUDA device", fn);
    ssm::SsdDecodeArgs a{};
    a.batch = batch;
    a.n_heads = n_heads;
    a.n_groups = n_groups;
    a.n_slots = n_slots;
    a.xBC = xBC;
    a.z = z;
    a.dt = dt;
    a.conv_w = conv_w;
    a.conv_b = conv_b;
    a.A = A;
    a.Dskip = Dskip;
    a.dt_bias = dt_bias;
    a.conv_state = conv_state;
    a.ssm_state = ssm_state;
    a.state_slot = state_slot;
    a.out = out;
    a.status = status;
    const char* why = "";
    if (ssm::launch_ssd_decode(a, in_dtype == SSM_BF16, out_dtype == SSM_BF16, static_cast<cudaStream_t>(cuda_stream),
                               &why) != 0)
        return fail(SSM_ERR_CUDA, "%s: %s", fn, why);
    return SSM_OK;
}

int ssm_selftest_expire_wait(int limit_us, void* cuda_stream) {
    static const char* fn = "ssm_selftest_expire_wait";
    g_err[0] = 0;
    if (limit_us < 1 || limit_us > 2000000) return fail(SSM_ERR_INVALID_ARG, "%s: limit_us %d not in [1, 2e6]", fn, limit_us);
    int serr = 0;
    unsigned int* status = status_ptr(&serr);
    if (serr) return fail(SSM_ERR_CUDA, "%s: no usable CUDA device", fn);
    const char* why = "";
    if (ssm::launch_expire_wait(status, (uint64_t)limit_us * 1000u, static_cast<cudaStream_t>(cuda_stream), &why) != 0)
        return fail(SSM_ERR_CUDA, "%s: %s", fn, why);
    return SSM_OK;
}

size_t ssm_prefill_workspace_bytes(int batch, int seqlen, int d_inner, int seg_len) {
    if (batch < 1 || seqlen < 1 || d_inner < 1 || seg_len < 1) return 0;
    const int64_t n_seg = ((int64_t)seqlen + seg_len - 1) / seg_len;
    return (size_t)(n_seg - 1) * (size_t)batch * (size_t)d_inner * 32 * sizeof(float);
}

int ssm_prefill_segmented(int batch, int seqlen, int d_inner, int d_state, int d_conv,
                          ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                          const void* x, const void* z, const void* dt,
                          int64_t in_stride_b, int64_t in_stride_t,
                          const void* Bmat, const void* Cmat,
                          const float* A, const float* Dskip, const float* dt_bias,
                          const float* conv_w, const float* conv_b,
                          const float* conv_state_in, const float* ssm_state_in,
                          int64_t conv_state_ld, int64_t ssm_state_stride_b,
                          void* out, int64_t out_stride_b, int64_t out_stride_t,
                          float* conv_state_out, float* ssm_state_out,
                          int seg_len, void* workspace, size_t workspace_bytes,
                          void* cuda_stream) {
    return prefill_impl("ssm_prefill_segmented", batch, seqlen, d_inner, d_state, d_conv, in_dtype, out_dtype,
                        x, z, dt, in_stride_b, in_stride_t, Bmat, Cmat, A, Dskip, dt_bias, conv_w, conv_b,
                        conv_state_in, ssm_state_in, conv_state_ld, ssm_state_stride_b, out, out_stride_b,
                        out_stride_t, conv_state_out, ssm_state_out, seg_len, workspace, workspace_bytes,
                        cuda_stream);
}

}  // extern "C"

namespace {

// Shared by ssm_decode_step (one token) and ssm_decode_tokens (T tokens).
int decode_impl(const char* fn, int batch, int n_tokens, int d_inner, int d_state, int d_conv,
                ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                const void* x, const void* z, const void* dt, int64_t in_stride_b, int64_t in_stride_t,
                const void* Bmat, const void* Cmat,
                const float* A, const float* Dskip, const float* dt_bias,
                const float* conv_w, const float* conv_b,
                float* conv_state, float* ssm_state,
                int64_t conv_state_ld, int64_t ssm_state_stride_b,
                int n_slots, const int32_t* state_slot,
                void* out, int64_t out_stride_b, int64_t out_stride_t,
                void* cuda_stream) {
    g_err[0] = 0;
    if (batch < 1 || batch > 65535) return fail(SSM_ERR_INVALID_ARG, "%s: batch %lld not in [1, 65535]", fn, (long long)batch);
    if (n_tokens < 1 || n_tokens > 4096) return fail(SSM_ERR_INVALID_ARG, "%s: n_tokens %lld not in [1, 4096]", fn, (long long)n_tokens);
    if (d_inner < 1) return fail(SSM_ERR_INVALID_ARG, "%s: d_inner %lld < 1", fn, (long long)d_inner);
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return fail(SSM_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    if (d_state != 16) return fail(SSM_ERR_UNSUPPORTED, "%s: d_state %lld unsupported (16 only)", fn, (long long)d_state);
    if (d_conv != 4) return fail(SSM_ERR_UNSUPPORTED, "%s: d_conv %lld unsupported (4 only)", fn, (long long)d_conv);
    if (d_inner % 8 != 0) return fail(SSM_ERR_UNSUPPORTED, "%s: d_inner %lld is not a multiple of 8", fn, (long long)d_inner);
    if (!x || !z || !dt || !Bmat || !Cmat || !A || !Dskip || !dt_bias || !conv_w || !conv_b || !conv_state ||
        !ssm_state || !out)
        return fail(SSM_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (n_tokens > 1 && in_stride_t < d_inner) return fail(SSM_ERR_INVALID_ARG, "%s: in_stride_t %lld < d_inner", fn, (long long)in_stride_t);
    if (n_tokens > 1 && out_stride_t < d_inner) return fail(SSM_ERR_INVALID_ARG, "%s: out_stride_t %lld < d_inner", fn, (long long)out_stride_t);
    const int64_t in_row = n_tokens > 1 ? (int64_t)(n_tokens - 1) * in_stride_t + d_inner : d_inner;
    const int64_t out_row = n_tokens > 1 ? (int64_t)(n_tokens - 1) * out_stride_t + d_inner : d_inner;
    if (batch > 1 && in_stride_b < in_row) return fail(SSM_ERR_INVALID_ARG, "%s: in_stride_b %lld too small", fn, (long long)in_stride_b);
    if (batch > 1 && out_stride_b < out_row) return fail(SSM_ERR_INVALID_ARG, "%s: out_stride_b %lld lets requests overlap", fn, (long long)out_stride_b);
    if (conv_state_ld < d_inner) return fail(SSM_ERR_INVALID_ARG, "%s: conv_state_ld %lld < d_inner", fn, (long long)conv_state_ld);
    if (ssm_state_stride_b < 16LL * d_inner)
        return fail(SSM_ERR_INVALID_ARG, "%s: ssm_state_stride_b %lld < 16*d_inner", fn, (long long)ssm_state_stride_b);
    if (n_slots < 1 || (!state_slot && n_slots < batch))
        return fail(SSM_ERR_INVALID_ARG, "%s: n_slots %lld too small", fn, (long long)n_slots);
    const int es = esize(in_dtype);
    if (!aligned(Bmat, 4 * es) || !aligned(Cmat, 4 * es))
        return fail(SSM_ERR_MISALIGNED, "%s: B and C must be aligned to 4 elements", fn);
    if (!aligned(A, 16) || !aligned(conv_w, 16) || !aligned(ssm_state, 16) || ssm_state_stride_b % 4 != 0)
        return fail(SSM_ERR_MISALIGNED, "%s: A, conv_w and ssm_state need 16-byte alignment", fn);
    if (!aligned(x, es) || !aligned(z, es) || !aligned(dt, es) || !aligned(out, esize(out_dtype)) ||
        !aligned(conv_state, 4) || (state_slot && !aligned(state_slot, 4)))
        return fail(SSM_ERR_MISALIGNED, "%s: a pointer is not element aligned", fn);

    int serr = 0;
    unsigned int* status = status_ptr(&serr);
    if (serr) return fail(SSM_ERR_CUDA, "%s: no usable CUDA device", fn);

    ssm::DecodeArgs a{};
    a.batch = batch;
    a.n_tokens = n_tokens;
    a.d_inner = d_inner;
    a.n_slots = n_slots;
    a.x = x;
    a.z = z;
    a.dt = dt;
    a.in_stride_b = in_stride_b;
    a.in_stride_t = in_stride_t;
    a.Bm = Bmat;
    a.Cm = Cmat;
    a.A = A;
    a.Dskip = Dskip;
    a.dt_bias = dt_bias;
    a.conv_w = conv_w;
    a.conv_b = conv_b;
    a.conv_state = conv_state;
    a.ssm_state = ssm_state;
    a.conv_state_ld = conv_state_ld;
    a.ssm_state_stride_b = ssm_state_stride_b;
    a.state_slot = state_slot;
    a.out = out;
    a.out_stride_b = out_stride_b;
    a.out_stride_t = out_stride_t;
    a.status = status;
    const char* why = "";
    if (ssm::launch_decode(a, in_dtype == SSM_BF16, out_dtype == SSM_BF16, static_cast<cudaStream_t>(cuda_stream),
                           &why) != 0)
        return fail(SSM_ERR_CUDA, "%s: %s", fn, why);
    return SSM_OK;
}

}  // namespace

extern "C" {

int ssm_decode_step(int batch, int d_inner, int d_state, int d_conv,
                    ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                    const void* x, const void* z, const void* dt, int64_t in_stride_b,
                    const void* Bmat, const void* Cmat,
                    const float* A, const float* Dskip, const float* dt_bias,
                    const float* conv_w, const float* conv_b,
                    float* conv_state, float* ssm_state,
                    int64_t conv_state_ld, int64_t ssm_state_stride_b,
                    int n_slots, const int32_t* state_slot,
                    void* out, int64_t out_stride_b,
                    void* cuda_stream) {
    return decode_impl("ssm_decode_step", batch, 1, d_inner, d_state, d_conv, in_dtype, out_dtype, x, z, dt,
                       in_stride_b, d_inner, Bmat, Cmat, A, Dskip, dt_bias, conv_w, conv_b, conv_state, ssm_state,
                       conv_state_ld, ssm_state_stride_b, n_slots, state_slot, out, out_stride_b, d_inner,
                       cuda_stream);
}

int ssm_decode_tokens(int batch, int n_tokens, int d_inner, int d_state, int d_conv,
                      ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                      const void* x, const void* z, const void* dt,
                      int64_t in_stride_b, int64_t in_stride_t,
                      const void* Bmat, const void* Cmat,
                      const float* A, const float* Dskip, const float* dt_bias,
                      const float* conv_w, const float* conv_b,
                      float* conv_state, float* ssm_state,
                      int64_t conv_state_ld, int64_t ssm_state_stride_b,
                      int n_slots, const int32_t* state_slot,
                      void* out, int64_t out_stride_b, int64_t out_stride_t,
                      void* cuda_stream) {
    return decode_impl("ssm_decode_tokens", batch, n_tokens, d_inner, d_state, d_conv, in_dtype, out_dtype, x, z,
                       dt, in_stride_b, in_stride_t, Bmat, Cmat, A, Dskip, dt_bias, conv_w, conv_b, conv_state,
                       ssm_state, conv_state_ld, ssm_state_stride_b, n_slots, state_slot, out, out_stride_b,
                       out_stride_t, cuda_stream);
}

int q8_reduce_partials(int P, const void* const* partials, ssm_dtype_t in_dtype, int64_t n, int block,
                       void* out, ssm_dtype_t out_dtype, int32_t* sums_out, float* scales_out,
                       void* cuda_stream) {
    g_err[0] = 0;
    if (P < 1 || P > ssm::kMaxPartials) return fail(SSM_ERR_UNSUPPORTED, "q8_reduce_partials: P %lld not in [1, 8]", (long long)(P));
    if (!partials) return fail(SSM_ERR_INVALID_ARG, "q8_reduce_partials: partials is NULL");
    if (n < 1) return fail(SSM_ERR_INVALID_ARG, "q8_reduce_partials: n %lld < 1", (long long)(n));
    if (block != 128) return fail(SSM_ERR_UNSUPPORTED, "q8_reduce_partials: block %lld unsupported (128 only)", (long long)(block));
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return fail(SSM_ERR_INVALID_ARG, "q8_reduce_partials: unknown dtype");
    if (!out) return fail(SSM_ERR_INVALID_ARG, "q8_reduce_partials: out is NULL");
    ssm::Q8Args a{};
    for (int p = 0; p < P; ++p) {
        if (!partials[p]) return fail(SSM_ERR_INVALID_ARG, "q8_reduce_partials: partials[%lld] is NULL", (long long)(p));
        if (!aligned(partials[p], 16)) return fail(SSM_ERR_MISALIGNED, "q8_reduce_partials: partials[%lld] not 16-byte aligned", (long long)(p));
        a.partials[p] = partials[p];
    }
    if (!aligned(out, 16) || (sums_out && !aligned(sums_out, 16)) || (scales_out && !aligned(scales_out, 4)))
        return fail(SSM_ERR_MISALIGNED, "q8_reduce_partials: out and sums must be 16-byte aligned");
    a.P = P;
    a.n = n;
    a.out = out;
    a.sums = sums_out;
    a.scales = scales_out;
    const char* why = "";
    if (ssm::launch_q8(a, in_dtype == SSM_BF16, out_dtype == SSM_BF16, static_cast<cudaStream_t>(cuda_stream), &why) != 0)
        return fail(SSM_ERR_CUDA, "q8_reduce_partials: %s", why);
    return SSM_OK;
}

int q8_block_absmax(const void* x, ssm_dtype_t in_dtype, int64_t n, int block, float* block_amax,
                    void* cuda_stream) {
    static const char* fn = "q8_block_absmax";
    g_err[0] = 0;
    if (!x || !block_amax) return fail(SSM_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (n < 1) return fail(SSM_ERR_INVALID_ARG, "%s: n %lld < 1", fn, (long long)n);
    if (block != 128) return fail(SSM_ERR_UNSUPPORTED, "%s: block %d unsupported (128 only)", fn, block);
    if (!dtype_ok(in_dtype)) return fail(SSM_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    if (!aligned(x, 16) || !aligned(block_amax, 4)) return fail(SSM_ERR_MISALIGNED, "%s: x must be 16-byte aligned", fn);
    const char* why = "";
    if (ssm::launch_q8_absmax(x, in_dtype == SSM_BF16, n, block_amax, static_cast<cudaStream_t>(cuda_stream), &why) != 0)
        return fail(SSM_ERR_CUDA, "%s: %s", fn, why);
    return SSM_OK;
}

int q8_quantize_shared(const void* x, ssm_dtype_t in_dtype, int64_t n, int block, const float* block_amax,
                       int8_t* codes, float* scales_out, void* cuda_stream) {
    static const char* fn = "q8_quantize_shared";
    g_err[0] = 0;
    if (!x || !block_amax || !codes) return fail(SSM_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (n < 1) return fail(SSM_ERR_INVALID_ARG, "%s: n %lld < 1", fn, (long long)n);
    if (block != 128) return fail(SSM_ERR_UNSUPPORTED, "%s: block %d unsupported (128 only)", fn, block);
    if (!dtype_ok(in_dtype)) return fail(SSM_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(block_amax, 4) || (scales_out && !aligned(scales_out, 4)))
        return fail(SSM_ERR_MISALIGNED, "%s: x and codes must be 16-byte aligned", fn);
    const char* why = "";
    if (ssm::launch_q8_quantize(x, in_dtype == SSM_BF16, n, block_amax, codes, scales_out,
                                static_cast<cudaStream_t>(cuda_stream), &why) != 0)
        return fail(SSM_ERR_CUDA, "%s: %s", fn, why);
    return SSM_OK;
}

int q8_sum_dequant(int P, const int8_t* const* codes, const float* scales, int64_t n, int block,
                   void* out, ssm_dtype_t out_dtype, int32_t* sums_out, void* cuda_stream) {
    static const char* fn = "q8_sum_dequant";
    g_err[0] = 0;
    if (P < 1 || P > ssm::kMaxPartials) return fail(SSM_ERR_UNSUPPORTED, "%s: P %d not in [1, 8]", fn, P);
    if (!codes || !scales || !out) return fail(SSM_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (n < 1) return fail(SSM_ERR_INVALID_ARG, "%s: n %lld < 1", fn, (long long)n);
    if (block != 128) return fail(SSM_ERR_UNSUPPORTED, "%s: block %d unsupported (128 only)", fn, block);
    if (!dtype_ok(out_dtype)) return fail(SSM_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    for (int p = 0; p < P; ++p) {
        if (!codes[p]) return fail(SSM_ERR_INVALID_ARG, "%s: codes[%d] is NULL", fn, p);
        if (!aligned(codes[p], 16)) return fail(SSM_ERR_MISALIGNED, "%s: codes[%d] not 16-byte aligned", fn, p);
    }
    if (!aligned(out, 16) || !aligned(scales, 4) || (sums_out && !aligned(sums_out, 16)))
        return fail(SSM_ERR_MISALIGNED, "%s: out and sums must be 16-byte aligned", fn);
    const char* why = "";
    if (ssm::launch_q8_sum(P, codes, scales, n, out, out_dtype == SSM_BF16, sums_out,
                           static_cast<cudaStream_t>(cuda_stream), &why) != 0)
        return fail(SSM_ERR_CUDA, "%s: %s", fn, why);
    return SSM_OK;
}

int ssm_device_status(uint32_t* status, int clear) {
    g_err[0] = 0;
    if (!status) return fail(SSM_ERR_INVALID_ARG, "ssm_device_status: status is NULL");
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof v) != cudaSuccess)
        return fail(SSM_ERR_CUDA, "ssm_device_status: cudaMemcpyFromSymbol failed");
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess)
            return fail(SSM_ERR_CUDA, "ssm_device_status: cudaMemcpyToSymbol failed");
    }
    *status = v;
    return SSM_OK;
}

}  // extern "C"
