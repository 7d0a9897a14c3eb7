/*
 * ssm.h -- C ABI of libssm: the selective state-space (SSM) mixer hot path on
 * one NVIDIA GB300 GPU (sm_103a).
 *
 * What is computed.  The pages this library follows ("Scaling State-Space Models
 * on Multiple GPUs with Tensor Parallelism", euno.news summary of arXiv
 * 2602.21144) describe a tensor-parallel SSM layer in which
 *   - every channel slice keeps its own hidden state, so the per-token recurrent
 *     update needs nothing from other channels (Methodology 2, "local recurrence");
 *   - the hidden state is cached at prefill and reused by token-by-token decode
 *     (Methodology 3, "state caching during prefill and decode");
 *   - partial outputs are quantized to 8 bits, summed and dequantized
 *     (Methodology 4, "quantized All-Reduce").
 * The pages do not print the mixer's equations; this library computes the
 * Mamba-style selective-scan mixer.  For batch row b, channel d, token t and
 * state n (N = d_state = 16, W = d_conv = 4):
 *
 *   xc_t    = conv_b[d] + sum_{k<W} conv_w[d][k] * x_{t-W+1+k}      (x_{<0}: conv_state_in or 0)
 *   u_t     = xc_t * sigmoid(xc_t)                                   (SiLU)
 *   delta_t = softplus(dt_t + dt_bias[d])
 *   h_t[n]  = exp(delta_t * A[d][n]) * h_{t-1}[n] + delta_t * B_t[n] * u_t
 *   y_t     = sum_n C_t[n] * h_t[n] + D[d] * u_t
 *   out_t   = y_t * z_t * sigmoid(z_t)
 *
 * Readings where the description leaves a step open: the "x" of the input and
 * skip terms is the post-conv, post-SiLU u; conv_w[d][W-1] multiplies the current
 * token; the conv state holds the last W-1 raw (pre-conv) inputs, oldest first;
 * B and C are per-token inputs shared by all channels; states start at zero when
 * no input state is given.
 *
 * Conventions for every call.
 *   - All pointers except `partials` (a host array) are DEVICE pointers owned by
 *     the caller.  The library allocates nothing and keeps no per-call state.
 *   - Calls are asynchronous on `cuda_stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Argument errors are found on the host before any launch
 *     and return a negative status synchronously; nothing is launched then.
 *   - Element strides are in ELEMENTS, channel stride is always 1.
 *   - Inputs and outputs must not alias, except the in-place decode states.
 *   - Supported: d_state == 16, d_conv == 4, d_inner % 8 == 0; token tensors
 *     16-byte aligned with 16-byte-multiple row strides.  Other shapes return
 *     SSM_ERR_UNSUPPORTED / SSM_ERR_MISALIGNED.
 *   - ssm_last_error() describes the last non-OK return on the calling thread.
 */
#ifndef SSM_H_
#define SSM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype_t;

enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = -1,   /* bad size, null required pointer, bad stride */
    SSM_ERR_UNSUPPORTED = -2,   /* valid but not implemented (d_state != 16, ...) */
    SSM_ERR_MISALIGNED = -3,    /* pointer or stride breaks the 16-byte rule */
    SSM_ERR_CUDA = -4,          /* a CUDA runtime/driver call or launch failed */
    SSM_ERR_DEVICE_TIMEOUT = -5 /* reported by ssm_device_status(): an in-kernel wait gave up */
};

/* Bits of the device status word (see ssm_device_status). */
enum {
    SSM_DEV_WAIT_TIMEOUT = 1u,  /* a bounded wait on a TMA copy expired; the block stopped early */
    SSM_DEV_BAD_SLOT = 2u,      /* a decode request named a state slot outside [0, n_slots) */
    SSM_DEV_SMEM_ALIGN = 4u     /* shared memory was not 128-byte aligned; the prefill did nothing */
};

/* ABI version of this header (major * 100 + minor). */
int ssm_abi_version(void);

/*
 * ssm_prefill -- run the mixer over `seqlen` tokens of every batch row and
 * return the outputs plus the final conv and SSM states (the cached state of
 * Methodology 3).  Channels are independent (Methodology 2): the result for a
 * channel does not depend on d_inner, on which other channels are in the call,
 * or on the launch shape, bit for bit.
 *
 *   batch, seqlen, d_inner       B >= 1, L >= 1, D >= 8 with D % 8 == 0
 *   d_state, d_conv              must be 16 and 4
 *   in_dtype                     SSM_BF16 or SSM_F32, for x, z, dt, Bmat, Cmat
 *   out_dtype                    SSM_F32 or SSM_BF16 (round to nearest even)
 *   x, z, dt                     [B][L][D] views: element (b, t, d) at
 *                                b*in_stride_b + t*in_stride_t + d; in_stride_t >= D
 *                                (a channel slice of a wider tensor is allowed);
 *                                base 16-byte aligned, strides*size multiples of 16
 *   Bmat, Cmat                   [B][L][16] contiguous, 16-byte aligned
 *   A, Dskip, dt_bias            [D][16], [D], [D] float32 (A row-major, rows of 16)
 *   conv_w, conv_b               [D][4], [D] float32
 *   conv_state_in                NULL (zeros) or [B][3][conv_state_ld] float32, oldest first
 *   ssm_state_in                 NULL (zeros) or [B][*][16] float32 with batch stride
 *                                ssm_state_stride_b (>= 16*D), channel stride 16
 *   conv_state_ld                row stride of conv_state_in/out, >= D
 *   ssm_state_stride_b           batch stride of ssm_state_in/out, >= 16*D
 *   out                          [B][L][D] view with out_stride_b, out_stride_t (>= D)
 *   conv_state_out, ssm_state_out required, same layouts as the inputs; may not
 *                                alias the inputs
 * Returns SSM_OK or a negative status.
 */
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
                void* cuda_stream);

/*
 * ssm_prefill_workspace_bytes -- bytes of device workspace that ssm_prefill_segmented
 * needs for these sizes: (ceil(seqlen / seg_len) - 1) * batch * d_inner * 128.  Zero when
 * the row is a single segment or an argument is not positive.
 */
size_t ssm_prefill_workspace_bytes(int batch, int seqlen, int d_inner, int seg_len);

/*
 * ssm_prefill_segmented -- ssm_prefill with every row cut into segments of seg_len
 * tokens that run in parallel.  The recurrence h_t = a_t h_{t-1} + b_t stays inside
 * its channel (Methodology 2) and composes associatively, so a segment is summed up
 * by the pair (product of its a_t, state reached from zero).  A carry pass over the
 * segments turns the pairs into every segment's start state.  That is the chunked
 * scan's carry across chunks, taken across thread blocks, and it hands each segment
 * the state that Methodology 3 caches at the end of the row.
 * Use it when there are too few rows to fill the GPU: batch * ceil(d_inner / 16)
 * well below three times the SM count, e.g. batch-1 long-context prefill.  It costs
 * about 1.4 times the arithmetic of ssm_prefill and enqueues three kernels.
 *
 *   every ssm_prefill argument   as for ssm_prefill
 *   seg_len                      tokens per segment, a positive multiple of 64, giving at
 *                                most 65535 segments; seg_len >= seqlen is ssm_prefill itself
 *   workspace, workspace_bytes   device buffer of at least ssm_prefill_workspace_bytes(...)
 *                                bytes, 16-byte aligned, owned by the caller (NULL allowed
 *                                for a single segment).  Its contents on entry do not matter;
 *                                on return they are scratch.  Calls that share a workspace
 *                                must not overlap on the GPU.
 * The result depends on seg_len and seqlen, never on d_inner or the launch shape: a
 * channel slice run with the same seg_len equals the unsplit run bit for bit.  It
 * differs from ssm_prefill by fp32 rounding only, because the start states are
 * composed in another order.
 * Returns SSM_OK or a negative status (SSM_ERR_INVALID_ARG for a bad seg_len or a
 * missing or short workspace).
 */
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
                          void* cuda_stream);

/* Size of the fixed scratch array behind ssm_prefill_segmented_noalloc: 4 MiB per GPU. */
#define SSM_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * ssm_prefill_segmented_noalloc -- ssm_prefill_segmented for callers that cannot allocate
 * device memory when they call.  Examples are a plugin running inside a host program that
 * owns every allocation on the GPU, and a serving loop that must not allocate once it has
 * started, because cudaMalloc can synchronize the device and can fail under memory
 * pressure.  The pages have no counterpart for this call: it only changes where the
 * segment scratch lives.
 *
 * The scratch is a fixed array of SSM_NOALLOC_SCRATCH_BYTES inside the library, which every
 * GPU that loads the library holds until the process exits; nothing is allocated per call.
 *   every argument               as for ssm_prefill_segmented, without the workspace
 *   limit                        ssm_prefill_workspace_bytes(batch, seqlen, d_inner, seg_len)
 *                                must not exceed SSM_NOALLOC_SCRATCH_BYTES, e.g. batch 1 with
 *                                d_inner 8192 and 4 segments (3 MiB).  Larger requests return
 *                                SSM_ERR_INVALID_ARG before anything runs.
 *   first call on a device       looks up the array's device address (cudaGetSymbolAddress)
 *                                with that device current and keeps it; make that first call
 *                                before any stream capture.
 *   sharing                      every call on a device uses the same array, and the array
 *                                keeps the last call's contents.  Nothing in it needs to
 *                                start at zero.  Calls that overlap on the GPU (other streams,
 *                                other host threads) race on it and must be ordered by the
 *                                caller.
 * The result equals ssm_prefill_segmented's for the same seg_len, bit for bit.
 */
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
                                  int seg_len, void* cuda_stream);

/*
 * ssm_decode_step -- one token per request, continuing from cached states that
 * are read and updated IN PLACE (Methodology 3: decode reuses the prefill state).
 * Equals one more token of ssm_prefill.
 *
 *   batch                        number of requests, 1..65535
 *   x, z, dt                     [batch][D] rows with row stride in_stride_b (>= D)
 *   Bmat, Cmat                   [batch][16] contiguous
 *   A .. conv_b                  as for ssm_prefill
 *   conv_state                   [n_slots][3][conv_state_ld] float32, in/out
 *   ssm_state                    [n_slots][*][16] float32, batch stride ssm_state_stride_b, in/out
 *   state_slot                   NULL (request r uses slot r; needs n_slots >= batch) or a
 *                                device array [batch] of slot indices; distinct requests must
 *                                name distinct slots.  An index outside [0, n_slots) skips
 *                                that request and sets SSM_DEV_BAD_SLOT in the status word.
 *   out                          [batch][D] with row stride out_stride_b (>= D)
 */
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
                    void* cuda_stream);

/*
 * ssm_decode_tokens -- n_tokens >= 1 tokens per request, continuing from the cached
 * states and updating them in place (Methodology 3): the same result as n_tokens
 * calls of ssm_decode_step, or as ssm_prefill over those tokens started from the
 * cached states.  Meant for short blocks (speculative or verification tokens,
 * 2..16); long prompts belong to ssm_prefill.  ssm_decode_step is n_tokens = 1.
 *
 *   batch, n_tokens              1..65535 requests, 1..4096 tokens each
 *   x, z, dt                     [batch][n_tokens][D] views: element (r, t, d) at
 *                                r*in_stride_b + t*in_stride_t + d (in_stride_t >= D)
 *   Bmat, Cmat                   [batch][n_tokens][16] contiguous
 *   conv_state, ssm_state,
 *   n_slots, state_slot          as for ssm_decode_step
 *   out                          [batch][n_tokens][D] view with out_stride_b, out_stride_t;
 *                                requests may not overlap
 */
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
                      void* cuda_stream);

/*
 * ssm_out_proj_partial -- one tensor-parallel rank's partial of the mixer's output
 * projection, on the tensor cores.  Methodology 1 splits the layer along the feature
 * dimension, so a rank holds the mixer output of its channel slice and the matching
 * columns of the projection weight.  Methodology 4 sums the ranks' partials through the
 * 8-bit all-reduce.
 *   out[m][n] = sum_k y[m][k] * W[n][k]     (bf16 products, fp32 accumulation)
 * When block_amax is not NULL: block_amax[j] = max |out_i| over block j of 128 consecutive
 * elements of the row-major [M][N] partial.  The maximum is taken over the values stored in
 * `out`, so it equals what q8_reduce_partials would find in them.  The all-reduce's
 * shared scale is the maximum of the ranks' block_amax.
 *
 *   M, N, K                  rows (batch x tokens), model width, channels of the slice;
 *                            N % 128 == 0, K % 8 == 0, M <= 65535 * 128, and
 *                            ceil(M/128) * ceil(N/128) * ceil(K/64) < 2^31
 *   y, ldy                   [M][K] bf16, row stride ldy >= K (a multiple of 8), 16-byte aligned
 *   W, ldw                   [N][K] bf16: the weight's columns for the slice, K contiguous
 *   out_dtype, out, ldo      [M][N] SSM_BF16 (round to nearest even) or SSM_F32, row
 *                            stride ldo >= N (a multiple of 8), 16-byte aligned
 *   block_amax               NULL or [M * N / 128] float32
 * Returns SSM_OK or a negative status.
 */
int ssm_out_proj_partial(int64_t M, int64_t N, int64_t K, const void* y, int64_t ldy,
                         const void* W, int64_t ldw, ssm_dtype_t out_dtype, void* out, int64_t ldo,
                         float* block_amax, void* cuda_stream);

/*
 * q8_reduce_partials -- the arithmetic of the pages' 8-bit quantized all-reduce
 * (Methodology 4), done locally over P partial buffers already in this GPU's
 * memory: quantize every partial to int8 with one scale per block of `block`
 * elements shared by all P partials (absolute maximum over the P partials / 127),
 * sum the int8 codes in int32, dequantize the sum with that scale.
 *
 * Per block j:  amax = max_{p,i in j} |x_p[i]|;  if amax == 0: codes and scale are 0;
 *   else inv = 127/amax and scale = amax/127 (IEEE fp32 division),
 *   q_p[i] = round_half_even(x_p[i] * inv) clamped to [-127, 127],
 *   S[i] = sum_p q_p[i] (int32),  out[i] = float(S[i]) * scale (fp32, then RNE to bf16
 *   when out_dtype is bf16).  The last block may be shorter than `block`.
 * Bit-exact: S and scale equal any IEEE-fp32 evaluation of the same steps, and
 * |out - sum_p x_p| <= P*scale/2 plus fp32 rounding.
 * Non-finite partials lie outside the method; they are handled as follows: a NaN
 * element is ignored by the block maximum and gets code 0; a block holding an
 * infinity gets scale +inf, codes 0 and NaN outputs.  Other blocks are unaffected.
 *
 *   P                            1..8
 *   partials                     HOST array of P device pointers, each to n elements of
 *                                in_dtype, 16-byte aligned
 *   n                            elements per partial (>= 1)
 *   block                        must be 128
 *   out                          [n] of out_dtype (device, 16-byte aligned)
 *   sums_out                     NULL or [n] int32       scales_out  NULL or [ceil(n/block)]
 */
int q8_reduce_partials(int P, const void* const* partials, ssm_dtype_t in_dtype, int64_t n,
                       int block, void* out, ssm_dtype_t out_dtype, int32_t* sums_out,
                       float* scales_out, void* cuda_stream);

/*
 * The rank-local halves of the 8-bit all-reduce (Methodology 4) for partials that live on
 * different GPUs.  q8_reduce_partials needs all P partials in one memory; a tensor-parallel
 * rank holds only its own.  The same arithmetic then runs as:
 *   1. q8_block_absmax on the rank's partial (ssm_out_proj_partial emits the same maxima);
 *   2. a MAX all-reduce of those maxima across the ranks (the caller's collective);
 *   3. q8_quantize_shared: the rank's int8 codes with the shared per-block scale;
 *   4. an all-gather of the ranks' codes (the caller's collective; 1 byte per element);
 *   5. q8_sum_dequant over the P code buffers.
 * Steps 5 o 3 with the maximum of step 1 over the ranks give q8_reduce_partials' sums,
 * scales and outputs bit for bit, because every step is the same correctly rounded fp32
 * operation.  Shapes as in q8_reduce_partials; block must be 128; every device pointer
 * 16-byte aligned; n >= 1.  Non-finite values: a NaN is ignored by the block maximum and
 * gets code 0; a block whose maximum is +inf gets codes 0, scale +inf and NaN outputs.
 */

/* block_amax[j] = max |x_i| over block j of 128 consecutive elements of x ([n] in_dtype);
 * block_amax holds ceil(n / 128) float32. */
int q8_block_absmax(const void* x, ssm_dtype_t in_dtype, int64_t n, int block, float* block_amax,
                    void* cuda_stream);

/* With the shared maxima amax[j] (the maximum of every rank's block_amax): codes[i] =
 * round_half_even(x_i * (127 / amax[j])) clamped to [-127, 127] (0 when amax[j] is 0);
 * scales_out (NULL or [ceil(n / 128)] float32) = amax[j] / 127 (IEEE fp32 division).
 * codes: [n] int8, written. */
int q8_quantize_shared(const void* x, ssm_dtype_t in_dtype, int64_t n, int block, const float* block_amax,
                       int8_t* codes, float* scales_out, void* cuda_stream);

/* S[i] = sum over the P code buffers of codes_p[i] (int32); out[i] = float(S[i]) * scales[j]
 * (fp32, then round to nearest even for bf16 out).  codes: HOST array of P (1..8) device
 * pointers to [n] int8; scales: [ceil(n / 128)] float32 from q8_quantize_shared (the same on
 * every rank); sums_out: NULL or [n] int32. */
int q8_sum_dequant(int P, const int8_t* const* codes, const float* scales, int64_t n, int block,
                   void* out, ssm_dtype_t out_dtype, int32_t* sums_out, void* cuda_stream);

/*
 * The SSD (Mamba-2-style) variant of the mixer.  The pages name the model families the
 * mixer serves (Overview: Mamba, Falcon-Mamba, Zamba) but print no equations for this
 * form; it follows the published Mamba-2 layer (Dao and Gu, "Transformers are SSMs",
 * 2024).  Per batch row b, head h of H, group g = h / (H / G), position p < 64 and
 * state n < 64:
 *   [x | B | C]_t = SiLU(conv_b + causal width-4 depthwise conv of the raw xBC channels)
 *   delta_t       = softplus(dt_t[h] + dt_bias[h])
 *   S_t[p][n]     = exp(delta_t A[h]) S_{t-1}[p][n] + delta_t x_t[h][p] B_t[g][n]
 *   out_t[h][p]   = (sum_n C_t[g][n] S_t[p][n] + D[h] x_t[h][p]) * SiLU(z_t[h][p])
 * The recurrence stays inside its head (Methodology 2) and the final states are the
 * cache that decode continues from (Methodology 3).
 *
 * Shapes (elements; channel stride 1):
 *   xBC      [batch][L][Cx], Cx = 64 H + 128 G: channel 64 h + p is x of head h,
 *            64 H + 64 g + n is B of group g, 64 H + 64 G + 64 g + n is C of group g
 *   z        [batch][L][64 H]          dt  [batch][L][H]
 *   conv_w   [Cx][4] (tap 3 multiplies the current token), conv_b [Cx]
 *   A, Dskip, dt_bias  [H]             (float32)
 *   conv_state [batch or slot][3][Cx]  the last three raw xBC inputs, oldest first (float32)
 *   ssm_state  [batch or slot][H][64][64]  (float32)
 * Supported: head_dim == 64, d_state == 64, d_conv == 4, H % G == 0.  Anything else
 * returns SSM_ERR_UNSUPPORTED.
 */

/* Bytes of device workspace ssd_prefill needs for these sizes (0 on a bad size): the B and C
 * channels after the conv as bf16 hi/lo operand planes, delta and the chunk-local decay sums,
 * and min(batch * n_heads, 256) fp32 [64][64] state slots with their ready flags, through
 * which a (row, head) pair cut between two CTAs of the chunk kernel passes its state. */
size_t ssd_prefill_workspace_bytes(int batch, int seqlen, int n_heads, int n_groups);

/*
 * ssd_prefill -- the SSD mixer over L tokens, on the tensor cores.  The recurrence is
 * computed chunk by chunk (128 tokens) in its matrix form: the products C B^T, M X, C S^T
 * and the state update run as tcgen05 MMAs on bf16 hi + lo operand pairs with fp32
 * accumulation, so every operand carries 16 significant bits.
 *
 *   batch, seqlen            1..65535 rows, 1..2^30 tokens
 *   n_heads, head_dim        1..65535 heads of 64
 *   n_groups, d_state        groups sharing B and C (n_heads % n_groups == 0), 64 states
 *   d_conv                   4
 *   in_dtype                 SSM_BF16 (xBC, z, dt); SSM_F32 returns SSM_ERR_UNSUPPORTED
 *   out_dtype                SSM_F32 or SSM_BF16
 *   xBC, xbc_stride_b/_t     view of [batch][L][Cx]: 16-byte aligned, strides multiples of 8,
 *                            xbc_stride_t >= Cx
 *   z, z_stride_b/_t         view of [batch][L][64 H]: same rules, z_stride_t >= 64 H
 *   dt, dt_stride_b/_t       view of [batch][L][H]: element aligned, dt_stride_t >= H
 *   conv_w (16-byte aligned), conv_b, A, Dskip, dt_bias
 *   conv_state_in, ssm_state_in   NULL (zeros) or [batch][3][Cx] / [batch][H][64][64],
 *                            contiguous; ssm_state_in 16-byte aligned
 *   out, out_stride_b/_t     view of [batch][L][64 H] in out_dtype: 16-byte aligned, strides
 *                            multiples of 16 bytes; rows may not overlap
 *   conv_state_out, ssm_state_out  [batch][3][Cx] / [batch][H][64][64] float32, contiguous;
 *                            ssm_state_out 16-byte aligned
 *   workspace, workspace_bytes     device memory of at least
 *                            ssd_prefill_workspace_bytes(batch, seqlen, n_heads, n_groups) bytes,
 *                            16-byte aligned, owned by the caller and not read afterwards
 * Asynchronous on cuda_stream (two kernels).  When batch * n_heads exceeds the CTAs the GPU
 * holds at once, the chunk kernel goes out as a cooperative launch of one CTA per resident
 * slot, each walking an equal share of all rows' chunks; a launch the device refuses returns
 * SSM_ERR_CUDA.  The result does not depend on how the rows were split.  Returns SSM_OK or a
 * negative status.
 */
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
                void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * ssd_decode_step -- one token per request of the SSD mixer, continuing from the cached
 * states of its slot and updating them in place (Methodology 3).
 *
 *   batch                    1..65535 requests
 *   n_heads .. d_conv        as for ssd_prefill
 *   in_dtype, out_dtype      SSM_F32 or SSM_BF16
 *   xBC, z, dt               [batch][Cx], [batch][64 H], [batch][H], contiguous, element aligned
 *   conv_w (16-byte aligned), conv_b, A, Dskip, dt_bias   as for ssd_prefill
 *   conv_state, ssm_state    [n_slots][3][Cx] / [n_slots][H][64][64] float32, in/out;
 *                            ssm_state 16-byte aligned
 *   n_slots, state_slot      request r uses slot state_slot[r] (NULL: slot r, then
 *                            n_slots >= batch); a slot outside [0, n_slots) is skipped and
 *                            sets SSM_DEV_BAD_SLOT; slots must be distinct
 *   out                      [batch][64 H] in out_dtype, contiguous
 * Asynchronous on cuda_stream (two kernels).  Returns SSM_OK or a negative status.
 */
int ssd_decode_step(int batch, int n_heads, int head_dim, int n_groups, int d_state, int d_conv,
                    ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                    const void* xBC, const void* z, const void* dt,
                    const float* conv_w, const float* conv_b,
                    const float* A, const float* Dskip, const float* dt_bias,
                    float* conv_state, float* ssm_state, int n_slots, const int32_t* state_slot,
                    void* out, void* cuda_stream);

/*
 * ssm_selftest_expire_wait -- a diagnostic with no counterpart in the pages: launches one
 * kernel that waits, through the library's bounded mbarrier wait, for a phase that nothing
 * completes.  After limit_us microseconds (1 .. 2e6) the wait gives up, the kernel sets
 * SSM_DEV_WAIT_TIMEOUT in the device status word and returns normally.  It shows on a given
 * GPU that an expired in-kernel wait is reported through ssm_device_status and that the
 * context stays usable, without faulting or hanging the GPU.
 */
int ssm_selftest_expire_wait(int limit_us, void* cuda_stream);

/*
 * ssm_device_status -- read (and if `clear` is nonzero, reset) the device status
 * word of the current device: an OR of SSM_DEV_* bits set by kernels that hit a
 * bounded-wait timeout or a bad state slot since the last clear.  Synchronises
 * the device.  Returns SSM_OK, or SSM_ERR_CUDA.
 */
int ssm_device_status(uint32_t* status, int clear);

/* Thread-local text for the last non-OK return on this thread ("" if none). */
const char* ssm_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_H_ */
