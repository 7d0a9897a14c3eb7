/*
 * ssm_oracle.c -- plain, slow, sequential fp64 CPU oracle for the selective
 * state-space (SSM) mixer: prefill, one decode step, and the 8-bit quantized
 * reduction of partial outputs.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test-suite, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or constant with the
 * CUDA path.
 *
 * Source of the method: "Scaling State-Space Models on Multiple GPUs with
 * Tensor Parallelism" (euno.news summary of arXiv 2602.21144):
 *   - Overview / Methodology 2 ("local recurrence"): every channel keeps its own
 *     slice of the hidden state and updates it token by token; nothing crosses
 *     channels, so each channel below is computed on its own.
 *   - Methodology 3 ("state caching during prefill and decode"): prefill returns
 *     the hidden state and decode continues from it without recomputing tokens.
 *   - Methodology 4 ("quantized All-Reduce"): partial outputs are quantized to
 *     8 bits before they are summed and dequantized afterwards.
 * The last function, oracle_ssd_prefill, is the Mamba-2-style (SSD) variant of the
 * same mixer; its own header states its source and readings.
 * The pages do not print the mixer's equations.  This file uses the
 * Mamba-style selective-scan mixer (width-4 causal depthwise conv + SiLU,
 * softplus step, diagonal recurrence, C readout, D skip, SiLU(z) gate), with
 * these readings where the description leaves a step open:
 *   - "x" in the Delta*B*x term and in the D*x skip is the post-conv, post-SiLU
 *     activation u;
 *   - the conv is a cross-correlation: conv_w[d][W-1] multiplies the current
 *     token, conv_w[d][0] the token W-1 steps back; tokens before the start come
 *     from conv_state_in (oldest first) or are zero;
 *   - conv_state holds the last W-1 RAW (pre-conv) inputs, oldest first;
 *   - B and C are per-token inputs [batch][L][N] shared by all channels;
 *   - states start at zero unless an input state is given;
 *   - softplus(v) = log(1 + e^v), evaluated as v + log1p(e^-v) for v > 0 and
 *     log1p(e^v) otherwise (both exact forms, no threshold).
 *
 * Every floating-point step below is the definition written out in double
 * precision, in the pages' order, with no blocking, fusion or reordering.
 *
 * Build: cc -O2 -ffp-contract=off -fopenmp -shared -fPIC (OpenMP is optional;
 * it only spreads independent channels over threads).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Widen element i of a float32 or bfloat16 array to double.  A bfloat16 is the
 * upper 16 bits of an IEEE binary32, so the widening is exact. */
static double widen(const void* p, int dtype, int64_t i)
{
    float f;
    if (dtype == ORACLE_F32) {
        f = ((const float*)p)[i];
    } else {
        uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
        memcpy(&f, &bits, sizeof f);
    }
    return (double)f;
}

static double silu(double v) { return v / (1.0 + exp(-v)); }

static double softplus(double v) { return v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v)); }

/*
 * One token of one channel: the body shared by prefill and decode.
 *   hist[0..W-2]  raw inputs of the W-1 previous tokens, oldest first (in/out)
 *   h[0..N-1]     hidden state of this channel (in/out)
 * Returns out_t.
 */
static double mixer_token(int N, int W, double xt, double zt, double dtt,
                          const double* Bt, const double* Ct,
                          const float* A_d, double D_d, double dt_bias_d,
                          const float* conv_w_d, double conv_b_d,
                          double* hist, double* h)
{
    /* causal depthwise conv over [hist..., x_t], then SiLU */
    double xc = conv_b_d;
    for (int k = 0; k < W - 1; ++k) xc += (double)conv_w_d[k] * hist[k];
    xc += (double)conv_w_d[W - 1] * xt;
    double u = silu(xc);

    /* step size */
    double delta = softplus(dtt + dt_bias_d);

    /* diagonal recurrence and readout */
    double y = 0.0;
    for (int n = 0; n < N; ++n) {
        double a = exp(delta * (double)A_d[n]);
        h[n] = a * h[n] + delta * Bt[n] * u;
        y += Ct[n] * h[n];
    }
    y += D_d * u;

    /* shift the conv window: drop the oldest, append the raw x_t */
    for (int k = 0; k + 1 < W - 1; ++k) hist[k] = hist[k + 1];
    if (W > 1) hist[W - 2] = xt;

    return y * silu(zt);
}

/*
 * Prefill over L tokens.  All arrays are contiguous and row-major:
 *   x, z, dt        [batch][L][Dn]   in_dtype
 *   Bm, Cm          [batch][L][N]    in_dtype
 *   A [Dn][N], Dskip [Dn], dt_bias [Dn], conv_w [Dn][W], conv_b [Dn]   float32
 *   conv_state_in   [batch][W-1][Dn] float64 or NULL (zeros)
 *   ssm_state_in    [batch][Dn][N]   float64 or NULL (zeros)
 * Outputs (float64): out [batch][L][Dn], conv_state_out [batch][W-1][Dn],
 * ssm_state_out [batch][Dn][N].
 * Returns 0, or -1 on a bad size.
 */
int oracle_prefill(int batch, int L, int Dn, int N, int W, int in_dtype,
                   const void* x, const void* z, const void* dt,
                   const void* Bm, const void* Cm,
                   const float* A, const float* Dskip, const float* dt_bias,
                   const float* conv_w, const float* conv_b,
                   const double* conv_state_in, const double* ssm_state_in,
                   double* out, double* conv_state_out, double* ssm_state_out,
                   int n_threads)
{
    if (batch < 0 || L < 0 || Dn < 0 || N < 1 || N > 256 || W < 1 || W > 64) return -1;
    if (n_threads < 1) n_threads = 1;
    int64_t jobs = (int64_t)batch * Dn;

#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
    for (int64_t job = 0; job < jobs; ++job) {
        int b = (int)(job / Dn), d = (int)(job % Dn);
        double hist[64], h[256], Bt[256], Ct[256];
        for (int k = 0; k < W - 1; ++k)
            hist[k] = conv_state_in ? conv_state_in[((int64_t)b * (W - 1) + k) * Dn + d] : 0.0;
        for (int n = 0; n < N; ++n)
            h[n] = ssm_state_in ? ssm_state_in[((int64_t)b * Dn + d) * N + n] : 0.0;

        for (int t = 0; t < L; ++t) {
            int64_t it = ((int64_t)b * L + t) * Dn + d;
            int64_t ib = ((int64_t)b * L + t) * N;
            for (int n = 0; n < N; ++n) {
                Bt[n] = widen(Bm, in_dtype, ib + n);
                Ct[n] = widen(Cm, in_dtype, ib + n);
            }
            out[it] = mixer_token(N, W, widen(x, in_dtype, it), widen(z, in_dtype, it),
                                  widen(dt, in_dtype, it), Bt, Ct, A + (int64_t)d * N,
                                  Dskip[d], dt_bias[d], conv_w + (int64_t)d * W, conv_b[d],
                                  hist, h);
        }
        for (int k = 0; k < W - 1; ++k) conv_state_out[((int64_t)b * (W - 1) + k) * Dn + d] = hist[k];
        for (int n = 0; n < N; ++n) ssm_state_out[((int64_t)b * Dn + d) * N + n] = h[n];
    }
    return 0;
}

/*
 * One decode step: the same token body, continuing from cached states which
 * are read and then overwritten in place.
 *   x, z, dt [batch][Dn], Bm, Cm [batch][N]   in_dtype
 *   conv_state [batch][W-1][Dn], ssm_state [batch][Dn][N]   float64, in/out
 *   out [batch][Dn] float64
 */
int oracle_decode_step(int batch, int Dn, int N, int W, int in_dtype,
                       const void* x, const void* z, const void* dt,
                       const void* Bm, const void* Cm,
                       const float* A, const float* Dskip, const float* dt_bias,
                       const float* conv_w, const float* conv_b,
                       double* conv_state, double* ssm_state, double* out)
{
    if (batch < 0 || Dn < 0 || N < 1 || N > 256 || W < 1 || W > 64) return -1;
    for (int b = 0; b < batch; ++b) {
        double Bt[256], Ct[256];
        for (int n = 0; n < N; ++n) {
            Bt[n] = widen(Bm, in_dtype, (int64_t)b * N + n);
            Ct[n] = widen(Cm, in_dtype, (int64_t)b * N + n);
        }
        for (int d = 0; d < Dn; ++d) {
            double hist[64];
            for (int k = 0; k < W - 1; ++k) hist[k] = conv_state[((int64_t)b * (W - 1) + k) * Dn + d];
            double* h = ssm_state + ((int64_t)b * Dn + d) * N;
            int64_t it = (int64_t)b * Dn + d;
            out[it] = mixer_token(N, W, widen(x, in_dtype, it), widen(z, in_dtype, it),
                                  widen(dt, in_dtype, it), Bt, Ct, A + (int64_t)d * N,
                                  Dskip[d], dt_bias[d], conv_w + (int64_t)d * W, conv_b[d],
                                  hist, h);
            for (int k = 0; k < W - 1; ++k) conv_state[((int64_t)b * (W - 1) + k) * Dn + d] = hist[k];
        }
    }
    return 0;
}

/*
 * The recurrence h_t = a_t * h_{t-1} + b_t written two ways, for the check that
 * the chunked associative scan equals the sequential one.
 *
 * Sequential: h[t] for t = 0..L-1 from h0.
 */
void oracle_scan_sequential(int64_t L, const double* a, const double* b, double h0, double* h)
{
    double s = h0;
    for (int64_t t = 0; t < L; ++t) {
        s = a[t] * s + b[t];
        h[t] = s;
    }
}

/*
 * Chunked: pairs (a, b) compose associatively as
 *   (a1, b1) then (a2, b2) = (a1*a2, a2*b1 + b2).
 * Pass 1 reduces every chunk of `chunk` tokens to one pair (its aggregate).
 * Pass 2 carries the state across chunks: carry_{c+1} = A_c * carry_c + B_c.
 * Pass 3 replays each chunk from its carried-in state.
 */
void oracle_scan_chunked(int64_t L, const double* a, const double* b, double h0, int64_t chunk,
                         double* h)
{
    if (chunk < 1) chunk = 1;
    int64_t nchunks = (L + chunk - 1) / chunk;
    double carry = h0;
    for (int64_t c = 0; c < nchunks; ++c) {
        int64_t t0 = c * chunk, t1 = t0 + chunk < L ? t0 + chunk : L;
        double Aagg = 1.0, Bagg = 0.0;
        for (int64_t t = t0; t < t1; ++t) {
            Bagg = a[t] * Bagg + b[t];
            Aagg = Aagg * a[t];
        }
        double s = carry;
        for (int64_t t = t0; t < t1; ++t) {
            s = a[t] * s + b[t];
            h[t] = s;
        }
        carry = Aagg * carry + Bagg;
    }
}

/* float32 -> bfloat16 bits, round to nearest, ties to even (finite inputs). */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

static float widen_f32(const void* p, int dtype, int64_t i) { return (float)widen(p, dtype, i); }

/*
 * 8-bit quantized reduction of P partial buffers (Methodology 4 of the pages:
 * quantize to 8 bits, sum, dequantize).  Defined in IEEE binary32 so that the
 * integer sums are reproducible bit for bit.  Readings (the pages give no
 * codec): one scale per block of `block` elements, shared by all P partials,
 * from the block's absolute maximum over every partial; symmetric int8 range
 * [-127, 127]; round to nearest, ties to even; an all-zero block has scale 0.
 * The last block may be shorter than `block`.
 *
 *   partials  host array of P pointers, each to n elements of in_dtype
 *   sums      [n] int32 (may be NULL)      scales [ceil(n/block)] (may be NULL)
 *   out_f32   [n] (may be NULL)            out_bf16 [n] bf16 bits (may be NULL)
 */
int oracle_q8_reduce(int P, const void* const* partials, int in_dtype, int64_t n, int block,
                     int32_t* sums, float* scales, float* out_f32, uint16_t* out_bf16)
{
    if (P < 1 || n < 0 || block < 1) return -1;
    for (int64_t j0 = 0; j0 < n; j0 += block) {
        int64_t j1 = j0 + block < n ? j0 + block : n;
        float amax = 0.0f;
        for (int p = 0; p < P; ++p)
            for (int64_t i = j0; i < j1; ++i) {
                float v = fabsf(widen_f32(partials[p], in_dtype, i));
                if (v > amax) amax = v;
            }
        float inv = 0.0f, scale = 0.0f;
        if (amax > 0.0f) {
            inv = 127.0f / amax;
            scale = amax / 127.0f;
        }
        if (scales) scales[j0 / block] = scale;
        for (int64_t i = j0; i < j1; ++i) {
            int32_t s = 0;
            for (int p = 0; p < P; ++p) {
                int32_t q = 0;
                if (amax > 0.0f) {
                    float t = widen_f32(partials[p], in_dtype, i) * inv;
                    float r = rintf(t);
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    q = (int32_t)r;
                }
                s += q;
            }
            float o = (float)s * scale;
            if (sums) sums[i] = s;
            if (out_f32) out_f32[i] = o;
            if (out_bf16) out_bf16[i] = f32_to_bf16_rne(o);
        }
    }
    return 0;
}

/*
 * The rank-local halves of the quantized all-reduce (Methodology 4) when every rank holds
 * only its own partial, in fp32 like oracle_q8_reduce (the last block may be shorter):
 *   oracle_q8_block_absmax:    amax[j] = max_{i in block j} |x_i|   (a NaN is ignored)
 *   oracle_q8_quantize_shared: given the maxima shared by all ranks (the maximum over the
 *       ranks of their amax), inv = 127/amax_j and scale_j = amax_j/127 (both 0 when
 *       amax_j is 0 or not a number), q_i = clamp(rint(x_i * inv), -127, 127), a NaN
 *       product giving 0
 *   oracle_q8_sum_dequant:     S_i = sum_p q_p,i (int32), out_i = (float)S_i * scale_j
 * Combining the ranks' maxima by max and composing the three gives the steps of
 * oracle_q8_reduce.
 */
int oracle_q8_block_absmax(const void* x, int in_dtype, int64_t n, int block, float* amax)
{
    if (n < 0 || block < 1) return -1;
    for (int64_t j0 = 0; j0 < n; j0 += block) {
        const int64_t j1 = j0 + block < n ? j0 + block : n;
        float m = 0.0f;
        for (int64_t i = j0; i < j1; ++i) {
            const float v = fabsf(widen_f32(x, in_dtype, i));
            if (v > m) m = v;
        }
        amax[j0 / block] = m;
    }
    return 0;
}

int oracle_q8_quantize_shared(const void* x, int in_dtype, int64_t n, int block, const float* amax,
                              int8_t* codes, float* scales)
{
    if (n < 0 || block < 1) return -1;
    for (int64_t j0 = 0; j0 < n; j0 += block) {
        const int64_t j1 = j0 + block < n ? j0 + block : n;
        const float a = amax[j0 / block];
        float inv = 0.0f, scale = 0.0f;
        if (a > 0.0f) {
            inv = 127.0f / a;
            scale = a / 127.0f;
        }
        if (scales) scales[j0 / block] = scale;
        for (int64_t i = j0; i < j1; ++i) {
            float r = rintf(widen_f32(x, in_dtype, i) * inv);
            if (r != r) r = 0.0f;
            r = r > 127.0f ? 127.0f : (r < -127.0f ? -127.0f : r);
            codes[i] = (int8_t)r;
        }
    }
    return 0;
}

int oracle_q8_sum_dequant(int P, const int8_t* const* codes, const float* scales, int64_t n, int block,
                          int32_t* sums, float* out_f32, uint16_t* out_bf16)
{
    if (P < 1 || n < 0 || block < 1) return -1;
    for (int64_t i = 0; i < n; ++i) {
        int32_t s = 0;
        for (int p = 0; p < P; ++p) s += codes[p][i];
        const float o = (float)s * scales[i / block];
        if (sums) sums[i] = s;
        if (out_f32) out_f32[i] = o;
        if (out_bf16) out_bf16[i] = f32_to_bf16_rne(o);
    }
    return 0;
}

/*
 * oracle_out_proj -- one tensor-parallel rank's partial of the mixer's output
 * projection, the operand of the quantized all-reduce ("Scaling State-Space
 * Models on Multiple GPUs with Tensor Parallelism", Methodology 1: the layer is
 * split along the feature dimension; Methodology 4: the ranks' partial outputs
 * are quantized, summed and dequantized).  The rank holds the mixer output of
 * its channel slice, y [M][K] (M = batch * tokens, K = channels of the slice),
 * and the matching columns of the projection weight, W [N][K] (N = model width).
 * Its partial is
 *   out[m][n] = sum_k y[m][k] * W[n][k]                          (double, k in order)
 * and, for the shared-scale codec, the absolute maximum of every block of 128
 * consecutive elements of the row-major [M][N] partial (the last block may be
 * shorter):
 *   amax[j] = max_{i in block j} |out_i|.
 * absdot[m][n] = sum_k |y[m][k]| * |W[n][k]| (nullable) bounds the rounding of
 * any fp32 evaluation of the same sum.
 *   y, W      in_dtype elements, row-major, contiguous
 *   out       [M][N] double;  amax  [ceil(M*N/128)] double (nullable)
 */
int oracle_out_proj(int64_t M, int64_t N, int64_t K, int in_dtype, const void* y, const void* W,
                    double* out, double* amax, double* absdot, int n_threads)
{
    if (M < 1 || N < 1 || K < 1) return -1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double yv = widen(y, in_dtype, m * K + k);
                const double wv = widen(W, in_dtype, n * K + k);
                s += yv * wv;
                a += fabs(yv) * fabs(wv);
            }
            out[m * N + n] = s;
            if (absdot) absdot[m * N + n] = a;
        }
    }
    if (amax) {
        const int64_t total = M * N;
        for (int64_t j0 = 0; j0 < total; j0 += 128) {
            const int64_t j1 = j0 + 128 < total ? j0 + 128 : total;
            double mx = 0.0;
            for (int64_t i = j0; i < j1; ++i)
                if (fabs(out[i]) > mx) mx = fabs(out[i]);
            amax[j0 / 128] = mx;
        }
    }
    return 0;
}

/*
 * oracle_ssd_prefill -- the structured-state-space-duality (SSD, Mamba-2-style)
 * variant of the mixer: the same local recurrence, with the decay a scalar per
 * head and B, C shared by the heads of a group.  The pages name the model
 * families this serves (Overview: Mamba, Falcon-Mamba and Zamba) but print no
 * equations for this form; it follows the published Mamba-2 layer (Dao and Gu,
 * "Transformers are SSMs", 2024), with these readings:
 *   - one width-W causal depthwise conv + SiLU runs over the concatenated input
 *     channels [x | B | C] (Cx = H*P + 2*G*N per token): channel h*P + p is x of
 *     head h, position p; H*P + g*N + n is B of group g; H*P + G*N + g*N + n is C;
 *   - head h belongs to group g(h) = h / (H / G) (contiguous blocks of heads);
 *   - Delta = softplus(dt + dt_bias[h]) per token and head; the decay is
 *     exp(Delta * A[h]);
 *   - state S[h][p][n] <- exp(Delta A[h]) S[h][p][n] + Delta x[h][p] B[g(h)][n];
 *   - y[h][p] = sum_n C[g(h)][n] S[h][p][n] + D[h] x[h][p], out = y * SiLU(z);
 *   - the gated normalisation that follows in Mamba-2 is a separate layer op and
 *     is not part of this mixer, like the output projection.
 * Every step is the definition written out in double precision, token by token.
 *   xBC [batch][L][Cx], z [batch][L][H*P], dt [batch][L][H]   in_dtype
 *   conv_w [Cx][W], conv_b [Cx], A [H], Dskip [H], dt_bias [H]  float32
 *   conv_state_in  [batch][W-1][Cx]  float64 or NULL (zeros), raw inputs, oldest first
 *   ssm_state_in   [batch][H][P][N]  float64 or NULL (zeros)
 *   heads          n_run head indices to evaluate, or NULL for all H heads; only their
 *                  rows of out / ssm_state_out and their x channels of
 *                  conv_state_out are written (B and C channels always are)
 * Outputs (float64): out [batch][L][H*P], conv_state_out [batch][W-1][Cx],
 * ssm_state_out [batch][H][P][N].  Returns 0, or -1 on a bad size.
 */
int oracle_ssd_prefill(int batch, int L, int H, int P, int G, int N, int W, int in_dtype,
                       const void* xBC, const void* z, const void* dt,
                       const float* conv_w, const float* conv_b,
                       const float* A, const float* Dskip, const float* dt_bias,
                       const double* conv_state_in, const double* ssm_state_in,
                       const int* heads, int n_run,
                       double* out, double* conv_state_out, double* ssm_state_out, int n_threads)
{
    if (batch < 0 || L < 0 || H < 1 || P < 1 || G < 1 || N < 1 || W < 1 || W > 64) return -1;
    if (H % G != 0) return -1;
    if (!heads) n_run = H;
    if (n_threads < 1) n_threads = 1;
    const int64_t Cx = (int64_t)H * P + 2 * (int64_t)G * N;
    const int hpg = H / G;
    const int64_t jobs = (int64_t)batch * n_run;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
    for (int64_t job = 0; job < jobs; ++job) {
        const int b = (int)(job / n_run);
        const int h = heads ? heads[job % n_run] : (int)(job % n_run);
        if (h < 0 || h >= H) {
            bad = 1;
            continue;
        }
        const int g = h / hpg;
        /* the channels this head reads: its P x channels, then its group's N B and N C channels */
        const int nch = P + 2 * N;
        int64_t* ch = (int64_t*)malloc(sizeof(int64_t) * nch);
        double* hist = (double*)malloc(sizeof(double) * nch * (W > 1 ? W - 1 : 1));
        double* u = (double*)malloc(sizeof(double) * nch);
        double* S = (double*)malloc(sizeof(double) * (size_t)P * N);
        if (!ch || !hist || !u || !S) {
            free(ch); free(hist); free(u); free(S);
            bad = 1;
            continue;
        }
        for (int p = 0; p < P; ++p) ch[p] = (int64_t)h * P + p;
        for (int n = 0; n < N; ++n) {
            ch[P + n] = (int64_t)H * P + (int64_t)g * N + n;
            ch[P + N + n] = (int64_t)H * P + (int64_t)G * N + (int64_t)g * N + n;
        }
        for (int c = 0; c < nch; ++c)
            for (int k = 0; k < W - 1; ++k)
                hist[c * (W - 1) + k] = conv_state_in ? conv_state_in[((int64_t)b * (W - 1) + k) * Cx + ch[c]] : 0.0;
        for (int64_t e = 0; e < (int64_t)P * N; ++e)
            S[e] = ssm_state_in ? ssm_state_in[((int64_t)b * H + h) * P * N + e] : 0.0;

        for (int t = 0; t < L; ++t) {
            const int64_t row = (int64_t)b * L + t;
            /* causal depthwise conv over [hist..., xBC_t] and SiLU, channel by channel */
            for (int c = 0; c < nch; ++c) {
                const double xt = widen(xBC, in_dtype, row * Cx + ch[c]);
                double xc = (double)conv_b[ch[c]];
                for (int k = 0; k < W - 1; ++k) xc += (double)conv_w[ch[c] * W + k] * hist[c * (W - 1) + k];
                xc += (double)conv_w[ch[c] * W + W - 1] * xt;
                u[c] = silu(xc);
                for (int k = 0; k + 1 < W - 1; ++k) hist[c * (W - 1) + k] = hist[c * (W - 1) + k + 1];
                if (W > 1) hist[c * (W - 1) + W - 2] = xt;
            }
            const double* xh = u;          /* x[h][0..P-1] */
            const double* Bg = u + P;      /* B[g][0..N-1] */
            const double* Cg = u + P + N;  /* C[g][0..N-1] */
            const double delta = softplus(widen(dt, in_dtype, row * H + h) + (double)dt_bias[h]);
            const double a = exp(delta * (double)A[h]);
            for (int p = 0; p < P; ++p) {
                double y = 0.0;
                for (int n = 0; n < N; ++n) {
                    S[(int64_t)p * N + n] = a * S[(int64_t)p * N + n] + delta * xh[p] * Bg[n];
                    y += Cg[n] * S[(int64_t)p * N + n];
                }
                y += (double)Dskip[h] * xh[p];
                const double zt = widen(z, in_dtype, row * H * P + (int64_t)h * P + p);
                out[row * H * P + (int64_t)h * P + p] = y * silu(zt);
            }
        }
        /* x channels belong to this head; B and C channels are written by the first evaluated
         * head of the group (every head of a group computes the same B and C history) */
        int first_of_group = heads ? 1 : (h % hpg == 0);
        if (heads)
            for (int64_t q = 0; q < job % n_run; ++q)
                if (heads[q] >= 0 && heads[q] < H && heads[q] / hpg == g) first_of_group = 0;
        for (int c = 0; c < nch; ++c) {
            if (c >= P && !first_of_group) continue;
            for (int k = 0; k < W - 1; ++k)
                conv_state_out[((int64_t)b * (W - 1) + k) * Cx + ch[c]] = hist[c * (W - 1) + k];
        }
        for (int64_t e = 0; e < (int64_t)P * N; ++e)
            ssm_state_out[((int64_t)b * H + h) * P * N + e] = S[e];
        free(ch); free(hist); free(u); free(S);
    }
    return bad ? -1 : 0;
}
