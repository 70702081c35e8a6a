/*
 * qerl_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU restatement of what the NVFP4 weight-only LoRA linear path
 * computes, used to check the CUDA library.  Single-threaded unless
 * orc_set_threads asks for more: the linear forward then hands whole output
 * features to threads (OpenMP), each element computed exactly as alone.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code, header, table or constant generator with the CUDA library.
 *
 * Sources (web pages about QeRL; cited by page title and section):
 *  [NVFP4]  "QeRL: NVFP4-Quantized Reinforcement Learning -- Redefining Efficiency
 *           in AI Training and Inference", section "NVFP4: NVIDIA's FP4 Format":
 *           blocks of 16 values along a row, one FP8 E4M3 scale per block, one
 *           FP32 tensor-wise scale; the cuDNN block-scaling recipe: block scale
 *           = quantize_round_up(amax(vals)/vmax), value = round_to_even(v/scale).
 *  [LoRA]   same page, LoRA paragraph: frozen W plus a trainable low-rank update
 *           kept in higher precision (e.g. FP16 or FP32).
 *  [MX]     same page, "NVFP4" section: NVFP4 against MXFP4, whose blocks are 32
 *           values with a power-of-two (E8M0) scale.  The block-scale rule is
 *           the OCP Microscaling (MX) v1.0 one: shared exponent =
 *           floor(log2(amax)) - emax of the element type (2 for E2M1).
 *  [Impl]   same page, "Implementation and Practical Details": weight-only
 *           quantization; activations and gradients stay in high precision.
 *  [AQN-S]  "QeRL: Beyond Efficiency -- Quantization-enhanced Reinforcement
 *           Learning for LLMs" (summary): AQN injects channel-wise Gaussian noise
 *           via the normalization layer with an exponential decay schedule.
 *  [AQN-M]  "QERL: NVFP4-intensive learning (RL) brings 32B LLM training to H100",
 *           AQN paragraph: the Gaussian noise lives in the norm's scale
 *           parameters, driven by an exponential schedule.
 *  [Hints]  "QeRL" README mirror, "Hints for QeRL training" item 3: noise knobs
 *           sigma_start, sigma_end, num_stages.
 *
 * Readings where the pages are silent (each applied identically by the CUDA
 * library, which is written separately):
 *  - tensor scale s_t = amax(|W|) / (6 * 448) in FP32 (1.0 for an all-zero W);
 *  - block scale = smallest finite E4M3 value >= amax_b / (6 * s_t) ("round up"),
 *    saturating at 448; an optional round-to-nearest-even mode clips at 448;
 *  - element code = E2M1 nearest value of w / (scale * s_t), ties to the even
 *    code, saturating at 6; a value that rounds to zero gets code 0 (no -0);
 *  - packing: byte j of a row holds element 2j in bits 0-3, element 2j+1 in
 *    bits 4-7; scales are a row-major [N, K/16] byte array;
 *  - AQN: y = x / sqrt(mean(x^2) + eps) * (gamma + sigma * z), z[c] ~ N(0,1) per
 *    channel, drawn from Philox4x64-10 (Salmon et al., SC'11) with key
 *    (seed, layer) and counter (c / 4, step, 0, 0), Box-Muller per word pair;
 *  - sigma schedule: stage k = min(floor(step * S / total), S - 1),
 *    sigma_k = sigma_start * (sigma_end / sigma_start)^(k / (S - 1)).
 *
 * Build flags must keep IEEE single-precision semantics: -ffp-contract=off,
 * no -ffast-math.  The quantizer's decisions are taken in FP32, as the format's
 * scales are FP32/FP8 numbers; everything else is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_SHAPE 2
#define ORC_ERR_NONFINITE 4

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 bit pattern -> float (exact: bf16 is the top half of an IEEE single). */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

double orc_bf16_value(uint16_t h) { return (double)bf16_bits_to_float(h); }

/* FP8 E4M3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, S.1111.111 is NaN, exponent field 0 is subnormal m*2^-9. */
double orc_e4m3_value(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* FP4 E2M1: 1 sign bit (bit 3), 2 exponent bits with bias 1, 1 mantissa bit;
 * exponent field 0 is subnormal m*0.5.  Magnitudes 0,.5,1,1.5,2,3,4,6. */
double orc_e2m1_value(uint8_t c)
{
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 3;
    int m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + m / 2.0, e - 1);
    return sign ? -v : v;
}

/* Block scale, "quantize_round_up" [NVFP4]: the smallest finite non-negative
 * E4M3 value that is >= t, found by scanning the 127 non-negative finite codes
 * in increasing order.  t <= 0 gives code 0; t above 448 saturates to 448. */
uint8_t orc_e4m3_round_up(float t)
{
    int b;
    if (!(t > 0.0f))
        return 0;
    for (b = 0; b <= 126; ++b)
        if (orc_e4m3_value((uint8_t)b) >= (double)t)
            return (uint8_t)b;
    return 126;
}

/* Optional block-scale mode: nearest E4M3 value, ties to the even code
 * (mantissa LSB = code LSB), clipped at 448. */
uint8_t orc_e4m3_round_rne(float t)
{
    int b, best = 0;
    double bestd;
    if (!(t > 0.0f))
        return 0;
    if (t >= 448.0f)
        return 126;
    bestd = (double)t;
    for (b = 1; b <= 126; ++b) {
        double d = fabs(orc_e4m3_value((uint8_t)b) - (double)t);
        if (d < bestd || (d == bestd && (b & 1) == 0)) {
            best = b;
            bestd = d;
        }
    }
    return (uint8_t)best;
}

/* Element code, "round_to_even(vals/scale)" [NVFP4]: nearest E2M1 magnitude to
 * |q| by scanning the 8 magnitudes, ties to the even code; |q| >= 6 saturates
 * to 6, the nearest magnitude (tested before the scan, whose fp64 distances
 * would tie for |q| beyond 2^53).  Zero is always code 0. */
uint8_t orc_e2m1_round(float q)
{
    double a = fabs((double)q);
    int c, best = 0;
    double bestd = a; /* distance to magnitude 0 */
    if (a >= 6.0) /* 6 is the largest magnitude, so the nearest one from above */
        return (uint8_t)((q < 0.0f ? 8 : 0) | 7);
    for (c = 1; c < 8; ++c) {
        double d = fabs(orc_e2m1_value((uint8_t)c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    if (best == 0)
        return 0;
    return (uint8_t)((q < 0.0f ? 8 : 0) | best);
}

/* ------------------------------------------------------------------ */
/* NVFP4 quantize / dequantize                                         */
/* ------------------------------------------------------------------ */

/* Two-level NVFP4 quantization of a bf16 [N, K] row-major matrix (row stride
 * ldw elements) [NVFP4].  Outputs codes [N, K/2] (two per byte, even element in
 * the low nibble), block-scale bytes [N, K/16] and the FP32 tensor scale.
 * scale_mode 0 = round up (the recipe's), 1 = round to nearest even.
 * Returns ORC_ERR_SHAPE if K is not a multiple of 16 and ORC_ERR_NONFINITE if
 * W holds an Inf or NaN (nothing is written then). */
int orc_nvfp4_quantize(const uint16_t *W, int64_t N, int64_t K, int64_t ldw,
                       uint8_t *codes, uint8_t *scales, float *tensor_scale,
                       int scale_mode)
{
    int64_t n, k, b;
    float amax = 0.0f, s_t;
    if (K % 16 != 0 || N < 0 || ldw < K)
        return ORC_ERR_SHAPE;

    /* Step 1: tensor amax and the FP32 tensor-wise scale. */
    for (n = 0; n < N; ++n)
        for (k = 0; k < K; ++k) {
            float w = bf16_bits_to_float(W[n * ldw + k]);
            if (!isfinite(w))
                return ORC_ERR_NONFINITE;
            if (fabsf(w) > amax)
                amax = fabsf(w);
        }
    s_t = (amax > 0.0f) ? amax / 2688.0f : 1.0f; /* 2688 = 6 * 448 */
    *tensor_scale = s_t;

    memset(codes, 0, (size_t)(N * (K / 2)));
    for (n = 0; n < N; ++n) {
        for (b = 0; b < K / 16; ++b) {
            const uint16_t *blk = W + n * ldw + b * 16;
            float amax_b = 0.0f, d, t, sc, denom;
            uint8_t sb;
            int i;
            /* Step 2: block amax -> E4M3 block scale. */
            for (i = 0; i < 16; ++i) {
                float a = fabsf(bf16_bits_to_float(blk[i]));
                if (a > amax_b)
                    amax_b = a;
            }
            d = 6.0f * s_t;
            t = amax_b / d;
            sb = (scale_mode == 1) ? orc_e4m3_round_rne(t) : orc_e4m3_round_up(t);
            scales[n * (K / 16) + b] = sb;

            /* Step 3: element codes, divided by (block scale * tensor scale). */
            sc = (float)orc_e4m3_value(sb);
            denom = sc * s_t;
            for (i = 0; i < 16; ++i) {
                uint8_t c = 0;
                int64_t kk = b * 16 + i;
                if (sb != 0)
                    c = orc_e2m1_round(bf16_bits_to_float(blk[i]) / denom);
                /* Step 4: pack two codes per byte, even element low. */
                if (kk % 2 == 0)
                    codes[n * (K / 2) + kk / 2] |= c;
                else
                    codes[n * (K / 2) + kk / 2] |= (uint8_t)(c << 4);
            }
        }
    }
    return ORC_OK;
}

/* The code of element (n, k) in a packed [N, K/2] array. */
static uint8_t code_at(const uint8_t *codes, int64_t K, int64_t n, int64_t k)
{
    uint8_t byte = codes[n * (K / 2) + k / 2];
    return (k % 2 == 0) ? (uint8_t)(byte & 15) : (uint8_t)(byte >> 4);
}

/* w_hat(n, k) = e2m1(code) * e4m3(block scale) * s_t, in fp64 (exact). */
static double w_hat(const uint8_t *codes, const uint8_t *scales, double s_t,
                    int64_t K, int64_t n, int64_t k)
{
    return orc_e2m1_value(code_at(codes, K, n, k)) *
           orc_e4m3_value(scales[n * (K / 16) + k / 16]) * s_t;
}

/* Dequantize rows [0, N) into out [N, K] (fp64). */
/* E8M0 scale byte [MX]: 2^(b - 127); 0xFF is NaN (never emitted). */
double orc_e8m0_value(uint8_t b) { return b == 0xFF ? NAN : ldexp(1.0, (int)b - 127); }

/* MXFP4 quantizer [MX]: per block of 32 consecutive k, e = floor(log2(amax_b))
 * - 2 clamped to [-127, 127] (all-zero block: e = -127), scale byte e + 127,
 * element code = E2M1 nearest value of w * 2^-e (ties to the even code,
 * saturating at 6, zero as code 0).  Codes pack as for NVFP4; scales are a
 * row-major [N, K/32] byte array.  No tensor scale. */
int orc_mxfp4_quantize(const uint16_t *W, int64_t N, int64_t K, int64_t ldw,
                       uint8_t *codes, uint8_t *scales)
{
    int64_t n, k, b;
    if (K % 32 != 0 || N < 0 || ldw < K)
        return ORC_ERR_SHAPE;
    for (n = 0; n < N; ++n)
        for (k = 0; k < K; ++k)
            if (!isfinite(bf16_bits_to_float(W[n * ldw + k])))
                return ORC_ERR_NONFINITE;
    memset(codes, 0, (size_t)(N * (K / 2)));
    for (n = 0; n < N; ++n)
        for (b = 0; b < K / 32; ++b) {
            const uint16_t *blk = W + n * ldw + b * 32;
            float amax = 0.0f;
            int i, e = -127, ex;
            for (i = 0; i < 32; ++i) {
                float a = fabsf(bf16_bits_to_float(blk[i]));
                if (a > amax)
                    amax = a;
            }
            if (amax > 0.0f) {
                frexpf(amax, &ex); /* amax = m 2^ex, m in [0.5, 1): floor(log2) = ex - 1 */
                e = ex - 1 - 2;
                if (e < -127)
                    e = -127;
                if (e > 127)
                    e = 127;
            }
            scales[n * (K / 32) + b] = (uint8_t)(e + 127);
            for (i = 0; i < 32; ++i) {
                int64_t kk = b * 32 + i;
                uint8_t c = orc_e2m1_round(ldexpf(bf16_bits_to_float(blk[i]), -e));
                if (kk % 2 == 0)
                    codes[n * (K / 2) + kk / 2] |= c;
                else
                    codes[n * (K / 2) + kk / 2] |= (uint8_t)(c << 4);
            }
        }
    return ORC_OK;
}

/* w_hat = e2m1(code) * 2^(scale byte - 127) of an MXFP4 weight, fp64 [N, K]. */
void orc_mxfp4_dequantize(const uint8_t *codes, const uint8_t *scales, int64_t N, int64_t K, double *out)
{
    int64_t n, k;
    for (n = 0; n < N; ++n)
        for (k = 0; k < K; ++k)
            out[n * K + k] = orc_e2m1_value(code_at(codes, K, n, k)) * orc_e8m0_value(scales[n * (K / 32) + k / 32]);
}

void orc_nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales,
                          float tensor_scale, int64_t N, int64_t K, double *out)
{
    int64_t n, k;
    for (n = 0; n < N; ++n)
        for (k = 0; k < K; ++k)
            out[n * K + k] = w_hat(codes, scales, (double)tensor_scale, K, n, k);
}

/* ------------------------------------------------------------------ */
/* Linear + LoRA, forward and backward                                 */
/* ------------------------------------------------------------------ */

/* Forward [LoRA][Impl]: y = x * W_hat^T + s * (x * A^T) * B^T, fp64.
 * x bf16 [M, K]; A bf16 [r, K]; B bf16 [N, r].  Only the nrows token rows listed
 * in rows[] are computed; y is [nrows, N] and t (optional) is [nrows, r] holding
 * x * A^T for those rows. */
/* Threads the linear forward may use (1 = single-threaded, the default). */
static int g_threads = 1;
void orc_set_threads(int n) { g_threads = n > 0 ? n : 1; }

/* A weight element of format fmt (0: NVFP4 with tensor scale s_t; 1: MXFP4). */
static double weight_value(int fmt, const uint8_t *codes, const uint8_t *scales, double s_t, int64_t K,
                           int64_t n, int64_t k)
{
    if (fmt == 1)
        return orc_e2m1_value(code_at(codes, K, n, k)) * orc_e8m0_value(scales[n * (K / 32) + k / 32]);
    return w_hat(codes, scales, s_t, K, n, k);
}
/* An adapter element: bf16 bit patterns, or FP32 values when f32. */
static double adapter_value(const void *p, int f32, int64_t i)
{
    return f32 ? (double)((const float *)p)[i] : orc_bf16_value(((const uint16_t *)p)[i]);
}

/* y[i, n] = sum_k x[rows[i], k] w_hat[n, k] + s * sum_j t[i, j] B[n, j],
 * t[i, j] = sum_k x[rows[i], k] A[j, k], in fp64 [LoRA][Impl]. */
static void lora_fwd(int fmt, int f32_adapters, const uint16_t *x, int64_t K, int64_t N, const uint8_t *codes,
                     const uint8_t *scales, float tensor_scale, const void *A, const void *B, int r,
                     double lora_scale, const int64_t *rows, int64_t nrows, double *y, double *t)
{
    int64_t i, k;
    int j;
    double *tt = (double *)calloc((size_t)(nrows * (r > 0 ? r : 1)), sizeof(double));

    /* t = x * A^T for the selected rows. */
    for (i = 0; i < nrows; ++i)
        for (j = 0; j < r; ++j) {
            double acc = 0.0;
            for (k = 0; k < K; ++k)
                acc += orc_bf16_value(x[rows[i] * K + k]) * adapter_value(A, f32_adapters, (int64_t)j * K + k);
            tt[i * r + j] = acc;
        }

    /* Output features are independent: with threads, each takes whole features
     * (its own dequantized row), the sums over k run in the same order. */
#pragma omp parallel num_threads(g_threads) if (g_threads > 1)
    {
        double *wrow = (double *)malloc((size_t)K * sizeof(double));
        int64_t nn, ii, kk;
        int jj;
#pragma omp for schedule(static)
        for (nn = 0; nn < N; ++nn) {
            for (kk = 0; kk < K; ++kk)
                wrow[kk] = weight_value(fmt, codes, scales, (double)tensor_scale, K, nn, kk);
            for (ii = 0; ii < nrows; ++ii) {
                double acc = 0.0, lora = 0.0;
                for (kk = 0; kk < K; ++kk)
                    acc += orc_bf16_value(x[rows[ii] * K + kk]) * wrow[kk];
                for (jj = 0; jj < r; ++jj)
                    lora += tt[ii * r + jj] * adapter_value(B, f32_adapters, nn * r + jj);
                y[ii * N + nn] = acc + lora_scale * lora;
            }
        }
        free(wrow);
    }
    if (t)
        memcpy(t, tt, (size_t)(nrows * r) * sizeof(double));
    free(tt);
}

void orc_lora_linear_fwd(const uint16_t *x, int64_t M, int64_t K, int64_t N, const uint8_t *codes,
                         const uint8_t *scales, float tensor_scale, const uint16_t *A, const uint16_t *B, int r,
                         double lora_scale, const int64_t *rows, int64_t nrows, double *y, double *t)
{
    (void)M;
    lora_fwd(0, 0, x, K, N, codes, scales, tensor_scale, A, B, r, lora_scale, rows, nrows, y, t);
}

/* The forward with FP32 LoRA adapters A [r, K] and B [N, r] [LoRA]. */
void orc_lora_linear_fwd_f32ab(const uint16_t *x, int64_t M, int64_t K, int64_t N, const uint8_t *codes,
                               const uint8_t *scales, float tensor_scale, const float *A, const float *B, int r,
                               double lora_scale, const int64_t *rows, int64_t nrows, double *y, double *t)
{
    (void)M;
    lora_fwd(0, 1, x, K, N, codes, scales, tensor_scale, A, B, r, lora_scale, rows, nrows, y, t);
}

/* The forward with an MXFP4 weight (codes, E8M0 scales [N, K/32]) [MX]. */
void orc_mxfp4_lora_linear_fwd(const uint16_t *x, int64_t M, int64_t K, int64_t N, const uint8_t *codes,
                               const uint8_t *scales, const uint16_t *A, const uint16_t *B, int r, double lora_scale,
                               const int64_t *rows, int64_t nrows, double *y, double *t)
{
    (void)M;
    lora_fwd(1, 0, x, K, N, codes, scales, 1.0f, A, B, r, lora_scale, rows, nrows, y, t);
}

/* Backward with W_hat frozen [LoRA][Impl]:
 *   v  = dy * B                      [M, r]
 *   dx = dy * W_hat + s * v * A      (rows dx_rows only)  -> dx [n_dx, K]
 *   dA = s * v^T * x                 (columns dA_cols only) -> dA [r, n_dA]
 *   dB = s * dy^T * (x * A^T)        (rows dB_rows only)  -> dB [n_dB, r]
 * dy bf16 [M, N], x bf16 [M, K].  Any output pointer may be NULL. */
void orc_lora_linear_bwd(const uint16_t *dy, const uint16_t *x, int64_t M,
                         int64_t K, int64_t N, const uint8_t *codes,
                         const uint8_t *scales, float tensor_scale,
                         const uint16_t *A, const uint16_t *B, int r,
                         double lora_scale, const int64_t *dx_rows,
                         int64_t n_dx, double *dx, const int64_t *dA_cols,
                         int64_t n_dA, double *dA, const int64_t *dB_rows,
                         int64_t n_dB, double *dB)
{
    int64_t m, n, k, i;
    int j;
    double *v = (double *)calloc((size_t)(M * r + 1), sizeof(double));
    double *u = (double *)calloc((size_t)(M * r + 1), sizeof(double));

    /* v = dy * B, u = x * A^T over all tokens. */
    for (m = 0; m < M; ++m)
        for (j = 0; j < r; ++j) {
            double acc = 0.0;
            for (n = 0; n < N; ++n)
                acc += orc_bf16_value(dy[m * N + n]) * orc_bf16_value(B[n * r + j]);
            v[m * r + j] = acc;
            acc = 0.0;
            for (k = 0; k < K; ++k)
                acc += orc_bf16_value(x[m * K + k]) * orc_bf16_value(A[(int64_t)j * K + k]);
            u[m * r + j] = acc;
        }

    if (dx) {
        for (i = 0; i < n_dx; ++i) {
            m = dx_rows[i];
            for (k = 0; k < K; ++k) {
                double acc = 0.0, lora = 0.0;
                for (n = 0; n < N; ++n)
                    acc += orc_bf16_value(dy[m * N + n]) *
                           w_hat(codes, scales, (double)tensor_scale, K, n, k);
                for (j = 0; j < r; ++j)
                    lora += v[m * r + j] * orc_bf16_value(A[(int64_t)j * K + k]);
                dx[i * K + k] = acc + lora_scale * lora;
            }
        }
    }
    if (dA) {
        for (j = 0; j < r; ++j)
            for (i = 0; i < n_dA; ++i) {
                double acc = 0.0;
                k = dA_cols[i];
                for (m = 0; m < M; ++m)
                    acc += v[m * r + j] * orc_bf16_value(x[m * K + k]);
                dA[(int64_t)j * n_dA + i] = lora_scale * acc;
            }
    }
    if (dB) {
        for (i = 0; i < n_dB; ++i) {
            n = dB_rows[i];
            for (j = 0; j < r; ++j) {
                double acc = 0.0;
                for (m = 0; m < M; ++m)
                    acc += orc_bf16_value(dy[m * N + n]) * u[m * r + j];
                dB[i * r + j] = lora_scale * acc;
            }
        }
    }
    free(v);
    free(u);
}

/* ------------------------------------------------------------------ */
/* Adaptive Quantization Noise (AQN) RMSNorm                           */
/* ------------------------------------------------------------------ */

/* Philox4x64-10 block cipher (Salmon, Moraes, Dror, Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3", SC'11): ten rounds of two 64x64->128 multiplies
 * by the published multipliers, with the Weyl key schedule (golden ratio and
 * sqrt(3)-1 increments) applied between rounds. */
void orc_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2],
                       uint64_t out[4])
{
    const uint64_t M0 = 0xD2E7470EE14C6C93ULL, M1 = 0xCA5A826395121157ULL;
    const uint64_t W0 = 0x9E3779B97F4A7C15ULL, W1 = 0xBB67AE8584CAA73BULL;
    uint64_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint64_t k0 = key_in[0], k1 = key_in[1];
    int round;
    for (round = 0; round < 10; ++round) {
        unsigned __int128 p0 = (unsigned __int128)M0 * c0;
        unsigned __int128 p1 = (unsigned __int128)M1 * c2;
        uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
        uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
        uint64_t n0 = hi1 ^ c1 ^ k0;
        uint64_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += W0;
        k1 += W1;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* Channel-wise noise z[c] ~ N(0,1), c in [0, H) [AQN-S][AQN-M].
 * Block i = c / 4 uses counter (i, step, 0, 0) and key (seed, layer); its four
 * words w0..w3 give two Box-Muller pairs: (w0, w1) -> z[4i], z[4i+1] and
 * (w2, w3) -> z[4i+2], z[4i+3], with u1 = ((w >> 11) + 1) * 2^-53 in (0, 1] and
 * u2 = (w' >> 11) * 2^-53 in [0, 1). */
void orc_aqn_noise(int64_t H, uint64_t seed, uint64_t step, uint32_t layer,
                   double *z, uint64_t *raw)
{
    int64_t i, c;
    const double two53 = 9007199254740992.0; /* 2^53 */
    const double pi = 3.14159265358979323846;
    for (i = 0; i * 4 < H; ++i) {
        uint64_t ctr[4] = {(uint64_t)i, step, 0, 0};
        uint64_t key[2] = {seed, (uint64_t)layer};
        uint64_t w[4];
        double zz[4];
        int p;
        orc_philox4x64_10(ctr, key, w);
        for (p = 0; p < 2; ++p) {
            double u1 = ((double)(w[2 * p] >> 11) + 1.0) / two53;
            double u2 = (double)(w[2 * p + 1] >> 11) / two53;
            double rad = sqrt(-2.0 * log(u1));
            zz[2 * p] = rad * cos(2.0 * pi * u2);
            zz[2 * p + 1] = rad * sin(2.0 * pi * u2);
        }
        for (p = 0; p < 4; ++p) {
            c = 4 * i + p;
            if (c < H) {
                z[c] = zz[p];
                if (raw)
                    raw[c] = w[p];
            }
        }
    }
}

/* AQN-RMSNorm: y[m, c] = x[m, c] / sqrt(mean_c x^2 + eps) * (gamma[c] + sigma * z[c])
 * [AQN-S][AQN-M], fp64, for the nrows token rows listed in rows[]; y is
 * [nrows, H]. */
/* AQN-RMSNorm with the noise on the scale parameter, in one of the two
 * readings of "Gaussian noise in the LayerNorm scale" (dataforcee, AQN
 * paragraph): mult = 0 adds it, scale gamma + sigma z; mult = 1 scales by it,
 * gamma (1 + sigma z). */
void orc_aqn_rmsnorm_mode(const uint16_t *x, int64_t M, int64_t H,
                          const uint16_t *gamma, double eps, double sigma,
                          uint64_t seed, uint64_t step, uint32_t layer, int mult,
                          const int64_t *rows, int64_t nrows, double *y)
{
    int64_t i, c;
    double *z = (double *)malloc((size_t)(H > 0 ? H : 1) * sizeof(double));
    (void)M;
    orc_aqn_noise(H, seed, step, layer, z, NULL);
    for (i = 0; i < nrows; ++i) {
        const uint16_t *row = x + rows[i] * H;
        double ss = 0.0, inv;
        for (c = 0; c < H; ++c)
            ss += orc_bf16_value(row[c]) * orc_bf16_value(row[c]);
        inv = 1.0 / sqrt(ss / (double)H + eps);
        for (c = 0; c < H; ++c) {
            const double g = orc_bf16_value(gamma[c]);
            const double scale = mult ? g * (1.0 + sigma * z[c]) : g + sigma * z[c];
            y[i * H + c] = orc_bf16_value(row[c]) * inv * scale;
        }
    }
    free(z);
}

/* The additive reading (the library's default). */
void orc_aqn_rmsnorm(const uint16_t *x, int64_t M, int64_t H,
                     const uint16_t *gamma, double eps, double sigma,
                     uint64_t seed, uint64_t step, uint32_t layer,
                     const int64_t *rows, int64_t nrows, double *y)
{
    orc_aqn_rmsnorm_mode(x, M, H, gamma, eps, sigma, seed, step, layer, 0, rows, nrows, y);
}

/* Exponential-decay noise schedule [AQN-S][Hints]: num_stages equal stages over
 * total_steps; stage k uses sigma_start * (sigma_end / sigma_start)^(k/(S-1)). */
double orc_aqn_sigma(int64_t step, int64_t total_steps, double sigma_start,
                     double sigma_end, int num_stages)
{
    int64_t k;
    if (num_stages <= 1 || total_steps <= 0 || sigma_start == 0.0)
        return sigma_start;
    if (step < 0)
        step = 0;
    k = (step * num_stages) / total_steps;
    if (k > num_stages - 1)
        k = num_stages - 1;
    return sigma_start * pow(sigma_end / sigma_start, (double)k / (double)(num_stages - 1));
}
