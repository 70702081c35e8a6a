/*
 * qerl.h -- C ABI of the GB300 (sm_103a) NVFP4 weight-only LoRA linear library.
 *
 * What it computes (sources are web pages about QeRL, cited by title/section):
 *  - "QeRL: NVFP4-Quantized Reinforcement Learning -- Redefining Efficiency in AI
 *    Training and Inference" (bitsofall), section "NVFP4: NVIDIA's FP4 Format":
 *    16-element blocks along a row, an FP8 E4M3 scale per block plus one FP32
 *    tensor scale (about 4.5 bits per weight), block scale = round_up(amax/vmax),
 *    element = round_to_even(value/scale).  Same page, LoRA paragraph and
 *    "Implementation and Practical Details": a frozen quantized W plus a
 *    trainable low-rank adapter in higher precision; weight-only quantization,
 *    activations and gradients stay high precision.
 *  - "QERL: NVFP4-intensive learning (RL) brings 32B LLM training to H100"
 *    (dataforcee), sections on the RL loop and on AQN: weight-only FP4 with
 *    FP4 x BF16 kernels; AQN adds channel-wise Gaussian noise to the norm's scale
 *    parameters under an exponential schedule.
 *  - "QeRL: Beyond Efficiency -- Quantization-enhanced Reinforcement Learning for
 *    LLMs" (1kpapers), summary: channel-wise Gaussian noise via the norm layer,
 *    exponential decay.  "QeRL" README mirror, "Hints for QeRL training" 2-3:
 *    prefill still dequantizes; sigma_start, sigma_end, num_stages.
 *
 * Conventions for every entry point:
 *  - Pointers marked (device) are CUDA device pointers on the current device;
 *    (host) pointers are host memory.  The caller owns and allocates every
 *    buffer, including workspaces; the library allocates nothing per call.
 *  - All matrices are dense row-major.  bf16 buffers are 16-bit IEEE bfloat16.
 *  - Work is enqueued asynchronously on `stream` (NULL = legacy default stream).
 *    Calls never synchronize, except qerl_get_error.
 *  - Argument errors are returned synchronously and nothing is launched.  Errors
 *    found by kernels (non-finite weights, a bounded wait that ran out) are
 *    latched on the device and reported by qerl_get_error.
 *  - The library runs only on compute capability 10.3 (GB300); elsewhere every
 *    launching call returns QERL_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef QERL_H
#define QERL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *qerl_stream_t;

typedef enum {
    QERL_OK = 0,
    QERL_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad flag */
    QERL_ERR_SHAPE = 2,              /* K % 16 != 0, r out of [1, 256], ... */
    QERL_ERR_ALIGN = 3,              /* a pointer or row stride not 16-byte aligned */
    QERL_ERR_NONFINITE = 4,          /* the weight held an Inf or NaN (latched) */
    QERL_ERR_CUDA = 5,               /* a CUDA runtime call failed */
    QERL_ERR_TIMEOUT = 6,            /* a bounded device-side wait ran out (latched) */
    QERL_ERR_UNSUPPORTED_DEVICE = 7, /* current device is not compute capability 10.3 */
    QERL_ERR_WORKSPACE = 8,          /* workspace missing or smaller than required */
    QERL_ERR_TOO_LARGE = 9           /* needs more scratch than the fixed no-allocation buffer */
} qerl_status;

/* Size of the fixed device scratch buffer behind qerl_nvfp4_lora_linear_fwd_noalloc. */
#define QERL_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Block-scale rounding of the quantizer. */
enum { QERL_SCALE_ROUND_UP = 0, QERL_SCALE_ROUND_NEAREST_EVEN = 1 };

typedef struct {
    int scale_round; /* QERL_SCALE_ROUND_UP (default) or QERL_SCALE_ROUND_NEAREST_EVEN */
} qerl_quant_opts;

/* Operations for qerl_workspace_bytes. */
enum {
    QERL_OP_QUANTIZE = 0,
    QERL_OP_LINEAR_FWD = 1,
    QERL_OP_LINEAR_BWD = 2,
    QERL_OP_AQN_RMSNORM = 3,
    QERL_OP_MXFP4_FWD = 4,        /* qerl_mxfp4_lora_linear_fwd */
    QERL_OP_LINEAR_FWD_F32AB = 5  /* qerl_nvfp4_lora_linear_fwd_f32ab */
};

/* Linear algorithm selection (qerl_set_linear_algo); AUTO is the default.
 * AUTO: a single-token forward on a weight of at most 24M values runs the
 * CUDA-core GEMV (where it applies: K % 32 == 0, r <= 256, M * (K + r) * 4
 * bytes <= 200 KiB; not in grouped calls); other calls run the tensor-core
 * kernels where they apply, else the CUDA-core GEMM.  GEMV selects the GEMV
 * for every forward of one or two tokens it applies to.  The format-variant
 * forwards (MXFP4 weights, FP32 adapters) have no GEMV: every selection but
 * SIMT runs them on the tensor-core kernel where it applies. */
enum { QERL_ALGO_AUTO = 0, QERL_ALGO_SIMT = 1, QERL_ALGO_TCGEN05 = 2, QERL_ALGO_GEMV = 3 };

/*
 * NVFP4 quantization of a bf16 weight (bitsofall, "NVFP4: NVIDIA's FP4 Format":
 * two-level scaling, cuDNN block-scaling recipe).
 *   W            (device) bf16 [N, K], row stride ldw elements (ldw >= K,
 *                ldw*2 and W 16-byte aligned).
 *   codes        (device) out, uint8 [N, K/2]: element 2j of a row in bits 0-3 of
 *                byte j, element 2j+1 in bits 4-7; E2M1 code = sign bit 3,
 *                magnitude index 0..7 of {0, .5, 1, 1.5, 2, 3, 4, 6}; zero is 0x0.
 *   scales       (device) out, uint8 [N, K/16] E4M3 block scales, row-major.
 *   tensor_scale (device) out, one float: s_t = amax|W| / (6*448), 1.0 if W == 0.
 *   Block scale = smallest E4M3 >= amax_block / (6*s_t) (or nearest-even with
 *   opts->scale_round), saturated at 448; code = nearest E2M1 of
 *   w / (scale*s_t), ties to the even code, saturated at 6.
 *   Dequantized weight: w_hat = e2m1(code) * e4m3(scale) * s_t.
 *   opts may be NULL (round up).  ws (device) >= qerl_workspace_bytes(
 *   QERL_OP_QUANTIZE, 0, N, K, 0) bytes of scratch, contents on entry ignored.
 *   K % 16 == 0 required (QERL_ERR_SHAPE).  An Inf/NaN in W latches
 *   QERL_ERR_NONFINITE, sets *tensor_scale to NaN and leaves codes/scales
 *   undefined.
 */
qerl_status qerl_nvfp4_quantize(const void *W, int64_t N, int64_t K, int64_t ldw,
                                uint8_t *codes, uint8_t *scales, float *tensor_scale,
                                const qerl_quant_opts *opts, void *ws, size_t ws_bytes,
                                qerl_stream_t stream);

/*
 * Dequantization (test aid; bitsofall "NVFP4" section): W_out (device) bf16
 * [N, K] = e2m1(code) * e4m3(scale), times *tensor_scale when
 * apply_tensor_scale != 0 (then rounded to nearest-even bf16; without it the
 * product is exact in bf16).  Inputs as produced by qerl_nvfp4_quantize.
 */
qerl_status qerl_nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales,
                                  const float *tensor_scale, int64_t N, int64_t K,
                                  void *W_out, int apply_tensor_scale, qerl_stream_t stream);

/*
 * Forward of the frozen NVFP4 linear with its LoRA adapter (bitsofall, LoRA
 * paragraph and "Implementation and Practical Details"; dataforcee, RL-loop
 * section: weight-only FP4 x BF16):
 *     y = x * w_hat^T + lora_scale * (x * A^T) * B^T
 *   x      (device) bf16 [M, K]        A (device) bf16 [r, K]
 *   codes/scales/tensor_scale (device) NVFP4 weight of shape [N, K]
 *   B      (device) bf16 [N, r]        y (device) out bf16 [M, N]
 *   t_out  (device) optional out float [M, r] = x * A^T (for the backward); NULL ok
 *   Accumulation is FP32; the result is rounded to bf16 once.  1 <= r <= 256,
 *   K % 16 == 0, M, N >= 1; x, A, B, y and the codes rows 16-byte aligned.
 *   Kernels (see qerl_set_linear_algo): tcgen05 for K % 256 == 0; the CUDA-core
 *   GEMV for single-token calls on small weights (K % 32 == 0); the CUDA-core
 *   GEMM for the rest.  All compute the same result within rounding.
 *   ws (device) >= qerl_workspace_bytes(QERL_OP_LINEAR_FWD, M, N, K, r).
 */
qerl_status qerl_nvfp4_lora_linear_fwd(const void *x, int64_t M, int64_t K, int64_t N,
                                       const uint8_t *codes, const uint8_t *scales,
                                       const float *tensor_scale, const void *A, const void *B,
                                       int r, float lora_scale, void *y, float *t_out,
                                       void *ws, size_t ws_bytes, qerl_stream_t stream);

/*
 * The forward above without a caller-supplied workspace.  The pages have no
 * counterpart: this is an interface for callers that cannot allocate device
 * memory -- for example a host framework that owns every device byte through
 * its own pool and forbids allocations from outside it, or code that must not
 * call cudaMalloc mid-step because cudaMalloc can synchronize the device.
 * Computes exactly what qerl_nvfp4_lora_linear_fwd computes (same arguments
 * minus ws/ws_bytes), using a scratch buffer of QERL_NOALLOC_SCRATCH_BYTES that
 * lives in the library's own device memory: every GPU that loads the library
 * holds those bytes until the process exits.
 *   - Allocates nothing: no cudaMalloc/cudaFree, no allocating library call.
 *   - The first call on a device looks up that buffer's device address (with
 *     that device current) and caches it; make the first call on each device
 *     before any stream capture.
 *   - Shapes whose scratch need, qerl_workspace_bytes(QERL_OP_LINEAR_FWD, M, N,
 *     K, r), exceeds QERL_NOALLOC_SCRATCH_BYTES return QERL_ERR_TOO_LARGE with
 *     nothing launched.
 *   - Every call on a device shares the one buffer: calls whose kernels overlap
 *     on the GPU (other streams, other host threads) race and corrupt each
 *     other; serialize them.  The buffer holds the LoRA down-projection u and
 *     the split-K partial tiles; each call writes every part of it that it
 *     reads, so no part has to start at zero.
 */
qerl_status qerl_nvfp4_lora_linear_fwd_noalloc(const void *x, int64_t M, int64_t K, int64_t N,
                                               const uint8_t *codes, const uint8_t *scales,
                                               const float *tensor_scale, const void *A, const void *B,
                                               int r, float lora_scale, void *y, float *t_out,
                                               qerl_stream_t stream);

/*
 * Backward through the frozen NVFP4 weight into the LoRA adapter (bitsofall,
 * "Implementation and Practical Details": gradients flow through dequantized
 * weights; W itself is frozen so there is no dW):
 *     v  = dy * B                                   (FP32, internal)
 *     dx = dy * w_hat + lora_scale * v * A          (bf16 out [M, K])
 *     dA = lora_scale * v^T * x                     (float out [r, K])
 *     dB = lora_scale * dy^T * (x * A^T)            (float out [N, r])
 *   dy (device) bf16 [M, N]; x (device) bf16 [M, K]; t_saved (device) optional
 *   float [M, r] = x * A^T from the forward (recomputed when NULL).
 *   accumulate_grads != 0 adds into dA/dB instead of overwriting.  dx, dA or dB
 *   may be NULL to skip that output.  Shapes/alignment as the forward.
 *   ws (device) >= qerl_workspace_bytes(QERL_OP_LINEAR_BWD, M, N, K, r).
 */
qerl_status qerl_nvfp4_lora_linear_bwd(const void *dy, const void *x, int64_t M, int64_t K,
                                       int64_t N, const uint8_t *codes, const uint8_t *scales,
                                       const float *tensor_scale, const void *A, const void *B,
                                       int r, float lora_scale, const float *t_saved, void *dx,
                                       float *dA, float *dB, int accumulate_grads, void *ws,
                                       size_t ws_bytes, qerl_stream_t stream);

/*
 * Chained launches (default on).  The kernels of consecutive calls on a stream
 * are launched as programmatic dependents: a kernel may be scheduled before the
 * preceding work has finished, and it waits for that work (griddepcontrol.wait)
 * before it reads or writes memory the work touches -- with one exception: the
 * forward's main kernel starts reading the frozen weight (codes, scales,
 * tensor_scale) before the preceding work has finished.  Chaining hides the
 * launch gap between calls and overlaps each forward's weight stream with the
 * tail of the previous call.  Contract while on: a kernel that writes a
 * forward's codes, scales or tensor_scale must have completed before that
 * forward is enqueued, or be separated from it by any launch that does not
 * signal programmatic completion early (every library entry point that
 * writes weights -- quantize, pack, unpack -- is such a launch).  on = 0 turns
 * chaining off (every kernel waits for the preceding work to complete);
 * on = 1 turns it on; anything else returns QERL_ERR_INVALID_ARG.  Global.
 */
qerl_status qerl_set_launch_chaining(int on);

/*
 * Packed code layout for the tensor-core dequantizer.  The pages name Marlin as
 * the kernel that serves the NVFP4 x BF16 product ("QeRL" README mirror,
 * feature list; dataforcee, RL-loop section); kernels of that family lay the
 * frozen weight out once, when it is loaded, in the order their dequantizer
 * reads it.  This is that step for this library: a bit permutation inside each
 * little-endian 32-bit word of codes (eight codes of k = 8w .. 8w+7), so the
 * packed array has the same size and shape as the standard one [N, K/2]:
 *   elements 2p, 2p+1 form pair p = 0..3; the even element's mantissa, low
 *   exponent and high exponent bits sit at bits (6,7,8), (3,4,5), (0,1,2),
 *   (9,10,11) for p = 0,1,2,3 and its sign at bit 15, 12, 13, 14; the odd
 *   element uses the same positions + 16.
 * Scales and the tensor scale are unchanged.
 *   codes/packed (device) [N, K/2] bytes, 16-byte aligned; K % 16 == 0
 *   (QERL_ERR_SHAPE).  in == out (in place) is allowed; other overlaps return
 *   QERL_ERR_INVALID_ARG.
 */
qerl_status qerl_nvfp4_pack_codes(const uint8_t *codes, int64_t N, int64_t K, uint8_t *packed,
                                  qerl_stream_t stream);
qerl_status qerl_nvfp4_unpack_codes(const uint8_t *packed, int64_t N, int64_t K, uint8_t *codes,
                                    qerl_stream_t stream);

/*
 * Grouped forward: several linears that read the same x (in a decoder layer,
 * q|k|v and gate|up read one normalised input) in one call; the same result as
 * qerl_nvfp4_lora_linear_fwd (or _packed) on each group.  The pages have no
 * such call: it is an interface of this library that saves launches.  The
 * tensor-core path serves up to 3 groups in one launch (above 64 tokens, one
 * pass over x also computes every group's LoRA down-projection); more groups,
 * or shapes it does not cover, run the groups one after the other.
 *   groups (host) [n_groups], 1 <= n_groups <= 8: per group N, codes, scales,
 *   tensor_scale, A [r, K], B [N, r], y [M, N] out, t_out optional [M, r].
 *   x (device) bf16 [M, K]; r, lora_scale and packed (0: standard codes,
 *   1: packed layout) shared.  ws (device) >= qerl_lora_linear_fwd_grouped_ws_bytes.
 * Errors: QERL_ERR_INVALID_ARG for n_groups outside 1..8 or packed not 0/1;
 * each group is checked as in qerl_nvfp4_lora_linear_fwd (the same statuses,
 * nothing launched); QERL_ERR_WORKSPACE for a short ws.
 */
typedef struct qerl_lora_linear_group {
    int64_t N;
    const uint8_t *codes;
    const uint8_t *scales;
    const float *tensor_scale;
    const void *A;
    const void *B;
    void *y;
    float *t_out;
} qerl_lora_linear_group;
size_t qerl_lora_linear_fwd_grouped_ws_bytes(int64_t M, int64_t K, int r, const int64_t *N, int n_groups);
qerl_status qerl_nvfp4_lora_linear_fwd_grouped(const void *x, int64_t M, int64_t K, int r, float lora_scale,
                                               const qerl_lora_linear_group *groups, int n_groups, int packed,
                                               void *ws, size_t ws_bytes, qerl_stream_t stream);

/*
 * qerl_nvfp4_lora_linear_fwd and qerl_nvfp4_lora_linear_bwd with the codes in
 * the packed layout above: same arguments, same results, same workspace sizes.
 */
qerl_status qerl_nvfp4_lora_linear_fwd_packed(const void *x, int64_t M, int64_t K, int64_t N,
                                              const uint8_t *packed_codes, const uint8_t *scales,
                                              const float *tensor_scale, const void *A, const void *B,
                                              int r, float lora_scale, void *y, float *t_out,
                                              void *ws, size_t ws_bytes, qerl_stream_t stream);
qerl_status qerl_nvfp4_lora_linear_bwd_packed(const void *dy, const void *x, int64_t M, int64_t K,
                                              int64_t N, const uint8_t *packed_codes, const uint8_t *scales,
                                              const float *tensor_scale, const void *A, const void *B,
                                              int r, float lora_scale, const float *t_saved, void *dx,
                                              float *dA, float *dB, int accumulate_grads, void *ws,
                                              size_t ws_bytes, qerl_stream_t stream);

/*
 * AQN-RMSNorm (1kpapers summary; dataforcee AQN paragraph: channel-wise
 * Gaussian noise in the norm's scale parameters):
 *     y[m, c] = x[m, c] / sqrt(mean_c x[m, :]^2 + eps) * (gamma[c] + sigma * z[c])
 *   x (device) bf16 [M, H], gamma (device) bf16 [H], y (device) out bf16 [M, H].
 *   z[c] ~ N(0, 1) is one vector per (seed, step, layer_id), shared by all M
 *   tokens: Philox4x64-10 with key (seed, layer_id), counter (c/4, step, 0, 0),
 *   Box-Muller on word pairs (see qerl_aqn_noise).  sigma == 0 is plain RMSNorm.
 *   ws (device) >= qerl_workspace_bytes(QERL_OP_AQN_RMSNORM, M, 0, H, 0).
 *   One launch for H <= 16384 (each CTA draws the noisy scale into shared
 *   memory); wider rows draw it into ws first.
 */
qerl_status qerl_aqn_rmsnorm(const void *x, int64_t M, int64_t H, const void *gamma, float eps,
                             float sigma, uint64_t seed, uint64_t step, uint32_t layer_id,
                             void *y, void *ws, size_t ws_bytes, qerl_stream_t stream);

/*
 * The same norm with the noise mode chosen (dataforcee, AQN paragraph: noise in
 * the norm's scale parameters, which reads two ways):
 *   QERL_AQN_NOISE_ADD  scale gamma[c] + sigma * z[c]   (qerl_aqn_rmsnorm)
 *   QERL_AQN_NOISE_MUL  scale gamma[c] * (1 + sigma * z[c])
 * Any other noise_mode returns QERL_ERR_INVALID_ARG.  Arguments, workspace and
 * launches as qerl_aqn_rmsnorm.
 */
enum { QERL_AQN_NOISE_ADD = 0, QERL_AQN_NOISE_MUL = 1 };
qerl_status qerl_aqn_rmsnorm_mode(const void *x, int64_t M, int64_t H, const void *gamma, float eps,
                                  float sigma, uint64_t seed, uint64_t step, uint32_t layer_id,
                                  int noise_mode, void *y, void *ws, size_t ws_bytes,
                                  qerl_stream_t stream);

/*
 * The AQN noise vector alone (test aid): z_out (device) float [H]; raw_out
 * (device, optional) uint64 [H], the Philox word each channel used:
 * block i = c/4 -> words w0..w3 of Philox4x64-10(counter (i, step, 0, 0),
 * key (seed, layer_id)); z[4i], z[4i+1] from (w0, w1) and z[4i+2], z[4i+3]
 * from (w2, w3) with u1 = ((wa >> 11) + 1) * 2^-53, u2 = (wb >> 11) * 2^-53,
 * z = sqrt(-2 ln u1) * (cos 2 pi u2, sin 2 pi u2); raw_out[c] = w_(c mod 4).
 * Computed in FP32 (ln u1 as log1p(u1 - 1) near 1); within a few 1e-6 of the
 * exact values.
 */
qerl_status qerl_aqn_noise(int64_t H, uint64_t seed, uint64_t step, uint32_t layer_id,
                           float *z_out, uint64_t *raw_out, qerl_stream_t stream);

/*
 * Noise schedule (host function; "QeRL" README "Hints" item 3, 1kpapers
 * summary: exponential decay): num_stages equal stages over total_steps;
 * stage k = min(floor(step * num_stages / total_steps), num_stages - 1);
 * sigma = sigma_start * (sigma_end / sigma_start)^(k / (num_stages - 1)).
 * num_stages <= 1 or total_steps <= 0 returns sigma_start.
 */
float qerl_aqn_sigma(int64_t step, int64_t total_steps, float sigma_start, float sigma_end,
                     int num_stages);

/*
 * Format variants (bitsofall "QeRL: NVFP4-Quantized Reinforcement Learning",
 * "NVFP4" section, which sets NVFP4 against MXFP4, whose blocks are 32 values
 * with a power-of-two scale; and its LoRA paragraph, which keeps the adapters
 * in higher precision, e.g. FP32).
 *
 * The two variant forwards run on the tcgen05 kernel of the NVFP4 forward
 * when K % 256 == 0 and x, y, codes, scales, A, B (and t_out) are 16-byte
 * aligned, unless qerl_set_linear_algo selected QERL_ALGO_SIMT; otherwise on
 * the CUDA-core GEMM.  ws (device) >= qerl_workspace_bytes(QERL_OP_MXFP4_FWD
 * or QERL_OP_LINEAR_FWD_F32AB, M, N, K, r) bytes, contents on entry ignored
 * (QERL_ERR_WORKSPACE otherwise).
 *
 * MXFP4 quantizer: W (device) bf16 [N, K] (row stride ldw elements), K % 32 ==
 * 0 -> codes (device, 16-byte aligned) u8 [N, K/2] (element 2j in the low
 * nibble of byte j, E2M1 codes as for NVFP4) and scales (device) u8 [N, K/32]
 * E8M0 bytes: for each block of 32, e = floor(log2(amax)) - 2 (the OCP MX
 * rule: 2 is the exponent of E2M1's largest value 6 = 1.5 * 2^2) clamped to
 * [-127, 127] (-127 for an all-zero block), byte e + 127, and each code the
 * E2M1 value nearest w * 2^-e (ties to the even code, saturating at 6, zero as
 * code 0).  No tensor scale.  A non-finite weight latches QERL_ERR_NONFINITE.
 */
qerl_status qerl_mxfp4_quantize(const void *W, int64_t N, int64_t K, int64_t ldw, uint8_t *codes,
                                uint8_t *scales, qerl_stream_t stream);

/* y = x w_hat^T + s (x A^T) B^T with an MXFP4 weight, w_hat = e2m1(code) *
 * 2^(scale byte - 127); x bf16 [M, K], A bf16 [r, K], B bf16 [N, r], y bf16
 * [M, N], t_out (optional) FP32 [M, r].  K % 32 == 0, 1 <= r <= 256.
 * Tensor-core path: each call first writes the scales into ws at one byte per
 * 16 values (the NVFP4 scale layout), and the dequantizer multiplies the
 * E2M1 value by 2^(b - 127) in bf16, exact for every scale byte b <= 252 (the
 * weight itself overflows bf16 and FP32 above); accumulation in FP32. */
qerl_status qerl_mxfp4_lora_linear_fwd(const void *x, int64_t M, int64_t K, int64_t N,
                                       const uint8_t *codes, const uint8_t *scales, const void *A,
                                       const void *B, int r, float lora_scale, void *y, float *t_out,
                                       void *ws, size_t ws_bytes, qerl_stream_t stream);

/* qerl_nvfp4_lora_linear_fwd (standard code layout) with FP32 LoRA adapters:
 * A (device) float [r, K], B (device) float [N, r]; t = x A^T is accumulated
 * in FP32.  The LoRA term: FP32 on the CUDA-core GEMM; on the tensor-core
 * path, with u = s t / (s_t 2^c) split as u_hi = bf16(u), u_lo = bf16(u - u_hi)
 * and B likewise, the three products B_hi u_hi + B_hi u_lo + B_lo u_hi
 * accumulated in FP32 (relative error about 2^-16 of the term). */
qerl_status qerl_nvfp4_lora_linear_fwd_f32ab(const void *x, int64_t M, int64_t K, int64_t N,
                                             const uint8_t *codes, const uint8_t *scales,
                                             const float *tensor_scale, const float *A, const float *B,
                                             int r, float lora_scale, void *y, float *t_out, void *ws,
                                             size_t ws_bytes, qerl_stream_t stream);

/*
 * Decoder-layer chain at decode batch sizes: every NVFP4 + LoRA linear of n
 * Qwen2.5-style decoder layers, with the AQN-RMSNorms, the residual adds and
 * SwiGLU between them, in one persistent launch (one CTA per SM).  The chain
 * is the rollout forward the pages put the NVFP4 speed-up in ("QeRL" README
 * "Highlights": rollout phase; 1kpapers abstract: 32B RL on one GPU); the
 * norm is AQN-RMSNorm (1kpapers abstract; dataforcee "QERL: NVFP4-intensive
 * learning", AQN paragraph: the noise lives in the norm's scale).  Per layer:
 *     h1 = h0 + attn W_o^T (+ LoRA),   q,k,v = N1(h0) W_{q,k,v}^T (+ LoRA),
 *     h2 = h1 + (silu(N2(h1) W_gate^T) * N2(h1) W_up^T) W_down^T (+ LoRA each),
 * N_i(h) = h * rsqrt(mean(h^2) + eps) * (gamma_i + sigma z_i), z ~ N(0,1) per
 * channel from Philox4x64-10 (key (seed, 2*layer + i - 1), counter
 * (channel / 4, step, 0, 0)), as qerl_aqn_rmsnorm.
 * Attention itself is outside the path: `attn` is its output, given.  Each
 * linear's output is rounded to bf16, residual sums are rounded to bf16.
 * The norm is fused: its producer writes bf16(h * (gamma + sigma z)) and the
 * consumer scales its output rows by rsqrt(mean(h^2) + eps).
 */
typedef struct {
    const uint8_t *codes;       /* [N, K/2] E2M1 codes, packed layout (qerl_nvfp4_pack_codes) */
    const uint8_t *scales;      /* [N, K/16] E4M3 block scales */
    const float *tensor_scale;  /* device, 1 */
    const void *A;              /* bf16 [r, K] LoRA down */
    const void *B;              /* bf16 [N, r] LoRA up */
} qerl_linear_weights;

typedef struct {
    qerl_linear_weights q, k, v, o, gate, up, down;
    const void *gamma_attn;     /* bf16 [hidden]: scale of the norm before q, k, v */
    const void *gamma_mlp;      /* bf16 [hidden]: scale of the norm before gate, up */
    const void *attn;           /* bf16 [M, hidden]: attention output, the o input */
    void *q_out, *k_out, *v_out;  /* bf16 [M, q_dim], [M, kv_dim] x 2, or NULL (scratch) */
} qerl_decoder_layer;

typedef struct {
    int64_t M;                  /* tokens, 1..64 */
    int64_t hidden;             /* multiple of 256; q_dim == hidden */
    int64_t q_dim, kv_dim;      /* multiples of 128 */
    int64_t intermediate;       /* multiple of 256 */
    int r;                      /* LoRA rank: 8..64, multiple of 8 */
    float lora_scale, eps;
} qerl_decoder_dims;

typedef struct qerl_chain qerl_chain;

/* Workspace bytes of a chain of n_layers (0 if the dimensions are not covered). */
size_t qerl_decoder_chain_ws_bytes(const qerl_decoder_dims *dims, int n_layers);

/*
 * Builds the chain's tables (jobs, tensor maps, buffers) in `ws` (caller
 * owned, qerl_decoder_chain_ws_bytes bytes, 16-byte aligned) with blocking
 * copies, and returns a host handle.  Call it outside stream capture; the
 * pointers it is given (weights, x_in, x_out, attn, outputs) must stay valid
 * while the handle is used.  x_in, x_out: bf16 [M, hidden] device.  After a
 * run that reported an error, build the plan again (it resets the counters in
 * ws).  Errors: QERL_ERR_INVALID_ARG, QERL_ERR_ALIGN, QERL_ERR_WORKSPACE,
 * QERL_ERR_SHAPE, QERL_ERR_CUDA; nothing is launched on error.
 */
qerl_status qerl_decoder_chain_plan(const qerl_decoder_layer *layers, int n_layers,
                                    const qerl_decoder_dims *dims, const void *x_in, void *x_out,
                                    void *ws, size_t ws_bytes, qerl_chain **plan);

/* Runs a planned chain on `stream` (one cooperative launch; capturable).  sigma,
 * seed and step set the AQN noise of every norm; the chain's layer l is model
 * layer first_layer + l, whose norms use noise keys 2 (first_layer + l) (before
 * q/k/v) and 2 (first_layer + l) + 1 (before gate/up), so a model split over
 * several chains draws the same noise as one chain.  Timeouts latch
 * QERL_ERR_TIMEOUT (qerl_get_error). */
qerl_status qerl_decoder_chain_run(const qerl_chain *plan, float sigma, uint64_t seed, uint64_t step,
                                   uint32_t first_layer, qerl_stream_t stream);

/* Frees the host handle (the workspace stays the caller's). */
void qerl_decoder_chain_destroy(qerl_chain *plan);

/*
 * Decoder-layer glue between the per-linear calls (the pages have no
 * counterpart: these are the Qwen2.5 layer's residual add and SwiGLU, the
 * operations the decoder chain fuses).  Elementwise over n bf16 values
 * (device), each result rounded to bf16 once: out[i] = bf16(h[i] + y[i]), or
 * bf16(silu(g[i]) * u[i]) with silu(g) = g / (1 + e^-g), computed in FP32 as
 * g * sigmoid(g) from e^-|g| (no intermediate overflows).
 * out may alias an input.  16-byte vector accesses when every pointer is
 * 16-byte aligned and n % 8 == 0, else scalar ones.  Chained launches wait
 * for the preceding work.  n = 0 launches nothing; NULL pointers or n < 0
 * return QERL_ERR_INVALID_ARG.
 */
qerl_status qerl_residual_add(const void *h, const void *y, int64_t n, void *out, qerl_stream_t stream);
qerl_status qerl_swiglu(const void *g, const void *u, int64_t n, void *out, qerl_stream_t stream);

/* Scratch bytes an operation needs (0 if none).  Sizes as in the calls. */
size_t qerl_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, int r);

/* Waits for `stream`, then returns (and clears) the first error latched by a
 * kernel on the current device, or a CUDA error, or QERL_OK. */
qerl_status qerl_get_error(qerl_stream_t stream);

/* Static description of a status code. */
const char *qerl_status_string(qerl_status status);

/* Selects the linear kernels (process-wide): QERL_ALGO_AUTO, _SIMT, _TCGEN05 or
 * _GEMV.  TCGEN05 falls back to SIMT for shapes it does not cover; GEMV (the
 * forward only; the backward runs as under AUTO) falls back to the AUTO choice
 * among the other two. */
qerl_status qerl_set_linear_algo(int algo);

/* Number of kernels this library launched since load (host-side counter). */
uint64_t qerl_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* QERL_H */
