// Adaptive Quantization Noise (AQN) RMSNorm.
//
// 1kpapers summary of "QeRL: Beyond Efficiency": AQN injects channel-wise
// Gaussian noise via the normalization layer with an exponential decay
// schedule; dataforcee "QERL: NVFP4-intensive learning" AQN paragraph: the noise
// lives in the norm's scale parameters.  So the norm uses gamma + sigma * z with
// one z[H] ~ N(0, 1) per (seed, step, layer), shared by every token; the other
// reading of that sentence, gamma (1 + sigma z), is the multiplicative mode.
//
// One kernel for hidden sizes up to kFusedMaxH: every CTA draws the noisy scale
// vector gamma + sigma z into shared memory (Philox4x64-10, Box-Muller in FP32)
// and normalizes its token rows with it.  Wider rows take two kernels: the
// noisy scale vector into the workspace, then the norm.
#include "common.cuh"

namespace qerl {
namespace {

// Philox4x64-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11): ten rounds of two 64x64->128-bit products with the published
// multipliers; the key is bumped by the Weyl constants after every round.
__device__ __forceinline__ void philox4x64_10(uint64_t c[4], uint64_t k0, uint64_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint64_t a0 = 0xD2E7470EE14C6C93ull * c[0], h0 = __umul64hi(0xD2E7470EE14C6C93ull, c[0]);
        const uint64_t a1 = 0xCA5A826395121157ull * c[2], h1 = __umul64hi(0xCA5A826395121157ull, c[2]);
        const uint64_t n0 = h1 ^ c[1] ^ k0, n2 = h0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = a1;
        c[2] = n2;
        c[3] = a0;
        k0 += 0x9E3779B97F4A7C15ull;
        k1 += 0xBB67AE8584CAA73Bull;
    }
}

// Box-Muller in FP32 from two Philox words: u1 = ((w0 >> 11) + 1) 2^-53 in
// (0, 1], u2 = (w1 >> 11) 2^-53 in [0, 1); z = sqrt(-2 ln u1) (cos, sin)(2 pi u2).
// ln u1 is taken as log1p(-(1 - u1)) near 1, where 1 - u1 (formed exactly in
// integers) would round away in FP32.
__device__ __forceinline__ void box_muller(uint64_t w0, uint64_t w1, float &z0, float &z1)
{
    const uint64_t a = (w0 >> 11) + 1ull;                 // u1 = a 2^-53, 1 <= a <= 2^53
    const float lnu1 = a > (1ull << 52) ? log1pf(-(float)((1ull << 53) - a) * 0x1p-53f) : logf((float)a * 0x1p-53f);
    const float rad = sqrtf(-2.0f * lnu1);
    float sn, cs;
    sincospif(2.0f * ((float)(w1 >> 11) * 0x1p-53f), &sn, &cs);
    z0 = rad * cs;
    z1 = rad * sn;
}

// The four normals of Philox block i (channels 4i .. 4i+3).
__device__ __forceinline__ void noise4(uint64_t i, uint64_t seed, uint64_t step, uint32_t layer, float z[4],
                                       uint64_t w[4])
{
    w[0] = i;
    w[1] = step;
    w[2] = 0ull;
    w[3] = 0ull;
    philox4x64_10(w, seed, (uint64_t)layer);
    box_muller(w[0], w[1], z[0], z[1]);
    box_muller(w[2], w[3], z[2], z[3]);
}

// Noisy scale of channel c: gamma + sigma z (additive) or gamma (1 + sigma z).
__device__ __forceinline__ float noisy_scale(float g, float sigma, float z, int mult)
{
    return mult ? g * (1.0f + sigma * z) : g + sigma * z;
}

// One thread per Philox block: channels 4i .. 4i+3.  Writes any of z_out /
// raw_out / scale_out given.

__global__ void aqn_noise_kernel(int64_t H, uint64_t seed, uint64_t step, uint32_t layer,
                                 const __nv_bfloat16 *__restrict__ gamma, float sigma, int mult,
                                 float *__restrict__ scale_out, float *__restrict__ z_out,
                                 uint64_t *__restrict__ raw_out)
{
    pdl_trigger();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (4 * i >= H) return;
    float z[4];
    uint64_t w[4];
    noise4((uint64_t)i, seed, step, layer, z, w);
    // The draws need no input: only the writes (and gamma) wait for the
    // preceding work when the launch is chained.
    pdl_wait();
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int64_t c = 4 * i + e;
        if (c >= H) break;
        if (z_out) z_out[c] = z[e];
        if (raw_out) raw_out[c] = w[e];
        if (scale_out) scale_out[c] = noisy_scale(bf16f(gamma[c]), sigma, z[e], mult);
    }
}

constexpr int kNormThreads = 256;

__device__ __forceinline__ float block_sum(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    return red[0];
}

// y = x * rsqrt(mean(x^2) + eps) * g, g = noisy scale (float) or gamma (bf16).
// Rows are strided over the grid; 16-byte vectors when H % 8 == 0.
__global__ void __launch_bounds__(kNormThreads)
    rmsnorm_kernel(const __nv_bfloat16 *__restrict__ x, int64_t M, int64_t H, const float *__restrict__ gscale,
                   const __nv_bfloat16 *__restrict__ gamma, float eps, __nv_bfloat16 *__restrict__ y)
{
    __shared__ float red[32];
    pdl_trigger();
    pdl_wait();
    const bool vec = (H % 8) == 0;
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const __nv_bfloat16 *row = x + m * H;
        __nv_bfloat16 *out = y + m * H;
        float ss = 0.0f;
        if (vec) {
            for (int64_t v = threadIdx.x; v < H / 8; v += blockDim.x) {
                const uint4 u = reinterpret_cast<const uint4 *>(row)[v];
                const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float a = bf16lo(wd[i]), b = bf16hi(wd[i]);
                    ss = fmaf(a, a, ss);
                    ss = fmaf(b, b, ss);
                }
            }
        } else {
            for (int64_t c = threadIdx.x; c < H; c += blockDim.x) {
                const float a = bf16f(row[c]);
                ss = fmaf(a, a, ss);
            }
        }
        ss = block_sum(ss, red);
        const float inv = rsqrtf(ss / (float)H + eps);
        if (vec) {
            for (int64_t v = threadIdx.x; v < H / 8; v += blockDim.x) {
                const uint4 u = reinterpret_cast<const uint4 *>(row)[v];
                const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int64_t c = v * 8 + 2 * i;
                    const float g0 = gscale ? gscale[c] : bf16f(gamma[c]);
                    const float g1 = gscale ? gscale[c + 1] : bf16f(gamma[c + 1]);
                    const __nv_bfloat162 p = __floats2bfloat162_rn(bf16lo(wd[i]) * inv * g0, bf16hi(wd[i]) * inv * g1);
                    o[i] = *reinterpret_cast<const uint32_t *>(&p);
                }
                reinterpret_cast<uint4 *>(out)[v] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        } else {
            for (int64_t c = threadIdx.x; c < H; c += blockDim.x) {
                const float g = gscale ? gscale[c] : bf16f(gamma[c]);
                out[c] = __float2bfloat16_rn(bf16f(row[c]) * inv * g);
            }
        }
        __syncthreads();  // red[] is reused by the next row
    }
}

// AQN-RMSNorm in one launch: the CTA draws the noisy scale (gamma + sigma z,
// or gamma (1 + sigma z)) for all H channels into shared memory (sigma = 0:
// gamma), then normalizes token rows m =
// blockIdx.x, blockIdx.x + gridDim.x, ...
constexpr int64_t kFusedMaxH = 16384;
constexpr int kFusedThreads = 512;  // the noise of H = 3584 (896 Philox blocks) in at most two rounds
__global__ void __launch_bounds__(kFusedThreads)
    aqn_rmsnorm_fused_kernel(const __nv_bfloat16 *__restrict__ x, int64_t M, int64_t H,
                             const __nv_bfloat16 *__restrict__ gamma, float eps, float sigma, uint64_t seed,
                             uint64_t step, uint32_t layer, int mult, __nv_bfloat16 *__restrict__ y)
{
    extern __shared__ float gs[];  // [H]
    __shared__ float red[32];
    pdl_trigger();
    // The draws need no input: z goes to shared memory before the wait for the
    // preceding work (x, gamma and y follow it when the launch is chained).
    const int64_t nb = (H + 3) / 4;
    const bool noisy = sigma != 0.0f;
    if (noisy) {
        for (int64_t i = threadIdx.x; i < nb; i += blockDim.x) {
            float z[4];
            uint64_t w[4];
            noise4((uint64_t)i, seed, step, layer, z, w);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (4 * i + e < H) gs[4 * i + e] = z[e];
        }
    }
    pdl_wait();
    for (int64_t i = threadIdx.x; i < nb; i += blockDim.x) {  // the same channels as drawn above
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int64_t c = 4 * i + e;
            if (c < H) gs[c] = noisy ? noisy_scale(bf16f(gamma[c]), sigma, gs[c], mult) : bf16f(gamma[c]);
        }
    }
    __syncthreads();
    const bool vec = (H % 8) == 0;
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const __nv_bfloat16 *row = x + m * H;
        __nv_bfloat16 *out = y + m * H;
        float ss = 0.0f;
        if (vec) {
            for (int64_t v = threadIdx.x; v < H / 8; v += blockDim.x) {
                const uint4 u = reinterpret_cast<const uint4 *>(row)[v];
                const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float a = bf16lo(wd[i]), b = bf16hi(wd[i]);
                    ss = fmaf(a, a, ss);
                    ss = fmaf(b, b, ss);
                }
            }
        } else {
            for (int64_t c = threadIdx.x; c < H; c += blockDim.x) {
                const float a = bf16f(row[c]);
                ss = fmaf(a, a, ss);
            }
        }
        ss = block_sum(ss, red);
        const float inv = rsqrtf(ss / (float)H + eps);
        if (vec) {
            for (int64_t v = threadIdx.x; v < H / 8; v += blockDim.x) {
                const uint4 u = reinterpret_cast<const uint4 *>(row)[v];
                const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int64_t c = v * 8 + 2 * i;
                    const __nv_bfloat162 p = __floats2bfloat162_rn(bf16lo(wd[i]) * inv * gs[c], bf16hi(wd[i]) * inv * gs[c + 1]);
                    o[i] = *reinterpret_cast<const uint32_t *>(&p);
                }
                reinterpret_cast<uint4 *>(out)[v] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        } else {
            for (int64_t c = threadIdx.x; c < H; c += blockDim.x) out[c] = __float2bfloat16_rn(bf16f(row[c]) * inv * gs[c]);
        }
        __syncthreads();  // red[] is reused by the next row
    }
}

}  // namespace
}  // namespace qerl

using namespace qerl;

extern "C" qerl_status qerl_aqn_noise(int64_t H, uint64_t seed, uint64_t step, uint32_t layer_id, float *z_out,
                                      uint64_t *raw_out, qerl_stream_t stream)
{
    if (H < 1 || !z_out) return QERL_ERR_INVALID_ARG;
    QERL_TRY(check_device());
    const int64_t n = (H + 3) / 4;
    aqn_noise_kernel<<<(unsigned)((n + 63) / 64), 64, 0, as_cuda(stream)>>>(H, seed, step, layer_id, nullptr, 0.0f,
                                                                          0, nullptr, z_out, raw_out);
    return launched();
}

extern "C" qerl_status qerl_aqn_rmsnorm_mode(const void *x, int64_t M, int64_t H, const void *gamma, float eps,
                                             float sigma, uint64_t seed, uint64_t step, uint32_t layer_id,
                                             int noise_mode, void *y, void *ws, size_t ws_bytes,
                                             qerl_stream_t stream)
{
    if (noise_mode != QERL_AQN_NOISE_ADD && noise_mode != QERL_AQN_NOISE_MUL) return QERL_ERR_INVALID_ARG;
    const int mult = noise_mode == QERL_AQN_NOISE_MUL ? 1 : 0;
    if (!gamma || M < 0 || H < 1 || !(eps >= 0.0f)) return QERL_ERR_INVALID_ARG;
    if (M == 0) return QERL_OK;  // x and y may be NULL for an empty batch
    if (!x || !y) return QERL_ERR_INVALID_ARG;
    if ((H % 8 == 0) && (!aligned16(x) || !aligned16(y))) return QERL_ERR_ALIGN;
    const bool noisy = sigma != 0.0f;
    if (noisy && (!ws || ws_bytes < qerl_workspace_bytes(QERL_OP_AQN_RMSNORM, M, 0, H, 0))) return QERL_ERR_WORKSPACE;
    QERL_TRY(check_device());
    cudaStream_t s = as_cuda(stream);
    if (H <= kFusedMaxH) {  // one launch: every CTA draws the noisy scale into shared memory
        int64_t g = M;
        if (g > 2 * num_sms()) g = 2 * num_sms();
        const size_t smem = (size_t)H * sizeof(float);
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(aqn_rmsnorm_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess)
            return QERL_ERR_CUDA;
        return launched(launch_k(aqn_rmsnorm_fused_kernel, dim3((unsigned)g), dim3(kFusedThreads), smem, s,
                                 g_chain.load() != 0, static_cast<const __nv_bfloat16 *>(x), M, H,
                                 static_cast<const __nv_bfloat16 *>(gamma), eps, sigma, seed, step, layer_id, mult,
                                 static_cast<__nv_bfloat16 *>(y)));
    }
    float *gscale = nullptr;
    if (noisy) {
        gscale = static_cast<float *>(ws);
        const int64_t n = (H + 3) / 4;
        QERL_TRY(launched(launch_k(aqn_noise_kernel, dim3((unsigned)((n + 63) / 64)), dim3(64), 0, s,
                                   g_chain.load() != 0, H, seed, step, layer_id,
                                   static_cast<const __nv_bfloat16 *>(gamma), sigma, mult, gscale,
                                   (float *)nullptr, (uint64_t *)nullptr)));
    }
    int64_t g = M;
    if (g > 8 * num_sms()) g = 8 * num_sms();
    return launched(launch_k(rmsnorm_kernel, dim3((unsigned)g), dim3(kNormThreads), 0, s, g_chain.load() != 0,
                             static_cast<const __nv_bfloat16 *>(x), M, H, (const float *)gscale,
                             static_cast<const __nv_bfloat16 *>(gamma), eps, static_cast<__nv_bfloat16 *>(y)));
}

extern "C" qerl_status qerl_aqn_rmsnorm(const void *x, int64_t M, int64_t H, const void *gamma, float eps,
                                        float sigma, uint64_t seed, uint64_t step, uint32_t layer_id, void *y,
                                        void *ws, size_t ws_bytes, qerl_stream_t stream)
{
    return qerl_aqn_rmsnorm_mode(x, M, H, gamma, eps, sigma, seed, step, layer_id, QERL_AQN_NOISE_ADD, y, ws,
                                 ws_bytes, stream);
}
