// NVFP4 quantizer and dequantizer.
//
// The quantizer reads W twice (the tensor amax first, then the blocks), but the
// second pass walks W backwards: it starts on the part the first pass read
// last, which is still in L2, so for W up to about the L2 size (129 MB) HBM
// sees a single read of W, and for larger W the second read is shorter by
// roughly what L2 holds.
//
// Format (bitsofall "QeRL: NVFP4-Quantized Reinforcement Learning", section
// "NVFP4: NVIDIA's FP4 Format"): 16-element blocks along a row, one E4M3 scale
// per block, one FP32 tensor scale; block scale rounded up, values rounded to
// nearest-even E2M1.  Every decision is taken in IEEE FP32 with explicitly
// rounded operations so that it is reproducible bit for bit.
#include "common.cuh"

namespace qerl {
namespace {

constexpr int kAmaxThreads = 256;
constexpr int kMaxAmaxBlocks = 1024;  // workspace = kMaxAmaxBlocks * 4 bytes
constexpr int kQuantThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// The same load marked evict-first in L2: the second pass's lines are not
// needed again, so the ones the first pass left behind stay longer.
__device__ __forceinline__ uint4 ld_last_use(const void *p, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Largest |bf16| magnitude pattern among the two halves of u.  Magnitude bit
// patterns of IEEE numbers order like their values; Inf/NaN patterns are
// >= 0x7F80 and so dominate any finite value.
__device__ __forceinline__ uint32_t mag2(uint32_t u)
{
    return max(u & 0x7FFFu, (u >> 16) & 0x7FFFu);
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    v = red[0];
    __syncthreads();
    return v;
}

// Pass 1: per-CTA maximum of |W| as a bf16 magnitude bit pattern.
__global__ void __launch_bounds__(kAmaxThreads) amax_kernel(const __nv_bfloat16 *__restrict__ W, int64_t N,
                                                            int64_t K, int64_t ldw, uint32_t *__restrict__ partial)
{
    __shared__ uint32_t red[32];
    const int64_t vpr = K / 8;  // 16-byte vectors per row
    const int64_t total = N * vpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    uint32_t m = 0;
    int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; v + 3 * stride < total; v += 4 * stride) {
        uint4 u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int64_t vi = v + i * stride, row = vi / vpr, c = vi - row * vpr;
            u[i] = ld_stream(W + row * ldw + c * 8);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) m = max(m, max(max(mag2(u[i].x), mag2(u[i].y)), max(mag2(u[i].z), mag2(u[i].w))));
    }
    for (; v < total; v += stride) {
        int64_t row = v / vpr, c = v - row * vpr;
        uint4 u = ld_stream(W + row * ldw + c * 8);
        m = max(m, max(max(mag2(u.x), mag2(u.y)), max(mag2(u.z), mag2(u.w))));
    }
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) partial[blockIdx.x] = m;
}

// Smallest non-negative finite E4M3 value >= t, as a byte (saturates at 448).
__device__ __forceinline__ uint32_t e4m3_ceil(float t)
{
    if (!(t > 0.0f)) return 0u;
    if (t > 448.0f) return 0x7Eu;
    const uint32_t u = __float_as_uint(t);
    const int e = (int)(u >> 23) - 127;
    if (e < -6) {
        // Subnormal E4M3 range m * 2^-9 (m = 8 is 2^-6, the first normal, whose
        // byte 0x08 continues the sequence).  t * 512 is exact.
        return (uint32_t)ceilf(t * 512.0f);
    }
    uint32_t m3 = (u >> 20) & 7u, E = (uint32_t)(e + 7);
    if (u & 0xFFFFFu) {  // bits below the 3 kept mantissa bits: round up
        if (++m3 == 8u) {
            m3 = 0u;
            ++E;
        }
    }
    return (E << 3) | m3;
}

// Nearest-even E4M3 with saturation at 448 (the hardware conversion).
__device__ __forceinline__ uint32_t e4m3_rne(float t)
{
    if (!(t > 0.0f)) return 0u;
    uint16_t pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f), "f"(t));
    return pair & 0xFFu;
}

// E2M1 code of q: nearest of {0,.5,1,1.5,2,3,4,6} in magnitude, ties to the even
// code (the midpoints .25,1.25,2.5,5 fall down, .75,1.75,3.5 fall up), > 6
// saturates; a zero result is code 0 whatever the sign.
__device__ __forceinline__ uint32_t e2m1_code(float q)
{
    const float a = fabsf(q);
    uint32_t c = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) + (uint32_t)(a >= 1.75f) +
                 (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.0f);
    return (c != 0u && q < 0.0f) ? (c | 8u) : c;
}

// Pass 2: reduce the partials to s_t, then quantize one 16-block per thread,
// from the last block of W to the first (the first pass ran front to back).
__global__ void __launch_bounds__(kQuantThreads)
    quantize_kernel(const __nv_bfloat16 *__restrict__ W, int64_t N, int64_t K, int64_t ldw,
                    const uint32_t *__restrict__ partial, int nparts, uint8_t *__restrict__ codes,
                    uint8_t *__restrict__ scales, float *__restrict__ tensor_scale, int round_mode,
                    unsigned int *err)
{
    __shared__ uint32_t red[32];
    uint32_t m = 0;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) m = max(m, partial[i]);
    m = block_max_u32(m, red);
    if (m >= 0x7F80u) {  // Inf or NaN somewhere in W
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            latch_error(err, QERL_ERR_NONFINITE);
            *tensor_scale = __uint_as_float(0x7FC00000u);
        }
        return;
    }
    const float amax = __uint_as_float(m << 16);
    const float s_t = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;  // 2688 = 6 * 448
    if (blockIdx.x == 0 && threadIdx.x == 0) *tensor_scale = s_t;
    const float d = __fmul_rn(6.0f, s_t);

    const int64_t bpr = K / 16;
    const int64_t nblk = N * bpr;
    const uint64_t pol = l2_evict_first_policy();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nblk; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t blk = nblk - 1 - i;
        const int64_t row = blk / bpr, b = blk - row * bpr;
        const __nv_bfloat16 *src = W + row * ldw + b * 16;
        const uint4 u0 = ld_last_use(src, pol), u1 = ld_last_use(src + 8, pol);
        const uint32_t wd[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        float w[16];
        float amax_b = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            w[2 * i] = bf16lo(wd[i]);
            w[2 * i + 1] = bf16hi(wd[i]);
            amax_b = fmaxf(amax_b, fmaxf(fabsf(w[2 * i]), fabsf(w[2 * i + 1])));
        }
        const float t = __fdiv_rn(amax_b, d);
        const uint32_t sb = round_mode == QERL_SCALE_ROUND_NEAREST_EVEN ? e4m3_rne(t) : e4m3_ceil(t);
        const float denom = __fmul_rn(e4m3_to_float(sb), s_t);
        uint32_t lo = 0, hi = 0;
        if (sb != 0u) {
#pragma unroll
            for (int i = 0; i < 8; ++i) lo |= e2m1_code(__fdiv_rn(w[i], denom)) << (4 * i);
#pragma unroll
            for (int i = 0; i < 8; ++i) hi |= e2m1_code(__fdiv_rn(w[8 + i], denom)) << (4 * i);
        }
        *reinterpret_cast<uint2 *>(codes + row * (K / 2) + b * 8) = make_uint2(lo, hi);
        scales[row * bpr + b] = (uint8_t)sb;
    }
}

// MXFP4 (bitsofall "NVFP4" section: MXFP4's blocks are 32 values with a
// power-of-two scale; OCP MX rule for that scale): one 32-block per thread,
// e = floor(log2(amax)) - 2 clamped to [-127, 127] (all-zero block: -127),
// scale byte e + 127, codes = E2M1 nearest of w * 2^-e.  One pass over W.
__global__ void __launch_bounds__(kQuantThreads)
    mx_quantize_kernel(const __nv_bfloat16 *__restrict__ W, int64_t N, int64_t K, int64_t ldw,
                       uint8_t *__restrict__ codes, uint8_t *__restrict__ scales, unsigned int *err)
{
    const int64_t bpr = K / 32;
    const int64_t nblk = N * bpr;
    for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nblk;
         blk += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = blk / bpr, b = blk - row * bpr;
        const __nv_bfloat16 *src = W + row * ldw + b * 32;
        uint4 u[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) u[v] = ld_stream(src + 8 * v);
        uint32_t m = 0;
#pragma unroll
        for (int v = 0; v < 4; ++v) m = max(max(m, mag2(u[v].x)), max(mag2(u[v].y), max(mag2(u[v].z), mag2(u[v].w))));
        if (m >= 0x7F80u) {  // Inf or NaN in the block
            latch_error(err, QERL_ERR_NONFINITE);
            continue;
        }
        int e = -127;
        if (m != 0u) {
            int ex;
            frexpf(__uint_as_float(m << 16), &ex);  // amax = f 2^ex, f in [0.5, 1)
            e = min(127, max(-127, ex - 3));
        }
        uint32_t wc[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint32_t wd[4] = {u[v].x, u[v].y, u[v].z, u[v].w};
            uint32_t c = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                c |= (e2m1_code(ldexpf(bf16lo(wd[i]), -e)) | (e2m1_code(ldexpf(bf16hi(wd[i]), -e)) << 4)) << (8 * i);
            wc[v] = c;
        }
        *reinterpret_cast<uint4 *>(codes + row * (K / 2) + b * 16) = make_uint4(wc[0], wc[1], wc[2], wc[3]);
        scales[row * bpr + b] = (uint8_t)(e + 127);
    }
}

__global__ void dequantize_kernel(const uint8_t *__restrict__ codes, const uint8_t *__restrict__ scales,
                                  const float *__restrict__ tensor_scale, int64_t N, int64_t K,
                                  __nv_bfloat16 *__restrict__ out, int apply_ts)
{
    const int64_t bpr = K / 16, nblk = N * bpr;
    const float s_t = apply_ts ? *tensor_scale : 1.0f;
    for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nblk;
         blk += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = blk / bpr, b = blk - row * bpr;
        const uint2 c = *reinterpret_cast<const uint2 *>(codes + row * (K / 2) + b * 8);
        const float sc = e4m3_to_float(scales[row * bpr + b]);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t word = i < 4 ? c.x : c.y;
            const uint32_t byte = (word >> (8 * (i & 3))) & 0xFFu;
            float v0 = e2m1_to_float(byte & 15u) * sc, v1 = e2m1_to_float(byte >> 4) * sc;
            if (apply_ts) {
                v0 = __fmul_rn(v0, s_t);
                v1 = __fmul_rn(v1, s_t);
            }
            const __nv_bfloat162 p = __floats2bfloat162_rn(v0, v1);
            o[i] = *reinterpret_cast<const uint32_t *>(&p);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(out + row * K + b * 16);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

}  // namespace

// Launches the two quantizer passes with partials in `partial_ws`
// (>= kMaxAmaxBlocks words).  Shared with the fixed-scratch entry point.
qerl_status launch_quantize(const void *W, int64_t N, int64_t K, int64_t ldw, uint8_t *codes, uint8_t *scales,
                            float *tensor_scale, int round_mode, uint32_t *partial_ws, cudaStream_t s)
{
    const int sms = num_sms();
    const int64_t vecs = N * (K / 8);
    int64_t g = (vecs + kAmaxThreads * 4 - 1) / (kAmaxThreads * 4);
    if (g > 4 * sms) g = 4 * sms;
    if (g > kMaxAmaxBlocks) g = kMaxAmaxBlocks;
    if (g < 1) g = 1;
    amax_kernel<<<(unsigned)g, kAmaxThreads, 0, s>>>(static_cast<const __nv_bfloat16 *>(W), N, K, ldw, partial_ws);
    QERL_TRY(launched());
    const int64_t nblk = N * (K / 16);
    int64_t q = (nblk + kQuantThreads - 1) / kQuantThreads;
    if (q > 16 * sms) q = 16 * sms;
    if (q < 1) q = 1;
    quantize_kernel<<<(unsigned)q, kQuantThreads, 0, s>>>(static_cast<const __nv_bfloat16 *>(W), N, K, ldw,
                                                            partial_ws, (int)g, codes, scales, tensor_scale,
                                                            round_mode, error_word());
    return launched();
}

qerl_status check_quantize_args(const void *W, int64_t N, int64_t K, int64_t ldw, const uint8_t *codes,
                                const uint8_t *scales, const float *tensor_scale, const qerl_quant_opts *opts)
{
    if (!W || !codes || !scales || !tensor_scale) return QERL_ERR_INVALID_ARG;
    if (N < 1 || K < 1 || ldw < K) return N < 0 || K < 0 ? QERL_ERR_INVALID_ARG : QERL_ERR_SHAPE;
    if (K % 16 != 0) return QERL_ERR_SHAPE;
    if (opts && opts->scale_round != QERL_SCALE_ROUND_UP && opts->scale_round != QERL_SCALE_ROUND_NEAREST_EVEN)
        return QERL_ERR_INVALID_ARG;
    if (!aligned16(W) || (ldw * 2) % 16 != 0 || (reinterpret_cast<uintptr_t>(codes) & 7u)) return QERL_ERR_ALIGN;
    return QERL_OK;
}

}  // namespace qerl

using namespace qerl;

extern "C" qerl_status qerl_nvfp4_quantize(const void *W, int64_t N, int64_t K, int64_t ldw, uint8_t *codes,
                                           uint8_t *scales, float *tensor_scale, const qerl_quant_opts *opts,
                                           void *ws, size_t ws_bytes, qerl_stream_t stream)
{
    QERL_TRY(check_quantize_args(W, N, K, ldw, codes, scales, tensor_scale, opts));
    if (!ws || ws_bytes < qerl_workspace_bytes(QERL_OP_QUANTIZE, 0, N, K, 0)) return QERL_ERR_WORKSPACE;
    QERL_TRY(check_device());
    return launch_quantize(W, N, K, ldw, codes, scales, tensor_scale, opts ? opts->scale_round : QERL_SCALE_ROUND_UP,
                           static_cast<uint32_t *>(ws), as_cuda(stream));
}

extern "C" qerl_status qerl_nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales, const float *tensor_scale,
                                             int64_t N, int64_t K, void *W_out, int apply_tensor_scale,
                                             qerl_stream_t stream)
{
    if (!codes || !scales || !W_out || (apply_tensor_scale && !tensor_scale)) return QERL_ERR_INVALID_ARG;
    if (N < 1 || K < 1) return N < 0 || K < 0 ? QERL_ERR_INVALID_ARG : QERL_ERR_SHAPE;
    if (K % 16 != 0) return QERL_ERR_SHAPE;
    if (!aligned16(W_out) || (reinterpret_cast<uintptr_t>(codes) & 7u)) return QERL_ERR_ALIGN;
    QERL_TRY(check_device());
    const int64_t nblk = N * (K / 16);
    int64_t g = (nblk + 255) / 256;
    if (g > 16 * num_sms()) g = 16 * num_sms();
    dequantize_kernel<<<(unsigned)g, 256, 0, as_cuda(stream)>>>(codes, scales, tensor_scale, N, K,
                                                                 static_cast<__nv_bfloat16 *>(W_out),
                                                                 apply_tensor_scale);
    return launched();
}

extern "C" qerl_status qerl_mxfp4_quantize(const void *W, int64_t N, int64_t K, int64_t ldw, uint8_t *codes,
                                           uint8_t *scales, qerl_stream_t stream)
{
    if (!W || !codes || !scales) return QERL_ERR_INVALID_ARG;
    if (N < 1 || K < 1 || ldw < K) return N < 0 || K < 0 ? QERL_ERR_INVALID_ARG : QERL_ERR_SHAPE;
    if (K % 32 != 0) return QERL_ERR_SHAPE;
    if (!aligned16(W) || (ldw * 2) % 16 != 0 || !aligned16(codes)) return QERL_ERR_ALIGN;
    QERL_TRY(check_device());
    const int64_t nblk = N * (K / 32);
    int64_t g = (nblk + kQuantThreads - 1) / kQuantThreads;
    if (g > 16 * num_sms()) g = 16 * num_sms();
    mx_quantize_kernel<<<(unsigned)g, kQuantThreads, 0, as_cuda(stream)>>>(static_cast<const __nv_bfloat16 *>(W), N, K,
                                                                          ldw, codes, scales, error_word());
    return launched();
}
