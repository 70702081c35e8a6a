// NVFP4 weight-only linear + LoRA: entry points, argument checks, and the
// CUDA-core (SIMT) kernels that cover every legal shape.
//
// Forward (bitsofall "QeRL: NVFP4-Quantized Reinforcement Learning", LoRA
// paragraph and "Implementation and Practical Details"):
//   y = s_t * x * w'^T + s * (x * A^T) * B^T,  w' = e2m1(code) * e4m3(scale)
// w' is exact in FP32 (and in bf16), so s_t is applied once, in FP32, in the
// epilogue.  Backward with the weight frozen:
//   v = dy * B,  dx = s_t * dy * w' + s * v * A,  dA = s * v^T * x,
//   dB = s * dy^T * (x * A^T).
#include <atomic>

#include "linear.cuh"
#include "packed_layout.cuh"

namespace qerl {
namespace {

std::atomic<int> g_algo{QERL_ALGO_AUTO};

// ------------------------------------------------------------ operand loaders
struct RowBF16 {  // (p, k) -> base[p * ld + k]
    const __nv_bfloat16 *base;
    int64_t ld;
    __device__ float operator()(int64_t p, int64_t k) const { return bf16f(base[p * ld + k]); }
};
struct ColBF16 {  // (p, k) -> base[k * ld + p]
    const __nv_bfloat16 *base;
    int64_t ld;
    __device__ float operator()(int64_t p, int64_t k) const { return bf16f(base[k * ld + p]); }
};
struct ColF32 {  // (p, k) -> base[k * ld + p]
    const float *base;
    int64_t ld;
    __device__ float operator()(int64_t p, int64_t k) const { return base[k * ld + p]; }
};
// w'(n, k) = e2m1(code) * e4m3(block scale), the weight without its tensor scale.
__device__ __forceinline__ float wprime(const uint8_t *codes, const uint8_t *scales, int64_t K, int64_t n, int64_t k,
                                        int packed)
{
    uint32_t c;
    if (packed) {
        const uint32_t w = reinterpret_cast<const uint32_t *>(codes)[n * (K / 8) + k / 8];
        c = packed_code(w, (int)(k & 7));
    } else {
        const uint32_t byte = codes[n * (K / 2) + k / 2];
        c = (k & 1) ? (byte >> 4) : (byte & 15u);
    }
    return e2m1_to_float(c) * e4m3_to_float(scales[n * (K / 16) + k / 16]);
}
struct WRow {  // (n, k)
    const uint8_t *codes, *scales;
    int64_t K;
    int packed;
    __device__ float operator()(int64_t n, int64_t k) const { return wprime(codes, scales, K, n, k, packed); }
};
struct WCol {  // (k, n)
    const uint8_t *codes, *scales;
    int64_t K;
    int packed;
    __device__ float operator()(int64_t k, int64_t n) const { return wprime(codes, scales, K, n, k, packed); }
};

// ------------------------------------------------------------ epilogues
struct StoreF32 {  // out[p, q] = (accumulate ? out : 0) + alpha * v
    float *out;
    int64_t ld;
    float alpha;
    int accumulate;
    __device__ void operator()(int64_t p, int64_t q, float v) const
    {
        float *o = out + p * ld + q;
        *o = accumulate ? fmaf(alpha, v, *o) : alpha * v;
    }
};
// y[m, n] = s_t * acc + s * sum_j t[m, j] * B[n, j]
struct FwdEpi {
    __nv_bfloat16 *y;
    int64_t N;
    const float *ts;
    const float *t;
    const __nv_bfloat16 *B;
    int r;
    float s;
    __device__ void operator()(int64_t m, int64_t n, float acc) const
    {
        float l = 0.0f;
        for (int j = 0; j < r; ++j) l = fmaf(t[m * r + j], bf16f(B[n * r + j]), l);
        y[m * N + n] = __float2bfloat16_rn(fmaf(s, l, *ts * acc));
    }
};
// dx[m, k] = s_t * acc + s * sum_j v[m, j] * A[j, k]
struct DxEpi {
    __nv_bfloat16 *dx;
    int64_t K;
    const float *ts;
    const float *v;
    const __nv_bfloat16 *A;
    int r;
    float s;
    __device__ void operator()(int64_t m, int64_t k, float acc) const
    {
        float l = 0.0f;
        for (int j = 0; j < r; ++j) l = fmaf(v[m * r + j], bf16f(A[(int64_t)j * K + k]), l);
        dx[m * K + k] = __float2bfloat16_rn(fmaf(s, l, *ts * acc));
    }
};

// C[p, q] = sum_k L(p, k) * R(q, k), 64x64 tiles, 16-deep k steps staged in
// shared memory as FP32, 4x4 outputs per thread.  Bounds-checked everywhere.
template <class LL, class LR, class EP>
__global__ void __launch_bounds__(256) simt_gemm(int64_t P, int64_t Q, int64_t Kd, LL lo, LR ro, EP ep)
{
    __shared__ float Ls[16][68];
    __shared__ float Rs[16][68];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int64_t p0 = (int64_t)blockIdx.y * 64, q0 = (int64_t)blockIdx.x * 64;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
    for (int64_t k0 = 0; k0 < Kd; k0 += 16) {
        for (int i = tid; i < 1024; i += 256) {
            const int pp = i >> 4, kk = i & 15;
            const int64_t k = k0 + kk, p = p0 + pp, q = q0 + pp;
            Ls[kk][pp] = (p < P && k < Kd) ? lo(p, k) : 0.0f;
            Rs[kk][pp] = (q < Q && k < Kd) ? ro(q, k) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = Ls[kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Rs[kk][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t p = p0 + ty + 16 * i, q = q0 + tx + 16 * j;
            if (p < P && q < Q) ep(p, q, acc[i][j]);
        }
}

template <class LL, class LR, class EP>
qerl_status run_gemm(int64_t P, int64_t Q, int64_t Kd, LL lo, LR ro, EP ep, cudaStream_t s)
{
    if (P <= 0 || Q <= 0) return QERL_OK;
    const dim3 grid((unsigned)((Q + 63) / 64), (unsigned)((P + 63) / 64));
    if (grid.y > 65535u) return QERL_ERR_SHAPE;
    simt_gemm<<<grid, 256, 0, s>>>(P, Q, Kd, lo, ro, ep);
    return launched();
}

qerl_status simt_fwd(const FwdArgs &a, char *ws, cudaStream_t s)
{
    float *t = a.t_out ? a.t_out : reinterpret_cast<float *>(ws);
    QERL_TRY(run_gemm(a.M, a.r, a.K, RowBF16{a.x, a.K}, RowBF16{a.A, a.K}, StoreF32{t, a.r, 1.0f, 0}, s));
    return run_gemm(a.M, a.N, a.K, RowBF16{a.x, a.K}, WRow{a.codes, a.scales, a.K, a.packed},
                    FwdEpi{a.y, a.N, a.tensor_scale, t, a.B, a.r, a.lora_scale}, s);
}

qerl_status simt_bwd(const BwdArgs &a, char *ws, cudaStream_t s)
{
    float *v = reinterpret_cast<float *>(ws);
    float *u = reinterpret_cast<float *>(ws + round256(size_t(a.M) * a.r * sizeof(float)));
    QERL_TRY(run_gemm(a.M, a.r, a.N, RowBF16{a.dy, a.N}, ColBF16{a.B, a.r}, StoreF32{v, a.r, 1.0f, 0}, s));
    if (a.dx)
        QERL_TRY(run_gemm(a.M, a.K, a.N, RowBF16{a.dy, a.N}, WCol{a.codes, a.scales, a.K, a.packed},
                          DxEpi{a.dx, a.K, a.tensor_scale, v, a.A, a.r, a.lora_scale}, s));
    if (a.dA)
        QERL_TRY(run_gemm((int64_t)a.r, a.K, a.M, ColF32{v, a.r}, ColBF16{a.x, a.K},
                          StoreF32{a.dA, a.K, a.lora_scale, a.accumulate}, s));
    if (a.dB) {
        const float *uu = a.t_saved;
        if (!uu) {
            QERL_TRY(run_gemm(a.M, a.r, a.K, RowBF16{a.x, a.K}, RowBF16{a.A, a.K}, StoreF32{u, a.r, 1.0f, 0}, s));
            uu = u;
        }
        QERL_TRY(run_gemm(a.N, (int64_t)a.r, a.M, ColBF16{a.dy, a.N}, ColF32{uu, a.r},
                          StoreF32{a.dB, a.r, a.lora_scale, a.accumulate}, s));
    }
    return QERL_OK;
}

qerl_status check_common(int64_t M, int64_t K, int64_t N, const uint8_t *codes, const uint8_t *scales,
                         const float *ts, const void *A, const void *B, int r)
{
    if (!codes || !scales || !ts || !A || !B) return QERL_ERR_INVALID_ARG;
    if (M < 0 || K < 1 || N < 1) return QERL_ERR_INVALID_ARG;
    if (K % 16 != 0 || r < 1 || r > 256) return QERL_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(codes) & 15u) || !aligned16(A) || !aligned16(B)) return QERL_ERR_ALIGN;
    return QERL_OK;
}

}  // namespace

size_t linear_fwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r)
{
    const size_t simt = round256(size_t(M) * r * sizeof(float));
    const size_t tc = tc_fwd_ws_bytes(M, N, K, r);
    return simt > tc ? simt : tc;
}

size_t linear_bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r)
{
    const size_t simt = 2 * round256(size_t(M) * r * sizeof(float));
    const size_t tc = tc_bwd_ws_bytes(M, N, K, r);
    return simt > tc ? simt : tc;
}

qerl_status linear_fwd_fixed_ws(const void *x, int64_t M, int64_t K, int64_t N, const uint8_t *codes,
                                const uint8_t *scales, const float *tensor_scale, const void *A, const void *B, int r,
                                float lora_scale, void *y, float *t_out, size_t ws_cap,
                                qerl_status (*get_ws)(void **), cudaStream_t s)
{
    QERL_TRY(check_common(M, K, N, codes, scales, tensor_scale, A, B, r));
    if (M == 0) return QERL_OK;
    if (!x || !y) return QERL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y) || (t_out && !aligned16(t_out))) return QERL_ERR_ALIGN;
    const size_t need = linear_fwd_ws_bytes(M, N, K, r);
    if (need > ws_cap) return QERL_ERR_TOO_LARGE;
    QERL_TRY(check_device());
    void *ws = nullptr;
    QERL_TRY(get_ws(&ws));
    const FwdArgs a{static_cast<const __nv_bfloat16 *>(x), M, K, N, codes, scales, tensor_scale,
                    static_cast<const __nv_bfloat16 *>(A), static_cast<const __nv_bfloat16 *>(B), r,
                    lora_scale, static_cast<__nv_bfloat16 *>(y), t_out};
    if (g_algo.load() != QERL_ALGO_SIMT) {
        const qerl_status st = tc_linear_fwd(a, static_cast<char *>(ws), ws_cap, s);
        if (st != QERL_ERR_SHAPE) return st;
    }
    return simt_fwd(a, static_cast<char *>(ws), s);
}

}  // namespace qerl

using namespace qerl;

extern "C" qerl_status qerl_set_linear_algo(int algo)
{
    if (algo != QERL_ALGO_AUTO && algo != QERL_ALGO_SIMT && algo != QERL_ALGO_TCGEN05) return QERL_ERR_INVALID_ARG;
    g_algo.store(algo);
    return QERL_OK;
}

namespace {

qerl_status fwd_entry(const void *x, int64_t M, int64_t K, int64_t N, const uint8_t *codes, const uint8_t *scales,
                      const float *tensor_scale, const void *A, const void *B, int r, float lora_scale, void *y,
                      float *t_out, void *ws, size_t ws_bytes, qerl_stream_t stream, int packed)
{
    QERL_TRY(check_common(M, K, N, codes, scales, tensor_scale, A, B, r));
    if (M == 0) return QERL_OK;  // x, y may be NULL for an empty batch
    if (!x || !y) return QERL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y) || (t_out && !aligned16(t_out))) return QERL_ERR_ALIGN;
    if (!ws || ws_bytes < linear_fwd_ws_bytes(M, N, K, r)) return QERL_ERR_WORKSPACE;
    QERL_TRY(check_device());
    const FwdArgs a{static_cast<const __nv_bfloat16 *>(x), M, K, N, codes, scales, tensor_scale,
                    static_cast<const __nv_bfloat16 *>(A), static_cast<const __nv_bfloat16 *>(B), r,
                    lora_scale, static_cast<__nv_bfloat16 *>(y), t_out, packed};
    cudaStream_t s = as_cuda(stream);
    if (g_algo.load() != QERL_ALGO_SIMT) {
        const qerl_status st = tc_linear_fwd(a, static_cast<char *>(ws), ws_bytes, s);
        if (st != QERL_ERR_SHAPE) return st;
    }
    return simt_fwd(a, static_cast<char *>(ws), s);
}

qerl_status bwd_entry(const void *dy, const void *x, int64_t M, int64_t K, int64_t N, const uint8_t *codes,
                      const uint8_t *scales, const float *tensor_scale, const void *A, const void *B, int r,
                      float lora_scale, const float *t_saved, void *dx, float *dA, float *dB, int accumulate_grads,
                      void *ws, size_t ws_bytes, qerl_stream_t stream, int packed)
{
    QERL_TRY(check_common(M, K, N, codes, scales, tensor_scale, A, B, r));
    if (M > 0 && (!dy || !x)) return QERL_ERR_INVALID_ARG;
    if ((M > 0 && (!aligned16(dy) || !aligned16(x))) || (dx && !aligned16(dx)) || (dA && !aligned16(dA)) ||
        (dB && !aligned16(dB)) || (t_saved && !aligned16(t_saved)))
        return QERL_ERR_ALIGN;
    if (M == 0) {  // empty sums: dA = 0, dB = 0 unless accumulating
        if (accumulate_grads) return QERL_OK;
        QERL_TRY(check_device());
        cudaStream_t s0 = as_cuda(stream);
        if (dA && cudaMemsetAsync(dA, 0, size_t(r) * K * sizeof(float), s0) != cudaSuccess) return QERL_ERR_CUDA;
        if (dB && cudaMemsetAsync(dB, 0, size_t(N) * r * sizeof(float), s0) != cudaSuccess) return QERL_ERR_CUDA;
        return QERL_OK;
    }
    if (!ws || ws_bytes < linear_bwd_ws_bytes(M, N, K, r)) return QERL_ERR_WORKSPACE;
    QERL_TRY(check_device());
    const BwdArgs a{static_cast<const __nv_bfloat16 *>(dy), static_cast<const __nv_bfloat16 *>(x), M, K, N, codes,
                    scales, tensor_scale, static_cast<const __nv_bfloat16 *>(A),
                    static_cast<const __nv_bfloat16 *>(B), r, lora_scale, t_saved,
                    static_cast<__nv_bfloat16 *>(dx), dA, dB, accumulate_grads, packed};
    cudaStream_t s = as_cuda(stream);
    if (g_algo.load() != QERL_ALGO_SIMT) {
        const qerl_status st = tc_linear_bwd(a, static_cast<char *>(ws), ws_bytes, s);
        if (st != QERL_ERR_SHAPE) return st;
    }
    return simt_bwd(a, static_cast<char *>(ws), s);
}

}  // namespace

extern "C" qerl_status qerl_nvfp4_lora_linear_fwd(const void *x, int64_t M, int64_t K, int64_t N,
                                                  const uint8_t *codes, const uint8_t *scales,
                                                  const float *tensor_scale, const void *A, const void *B, int r,
                                                  float lora_scale, void *y, float *t_out, void *ws, size_t ws_bytes,
                                                  qerl_stream_t stream)
{
    return fwd_entry(x, M, K, N, codes, scales, tensor_scale, A, B, r, lora_scale, y, t_out, ws, ws_bytes, stream, 0);
}

extern "C" qerl_status qerl_nvfp4_lora_linear_fwd_packed(const void *x, int64_t M, int64_t K, int64_t N,
                                                         const uint8_t *packed_codes, const uint8_t *scales,
                                                         const float *tensor_scale, const void *A, const void *B,
                                                         int r, float lora_scale, void *y, float *t_out, void *ws,
                                                         size_t ws_bytes, qerl_stream_t stream)
{
    return fwd_entry(x, M, K, N, packed_codes, scales, tensor_scale, A, B, r, lora_scale, y, t_out, ws, ws_bytes,
                     stream, 1);
}

extern "C" qerl_status qerl_nvfp4_lora_linear_bwd(const void *dy, const void *x, int64_t M, int64_t K, int64_t N,
                                                  const uint8_t *codes, const uint8_t *scales,
                                                  const float *tensor_scale, const void *A, const void *B, int r,
                                                  float lora_scale, const float *t_saved, void *dx, float *dA,
                                                  float *dB, int accumulate_grads, void *ws, size_t ws_bytes,
                                                  qerl_stream_t stream)
{
    return bwd_entry(dy, x, M, K, N, codes, scales, tensor_scale, A, B, r, lora_scale, t_saved, dx, dA, dB,
                     accumulate_grads, ws, ws_bytes, stream, 0);
}

extern "C" qerl_status qerl_nvfp4_lora_linear_bwd_packed(const void *dy, const void *x, int64_t M, int64_t K,
                                                         int64_t N, const uint8_t *packed_codes,
                                                         const uint8_t *scales, const float *tensor_scale,
                                                         const void *A, const void *B, int r, float lora_scale,
                                                         const float *t_saved, void *dx, float *dA, float *dB,
                                                         int accumulate_grads, void *ws, size_t ws_bytes,
                                                         qerl_stream_t stream)
{
    return bwd_entry(dy, x, M, K, N, packed_codes, scales, tensor_scale, A, B, r, lora_scale, t_saved, dx, dA, dB,
                     accumulate_grads, ws, ws_bytes, stream, 1);
}
