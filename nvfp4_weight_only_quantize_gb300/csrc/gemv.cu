// CUDA-core path of the forward for one or two tokens (rollout decode at the
// smallest batches):
//     y[m, n] = bf16(s_t 2^c * sum_k w''[n, k] x[m, k] + s * sum_j t[m, j] B[n, j])
// with w'' = e2m1 * e4m3 * 2^-c (exact bf16; the tensor-core kernels' dequant)
// and t = x A^T in FP32 from the LoRA down-projection kernel launched just
// before.  At one or two tokens there are one or two FMAs per weight, so the
// tensor cores would idle; this kernel streams the weight through registers.
//
// A warp owns GEMV_ROWS adjacent output rows at a time.  Lane l reads the
// 16-byte code chunks l, l + 32, ... of each row (32 weights per chunk, one
// coalesced 512-byte load per warp and row), GEMV_UNROLL chunks per row in
// flight.  x is staged once per CTA in shared memory as FP32, each run of 32
// values XOR-swizzled in 16-byte granules (granule g of chunk ch stored at
// g ^ (ch & 7)) so that 32 lanes reading 32 different chunks hit distinct bank
// groups; one staged read serves all rows of the warp.  Partial sums are
// reduced by warp shuffles in a fixed order (deterministic).
#include "dequant.cuh"
#include "linear.cuh"

namespace qerl {
namespace {

constexpr int GEMV_WARPS = 16;
constexpr int GEMV_ROWS = 2;    // output rows per warp
constexpr int GEMV_UNROLL = 4;  // code chunks in flight per lane and row
constexpr int GEMV_MAX_R = 256;

__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int MT, bool PACKED>
__global__ void __launch_bounds__(GEMV_WARPS * 32, 1)
    gemv_kernel(const __nv_bfloat16 *__restrict__ x, int K, int N, const uint8_t *__restrict__ codes,
                const uint8_t *__restrict__ scales, const float *__restrict__ ts, const float *__restrict__ t,
                const __nv_bfloat16 *__restrict__ B, int r, float s, __nv_bfloat16 *__restrict__ y)
{
    extern __shared__ float4 xs4[];  // [MT][K / 4] swizzled, then t [MT][r]
    float *t_s = reinterpret_cast<float *>(xs4 + (size_t)MT * (K / 4));
    const int chunks = K / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_step = gridDim.x * GEMV_WARPS * GEMV_ROWS;
    int n0 = (blockIdx.x * GEMV_WARPS + warp) * GEMV_ROWS;

    uint4 q[GEMV_ROWS][GEMV_UNROLL];
    uint32_t sc[GEMV_ROWS][GEMV_UNROLL];
    // Loads of one batch of chunks (rows past N read row N - 1; not stored).
    auto load = [&](int n, int base) {
#pragma unroll
        for (int i = 0; i < GEMV_ROWS; ++i) {
            const int nr = n + i < N ? n + i : N - 1;
            const uint8_t *crow = codes + (size_t)nr * (K / 2);
            const uint16_t *srow = reinterpret_cast<const uint16_t *>(scales + (size_t)nr * (K / 16));
#pragma unroll
            for (int u = 0; u < GEMV_UNROLL; ++u) {
                const int ch = base + u * 32 + lane;
                q[i][u] = ch < chunks ? ld_stream16(crow + (size_t)ch * 16) : make_uint4(0u, 0u, 0u, 0u);
                sc[i][u] = ch < chunks ? (uint32_t)__ldg(srow + ch) : 0u;
            }
        }
    };

    pdl_trigger();
    // The weight is frozen while a forward runs: its first batch is fetched
    // before waiting for the preceding work (x, t).
    if (n0 < N) load(n0, 0);
    pdl_wait();
    for (int i = threadIdx.x; i < MT * (K / 8); i += blockDim.x) {
        const int m = i / (K / 8), v = i % (K / 8);  // 8 values: granules 2v, 2v + 1 of the row
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)m * K) + v);
        const int ch = v >> 2, g0 = (v & 3) * 2;
        float4 *row = xs4 + (size_t)m * (K / 4) + ch * 8;
        row[g0 ^ (ch & 7)] = make_float4(bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y));
        row[(g0 + 1) ^ (ch & 7)] = make_float4(bf16lo(u.z), bf16hi(u.z), bf16lo(u.w), bf16hi(u.w));
    }
    for (int i = threadIdx.x; i < MT * r; i += blockDim.x) t_s[i] = t[i];
    __syncthreads();
    const float st = *ts;
    const int c = tc_exponent_offset(st);
    const float pow2 = pow2f(126 - c), ysc = st * pow2f(c);

    for (bool fetched = true; n0 < N; n0 += row_step, fetched = false) {
        float acc[GEMV_ROWS][MT];
#pragma unroll
        for (int i = 0; i < GEMV_ROWS; ++i)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[i][m] = 0.0f;
        for (int base = 0; base < chunks; base += 32 * GEMV_UNROLL) {
            if (base > 0 || !fetched) load(n0, base);  // the row's first batch came before the wait
#pragma unroll
            for (int u = 0; u < GEMV_UNROLL; ++u) {
                const int ch = base + u * 32 + lane;
                if (ch >= chunks) break;
                uint32_t w[GEMV_ROWS][16];
#pragma unroll
                for (int i = 0; i < GEMV_ROWS; ++i) {
                    const uint32_t f0 = scale_factor_bf16x2(sc[i][u] << 20, pow2);  // block 2 ch
                    const uint32_t f1 = scale_factor_bf16x2(sc[i][u] << 12, pow2);  // block 2 ch + 1
                    dequant_word<PACKED>(q[i][u].x, f0, w[i] + 0);
                    dequant_word<PACKED>(q[i][u].y, f0, w[i] + 4);
                    dequant_word<PACKED>(q[i][u].z, f1, w[i] + 8);
                    dequant_word<PACKED>(q[i][u].w, f1, w[i] + 12);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float4 *row = xs4 + (size_t)m * (K / 4) + ch * 8;
#pragma unroll
                    for (int g = 0; g < 8; ++g) {  // granule g: k = 32 ch + 4 g .. + 3 (pairs 2g, 2g + 1)
                        const float4 xv = row[g ^ (ch & 7)];
#pragma unroll
                        for (int i = 0; i < GEMV_ROWS; ++i) {
                            float a = acc[i][m];
                            a = fmaf(__uint_as_float(w[i][2 * g] << 16), xv.x, a);
                            a = fmaf(bf16hi(w[i][2 * g]), xv.y, a);
                            a = fmaf(__uint_as_float(w[i][2 * g + 1] << 16), xv.z, a);
                            a = fmaf(bf16hi(w[i][2 * g + 1]), xv.w, a);
                            acc[i][m] = a;
                        }
                    }
                }
            }
        }
        // fixed-order warp reductions, then the LoRA term s sum_j t[m, j] B[n, j]
#pragma unroll
        for (int i = 0; i < GEMV_ROWS; ++i) {
            const int n = n0 + i;
            if (n >= N) break;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float v = acc[i][m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                float l = 0.0f;
                for (int j = lane; j < r; j += 32) l = fmaf(t_s[m * r + j], bf16f(B[(size_t)n * r + j]), l);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
                if (lane == 0) y[(size_t)m * N + n] = __float2bfloat16_rn(fmaf(s, l, v * ysc));
            }
        }
    }
}

size_t gemv_smem(int64_t M, int64_t K, int r) { return (size_t)M * (K + r) * sizeof(float); }

template <int MT>
qerl_status launch_gemv(const FwdArgs &a, const float *t, cudaStream_t s)
{
    const size_t smem = gemv_smem(MT, a.K, a.r);
    auto kernel = a.packed ? gemv_kernel<MT, true> : gemv_kernel<MT, false>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return QERL_ERR_CUDA;
    int64_t g = (a.N + GEMV_WARPS * GEMV_ROWS - 1) / (GEMV_WARPS * GEMV_ROWS);
    if (g > num_sms()) g = num_sms();
    // always a programmatic dependent of the down-projection launched before it
    return launched(launch_k(kernel, dim3((unsigned)g), dim3(GEMV_WARPS * 32), smem, s, true, a.x, (int)a.K,
                             (int)a.N, a.codes, a.scales, a.tensor_scale, t, a.B, a.r, a.lora_scale, a.y));
}

inline int gemv_r_pad(int r) { return (r + 1) & ~1; }

}  // namespace

bool gemv_applies(int64_t M, int64_t N, int64_t K, int r)
{
    return M >= 1 && M <= 2 && N >= 1 && N < (int64_t(1) << 31) && K >= 32 && K % 32 == 0 && K < (1 << 30) &&
           r >= 1 && r <= GEMV_MAX_R && gemv_smem(M, K, r) <= 200 * 1024;
}

size_t gemv_ws_bytes(int64_t M, int64_t N, int64_t K, int r)
{
    if (!gemv_applies(M, N, K, r)) return 0;
    return round256(size_t(M) * r * sizeof(float)) + round256(size_t(M) * gemv_r_pad(r) * 2);
}

qerl_status gemv_fwd(const FwdArgs &a, char *ws, size_t ws_bytes, cudaStream_t s)
{
    if (!gemv_applies(a.M, a.N, a.K, a.r)) return QERL_ERR_SHAPE;
    if (ws_bytes < gemv_ws_bytes(a.M, a.N, a.K, a.r)) return QERL_ERR_WORKSPACE;
    float *t = a.t_out ? a.t_out : reinterpret_cast<float *>(ws);
    __nv_bfloat16 *u = reinterpret_cast<__nv_bfloat16 *>(ws + round256(size_t(a.M) * a.r * sizeof(float)));
    QERL_TRY(lora_down_small(a, gemv_r_pad(a.r), t, u, g_chain.load() != 0, s));
    return a.M == 1 ? launch_gemv<1>(a, t, s) : launch_gemv<2>(a, t, s);
}

}  // namespace qerl
