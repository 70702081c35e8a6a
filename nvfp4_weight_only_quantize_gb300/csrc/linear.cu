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
#include <algorithm>
#include <atomic>

#include "linear.cuh"
#include "packed_layout.cuh"

namespace qerl {
namespace {

std::atomic<int> g_algo{QERL_ALGO_AUTO};

// ------------------------------------------------------------ operand loaders
struct RowBF16 {  // (p, k) -> base[p * ld + k]
    static constexpr bool kVec8 = true;  // 8 consecutive k in one 16-byte load
    const __nv_bfloat16 *base;
    int64_t ld;
    __device__ float operator()(int64_t p, int64_t k) const { return bf16f(base[p * ld + k]); }
    __device__ bool vec_ok() const { return (ld & 7) == 0 && (reinterpret_cast<uintptr_t>(base) & 15) == 0; }
    __device__ uint4 load8(int64_t p, int64_t k) const
    {
        return __ldg(reinterpret_cast<const uint4 *>(base + p * ld + k));
    }
};
struct ColBF16 {  // (p, k) -> base[k * ld + p]
    static constexpr bool kColMajor = true;
    static constexpr bool kVec8 = true;  // 8 consecutive p in one 16-byte load
    const __nv_bfloat16 *base;
    int64_t ld;
    __device__ float operator()(int64_t p, int64_t k) const { return bf16f(base[k * ld + p]); }
    __device__ bool vec_ok() const { return (ld & 7) == 0 && (reinterpret_cast<uintptr_t>(base) & 15) == 0; }
    __device__ uint4 load8(int64_t p, int64_t k) const
    {
        return __ldg(reinterpret_cast<const uint4 *>(base + k * ld + p));
    }
};
struct ColF32 {  // (p, k) -> base[k * ld + p]
    static constexpr bool kColMajor = true;
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
// MXFP4 weight element: e2m1(code) * 2^(E8M0 byte - 127), blocks of 32 along k.
__device__ __forceinline__ float wprime_mx(const uint8_t *codes, const uint8_t *scales, int64_t K, int64_t n,
                                          int64_t k)
{
    const uint32_t byte = codes[n * (K / 2) + k / 2];
    const uint32_t c = (k & 1) ? (byte >> 4) : (byte & 15u);
    const uint32_t b = scales[n * (K / 32) + k / 32];
    // 2^(b-127); b = 0: 2^-127; b = 255: NaN (the OCP NaN scale)
    const float sc = b == 255u ? __uint_as_float(0x7FC00000u) : b != 0u ? __uint_as_float(b << 23) : __uint_as_float(1u << 22);
    return e2m1_to_float(c) * sc;
}
struct WRowMX {  // (n, k)
    const uint8_t *codes, *scales;
    int64_t K;
    __device__ float operator()(int64_t n, int64_t k) const { return wprime_mx(codes, scales, K, n, k); }
};
struct RowF32 {  // (p, k) -> base[p * ld + k]
    const float *base;
    int64_t ld;
    __device__ float operator()(int64_t p, int64_t k) const { return base[p * ld + k]; }
};
struct WRow {  // (n, k)
    const uint8_t *codes, *scales;
    int64_t K;
    int packed;
    __device__ float operator()(int64_t n, int64_t k) const { return wprime(codes, scales, K, n, k, packed); }
};
struct WCol {  // (k, n)
    static constexpr bool kColMajor = true;
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
    __device__ void operator()(int64_t p, int64_t q, float v, int) const
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
    __device__ void operator()(int64_t m, int64_t n, float acc, int) const
    {
        float l = 0.0f;
        for (int j = 0; j < r; ++j) l = fmaf(t[m * r + j], bf16f(B[n * r + j]), l);
        y[m * N + n] = __float2bfloat16_rn(fmaf(s, l, *ts * acc));
    }
};
// The forward's epilogue with FP32 LoRA B and/or no tensor scale (ts == null: 1).
struct FwdEpiF32 {
    __nv_bfloat16 *y;
    int64_t N;
    const float *ts;
    const float *t;
    const float *B32;            // FP32 [N, r], or null
    const __nv_bfloat16 *B16;    // bf16 [N, r] when B32 is null
    int r;
    float s;
    __device__ void operator()(int64_t m, int64_t n, float acc, int) const
    {
        float l = 0.0f;
        for (int j = 0; j < r; ++j) l = fmaf(t[m * r + j], B32 ? B32[n * r + j] : bf16f(B16[n * r + j]), l);
        y[m * N + n] = __float2bfloat16_rn(fmaf(s, l, (ts ? *ts : 1.0f) * acc));
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
    __device__ void operator()(int64_t m, int64_t k, float acc, int) const
    {
        float l = 0.0f;
        for (int j = 0; j < r; ++j) l = fmaf(v[m * r + j], bf16f(A[(int64_t)j * K + k]), l);
        dx[m * K + k] = __float2bfloat16_rn(fmaf(s, l, *ts * acc));
    }
};

// Operands contiguous along p (rather than k) are staged with consecutive
// threads on consecutive p, so that their loads coalesce.
template <class T, class = void>
struct col_major {
    static constexpr bool value = false;
};
template <class T>
struct col_major<T, decltype((void)T::kColMajor)> {
    static constexpr bool value = T::kColMajor;
};

template <class T, class = void>
struct vec8 {
    static constexpr bool value = false;
};
template <class T>
struct vec8<T, decltype((void)T::kVec8)> {
    static constexpr bool value = T::kVec8;
};

__device__ __forceinline__ void unpack8(uint4 u, float *f)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        f[2 * e] = __uint_as_float(w[e] << 16);
        f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}

template <class L>
__device__ __forceinline__ void stage16(float (&S)[16][68], const L &ld, int tid, int64_t p0, int64_t P, int64_t k0,
                                        int64_t kend)
{
    if constexpr (vec8<L>::value) {
        // A 64 x 16 block as 128 16-byte loads, one per thread of the first half;
        // rows past P read as zeros (for p-contiguous operands P % 8 == 0, so a
        // vector never straddles P).
        if (ld.vec_ok() && k0 + 16 <= kend && (!col_major<L>::value || (P & 7) == 0)) {
            if (tid < 128) {
                float f[8];
                if (col_major<L>::value) {  // 8 p at one k
                    const int kk = tid >> 3, pp = (tid & 7) * 8;
                    if (p0 + pp < P) {
                        unpack8(ld.load8(p0 + pp, k0 + kk), f);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = 0.0f;
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) S[kk][pp + e] = f[e];
                } else {  // 8 k at one p
                    const int pp = tid >> 1, kk = (tid & 1) * 8;
                    if (p0 + pp < P) {
                        unpack8(ld.load8(p0 + pp, k0 + kk), f);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = 0.0f;
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) S[kk + e][pp] = f[e];
                }
            }
            return;
        }
    }
    for (int i = tid; i < 1024; i += 256) {
        const int pp = col_major<L>::value ? (i & 63) : (i >> 4);
        const int kk = col_major<L>::value ? (i >> 6) : (i & 15);
        const int64_t k = k0 + kk, p = p0 + pp;
        S[kk][pp] = (p < P && k < kend) ? ld(p, k) : 0.0f;
    }
}

// C[p, q] = sum_k L(p, k) * R(q, k) over k in [kbeg, kend) with kbeg, kend from
// blockIdx.z (split k: each split writes its own partial), 64x64 tiles,
// 16-deep k steps staged in shared memory as FP32, 4x4 outputs per thread.
// Bounds-checked everywhere.
template <class LL, class LR, class EP>
__global__ void __launch_bounds__(256) simt_gemm(int64_t P, int64_t Q, int64_t Kd, int64_t kchunk, LL lo, LR ro,
                                                 EP ep)
{
    __shared__ float Ls[16][68];
    __shared__ float Rs[16][68];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int64_t p0 = (int64_t)blockIdx.y * 64, q0 = (int64_t)blockIdx.x * 64;
    const int64_t kbeg = (int64_t)blockIdx.z * kchunk;
    const int64_t kend = kbeg + kchunk < Kd ? kbeg + kchunk : Kd;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
    for (int64_t k0 = kbeg; k0 < kend; k0 += 16) {
        stage16(Ls, lo, tid, p0, P, k0, kend);
        stage16(Rs, ro, tid, q0, Q, k0, kend);
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
            if (p < P && q < Q) ep(p, q, acc[i][j], (int)blockIdx.z);
        }
}

// sum_{z < splits} p[z * stride], in z order, eight loads in flight at a time.
__device__ __forceinline__ float sum_splits(const float *p, int64_t stride, int splits)
{
    float acc = 0.0f;
    for (int z0 = 0; z0 < splits; z0 += 8) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = z0 + e < splits ? __ldcg(p + (int64_t)(z0 + e) * stride) : 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc += v[e];
    }
    return acc;
}

// Split-k partial: part[z][p][q] = acc.
struct PartialEpi {
    float *part;
    int64_t P, Q;
    __device__ void operator()(int64_t p, int64_t q, float v, int z) const { part[(z * P + p) * Q + q] = v; }
};
// Sum of the partials in split order (deterministic), then StoreF32's update.
__global__ void __launch_bounds__(256) split_reduce(const float *__restrict__ part, int splits, int64_t P, int64_t Q,
                                                    float *out, int64_t ld, float alpha, int accumulate)
{
    const int64_t n = P * Q;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = sum_splits(part + i, n, splits);
        float *o = out + (i / Q) * ld + (i % Q);
        *o = accumulate ? fmaf(alpha, v, *o) : alpha * v;
    }
}

template <class LL, class LR, class EP>
qerl_status run_gemm(int64_t P, int64_t Q, int64_t Kd, LL lo, LR ro, EP ep, cudaStream_t s)
{
    if (P <= 0 || Q <= 0) return QERL_OK;
    const dim3 grid((unsigned)((Q + 63) / 64), (unsigned)((P + 63) / 64));
    if (grid.y > 65535u) return QERL_ERR_SHAPE;
    simt_gemm<<<grid, 256, 0, s>>>(P, Q, Kd, Kd > 0 ? Kd : 1, lo, ro, ep);
    return launched();
}

// Split count for a StoreF32 product: enough 64x64 tiles x splits to fill the
// GPU twice over, at least 512 k per split, at most 32 splits.
int gemm_splits(int64_t P, int64_t Q, int64_t Kd)
{
    const int64_t tiles = ((P + 63) / 64) * ((Q + 63) / 64);
    int64_t sp = (2 * (int64_t)num_sms() + tiles - 1) / tiles;
    const int64_t kmax = Kd / 512;
    if (sp > kmax) sp = kmax;
    if (sp > 32) sp = 32;
    return sp < 1 ? 1 : (int)sp;
}
size_t gemm_split_ws(int64_t P, int64_t Q, int64_t Kd)
{
    const int sp = gemm_splits(P, Q, Kd);
    return sp > 1 ? round256(size_t(sp) * P * Q * sizeof(float)) : 0;
}

// C = StoreF32(sum_k L R) with k split over CTAs when the output is thin;
// part holds gemm_split_ws(P, Q, Kd) bytes.
template <class LL, class LR>
qerl_status run_gemm_store(int64_t P, int64_t Q, int64_t Kd, LL lo, LR ro, StoreF32 ep, float *part, cudaStream_t s)
{
    const int sp = gemm_splits(P, Q, Kd);
    if (sp == 1 || P <= 0 || Q <= 0) return run_gemm(P, Q, Kd, lo, ro, ep, s);
    const int64_t kchunk = ((Kd + sp - 1) / sp + 15) / 16 * 16;
    const int splits = (int)((Kd + kchunk - 1) / kchunk);
    const dim3 grid((unsigned)((Q + 63) / 64), (unsigned)((P + 63) / 64), (unsigned)splits);
    if (grid.y > 65535u) return QERL_ERR_SHAPE;
    simt_gemm<<<grid, 256, 0, s>>>(P, Q, Kd, kchunk, lo, ro, PartialEpi{part, P, Q});
    QERL_TRY(launched());
    int64_t g = (P * Q + 255) / 256;
    if (g > 8 * num_sms()) g = 8 * num_sms();
    split_reduce<<<(unsigned)g, 256, 0, s>>>(part, splits, P, Q, ep.out, ep.ld, ep.alpha, ep.accumulate);
    return launched();
}

qerl_status simt_fwd(const FwdArgs &a, char *ws, cudaStream_t s)
{
    float *t = a.t_out ? a.t_out : reinterpret_cast<float *>(ws);
    QERL_TRY(run_gemm(a.M, a.r, a.K, RowBF16{a.x, a.K}, RowBF16{a.A, a.K}, StoreF32{t, a.r, 1.0f, 0}, s));
    return run_gemm(a.M, a.N, a.K, RowBF16{a.x, a.K}, WRow{a.codes, a.scales, a.K, a.packed},
                    FwdEpi{a.y, a.N, a.tensor_scale, t, a.B, a.r, a.lora_scale}, s);
}

// ------------------------------------------------------------ thin products
// The LoRA products of the backward have one side of width r <= 64 and a long
// reduction; they are HBM-bound.  The tensor-core kernels of rank_tc.cu run
// them where their shape allows; these two CUDA-core kernels cover the rest,
// split over the reduction (partials summed in split order by split_reduce):
//   rows x rank:   P[z][m][j] = sum_{k in split z} X[m, k] * W(k, j)
//                  X bf16 [M, Kd] row-major; W(k, j) = Wkj[k * r + j] or Wjk[j * Kd + k]
//   wide x rank:   P[z][w][j] (or [j][w]) = sum_{m in split z} D[m, w] * T[m, j]
//                  D bf16 [M, Wd] row-major; T FP32 [M, r] row-major
constexpr int THIN_TK = 32;  // reduction depth per staged chunk
// rows (or wide columns) per CTA: 256 threads x 4 rows over r_pad / 8 rank groups
template <int R_PAD>
constexpr int thin_tr() { return 256 * 4 / (R_PAD / 8); }

// thin_tr<R_PAD>() rows x R_PAD (32 or 64) outputs per CTA; thread = 4 rows x 8 ranks.
template <bool WJK, int R_PAD>
__global__ void __launch_bounds__(256) thin_rows_kernel(const __nv_bfloat16 *__restrict__ X, int64_t M, int64_t Kd,
                                                        const __nv_bfloat16 *__restrict__ W, int r, int64_t kchunk,
                                                        float *__restrict__ part)
{
    constexpr int THIN_TR = thin_tr<R_PAD>(), r_pad = R_PAD;
    __shared__ __align__(16) __nv_bfloat16 Xs[THIN_TR][THIN_TK + 8];
    pdl_trigger();
    pdl_wait();  // chained launch: X and W follow the preceding work
    __shared__ __align__(16) float Ws[THIN_TK][68];
    const int tid = threadIdx.x;
    const int jg = tid % (r_pad / 8), rg = tid / (r_pad / 8);  // rank group (8), row group (4)
    const bool active = rg < THIN_TR / 4;
    const int64_t m0 = (int64_t)blockIdx.x * THIN_TR;
    const int64_t kbeg = (int64_t)blockIdx.y * kchunk;
    const int64_t kend = kbeg + kchunk < Kd ? kbeg + kchunk : Kd;
    float acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = 0.0f;
    // The next chunk is loaded into registers while the current one is used.
    constexpr int XV = THIN_TR * (THIN_TK / 8) / 256;  // 16-byte X vectors per thread
    constexpr int WV = THIN_TK * 64 / 256;             // W values per thread
    uint4 xr[XV];
    float wr[WV];
    auto load = [&](int64_t k0) {
#pragma unroll
        for (int e = 0; e < XV; ++e) {  // X: THIN_TR rows x 32 k (Kd % 8 == 0, chunks of 32 k)
            const int v = tid + 256 * e;
            const int row = v / (THIN_TK / 8), kk = (v % (THIN_TK / 8)) * 8;
            xr[e] = (m0 + row < M && k0 + kk < kend) ? __ldg(reinterpret_cast<const uint4 *>(X + (m0 + row) * Kd + k0 + kk))
                                                     : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int e = 0; e < WV; ++e) {  // W: 32 k x 64 ranks as FP32 (zeros past r and kend)
            const int i = tid + 256 * e;
            const int kk = WJK ? (i % THIN_TK) : (i / 64), j = WJK ? (i / THIN_TK) : (i % 64);
            wr[e] = (j < r && k0 + kk < kend) ? bf16f(WJK ? W[(int64_t)j * Kd + k0 + kk] : W[(k0 + kk) * r + j]) : 0.0f;
        }
    };
    if (kbeg < kend) load(kbeg);
    for (int64_t k0 = kbeg; k0 < kend; k0 += THIN_TK) {
#pragma unroll
        for (int e = 0; e < XV; ++e) {
            const int v = tid + 256 * e;
            *reinterpret_cast<uint4 *>(&Xs[v / (THIN_TK / 8)][(v % (THIN_TK / 8)) * 8]) = xr[e];
        }
#pragma unroll
        for (int e = 0; e < WV; ++e) {
            const int i = tid + 256 * e;
            Ws[WJK ? (i % THIN_TK) : (i / 64)][WJK ? (i / THIN_TK) : (i % 64)] = wr[e];
        }
        __syncthreads();
        if (k0 + THIN_TK < kend) load(k0 + THIN_TK);
        if (active) {
#pragma unroll
            for (int kk = 0; kk < THIN_TK; kk += 8) {
                float xv[4][8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(&Xs[rg * 4 + i][kk]);
                    unpack8(u, xv[i]);
                }
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8) {
                    const float4 w0 = *reinterpret_cast<const float4 *>(&Ws[kk + k8][jg * 8]);
                    const float4 w1 = *reinterpret_cast<const float4 *>(&Ws[kk + k8][jg * 8 + 4]);
                    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(xv[i][k8], wv[e], acc[i][e]);
                }
            }
        }
        __syncthreads();
    }
    if (!active) return;
    float *out = part + (int64_t)blockIdx.y * M * r;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + rg * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (jg * 8 + e < r) out[m * r + jg * 8 + e] = acc[i][e];
    }
}

// thin_tr<R_PAD>() wide columns x R_PAD ranks per CTA; thread = 4 wide x 8
// ranks.  Output partial [w][j] (WJ) or [j][w].
template <bool WJ, int R_PAD>
__global__ void __launch_bounds__(256) thin_wide_kernel(const __nv_bfloat16 *__restrict__ D, int64_t M, int64_t Wd,
                                                        const float *__restrict__ T, int r, int64_t mchunk,
                                                        float *__restrict__ part)
{
    constexpr int THIN_TR = thin_tr<R_PAD>(), r_pad = R_PAD;
    __shared__ __align__(16) __nv_bfloat16 Ds[THIN_TK][THIN_TR + 8];
    __shared__ __align__(16) float Ts[THIN_TK][68];
    const int tid = threadIdx.x;
    const int jg = tid % (r_pad / 8), wg = tid / (r_pad / 8);
    const bool active = wg < THIN_TR / 4;
    const int64_t w0 = (int64_t)blockIdx.x * THIN_TR;
    const int64_t mbeg = (int64_t)blockIdx.y * mchunk;
    const int64_t mend = mbeg + mchunk < M ? mbeg + mchunk : M;
    float acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = 0.0f;
    // The next chunk is loaded into registers while the current one is used.
    constexpr int DV = THIN_TK * (THIN_TR / 8) / 256;  // 16-byte D vectors per thread
    constexpr int TV = THIN_TK * 64 / 256;             // T values per thread
    uint4 dr[DV];
    float tr[TV];
    auto load = [&](int64_t mm0) {
#pragma unroll
        for (int e = 0; e < DV; ++e) {  // D: 32 m x THIN_TR w (Wd % 8 == 0)
            const int v = tid + 256 * e;
            const int mm = v / (THIN_TR / 8), ww = (v % (THIN_TR / 8)) * 8;
            dr[e] = (mm0 + mm < mend && w0 + ww < Wd) ? __ldg(reinterpret_cast<const uint4 *>(D + (mm0 + mm) * Wd + w0 + ww))
                                                       : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int e = 0; e < TV; ++e) {
            const int i = tid + 256 * e;
            const int mm = i / 64, j = i % 64;
            tr[e] = (j < r && mm0 + mm < mend) ? T[(mm0 + mm) * r + j] : 0.0f;
        }
    };
    if (mbeg < mend) load(mbeg);
    for (int64_t mm0 = mbeg; mm0 < mend; mm0 += THIN_TK) {
#pragma unroll
        for (int e = 0; e < DV; ++e) {
            const int v = tid + 256 * e;
            *reinterpret_cast<uint4 *>(&Ds[v / (THIN_TR / 8)][(v % (THIN_TR / 8)) * 8]) = dr[e];
        }
#pragma unroll
        for (int e = 0; e < TV; ++e) {
            const int i = tid + 256 * e;
            Ts[i / 64][i % 64] = tr[e];
        }
        __syncthreads();
        if (mm0 + THIN_TK < mend) load(mm0 + THIN_TK);
        if (active) {
#pragma unroll 8
            for (int mm = 0; mm < THIN_TK; ++mm) {
                const uint2 u = *reinterpret_cast<const uint2 *>(&Ds[mm][wg * 4]);
                const float dv[4] = {__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u)};
                const float4 t0 = *reinterpret_cast<const float4 *>(&Ts[mm][jg * 8]);
                const float4 t1 = *reinterpret_cast<const float4 *>(&Ts[mm][jg * 8 + 4]);
                const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(dv[i], tv[e], acc[i][e]);
            }
        }
        __syncthreads();
    }
    if (!active) return;
    float *out = part + (int64_t)blockIdx.y * Wd * r;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t w = w0 + wg * 4 + i;
        if (w >= Wd) continue;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = jg * 8 + e;
            if (j < r) out[WJ ? w * r + j : (int64_t)j * Wd + w] = acc[i][e];
        }
    }
}

// Splits of a thin product with `tiles` CTAs per split over a reduction of
// length L: fill the GPU about twice, at least 256 per split, at most 64 splits.
int thin_splits(int64_t tiles, int64_t L)
{
    int64_t sp = (2 * (int64_t)num_sms() + tiles - 1) / tiles;
    const int64_t lmax = L / 256;
    if (sp > lmax) sp = lmax;
    if (sp > 64) sp = 64;
    return sp < 1 ? 1 : (int)sp;
}
bool thin_ok(int64_t Kd_or_wd, int r) { return r <= 64 && (Kd_or_wd % 8) == 0; }

// out = alpha * X W (+ out if accumulate) over ranks: rows x rank product.
qerl_status thin_rows(const __nv_bfloat16 *X, int64_t M, int64_t Kd, const __nv_bfloat16 *W, bool wjk, int r,
                      StoreF32 ep, float *part, cudaStream_t s)
{
    const int tr = r <= 32 ? thin_tr<32>() : thin_tr<64>();
    const int64_t tiles = (M + tr - 1) / tr;
    const int sp = thin_splits(tiles, Kd);
    const int64_t kchunk = ((Kd + sp - 1) / sp + THIN_TK - 1) / THIN_TK * THIN_TK;
    const int splits = (int)((Kd + kchunk - 1) / kchunk);
    const dim3 grid((unsigned)tiles, (unsigned)splits);
    if (r <= 32) {
        if (wjk)
            thin_rows_kernel<true, 32><<<grid, 256, 0, s>>>(X, M, Kd, W, r, kchunk, part);
        else
            thin_rows_kernel<false, 32><<<grid, 256, 0, s>>>(X, M, Kd, W, r, kchunk, part);
    } else {
        if (wjk)
            thin_rows_kernel<true, 64><<<grid, 256, 0, s>>>(X, M, Kd, W, r, kchunk, part);
        else
            thin_rows_kernel<false, 64><<<grid, 256, 0, s>>>(X, M, Kd, W, r, kchunk, part);
    }
    QERL_TRY(launched());
    int64_t g = (M * r + 255) / 256;
    if (g > 8 * num_sms()) g = 8 * num_sms();
    split_reduce<<<(unsigned)g, 256, 0, s>>>(part, splits, M, r, ep.out, ep.ld, ep.alpha, ep.accumulate);
    return launched();
}

// out = alpha * D^T T (+ out): [Wd x r] when wj, else [r x Wd].
qerl_status thin_wide(const __nv_bfloat16 *D, int64_t M, int64_t Wd, const float *T, int r, bool wj, StoreF32 ep,
                      float *part, cudaStream_t s)
{
    const int tr = r <= 32 ? thin_tr<32>() : thin_tr<64>();
    const int64_t tiles = (Wd + tr - 1) / tr;
    const int sp = thin_splits(tiles, M);
    const int64_t mchunk = ((M + sp - 1) / sp + THIN_TK - 1) / THIN_TK * THIN_TK;
    const int splits = (int)((M + mchunk - 1) / mchunk);
    const dim3 grid((unsigned)tiles, (unsigned)splits);
    if (r <= 32) {
        if (wj)
            thin_wide_kernel<true, 32><<<grid, 256, 0, s>>>(D, M, Wd, T, r, mchunk, part);
        else
            thin_wide_kernel<false, 32><<<grid, 256, 0, s>>>(D, M, Wd, T, r, mchunk, part);
    } else {
        if (wj)
            thin_wide_kernel<true, 64><<<grid, 256, 0, s>>>(D, M, Wd, T, r, mchunk, part);
        else
            thin_wide_kernel<false, 64><<<grid, 256, 0, s>>>(D, M, Wd, T, r, mchunk, part);
    }
    QERL_TRY(launched());
    const int64_t P = wj ? Wd : r, Q = wj ? r : Wd;
    int64_t g = (P * Q + 255) / 256;
    if (g > 8 * num_sms()) g = 8 * num_sms();
    split_reduce<<<(unsigned)g, 256, 0, s>>>(part, splits, P, Q, ep.out, ep.ld, ep.alpha, ep.accumulate);
    return launched();
}
size_t thin_rows_ws(int64_t M, int64_t Kd, int r)
{
    const int tr = r <= 32 ? thin_tr<32>() : thin_tr<64>();
    return round256(size_t(thin_splits((M + tr - 1) / tr, Kd)) * M * r * sizeof(float));
}
size_t thin_wide_ws(int64_t M, int64_t Wd, int r)
{
    const int tr = r <= 32 ? thin_tr<32>() : thin_tr<64>();
    return round256(size_t(thin_splits((Wd + tr - 1) / tr, M)) * Wd * r * sizeof(float));
}

// Per group g (blockIdx.y): t = sum of the split partials (fixed order);
// t_out = t (optional); u = bf16(s t / (s_t 2^c)) as [M, r_pad], zeros past
// r: the LoRA operand of the tensor-core forward.
struct UReduceGroups {
    const float *part[RANK_MAX_G];
    const float *tensor_scale[RANK_MAX_G];
    float *t_out[RANK_MAX_G];
    __nv_bfloat16 *u[RANK_MAX_G];
};
__global__ void __launch_bounds__(256) u_reduce_kernel(const UReduceGroups grp, int splits, int64_t M, int r,
                                                       int r_pad, float s)
{
    pdl_trigger();
    pdl_wait();
    const int g = blockIdx.y;
    const float *part = grp.part[g];
    float *t_out = grp.t_out[g];
    __nv_bfloat16 *u = grp.u[g];
    const float st = *grp.tensor_scale[g];
    const float fac = s / (st * pow2f(tc_exponent_offset(st)));
    const int64_t n = M * r_pad;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / r_pad;
        const int j = (int)(i % r_pad);
        float t = 0.0f;
        if (j < r) {
            t = sum_splits(part + m * r + j, M * r, splits);
            if (t_out) t_out[m * r + j] = t;
        }
        u[i] = __float2bfloat16_rn(t * fac);
    }
}

// out = alpha * P (+ out if accumulate), P[w][j] (wj) or P[j][w] = sum over m
// of D[m, w] T[m, j]: the tensor-core wide product, then the split reduction.
qerl_status wide_rows(const __nv_bfloat16 *D, int64_t M, int64_t Wd, const float *T, int r, bool wj, StoreF32 ep,
                      __nv_bfloat16 *tb, bool tb_ready, float *part, cudaStream_t s)
{
    QERL_TRY(wide_tc(D, M, Wd, T, r, wj, tb, tb_ready, part, g_chain.load() != 0, s));
    const int64_t P = wj ? Wd : r, Q = wj ? r : Wd;
    int64_t g = (P * Q + 255) / 256;
    if (g > 8 * num_sms()) g = 8 * num_sms();
    split_reduce<<<(unsigned)g, 256, 0, s>>>(part, wide_tc_splits(M, Wd), P, Q, ep.out, ep.ld, ep.alpha,
                                             ep.accumulate);
    return launched();
}

// B [N, r] -> B^T [r, N] (the rank-side operand of v = dy B on tensor cores).
__global__ void __launch_bounds__(256) transpose_rank_kernel(const __nv_bfloat16 *__restrict__ B, int64_t N, int r,
                                                             __nv_bfloat16 *__restrict__ bt)
{
    for (int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; n < N; n += (int64_t)gridDim.x * blockDim.x)
        for (int j = 0; j < r; ++j) bt[(int64_t)j * N + n] = B[n * r + j];
}

// The sum T [M, r] of a rank product's split partials (split order) -> out, and
// in the same pass what the next products read: the bf16 pair Tb [M][2 RP] of
// the wide products (hi = bf16(T), lo = bf16(T - hi), zeros past r) when tb is
// given, and the dx kernel's LoRA operand v' = bf16(s T / (s_t 2^c)) [M, vp_pad]
// (zeros past r) when vp is given.
__global__ void __launch_bounds__(256) rank_reduce_kernel(const float *__restrict__ part, int splits, int64_t M, int r,
                                                          float *__restrict__ out, __nv_bfloat16 *__restrict__ tb,
                                                          int RP, __nv_bfloat16 *__restrict__ vp, int vp_pad, float s,
                                                          const float *__restrict__ tensor_scale)
{
    pdl_trigger();
    pdl_wait();
    const int jw = RP > vp_pad ? RP : vp_pad;  // columns per row (>= r)
    float fac = 0.0f;
    if (vp) {
        const float st = *tensor_scale;
        fac = s / (st * pow2f(tc_exponent_offset(st)));
    }
    const int64_t n = M * jw;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / jw;
        const int j = (int)(i % jw);
        float t = 0.0f;
        if (j < r) {
            t = sum_splits(part + m * r + j, M * r, splits);
            out[m * r + j] = t;
        }
        if (tb && j < RP) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(t);
            tb[m * 2 * RP + j] = hi;
            tb[m * 2 * RP + RP + j] = __float2bfloat16_rn(t - __bfloat162float(hi));
        }
        if (vp && j < vp_pad) vp[m * vp_pad + j] = __float2bfloat16_rn(j < r ? t * fac : 0.0f);
    }
}

// T = X W^T with W [r, Kd] on tensor cores, reduced by rank_reduce_kernel into
// out [M, r] (and Tb, v' where given).
qerl_status rank_rows_reduce(const __nv_bfloat16 *X, int64_t M, int64_t Kd, const __nv_bfloat16 *W, int r,
                             float *out, __nv_bfloat16 *tb, __nv_bfloat16 *vp, int vp_pad, float s,
                             const float *tensor_scale, float *part, cudaStream_t st)
{
    const bool chain = g_chain.load() != 0;
    const RankOut o{W, r, part};
    QERL_TRY(rank_tc(X, M, Kd, &o, 1, chain, st));
    const int RP = tb ? rank_tc_pad(r) : 0;
    const int jw = std::max(std::max(RP, vp ? vp_pad : 0), r);
    int64_t g = (M * jw + 255) / 256;
    if (g > 8 * num_sms()) g = 8 * num_sms();
    return launched(launch_k(rank_reduce_kernel, dim3((unsigned)g), dim3(256), 0, st, chain, (const float *)part,
                             rank_tc_splits(M, Kd), M, r, out, tb, RP > 0 ? RP : r, vp, vp ? vp_pad : 0, s,
                             tensor_scale));
}

// Scratch of the backward: v, t (when not saved), v' for the tensor-core dx,
// and the split-k partials of the thin products.
struct BwdWs {
    size_t vbytes, vp_bytes, bt_bytes, tb_bytes, part_bytes;
};
BwdWs bwd_ws(int64_t M, int64_t N, int64_t K, int r)
{
    BwdWs w;
    w.vbytes = round256(size_t(M) * r * sizeof(float));
    w.vp_bytes = tc_dx_ws_bytes(M, r);
    w.bt_bytes = r <= 64 ? round256(size_t(r) * N * 2) : 0;
    w.tb_bytes = r <= 64 ? wide_tc_tb_bytes(M, r) : 0;
    size_t pb = gemm_split_ws(M, r, N);                               // v = dy B
    pb = std::max(pb, gemm_split_ws(M, r, K));                         // t = x A^T
    pb = std::max(pb, gemm_split_ws(r, K, M));                         // dA
    pb = std::max(pb, gemm_split_ws(N, r, M));                         // dB
    if (thin_ok(N, r) && thin_ok(K, r)) {
        pb = std::max(pb, thin_rows_ws(M, N, r));
        pb = std::max(pb, thin_rows_ws(M, K, r));
        pb = std::max(pb, thin_wide_ws(M, K, r));
        pb = std::max(pb, thin_wide_ws(M, N, r));
        pb = std::max(pb, rank_tc_part_bytes(M, N, r));
        pb = std::max(pb, rank_tc_part_bytes(M, K, r));
        pb = std::max(pb, wide_tc_part_bytes(M, K, r));
        pb = std::max(pb, wide_tc_part_bytes(M, N, r));
    }
    w.part_bytes = pb;
    return w;
}

// v = dy B, dx, then dA = s v^T x and dB = s dy^T t.  Each product runs on the
// tensor cores where its shape allows (rank_tc.cu for the four rank-r products,
// split over their long reduction and summed in split order; tc_dx for dx),
// else on the CUDA-core kernels of this file.
qerl_status run_bwd(const BwdArgs &a, char *ws, cudaStream_t s)
{
    const BwdWs w = bwd_ws(a.M, a.N, a.K, a.r);
    float *v = reinterpret_cast<float *>(ws);
    float *u = reinterpret_cast<float *>(ws + w.vbytes);
    char *vp = ws + 2 * w.vbytes;
    __nv_bfloat16 *bt = reinterpret_cast<__nv_bfloat16 *>(vp + w.vp_bytes);
    __nv_bfloat16 *tb = reinterpret_cast<__nv_bfloat16 *>(vp + w.vp_bytes + w.bt_bytes);
    float *part = reinterpret_cast<float *>(vp + w.vp_bytes + w.bt_bytes + w.tb_bytes);
    // the thin products take the dedicated kernels when every operand is a
    // whole number of 16-byte vectors
    const bool thin = thin_ok(a.N, a.r) && thin_ok(a.K, a.r) && aligned16(a.dy) && aligned16(a.x) &&
                      aligned16(a.A) && aligned16(a.B);
    // the rows x rank products (v = dy B, t = x A^T) on tensor cores
    const bool rank = thin && g_algo.load() != QERL_ALGO_SIMT && rank_tc_applies(a.M, a.N, a.r, a.dy, bt) &&
                      rank_tc_applies(a.M, a.K, a.r, a.x, a.A);
    // the wide x rank products (dA, dB) on tensor cores
    const bool wide = thin && g_algo.load() != QERL_ALGO_SIMT && wide_tc_applies(a.M, a.K, a.r, a.x) &&
                      wide_tc_applies(a.M, a.N, a.r, a.dy);
    const bool dx_tc = a.dx && g_algo.load() != QERL_ALGO_SIMT && tc_dx_applies(a.M, a.N, a.K, a.r);
    bool vp_ready = false, tb_v = false;  // written by the reduction of v
    if (rank) {
        int64_t g = (a.N + 255) / 256;
        if (g > 4 * num_sms()) g = 4 * num_sms();
        transpose_rank_kernel<<<(unsigned)g, 256, 0, s>>>(a.B, a.N, a.r, bt);
        QERL_TRY(launched());
        // v, and in the same pass its bf16 pair (dA) and v' (dx)
        __nv_bfloat16 *tbv = wide && a.dA ? tb : nullptr;
        __nv_bfloat16 *vpv = dx_tc ? reinterpret_cast<__nv_bfloat16 *>(vp) : nullptr;
        QERL_TRY(rank_rows_reduce(a.dy, a.M, a.N, bt, a.r, v, tbv, vpv, tc_dx_rpad(a.r), a.lora_scale,
                                  a.tensor_scale, part, s));
        vp_ready = vpv != nullptr;
        tb_v = tbv != nullptr;
    } else if (thin)
        QERL_TRY(thin_rows(a.dy, a.M, a.N, a.B, false, a.r, StoreF32{v, a.r, 1.0f, 0}, part, s));
    else
        QERL_TRY(run_gemm_store(a.M, a.r, a.N, RowBF16{a.dy, a.N}, ColBF16{a.B, a.r}, StoreF32{v, a.r, 1.0f, 0},
                                part, s));
    if (a.dx) {
        if (dx_tc)
            QERL_TRY(tc_dx(a, v, vp, vp_ready, s));
        else
            QERL_TRY(run_gemm(a.M, a.K, a.N, RowBF16{a.dy, a.N}, WCol{a.codes, a.scales, a.K, a.packed},
                              DxEpi{a.dx, a.K, a.tensor_scale, v, a.A, a.r, a.lora_scale}, s));
    }
    if (a.dA) {
        const StoreF32 ep{a.dA, a.K, a.lora_scale, a.accumulate};
        if (wide)
            QERL_TRY(wide_rows(a.x, a.M, a.K, v, a.r, false, ep, tb, tb_v, part, s));
        else if (thin)
            QERL_TRY(thin_wide(a.x, a.M, a.K, v, a.r, false, ep, part, s));
        else
            QERL_TRY(run_gemm_store((int64_t)a.r, a.K, a.M, ColF32{v, a.r}, ColBF16{a.x, a.K}, ep, part, s));
    }
    if (a.dB) {
        const float *uu = a.t_saved;
        bool tb_t = false;  // written by the reduction of t
        if (!uu) {
            if (rank) {  // t, and in the same pass its bf16 pair (dB)
                __nv_bfloat16 *tbt = wide ? tb : nullptr;
                QERL_TRY(rank_rows_reduce(a.x, a.M, a.K, a.A, a.r, u, tbt, nullptr, 0, 0.0f, a.tensor_scale, part,
                                          s));
                tb_t = tbt != nullptr;
            } else if (thin)
                QERL_TRY(thin_rows(a.x, a.M, a.K, a.A, true, a.r, StoreF32{u, a.r, 1.0f, 0}, part, s));
            else
                QERL_TRY(run_gemm_store(a.M, a.r, a.K, RowBF16{a.x, a.K}, RowBF16{a.A, a.K},
                                        StoreF32{u, a.r, 1.0f, 0}, part, s));
            uu = u;
        }
        const StoreF32 ep{a.dB, a.r, a.lora_scale, a.accumulate};
        if (wide)
            QERL_TRY(wide_rows(a.dy, a.M, a.N, uu, a.r, true, ep, tb, tb_t, part, s));
        else if (thin)
            QERL_TRY(thin_wide(a.dy, a.M, a.N, uu, a.r, true, ep, part, s));
        else
            QERL_TRY(run_gemm_store(a.N, (int64_t)a.r, a.M, ColBF16{a.dy, a.N}, ColF32{uu, a.r}, ep, part, s));
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

// r <= 64: tensor cores or the CUDA-core fallback; 64 < r <= 128: tensor cores only
bool lora_down_rows_applies(int64_t K, int r) { return thin_ok(K, r) || (r <= 128 && K % 8 == 0 && K >= 64); }
size_t lora_down_rows_ws(int64_t M, int64_t K, int r, int G)
{
    return std::max(size_t(G) * rank_tc_part_bytes(M, K, r), r <= 64 ? thin_rows_ws(M, K, r) : size_t(0));
}

qerl_status lora_down_rows(const __nv_bfloat16 *x, int64_t M, int64_t K, const DownRowsGroup *grp, int G, int r,
                           int r_pad, float s, float *part, bool chain, cudaStream_t st)
{
    if (G < 1 || G > RANK_MAX_G) return QERL_ERR_INVALID_ARG;
    int64_t gred = (M * r_pad + 255) / 256;
    if (gred > 8 * num_sms()) gred = 8 * num_sms();
    UReduceGroups ug;
    for (int g = 0; g < RANK_MAX_G; ++g) {
        const DownRowsGroup &d = grp[g < G ? g : 0];
        ug.part[g] = nullptr;
        ug.tensor_scale[g] = d.tensor_scale;
        ug.t_out[g] = d.t_out;
        ug.u[g] = d.u;
    }
    bool tc = g_algo.load() != QERL_ALGO_SIMT;
    for (int g = 0; g < G && tc; ++g) tc = rank_tc_applies(M, K, r, x, grp[g].A);
    if (tc) {  // one pass over x for every group
        const size_t pb = rank_tc_part_bytes(M, K, r);
        RankOut outs[RANK_MAX_G];
        for (int g = 0; g < G; ++g) {
            outs[g] = RankOut{grp[g].A, r, reinterpret_cast<float *>(reinterpret_cast<char *>(part) + g * pb)};
            ug.part[g] = outs[g].part;
        }
        // groups per launch: their padded ranks fit the MMA's 256 columns
        const int per = std::min(G, 256 / rank_tc_pad(r));
        for (int g0 = 0; g0 < G; g0 += per)
            QERL_TRY(rank_tc(x, M, K, outs + g0, std::min(per, G - g0), chain, st));
        return launched(launch_k(u_reduce_kernel, dim3((unsigned)gred, (unsigned)G), dim3(256), 0, st, chain, ug,
                                 rank_tc_splits(M, K), M, r, r_pad, s));
    }
    if (r > 64) return QERL_ERR_SHAPE;  // the CUDA-core kernel covers r <= 64
    // CUDA cores, group by group through the same partials buffer
    const int tr = r <= 32 ? thin_tr<32>() : thin_tr<64>();
    const int64_t tiles = (M + tr - 1) / tr;
    const int sp = thin_splits(tiles, K);
    const int64_t kchunk = ((K + sp - 1) / sp + THIN_TK - 1) / THIN_TK * THIN_TK;
    const int splits = (int)((K + kchunk - 1) / kchunk);
    const dim3 grid((unsigned)tiles, (unsigned)splits);
    for (int g = 0; g < G; ++g) {
        const __nv_bfloat16 *A = grp[g].A;
        if (r <= 32)
            QERL_TRY(launched(launch_k(thin_rows_kernel<true, 32>, grid, dim3(256), 0, st, chain, x, M, K, A, r,
                                       kchunk, part)));
        else
            QERL_TRY(launched(launch_k(thin_rows_kernel<true, 64>, grid, dim3(256), 0, st, chain, x, M, K, A, r,
                                       kchunk, part)));
        UReduceGroups one = ug;
        one.part[0] = part;
        one.tensor_scale[0] = grp[g].tensor_scale;
        one.t_out[0] = grp[g].t_out;
        one.u[0] = grp[g].u;
        QERL_TRY(launched(launch_k(u_reduce_kernel, dim3((unsigned)gred, 1u), dim3(256), 0, st, chain, one, splits, M,
                                   r, r_pad, s)));
    }
    return QERL_OK;
}

size_t linear_fwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r)
{
    const size_t simt = round256(size_t(M) * r * sizeof(float));
    return std::max(std::max(simt, tc_fwd_ws_bytes(M, N, K, r)), gemv_ws_bytes(M, N, K, r));
}

// The CUDA-core GEMV takes one or two tokens when selected.  Under AUTO it
// takes single-token calls on weights of up to 24M values (13.5 MB), where its
// lower fixed cost per call beats the tensor-core kernel; on larger weights
// the tensor-core kernel streams faster (measured on Qwen2.5-7B shapes).
constexpr int64_t kGemvAutoMaxWeights = int64_t(24) << 20;
static bool use_gemv(const FwdArgs &a, bool grouped = false)
{
    const int algo = g_algo.load();
    const bool auto_pick = algo == QERL_ALGO_AUTO && !grouped && a.M == 1 && a.N * a.K <= kGemvAutoMaxWeights;
    return (algo == QERL_ALGO_GEMV || auto_pick) && gemv_applies(a.M, a.N, a.K, a.r);
}

// One forward: GEMV, tensor cores, or the CUDA-core GEMM, in that order of
// preference among the paths the selection allows and that cover the shape.
static qerl_status run_fwd(const FwdArgs &a, char *ws, size_t ws_bytes, cudaStream_t s, bool grouped = false)
{
    if (use_gemv(a, grouped)) {
        const qerl_status st = gemv_fwd(a, ws, ws_bytes, s);
        if (st != QERL_ERR_SHAPE) return st;
    }
    if (g_algo.load() != QERL_ALGO_SIMT) {
        const qerl_status st = tc_linear_fwd(a, ws, ws_bytes, s);
        if (st != QERL_ERR_SHAPE) return st;
    }
    return simt_fwd(a, ws, s);
}

size_t linear_bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r)
{
    const BwdWs w = bwd_ws(M, N, K, r);
    return 2 * w.vbytes + w.vp_bytes + w.bt_bytes + w.tb_bytes + w.part_bytes;
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
    return run_fwd(a, static_cast<char *>(ws), ws_cap, s);
}

}  // namespace qerl

using namespace qerl;

extern "C" qerl_status qerl_set_linear_algo(int algo)
{
    if (algo != QERL_ALGO_AUTO && algo != QERL_ALGO_SIMT && algo != QERL_ALGO_TCGEN05 && algo != QERL_ALGO_GEMV)
        return QERL_ERR_INVALID_ARG;
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
    return run_fwd(a, static_cast<char *>(ws), ws_bytes, as_cuda(stream));
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
    return run_bwd(a, static_cast<char *>(ws), as_cuda(stream));
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

extern "C" size_t qerl_lora_linear_fwd_grouped_ws_bytes(int64_t M, int64_t K, int r, const int64_t *N, int n_groups)
{
    if (!N || n_groups < 1 || n_groups > 8 || M < 0 || K < 0 || r < 0) return 0;
    size_t b = n_groups <= 3 ? tc_fwd_groups_ws_bytes(M, N, n_groups, K, r) : 0;
    for (int g = 0; g < n_groups; ++g) b = std::max(b, linear_fwd_ws_bytes(M, N[g], K, r));
    return b;
}

extern "C" qerl_status qerl_nvfp4_lora_linear_fwd_grouped(const void *x, int64_t M, int64_t K, int r, float lora_scale,
                                                          const qerl_lora_linear_group *groups, int n_groups,
                                                          int packed, void *ws, size_t ws_bytes, qerl_stream_t stream)
{
    if (!groups || n_groups < 1 || n_groups > 8 || (packed != 0 && packed != 1)) return QERL_ERR_INVALID_ARG;
    for (int g = 0; g < n_groups; ++g) {
        const qerl_lora_linear_group &q = groups[g];
        QERL_TRY(check_common(M, K, q.N, q.codes, q.scales, q.tensor_scale, q.A, q.B, r));
        if (M > 0 && !q.y) return QERL_ERR_INVALID_ARG;
        if ((q.y && !aligned16(q.y)) || (q.t_out && !aligned16(q.t_out))) return QERL_ERR_ALIGN;
    }
    if (M == 0) return QERL_OK;
    if (!x) return QERL_ERR_INVALID_ARG;
    if (!aligned16(x)) return QERL_ERR_ALIGN;
    int64_t Ns[8];
    for (int g = 0; g < n_groups; ++g) Ns[g] = groups[g].N;
    if (!ws || ws_bytes < qerl_lora_linear_fwd_grouped_ws_bytes(M, K, r, Ns, n_groups)) return QERL_ERR_WORKSPACE;
    QERL_TRY(check_device());
    FwdArgs a[8];
    for (int g = 0; g < n_groups; ++g) {
        const qerl_lora_linear_group &q = groups[g];
        a[g] = FwdArgs{static_cast<const __nv_bfloat16 *>(x), M, K, q.N, q.codes, q.scales, q.tensor_scale,
                       static_cast<const __nv_bfloat16 *>(q.A), static_cast<const __nv_bfloat16 *>(q.B), r,
                       lora_scale, static_cast<__nv_bfloat16 *>(q.y), q.t_out, packed};
    }
    cudaStream_t s = as_cuda(stream);
    char *w = static_cast<char *>(ws);
    // One tensor-core launch for all groups where it applies (AUTO keeps it at
    // one token too: one launch beats a GEMV per group); a GEMV per group when
    // the GEMV is selected.
    bool gemv = true;
    for (int g = 0; g < n_groups; ++g) gemv = gemv && use_gemv(a[g], true);
    if (!gemv && g_algo.load() != QERL_ALGO_SIMT && n_groups > 1 && n_groups <= 3) {
        const qerl_status st = tc_fwd_groups(a, n_groups, w, ws_bytes, s);
        if (st != QERL_ERR_SHAPE) return st;
    }
    for (int g = 0; g < n_groups; ++g) QERL_TRY(run_fwd(a[g], w, ws_bytes, s, true));  // one group after the other
    return QERL_OK;
}

namespace {
// Scratch of a format-variant forward: what the tensor-core path needs where
// it covers the shape, and at least t (FP32 [M, r]) for the CUDA-core GEMM.
size_t variant_ws_bytes(int64_t M, int64_t N, int64_t K, int r, bool mx, bool f32)
{
    return std::max(tc_fwd_variant_ws_bytes(M, N, K, r, mx, f32), round256(size_t(M) * r * sizeof(float)));
}

qerl_status variant_args(const void *x, int64_t M, int64_t K, int64_t N, const uint8_t *codes, const uint8_t *scales,
                         const void *A, const void *B, int r, void *y, void *ws, size_t ws_bytes, int kmul, bool mx)
{
    if (!codes || !scales || !A || !B) return QERL_ERR_INVALID_ARG;
    if (M < 0 || K < 1 || N < 1) return QERL_ERR_INVALID_ARG;
    if (K % kmul != 0 || r < 1 || r > 256) return QERL_ERR_SHAPE;
    if (M == 0) return QERL_OK;
    if (!x || !y) return QERL_ERR_INVALID_ARG;
    if (!ws || ws_bytes < variant_ws_bytes(M, N, K, r, mx, !mx)) return QERL_ERR_WORKSPACE;
    return QERL_OK;
}

// The tensor-core path takes a variant unless the CUDA-core GEMM is selected or
// an operand is not 16-byte aligned (its TMA maps and vector loads need that);
// it declines shapes it does not cover (K % 256 != 0) with QERL_ERR_SHAPE.
bool variant_tc_ok(const void *x, const void *y, const uint8_t *codes, const uint8_t *scales, const void *A,
                   const void *B, const float *t_out)
{
    return g_algo.load() != QERL_ALGO_SIMT && aligned16(x) && aligned16(y) && aligned16(codes) &&
           aligned16(scales) && aligned16(A) && aligned16(B) && (!t_out || aligned16(t_out));
}
}  // namespace

// MXFP4 weight (codes [N, K/2], E8M0 scales [N, K/32]), bf16 LoRA: tcgen05 with
// the E8M0 scale in the dequantizer, else the CUDA-core GEMM.
extern "C" qerl_status qerl_mxfp4_lora_linear_fwd(const void *x, int64_t M, int64_t K, int64_t N,
                                                  const uint8_t *codes, const uint8_t *scales, const void *A,
                                                  const void *B, int r, float lora_scale, void *y, float *t_out,
                                                  void *ws, size_t ws_bytes, qerl_stream_t stream)
{
    QERL_TRY(variant_args(x, M, K, N, codes, scales, A, B, r, y, ws, ws_bytes, 32, true));
    if (M == 0) return QERL_OK;
    QERL_TRY(check_device());
    cudaStream_t s = as_cuda(stream);
    const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
    const __nv_bfloat16 *Ab = static_cast<const __nv_bfloat16 *>(A), *Bb = static_cast<const __nv_bfloat16 *>(B);
    if (variant_tc_ok(x, y, codes, scales, A, B, t_out)) {
        const FwdArgs a{xb, M, K, N, codes, nullptr, nullptr, Ab, Bb, r, lora_scale, static_cast<__nv_bfloat16 *>(y),
                        t_out};
        const qerl_status st = tc_fwd_variant(a, scales, static_cast<char *>(ws), ws_bytes, s);
        if (st != QERL_ERR_SHAPE) return st;
    }
    float *t = t_out ? t_out : static_cast<float *>(ws);
    QERL_TRY(run_gemm(M, (int64_t)r, K, RowBF16{xb, K}, RowBF16{Ab, K}, StoreF32{t, r, 1.0f, 0}, s));
    return run_gemm(M, N, K, RowBF16{xb, K}, WRowMX{codes, scales, K},
                    FwdEpiF32{static_cast<__nv_bfloat16 *>(y), N, nullptr, t, nullptr, Bb, r, lora_scale}, s);
}

// NVFP4 weight with FP32 LoRA adapters A [r, K], B [N, r]: tcgen05 with the
// LoRA term as three bf16 products of hi/lo splits, else the CUDA-core GEMM.
extern "C" qerl_status qerl_nvfp4_lora_linear_fwd_f32ab(const void *x, int64_t M, int64_t K, int64_t N,
                                                        const uint8_t *codes, const uint8_t *scales,
                                                        const float *tensor_scale, const float *A, const float *B,
                                                        int r, float lora_scale, void *y, float *t_out, void *ws,
                                                        size_t ws_bytes, qerl_stream_t stream)
{
    if (!tensor_scale) return QERL_ERR_INVALID_ARG;
    QERL_TRY(variant_args(x, M, K, N, codes, scales, A, B, r, y, ws, ws_bytes, 16, false));
    if (M == 0) return QERL_OK;
    QERL_TRY(check_device());
    cudaStream_t s = as_cuda(stream);
    const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
    if (variant_tc_ok(x, y, codes, scales, A, B, t_out)) {
        FwdArgs a{xb, M, K, N, codes, scales, tensor_scale, nullptr, nullptr, r, lora_scale,
                  static_cast<__nv_bfloat16 *>(y), t_out};
        a.Af = A;
        a.Bf = B;
        const qerl_status st = tc_fwd_variant(a, nullptr, static_cast<char *>(ws), ws_bytes, s);
        if (st != QERL_ERR_SHAPE) return st;
    }
    float *t = t_out ? t_out : static_cast<float *>(ws);
    QERL_TRY(run_gemm(M, (int64_t)r, K, RowBF16{xb, K}, RowF32{A, K}, StoreF32{t, r, 1.0f, 0}, s));
    return run_gemm(M, N, K, RowBF16{xb, K}, WRow{codes, scales, K, 0},
                    FwdEpiF32{static_cast<__nv_bfloat16 *>(y), N, tensor_scale, t, B, nullptr, r, lora_scale}, s);
}

// Scratch of the format-variant forwards (QERL_OP_MXFP4_FWD, QERL_OP_LINEAR_FWD_F32AB).
size_t qerl::variant_fwd_ws_bytes(int op, int64_t M, int64_t N, int64_t K, int r)
{
    if (op == QERL_OP_MXFP4_FWD) return K % 32 == 0 ? variant_ws_bytes(M, N, K, r, true, false) : 0;
    return K % 16 == 0 ? variant_ws_bytes(M, N, K, r, false, true) : 0;
}
