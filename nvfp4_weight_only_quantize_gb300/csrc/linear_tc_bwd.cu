// Tensor-core (tcgen05) input gradient of the NVFP4 LoRA linear:
//     dx = dy * w_hat + lora_scale * v * A,   v = dy * B
// (bitsofall "QeRL: NVFP4-Quantized Reinforcement Learning", "Implementation
// and Practical Details": gradients flow through the dequantized frozen weight).
//
// One CTA computes a 256-token x 256-column tile of dx as two accumulators
// D0, D1 [128 tokens][256 columns] (TMEM, FP32, all 512 columns), so that each
// dequantized weight tile serves 256 tokens:
//   A operand = dy tile [256 tokens x 64 n] (one TMA box), K-major, each
//               accumulator reading its 128-row half;
//   B operand = w_hat^T tile [256 k x 64 n], K-major, written by the dequant
//               warps straight from the packed codes (each thread owns two
//               adjacent weight rows n, n+1 over 32 k, so that its shared-memory
//               stores are 32-bit {n, n+1} pairs of one k row: a full 128-byte
//               swizzled row per warp store, no bank conflicts);
//   extra K steps for the LoRA term: A = v' = bf16(lora_scale * v / (s_t 2^c))
//   (TMA), B = A^T tile copied from A by the same warps.
// The epilogue scales D by s_t * 2^c (c: the exponent offset of the forward)
// and stores bf16 dx.  Every wait is bounded; on a timeout the CTA latches
// QERL_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
//
// Warp roles (320 threads): warps 0-7 dequantize (warps 0-3 also run the
// epilogue), warp 8 issues every TMA load, warp 9 owns TMEM and issues MMAs.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <mutex>

#include "linear.cuh"
#include "sm100_ptx.cuh"

namespace qerl {
namespace {

using namespace ptx;

constexpr int BX_M = 128;   // tokens per accumulator (MMA M)
constexpr int BX_MT = 2;    // accumulators (token tiles) per CTA sharing each weight tile
constexpr int BX_K = 256;   // dx columns per tile (MMA N)
constexpr int BX_N = 64;    // reduction (weight rows n) per step
constexpr int BX_THREADS = 320;
constexpr int BX_WARP_TMA = 8, BX_WARP_MMA = 9;
constexpr int BX_DQ_WARPS = 8;
constexpr int BX_SA = 2;    // dy / v' stages (256 tokens each)
constexpr int BX_SB = 3;    // w_hat^T / A^T stages
constexpr int BX_R = 4;     // raw (codes + scales) stages
constexpr int BX_A_BYTES = BX_MT * BX_M * BX_N * 2;  // 32 KB
constexpr int BX_B_BYTES = BX_K * BX_N * 2;          // 32 KB
constexpr int BX_CODES = BX_N * (BX_K / 2);          // 64 rows x 128 B = 8 KB
constexpr int BX_RAW = BX_CODES + BX_N * (BX_K / 16);  // + 64 rows x 16 B of scales
constexpr int BX_RAW_STRIDE = 9216;                  // raw stages 1024-byte aligned
constexpr int BX_SMEM = BX_SA * BX_A_BYTES + BX_SB * BX_B_BYTES + BX_R * BX_RAW_STRIDE + 1024 + 1024;

struct TcDxParams {
    int M, N, K;
    int n_steps;     // N / 64
    int lora_steps;  // r_pad / 64
    int r;
    int k_tiles;     // K / 256
    const __nv_bfloat16 *A;  // [r, K]
    const float *tensor_scale;
    __nv_bfloat16 *dx;
    unsigned int *err;
    unsigned long long timeout_ns;
};


// {f, f}, f = e4m3(b) * pow2 with b in bits 20..27 of b20 (see the forward).
__device__ __forceinline__ uint32_t bx_scale(uint32_t b20, float pow2)
{
    const float f = __uint_as_float(b20 & 0x0FF00000u) * pow2f(120) * pow2;
    const uint32_t u = __float_as_uint(f);
    return prmt(u, u, 0x3232u);
}

// Eight codes of one word -> four bf16x2 {k, k+1} words (standard or packed
// code layout), as in the forward kernel.
template <bool PACKED>
__device__ __forceinline__ void bx_dequant_word(uint32_t q, uint32_t f2, uint32_t *out)
{
    if (PACKED) {
        out[0] = bf16x2_mul(q & 0x81C081C0u, f2);
        out[1] = bf16x2_mul((q << 3) & 0x81C081C0u, f2);
        out[2] = bf16x2_mul(((q << 6) & 0x01C001C0u) | ((q << 2) & 0x80008000u), f2);
        out[3] = bf16x2_mul(((q >> 3) & 0x01C001C0u) | ((q << 1) & 0x80008000u), f2);
        return;
    }
    const uint32_t q4 = q << 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t u = prmt(q4, q, 0x4400u + 0x1111u * (uint32_t)j);
        const uint32_t raw = (u & 0x80008000u) | ((u >> 6) & 0x01C001C0u);
        out[j] = bf16x2_mul(raw, f2);
    }
}

// Byte offset of the 32-bit word holding elements {n, n+1} (n even) of row k
// in a K-major, 128-byte-swizzled tile of 128-byte rows.
__device__ __forceinline__ uint32_t bx_b_offset(int k, int n)
{
    return (uint32_t)((k >> 3) * 1024 + (k & 7) * 128 + ((((n >> 3) ^ (k & 7)) << 4) | ((n & 7) << 1)));
}

template <bool PACKED>
__global__ void __launch_bounds__(BX_THREADS, 1)
    tc_dx_kernel(const __grid_constant__ CUtensorMap dy_map, const __grid_constant__ CUtensorMap v_map,
                 const __grid_constant__ CUtensorMap codes_map, const __grid_constant__ CUtensorMap scl_map,
                 const TcDxParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *A_ring = smem;                                  // BX_SA x 16 KB
    uint8_t *B_ring = A_ring + BX_SA * BX_A_BYTES;           // BX_SB x 32 KB
    uint8_t *R_ring = B_ring + BX_SB * BX_B_BYTES;           // BX_R x 9 KB (1024-aligned)
    uint64_t *bars = reinterpret_cast<uint64_t *>(R_ring + BX_R * BX_RAW_STRIDE);
    uint64_t *a_full = bars, *a_empty = a_full + BX_SA;
    uint64_t *b_full = a_empty + BX_SA, *b_empty = b_full + BX_SB;
    uint64_t *raw_full = b_empty + BX_SB, *raw_empty = raw_full + BX_R;
    uint64_t *acc_full = raw_empty + BX_R;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *ep_ok = abort_flag + 1;  // [4]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // blockIdx.x = m_tile * k_tiles + k_tile: a wave shares its dy tiles (L2)
    const int k_tile = blockIdx.x % p.k_tiles, m_tile = blockIdx.x / p.k_tiles;
    const int k0 = k_tile * BX_K, m0 = m_tile * (BX_MT * BX_M);
    const int n_total = p.n_steps + p.lora_steps;

    if (threadIdx.x == 0) {
        for (int i = 0; i < BX_SA; ++i) {
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < BX_SB; ++i) {
            mbar_init(&b_full[i], BX_DQ_WARPS);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < BX_R; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], BX_DQ_WARPS);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == BX_WARP_TMA && lane == 0) {
        prefetch_tensormap(&dy_map);
        prefetch_tensormap(&v_map);
        prefetch_tensormap(&codes_map);
        prefetch_tensormap(&scl_map);
    }
    if (warp == BX_WARP_MMA) {
        tmem_alloc(tmem_slot, BX_MT * BX_K);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const unsigned long long deadline = globaltimer_ns() + p.timeout_ns;

    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        for (;;) {
            if (*abort_flag) return false;
            __nanosleep(64);
            if (mbar_try_wait(bar, parity)) return true;
            if (globaltimer_ns() > deadline) {
                *abort_flag = 1;
                latch_error(p.err, QERL_ERR_TIMEOUT);
                return false;
            }
        }
    };
    auto drain_wait = [&](uint64_t *bar, uint32_t parity) {
        const unsigned long long until = globaltimer_ns() + 100000000ull;  // 100 ms
        while (!mbar_try_wait(bar, parity) && globaltimer_ns() < until) {
        }
    };

    if (warp == BX_WARP_TMA) {
        // ------------------------------------------- all TMA loads, one lane
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_last(), pol_a = policy_evict_first();
            int issued_a = 0, issued_r = 0;
            bool ok = true;
            for (int j = 0; j < n_total && ok; ++j) {
                if (j < p.n_steps) {  // raw codes + scales of weight rows 64j .. 64j+63, columns k0 .. k0+255
                    const int rs = j % BX_R;
                    if (j >= BX_R && !wait(&raw_empty[rs], (uint32_t)((j / BX_R) - 1) & 1u)) { ok = false; break; }
                    uint8_t *dst = R_ring + rs * BX_RAW_STRIDE;
                    mbar_arrive_expect_tx(&raw_full[rs], BX_RAW);
                    tma_load_2d_hint(dst, &codes_map, &raw_full[rs], k0 / 2, j * BX_N, pol_w);
                    tma_load_2d_hint(dst + BX_CODES, &scl_map, &raw_full[rs], k0 / 16, j * BX_N, pol_w);
                    issued_r = j + 1;
                }
                const int as = j % BX_SA;
                if (j >= BX_SA && !wait(&a_empty[as], (uint32_t)((j / BX_SA) - 1) & 1u)) { ok = false; break; }
                mbar_arrive_expect_tx(&a_full[as], BX_A_BYTES);
                if (j < p.n_steps)
                    tma_load_2d_hint(A_ring + as * BX_A_BYTES, &dy_map, &a_full[as], j * BX_N, m0, pol_a);
                else
                    tma_load_2d_hint(A_ring + as * BX_A_BYTES, &v_map, &a_full[as], (j - p.n_steps) * BX_N, m0, pol_a);
                issued_a = j + 1;
            }
            if (*abort_flag) {  // let the copies already issued land before the CTA exits
                for (int j = issued_r > BX_R ? issued_r - BX_R : 0; j < issued_r; ++j)
                    drain_wait(&raw_full[j % BX_R], (uint32_t)(j / BX_R) & 1u);
                for (int j = issued_a > BX_SA ? issued_a - BX_SA : 0; j < issued_a; ++j)
                    drain_wait(&a_full[j % BX_SA], (uint32_t)(j / BX_SA) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == BX_WARP_MMA) {
        // ------------------------------------------- MMA issue (whole warp, one elected lane)
        constexpr uint32_t idesc = idesc_bf16_f32(BX_M, BX_K);
        bool ready = n_total > 0;
        for (int j = 0; j < n_total && ready; ++j) {
            const int as = j % BX_SA, bs = j % BX_SB;
            ready = __all_sync(0xFFFFFFFFu, wait(&a_full[as], (uint32_t)(j / BX_SA) & 1u) &&
                                                wait(&b_full[bs], (uint32_t)(j / BX_SB) & 1u));
            if (!ready) break;
            tc_fence_after();
            if (elect_one()) {
                const uint64_t ad = desc_kmajor_sw128(smem_u32(A_ring + as * BX_A_BYTES));
                const uint64_t bd = desc_kmajor_sw128(smem_u32(B_ring + bs * BX_B_BYTES));
#pragma unroll
                for (int t = 0; t < BX_MT; ++t)  // accumulator t: tokens 128 t .. 128 t + 127 (16 KB in)
#pragma unroll
                    for (int kk = 0; kk < BX_N / 16; ++kk)  // 16 n = 32 bytes of each K-major row
                        umma_bf16(tmem + (uint32_t)(t * BX_K), ad + (uint64_t)((t * BX_M * 128) >> 4) + 2u * kk,
                                  bd + 2u * kk, idesc, (j > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&a_empty[as]);
                umma_commit(&b_empty[bs]);
            }
            __syncwarp();
        }
        if (elect_one()) umma_commit(acc_full);  // once every MMA issued above has completed
        __syncwarp();
    } else {
        // ------------------------------------------- w_hat^T (and A^T) tiles
        // Thread: weight rows n = 2*lane, 2*lane + 1 of the step, columns
        // k = 32*warp .. +31 of the tile.
        const int n0l = 2 * lane, kw = 32 * warp;
        const float pow2 = pow2f(126 - tc_exponent_offset(*p.tensor_scale));
        for (int j = 0; j < n_total; ++j) {
            const int bs = j % BX_SB;
            if (j >= BX_SB && !__all_sync(0xFFFFFFFFu, wait(&b_empty[bs], (uint32_t)((j / BX_SB) - 1) & 1u))) break;
            uint32_t w0[16], w1[16];  // {k, k+1} pairs of rows n0l and n0l + 1, k = kw + 2i
            if (j < p.n_steps) {
                const int rs = j % BX_R;
                if (!__all_sync(0xFFFFFFFFu, wait(&raw_full[rs], (uint32_t)(j / BX_R) & 1u))) break;
                const uint32_t raw = smem_u32(R_ring + rs * BX_RAW_STRIDE);
                // codes: 128-byte rows, logical 16-byte chunk `warp` stored at chunk ^ (row % 8)
                const uint4 c0 = ld_shared_v4(raw + n0l * 128 + ((warp ^ (n0l & 7)) << 4));
                const uint4 c1 = ld_shared_v4(raw + (n0l + 1) * 128 + ((warp ^ ((n0l + 1) & 7)) << 4));
                // scales: 16-byte rows; blocks 2*warp and 2*warp + 1 of each row
                const uint32_t s0 = ld_shared_u32(raw + BX_CODES + n0l * 16 + (warp >> 1) * 4) >> ((warp & 1) * 16);
                const uint32_t s1 = ld_shared_u32(raw + BX_CODES + (n0l + 1) * 16 + (warp >> 1) * 4) >> ((warp & 1) * 16);
                const uint32_t f0a = bx_scale(s0 << 20, pow2), f0b = bx_scale(s0 << 12, pow2);
                const uint32_t f1a = bx_scale(s1 << 20, pow2), f1b = bx_scale(s1 << 12, pow2);
                bx_dequant_word<PACKED>(c0.x, f0a, w0 + 0);
                bx_dequant_word<PACKED>(c0.y, f0a, w0 + 4);
                bx_dequant_word<PACKED>(c0.z, f0b, w0 + 8);
                bx_dequant_word<PACKED>(c0.w, f0b, w0 + 12);
                bx_dequant_word<PACKED>(c1.x, f1a, w1 + 0);
                bx_dequant_word<PACKED>(c1.y, f1a, w1 + 4);
                bx_dequant_word<PACKED>(c1.z, f1b, w1 + 8);
                bx_dequant_word<PACKED>(c1.w, f1b, w1 + 12);
                __syncwarp();
                if (lane == 0) mbar_arrive(&raw_empty[rs]);
            } else {
                // LoRA step l: B rows k, columns jj = LoRA index 64 l + jj: A[64 l + jj][k0 + k]
                const int jr = (j - p.n_steps) * BX_N + n0l;
                const __nv_bfloat16 *a0 = p.A + (size_t)jr * p.K + k0 + kw;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v0 = jr < p.r ? __ldg(reinterpret_cast<const uint4 *>(a0) + q) : make_uint4(0, 0, 0, 0);
                    const uint4 v1 = jr + 1 < p.r ? __ldg(reinterpret_cast<const uint4 *>(a0 + p.K) + q)
                                                  : make_uint4(0, 0, 0, 0);
                    w0[4 * q] = v0.x; w0[4 * q + 1] = v0.y; w0[4 * q + 2] = v0.z; w0[4 * q + 3] = v0.w;
                    w1[4 * q] = v1.x; w1[4 * q + 1] = v1.y; w1[4 * q + 2] = v1.z; w1[4 * q + 3] = v1.w;
                }
            }
            const uint32_t bt = smem_u32(B_ring + bs * BX_B_BYTES);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t lo = prmt(w0[i], w1[i], 0x5410u);  // {n, n+1} at k = kw + 2i
                const uint32_t hi = prmt(w0[i], w1[i], 0x7632u);  // {n, n+1} at k = kw + 2i + 1
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(bt + bx_b_offset(kw + 2 * i, n0l)), "r"(lo) : "memory");
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(bt + bx_b_offset(kw + 2 * i + 1, n0l)), "r"(hi) : "memory");
            }
            fence_proxy_async_smem();  // the tensor core reads these through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&b_full[bs]);
        }

        // ------------------------------------------- epilogue (warps 0-3)
        if (warp < 4) {
            const bool ok_warp = __all_sync(0xFFFFFFFFu, wait(acc_full, 0));
            if (lane == 0) ep_ok[warp] = ok_warp ? 1 : 0;
            named_bar_sync(1, 128);
            const bool ok = ep_ok[0] && ep_ok[1] && ep_ok[2] && ep_ok[3] && !*abort_flag;
            tc_fence_after();
            if (ok) {
                const float st = *p.tensor_scale;
                const float ysc = st * pow2f(tc_exponent_offset(st));
                for (int c = 0; c < BX_MT * BX_K; c += 16) {
                    const int t = c / BX_K, c0 = c % BX_K;
                    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(t * BX_K);
                    const int m = m0 + t * BX_M + warp * 32 + lane;
                    __nv_bfloat16 *dst = p.dx + (size_t)m * p.K + k0;
                    uint32_t r[16];
                    tmem_ld16(taddr + (uint32_t)c0, r);
                    tmem_wait_ld();
                    uint32_t o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * e]) * ysc,
                                                                       __uint_as_float(r[2 * e + 1]) * ysc);
                        o[e] = *reinterpret_cast<const uint32_t *>(&h);
                    }
                    if (m < p.M) {
                        reinterpret_cast<uint4 *>(dst + c0)[0] = make_uint4(o[0], o[1], o[2], o[3]);
                        reinterpret_cast<uint4 *>(dst + c0)[1] = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == BX_WARP_MMA) {
        if (lane == 0) drain_wait(acc_full, 0);  // every issued MMA has finished (no-op unless aborted)
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, BX_MT * BX_K);
    }
}

// v' = bf16(lora_scale * v / (s_t 2^c)) as [M, r_pad] (zeros past r): the A
// operand of the LoRA steps, in the units of the weight product.
__global__ void __launch_bounds__(256) vprime_kernel(const float *__restrict__ v, int M, int r, int r_pad, float s,
                                                     const float *__restrict__ tensor_scale,
                                                     __nv_bfloat16 *__restrict__ vp)
{
    const float st = *tensor_scale;
    const float fac = s / (st * pow2f(tc_exponent_offset(st)));
    const int64_t total = (int64_t)M * r_pad;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / r_pad;
        const int j = (int)(i % r_pad);
        vp[i] = __float2bfloat16_rn(j < r ? v[m * r + j] * fac : 0.0f);
    }
}

struct BxEnv {
    unsigned long long timeout_ns = 2000000000ull;  // 2 s
};

}  // namespace

bool tc_dx_applies(int64_t M, int64_t N, int64_t K, int r)
{
    return M >= 1 && K >= BX_K && K % BX_K == 0 && N >= BX_N && N % BX_N == 0 && r >= 1 && r <= 256 &&
           M <= (1 << 30) && N <= (1 << 30) && K <= (1 << 30);
}

int tc_dx_rpad(int r) { return (r + BX_N - 1) / BX_N * BX_N; }

size_t tc_dx_ws_bytes(int64_t M, int r) { return round256(size_t(M) * tc_dx_rpad(r) * 2); }

qerl_status tc_dx(const BwdArgs &a, const float *v, char *vp_ws, bool vp_ready, cudaStream_t s)
{
    const int r_pad = tc_dx_rpad(a.r);
    __nv_bfloat16 *vp = reinterpret_cast<__nv_bfloat16 *>(vp_ws);
    if (!vp_ready) {
        int64_t g = (a.M * r_pad + 255) / 256;
        if (g > 4 * num_sms()) g = 4 * num_sms();
        vprime_kernel<<<(unsigned)g, 256, 0, s>>>(v, (int)a.M, a.r, r_pad, a.lora_scale, a.tensor_scale, vp);
        QERL_TRY(launched());
    }
    CUtensorMap dym, vm, cm, sm;
    // dy: [M, N] bf16, 64 x 128 boxes; v': [M, r_pad]; codes: 64 rows x 128 bytes
    // (256 columns), 128-byte swizzle; scales: 64 rows x 16 bytes.
    if (!make_map_2d(&dym, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.dy, a.N, a.M, a.N * 2, BX_N, BX_MT * BX_M,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, vp, r_pad, a.M, r_pad * 2, BX_N, BX_MT * BX_M,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&cm, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.codes, a.K / 2, a.N, a.K / 2, BX_K / 2, BX_N,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&sm, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.scales, a.K / 16, a.N, a.K / 16, BX_K / 16, BX_N,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
        return QERL_ERR_CUDA;
    TcDxParams p;
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.n_steps = (int)(a.N / BX_N);
    p.lora_steps = r_pad / BX_N;
    p.r = a.r;
    p.k_tiles = (int)(a.K / BX_K);
    p.A = a.A;
    p.tensor_scale = a.tensor_scale;
    p.dx = a.dx;
    p.err = error_word();
    static const BxEnv env;
    p.timeout_ns = env.timeout_ns;
    const int64_t m_tiles = (a.M + BX_MT * BX_M - 1) / (BX_MT * BX_M);
    const int64_t grid = m_tiles * p.k_tiles;
    if (grid > 0x7FFFFFFF) return QERL_ERR_SHAPE;
    auto kernel = a.packed ? tc_dx_kernel<true> : tc_dx_kernel<false>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BX_SMEM) != cudaSuccess)
        return QERL_ERR_CUDA;
    kernel<<<(unsigned)grid, BX_THREADS, BX_SMEM, s>>>(dym, vm, cm, sm, p);
    return launched();
}

}  // namespace qerl
