// Tensor-core (tcgen05) rank-r products of the LoRA branch that have a long
// reduction (bitsofall "QeRL: NVFP4-Quantized Reinforcement Learning", LoRA
// paragraph: the adapter path x A^T runs beside the NVFP4 product; its
// backward needs v = dy B and t = x A^T):
//     P_g[z][m][j] = sum over k in split z of X[m, k] * W_g[j, k],   j < r_g,
// for up to three W_g sharing one X.  X bf16 [M, Kd] row-major (x or dy); W_g
// bf16 [r_g, Kd] row-major (A, or B^T); P_g FP32 [splits][M][r_g]: the split
// partials, summed in split order by the caller's reduction kernel.
//
// One CTA: 128 tokens (MMA M) x G * RP ranks (MMA N <= 256, RP = 32, 64 or 128;
// rows r_g .. RP-1 of each group are the TMA zero fill) over one split of the reduction, 64 k per stage
// (one X box of 128 x 64 and one RP x 64 box per group, K-major, 128-byte
// swizzle).  The accumulator sits in TMEM, lane = token.  Warp 0 issues the TMA
// loads, warp 1 owns TMEM and issues the MMAs, all four warps run the epilogue.
// One pass over X serves every group, which bounds the product by HBM.  Every
// wait is bounded; on a timeout the CTA latches QERL_ERR_TIMEOUT, lets its
// copies and MMAs land, frees TMEM and exits.
#include <cudaTypedefs.h>

#include "linear.cuh"
#include "sm100_ptx.cuh"

namespace qerl {
namespace {

using namespace ptx;

constexpr int RK_M = 128;  // tokens per CTA (MMA M)
constexpr int RK_K = 64;   // reduction per stage: one 128-byte swizzled row
constexpr int RK_THREADS = 128;
constexpr int RK_MAX_S = 6;
constexpr int RK_X_BYTES = RK_M * RK_K * 2;  // 16 KB
constexpr int RK_SMEM_BUDGET = 110 * 1024;   // two CTAs per SM
constexpr int RK_OVERHEAD_KB = 3;            // per-CTA start-up, in k blocks (split choice)

struct RankMaps {
    CUtensorMap x;
    CUtensorMap w[RANK_MAX_G];
};

struct RankParams {
    int64_t M;
    int G, S;            // groups, pipeline stages
    int kb, kb_split;    // 64-wide k blocks in all / per split
    int m_tiles;
    int r[RANK_MAX_G];
    float *part[RANK_MAX_G];
    unsigned int *err;
    unsigned long long timeout_ns;
};

template <int RP>
__global__ void __launch_bounds__(RK_THREADS) rank_tc_kernel(const __grid_constant__ RankMaps maps,
                                                             const RankParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int N = p.G * RP;
    const int stage_bytes = RK_X_BYTES + N * 128;  // 1024-byte multiple: RP is a multiple of 8 rows
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.S * stage_bytes);
    uint64_t *empty = full + RK_MAX_S;
    uint64_t *acc_full = empty + RK_MAX_S;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *ep_ok = abort_flag + 1;  // [4]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tile = blockIdx.x % p.m_tiles, split = blockIdx.x / p.m_tiles;
    const int kb0 = split * p.kb_split;
    const int nkb = p.kb - kb0 < p.kb_split ? p.kb - kb0 : p.kb_split;  // >= 1: no empty split
    const int m0 = m_tile * RK_M;
    const uint32_t tcols = N <= 32 ? 32u : N <= 64 ? 64u : N <= 128 ? 128u : 256u;

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&maps.x);
        for (int g = 0; g < p.G; ++g) prefetch_tensormap(&maps.w[g]);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tcols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // chained launch: X is written, and the partials read, by preceding work
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

    if (warp == 0) {
        // ------------------------------------------- TMA loads, one lane
        if (lane == 0) {
            const uint64_t pol_x = policy_evict_first(), pol_w = policy_evict_last();
            int s = 0, issued = 0;
            uint32_t ph = 0;
            for (int i = 0; i < nkb; ++i) {
                if (i >= p.S && !wait(&empty[s], ph ^ 1u)) break;
                uint8_t *st = smem + s * stage_bytes;
                const int kx = (kb0 + i) * RK_K;
                mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
                tma_load_2d_hint(st, &maps.x, &full[s], kx, m0, pol_x);
                for (int g = 0; g < p.G; ++g)
                    tma_load_2d_hint(st + RK_X_BYTES + g * RP * 128, &maps.w[g], &full[s], kx, 0, pol_w);
                issued = i + 1;
                if (++s == p.S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (*abort_flag)  // let the copies already issued land before the CTA exits
                for (int j = issued > p.S ? issued - p.S : 0; j < issued; ++j)
                    drain_wait(&full[j % p.S], (uint32_t)(j / p.S) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------- MMA issue (one elected lane)
        const uint32_t idesc = idesc_bf16_f32(RK_M, N);
        int s = 0;
        uint32_t ph = 0;
        for (int i = 0; i < nkb; ++i) {
            if (!__all_sync(0xFFFFFFFFu, wait(&full[s], ph))) break;
            tc_fence_after();
            if (elect_one()) {
                const uint32_t st = smem_u32(smem + s * stage_bytes);
                const uint64_t ad = desc_kmajor_sw128(st);
                const uint64_t bd = desc_kmajor_sw128(st + RK_X_BYTES);
#pragma unroll
                for (int kk = 0; kk < RK_K / 16; ++kk)  // 16 k = 32 bytes of each K-major row
                    umma_bf16(tmem, ad + 2u * kk, bd + 2u * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&empty[s]);
            }
            __syncwarp();
            if (++s == p.S) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (elect_one()) umma_commit(acc_full);  // once every MMA issued above has completed
        __syncwarp();
    }

    // ------------------------------------------- epilogue: TMEM lane = token
    {
        const bool ok_warp = __all_sync(0xFFFFFFFFu, wait(acc_full, 0));
        if (lane == 0) ep_ok[warp] = ok_warp ? 1 : 0;
        __syncthreads();
        const bool ok = ep_ok[0] && ep_ok[1] && ep_ok[2] && ep_ok[3] && !*abort_flag;
        tc_fence_after();
        if (ok) {
            const int64_t m = (int64_t)m0 + warp * 32 + lane;
            for (int c = 0; c < N; c += 16) {  // a 16-column chunk lies in one group (RP % 16 == 0)
                const int g = c / RP, j0 = c % RP, rg = p.r[g];
                if (j0 >= rg) continue;  // uniform over the warp
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
                tmem_wait_ld();
                if (m >= p.M) continue;
                float *dst = p.part[g] + ((int64_t)split * p.M + m) * rg + j0;
                const int n = rg - j0 < 16 ? rg - j0 : 16;
                if ((rg & 3) == 0) {
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        if (e < n)
                            *reinterpret_cast<float4 *>(dst + e) =
                                make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                            __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (e < n) dst[e] = __uint_as_float(v[e]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) drain_wait(acc_full, 0);  // every issued MMA has finished (no-op unless aborted)
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, tcols);
    }
}

// ------------------------------------------------------------------ wide x rank
// P[z][w][j] (or [z][j][w]) = sum over m in split z of D[m, w] * T[m, j]: the
// weight gradients dA = s v^T x (D = x) and dB = s dy^T t (D = dy).  The
// reduction runs over tokens, the outer dimension of both row-major operands,
// so both are MN-major: D tile [64 tokens][128 w] as two 64-column swizzled
// boxes (MMA M = w), T as the bf16 pair Tb [M][2 RP] = (hi, lo), hi = bf16(T),
// lo = bf16(T - hi), zeros past r (MMA N = 2 RP; hi + lo carries T to about
// 2^-17, so the product keeps FP32 accuracy).  The epilogue adds the hi and lo
// columns.
constexpr int WD_W = 128;         // w per CTA (MMA M)
constexpr int WD_MB = 64;         // tokens per stage
constexpr int WD_BLOCK = 8192;    // one 64-column box of 64 token rows
constexpr int WD_SLACK = 16384;   // shared memory past the last stage (see below)

// Tb = (bf16(T), bf16(T - bf16(T))) as [M][2 RP], zeros past r.
__global__ void __launch_bounds__(256) hilo_kernel(const float *__restrict__ T, int64_t M, int r, int RP,
                                                   __nv_bfloat16 *__restrict__ tb)
{
    pdl_trigger();
    pdl_wait();
    const int64_t n = M * RP;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / RP;
        const int j = (int)(i % RP);
        const float t = j < r ? T[m * r + j] : 0.0f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(t);
        tb[m * 2 * RP + j] = hi;
        tb[m * 2 * RP + RP + j] = __float2bfloat16_rn(t - __bfloat162float(hi));
    }
}

struct WideParams {
    int64_t M, Wd;
    int r, S, mb, mb_split, w_tiles, wj;
    float *part;
    unsigned int *err;
    unsigned long long timeout_ns;
};

template <int RP>
__global__ void __launch_bounds__(RK_THREADS) wide_tc_kernel(const __grid_constant__ CUtensorMap d_map,
                                                             const __grid_constant__ CUtensorMap tb_map,
                                                             const WideParams p)
{
    constexpr int N = 2 * RP;                        // hi and lo columns
    constexpr int B_BYTES = (N / 64) * WD_BLOCK;     // Tb: one or two 64-column boxes
    constexpr int STAGE = 2 * WD_BLOCK + B_BYTES;    // D: two 64-column boxes
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // The barriers follow WD_SLACK bytes past the last stage, so that every
    // operand address the descriptors can form stays inside this allocation.
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.S * STAGE + WD_SLACK);
    uint64_t *empty = full + RK_MAX_S;
    uint64_t *acc_full = empty + RK_MAX_S;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *ep_ok = abort_flag + 1;  // [4]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w_tile = blockIdx.x % p.w_tiles, split = blockIdx.x / p.w_tiles;
    const int mb0 = split * p.mb_split;
    const int nmb = p.mb - mb0 < p.mb_split ? p.mb - mb0 : p.mb_split;  // >= 1: no empty split
    const int w0 = w_tile * WD_W;

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&d_map);
        prefetch_tensormap(&tb_map);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, N);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // chained launch: D and Tb are written, the partials read, by preceding work
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

    if (warp == 0) {
        // ------------------------------------------- TMA loads, one lane
        if (lane == 0) {
            const uint64_t pol_d = policy_evict_first(), pol_t = policy_evict_last();
            int s = 0, issued = 0;
            uint32_t ph = 0;
            for (int i = 0; i < nmb; ++i) {
                if (i >= p.S && !wait(&empty[s], ph ^ 1u)) break;
                uint8_t *st = smem + s * STAGE;
                const int m = (mb0 + i) * WD_MB;
                mbar_arrive_expect_tx(&full[s], (uint32_t)STAGE);
                tma_load_2d_hint(st, &d_map, &full[s], w0, m, pol_d);
                tma_load_2d_hint(st + WD_BLOCK, &d_map, &full[s], w0 + 64, m, pol_d);
#pragma unroll
                for (int b = 0; b < N / 64; ++b)
                    tma_load_2d_hint(st + 2 * WD_BLOCK + b * WD_BLOCK, &tb_map, &full[s], 64 * b, m, pol_t);
                issued = i + 1;
                if (++s == p.S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (*abort_flag)  // let the copies already issued land before the CTA exits
                for (int j = issued > p.S ? issued - p.S : 0; j < issued; ++j)
                    drain_wait(&full[j % p.S], (uint32_t)(j / p.S) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------- MMA issue (one elected lane)
        constexpr uint32_t idesc = idesc_bf16_f32_mn(WD_W, N);
        int s = 0;
        uint32_t ph = 0;
        for (int i = 0; i < nmb; ++i) {
            if (!__all_sync(0xFFFFFFFFu, wait(&full[s], ph))) break;
            tc_fence_after();
            if (elect_one()) {
                const uint32_t st = smem_u32(smem + s * STAGE);
#pragma unroll
                for (int kk = 0; kk < WD_MB / 16; ++kk) {  // 16 tokens = two 8-row groups = 2048 bytes
                    const uint64_t ad = desc_mnmajor_sw128(st + 2048u * kk, WD_BLOCK, 1024);
                    const uint64_t bd = desc_mnmajor_sw128(st + 2 * WD_BLOCK + 2048u * kk, WD_BLOCK, 1024);
                    umma_bf16(tmem, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&empty[s]);
            }
            __syncwarp();
            if (++s == p.S) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (elect_one()) umma_commit(acc_full);
        __syncwarp();
    }

    // ------------------------------------------- epilogue: TMEM lane = w, P = hi + lo
    {
        const bool ok_warp = __all_sync(0xFFFFFFFFu, wait(acc_full, 0));
        if (lane == 0) ep_ok[warp] = ok_warp ? 1 : 0;
        __syncthreads();
        const bool ok = ep_ok[0] && ep_ok[1] && ep_ok[2] && ep_ok[3] && !*abort_flag;
        tc_fence_after();
        if (ok) {
            const int64_t w = (int64_t)w0 + warp * 32 + lane;
            const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
            for (int c = 0; c < RP && c < p.r; c += 16) {
                uint32_t hi[16], lo[16];
                tmem_ld16(lane_addr + (uint32_t)c, hi);
                tmem_ld16(lane_addr + (uint32_t)(RP + c), lo);
                tmem_wait_ld();
                if (w >= p.Wd) continue;
                const int n = p.r - c < 16 ? p.r - c : 16;
                if (p.wj) {  // [split][w][j]
                    float *dst = p.part + ((int64_t)split * p.Wd + w) * p.r + c;
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (e < n) dst[e] = __uint_as_float(hi[e]) + __uint_as_float(lo[e]);
                } else {  // [split][j][w]: consecutive lanes, consecutive w
                    float *dst = p.part + ((int64_t)split * p.r + c) * p.Wd + w;
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (e < n) dst[(int64_t)e * p.Wd] = __uint_as_float(hi[e]) + __uint_as_float(lo[e]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) drain_wait(acc_full, 0);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, N);
    }
}

// Split count that fills two CTAs per SM in the fewest waves of (start-up +
// stages), for `tiles` CTAs per split over `blocks` reduction stages.
int fill_splits(int64_t tiles, int blocks)
{
    const int64_t slots = 2 * (int64_t)num_sms();
    int best = 1;
    int64_t best_cost = -1;
    for (int s = 1; s <= blocks && s <= 64; ++s) {
        const int64_t waves = (tiles * s + slots - 1) / slots;
        const int64_t cost = waves * ((blocks + s - 1) / s + RK_OVERHEAD_KB);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

struct WidePlan {
    int RP, S, mb, mb_split, splits, w_tiles;
    size_t smem;
};

WidePlan wide_plan(int64_t M, int64_t Wd, int r)
{
    WidePlan pl;
    pl.RP = r <= 32 ? 32 : 64;
    const int stage = 2 * WD_BLOCK + (2 * pl.RP / 64) * WD_BLOCK;
    pl.S = (RK_SMEM_BUDGET - WD_SLACK - 2048) / stage;
    if (pl.S > RK_MAX_S) pl.S = RK_MAX_S;
    pl.w_tiles = (int)((Wd + WD_W - 1) / WD_W);
    pl.mb = (int)((M + WD_MB - 1) / WD_MB);
    const int s = fill_splits(pl.w_tiles, pl.mb);
    pl.mb_split = (pl.mb + s - 1) / s;
    pl.splits = (pl.mb + pl.mb_split - 1) / pl.mb_split;
    pl.smem = (size_t)pl.S * stage + WD_SLACK + 1024 + 256;
    return pl;
}

struct RankPlan {
    int RP, S, kb, kb_split, splits, m_tiles;
    size_t smem;
};

RankPlan rank_plan(int64_t M, int64_t Kd, int r_max, int G)
{
    RankPlan pl;
    pl.RP = rank_tc_pad(r_max);
    const int stage = RK_X_BYTES + G * pl.RP * 128;
    pl.S = (RK_SMEM_BUDGET - 2048) / stage;
    if (pl.S > RK_MAX_S) pl.S = RK_MAX_S;
    pl.m_tiles = (int)((M + RK_M - 1) / RK_M);
    pl.kb = (int)((Kd + RK_K - 1) / RK_K);
    const int best = fill_splits(pl.m_tiles, pl.kb);
    pl.kb_split = (pl.kb + best - 1) / best;
    pl.splits = (pl.kb + pl.kb_split - 1) / pl.kb_split;  // no empty split
    pl.smem = (size_t)pl.S * stage + 1024 + 256;
    return pl;
}

struct RankEnv {
    unsigned long long timeout_ns = 2000000000ull;  // 2 s
};

}  // namespace

bool rank_tc_applies(int64_t M, int64_t Kd, int r, const void *X, const void *W)
{
    // Kd >= 64: the X box is never wider than the tensor
    return M >= 1 && Kd >= RK_K && Kd % 8 == 0 && r >= 1 && r <= 128 && aligned16(X) && aligned16(W) &&
           (M + RK_M - 1) / RK_M * 64 <= 0x7FFFFFFF && Kd <= (int64_t(1) << 31);
}

int rank_tc_splits(int64_t M, int64_t Kd) { return rank_plan(M, Kd, 32, 1).splits; }

size_t rank_tc_part_bytes(int64_t M, int64_t Kd, int r)
{
    return round256(size_t(rank_tc_splits(M, Kd)) * size_t(M) * size_t(r) * sizeof(float));
}

qerl_status rank_tc(const __nv_bfloat16 *X, int64_t M, int64_t Kd, const RankOut *outs, int G, bool chain,
                    cudaStream_t s)
{
    if (G < 1 || G > RANK_MAX_G) return QERL_ERR_INVALID_ARG;
    int r_max = 0;
    for (int g = 0; g < G; ++g) {
        if (!rank_tc_applies(M, Kd, outs[g].r, X, outs[g].W)) return QERL_ERR_SHAPE;
        r_max = outs[g].r > r_max ? outs[g].r : r_max;
    }
    if (G * rank_tc_pad(r_max) > 256) return QERL_ERR_SHAPE;  // MMA N and TMEM columns
    const RankPlan pl = rank_plan(M, Kd, r_max, G);
    RankMaps maps;
    // X: [M, Kd] bf16, 128 tokens x 64 k per box; W_g: [r_g, Kd], RP rows x 64 k
    // (rows past r_g read as zero); both with the 128-byte swizzle.
    if (!make_map_2d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)Kd, (uint64_t)M, (uint64_t)Kd * 2,
                     RK_K, RK_M, CU_TENSOR_MAP_SWIZZLE_128B))
        return QERL_ERR_CUDA;
    RankParams p;
    p.M = M;
    p.G = G;
    p.S = pl.S;
    p.kb = pl.kb;
    p.kb_split = pl.kb_split;
    p.m_tiles = pl.m_tiles;
    for (int g = 0; g < RANK_MAX_G; ++g) {
        const RankOut &o = outs[g < G ? g : 0];  // unused slots repeat group 0
        if (!make_map_2d(&maps.w[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, o.W, (uint64_t)Kd, (uint64_t)o.r,
                         (uint64_t)Kd * 2, RK_K, pl.RP, CU_TENSOR_MAP_SWIZZLE_128B))
            return QERL_ERR_CUDA;
        p.r[g] = o.r;
        p.part[g] = o.part;
    }
    p.err = error_word();
    static const RankEnv env;
    p.timeout_ns = env.timeout_ns;
    const unsigned grid = (unsigned)((int64_t)pl.m_tiles * pl.splits);
    auto kernel = pl.RP == 32 ? rank_tc_kernel<32> : pl.RP == 64 ? rank_tc_kernel<64> : rank_tc_kernel<128>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem) != cudaSuccess)
        return QERL_ERR_CUDA;
    return launched(launch_k(kernel, dim3(grid), dim3(RK_THREADS), pl.smem, s, chain, maps, p));
}

bool wide_tc_applies(int64_t M, int64_t Wd, int r, const void *D)
{
    // Wd >= 64: the D boxes are never wider than the tensor
    return M >= 1 && Wd >= 64 && Wd % 8 == 0 && r >= 1 && r <= 64 && aligned16(D) &&
           (Wd + WD_W - 1) / WD_W * 64 <= 0x7FFFFFFF && M <= (int64_t(1) << 31);
}

int wide_tc_splits(int64_t M, int64_t Wd) { return wide_plan(M, Wd, 32).splits; }

size_t wide_tc_part_bytes(int64_t M, int64_t Wd, int r)
{
    return round256(size_t(wide_tc_splits(M, Wd)) * size_t(Wd) * size_t(r) * sizeof(float));
}

size_t wide_tc_tb_bytes(int64_t M, int r) { return round256(size_t(M) * 2 * (r <= 32 ? 32 : 64) * 2); }

qerl_status wide_tc(const __nv_bfloat16 *D, int64_t M, int64_t Wd, const float *T, int r, bool wj,
                    __nv_bfloat16 *tb, bool tb_ready, float *part, bool chain, cudaStream_t s)
{
    if (!wide_tc_applies(M, Wd, r, D)) return QERL_ERR_SHAPE;
    const WidePlan pl = wide_plan(M, Wd, r);
    if (!tb_ready) {
        int64_t g = (M * pl.RP + 255) / 256;
        if (g > 4 * num_sms()) g = 4 * num_sms();
        QERL_TRY(launched(launch_k(hilo_kernel, dim3((unsigned)g), dim3(256), 0, s, chain, T, M, r, pl.RP, tb)));
    }
    CUtensorMap dm, tm;
    // D: [M, Wd] bf16, 64 columns x 64 tokens per box; Tb: [M, 2 RP], the same
    // box; both with the 128-byte swizzle (MN-major operands).
    if (!make_map_2d(&dm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)Wd, (uint64_t)M, (uint64_t)Wd * 2, 64,
                     WD_MB, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, tb, (uint64_t)(2 * pl.RP), (uint64_t)M,
                     (uint64_t)(4 * pl.RP), 64, WD_MB, CU_TENSOR_MAP_SWIZZLE_128B))
        return QERL_ERR_CUDA;
    WideParams p;
    p.M = M;
    p.Wd = Wd;
    p.r = r;
    p.S = pl.S;
    p.mb = pl.mb;
    p.mb_split = pl.mb_split;
    p.w_tiles = pl.w_tiles;
    p.wj = wj ? 1 : 0;
    p.part = part;
    p.err = error_word();
    static const RankEnv env;
    p.timeout_ns = env.timeout_ns;
    const unsigned grid = (unsigned)((int64_t)pl.w_tiles * pl.splits);
    auto kernel = pl.RP == 32 ? wide_tc_kernel<32> : wide_tc_kernel<64>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem) != cudaSuccess)
        return QERL_ERR_CUDA;
    return launched(launch_k(kernel, dim3(grid), dim3(RK_THREADS), pl.smem, s, chain, dm, tm, p));
}

}  // namespace qerl
