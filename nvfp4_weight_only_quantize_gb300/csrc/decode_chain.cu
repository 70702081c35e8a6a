// Persistent decoder-chain kernel: every NVFP4 + LoRA linear of a chain of
// decoder layers at decode batch sizes (M <= 64 tokens), with the AQN-RMSNorm,
// residual and SwiGLU steps between them, in one launch of one CTA per SM.
//
// Per layer (Qwen2.5 decoder layer; attention itself is outside the path and
// its output is an input):
//     a = AQN-RMSNorm(h0)        q, k, v = a W_{q,k,v}^T (+ LoRA)
//     h1 = h0 + attn W_o^T       b = AQN-RMSNorm(h1)
//     g, u = b W_{gate,up}^T     m = silu(g) * u
//     h2 = h1 + m W_down^T       (h2 feeds the next layer)
// The AQN noise enters the norm's scale (dataforcee "QERL: NVFP4-intensive
// learning", AQN paragraph: the noise lives in the norm's scale parameters so
// that kernel fusion stays small), so the norm folds into its neighbours:
//   - the producer of h (o_proj, down_proj) writes xn = bf16(h * (gamma +
//     sigma z)) and the sum of squares of h per token over its 128 columns;
//   - the consumer (q/k/v, gate/up) runs the linear on xn and scales each
//     token's output row by rs = rsqrt(mean h^2 + eps): the linear and its
//     LoRA branch are both linear in the input, so y = rs * (xn W^T + s (xn
//     A^T) B^T) equals the linear of the normalized input.
//
// Work is split into phases (noise, first norm, then per layer q|k|v|o,
// gate|up, SwiGLU, down); a phase starts consuming activations once every unit
// of the phase before it has completed (global counters, bounded waits, a
// cooperative launch so that every CTA is resident).  The weight stream never
// waits on activations: each CTA's producer streams the codes of all its jobs
// back to back, so a phase boundary costs only the dependency latency.
//
// Each phase's (tile, 256-k chunk) units are divided evenly over the CTAs; a
// tile split across CTAs is summed by the last of its parts to finish, in part
// order (deterministic).  Each part also runs its own LoRA down-projection on
// its k-range (t_s = x A^T on tensor cores) and adds s t_s B^T; the sum over
// parts is the LoRA term.
//
// Warp roles (480 threads, one CTA per SM):
//   warps 0-7   dequantize (two groups of four, alternate stages) into TMEM
//   warp 8      TMA: packed codes + block scales, one 256-k stage at a time
//   warp 9      TMA: input tiles x and LoRA A rows, after the phase dependency
//   warp 10     TMEM owner, MMA issue (main, t_s and LoRA up-projection)
//   warps 11-14 epilogue: builds u_s, drains the accumulator, sums parts, the
//               fused norm / residual output, and the glue steps
// Every wait is bounded (global timer); on expiry the CTA latches
// QERL_ERR_TIMEOUT, every role leaves its loop, TMEM is freed and the CTA exits.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <vector>

#include "chain.cuh"
#include "dequant.cuh"
#include "linear.cuh"
#include "sm100_ptx.cuh"

namespace qerl {
namespace chain {
namespace {

using namespace ptx;

constexpr int BK = 64;                               // k per MMA k-step
constexpr int GK = KC / BK;                          // k-steps per stage
constexpr int RAW_CODES = TILE_N * KC / 2;           // 16 KB
constexpr int RAW_SCALES = TILE_N * KC / 16;         // 2 KB
constexpr int RAW_STAGE = RAW_CODES + RAW_SCALES;    // 18 KB
constexpr int DQG = 2;                               // dequant groups
constexpr int NUM_DQ_WARPS = 4 * DQG;
constexpr int WARP_RAW = 8, WARP_X = 9, WARP_MMA = 10, WARP_EPI = 11;
constexpr int NUM_THREADS = 15 * 32;
constexpr int EPI_THREADS = 128;
constexpr int S = 3;                                 // A slots (256 k = 128 TMEM columns)
constexpr int ACC_COL = 0, T_COL = 64, A_COL0 = 128, TMEM_COLS = 512;
constexpr int X_STEP = BN * BK * 2;                  // 8 KB
constexpr int X_STAGE = X_STEP * GK;                 // 32 KB
constexpr int Y_BYTES = BN * TILE_N * 2;             // bf16 output staging [64 tokens][128 rows]
constexpr int BAR_BYTES = 2048;
constexpr int BAR_EPI = 1;                           // named barrier of the epilogue warps

template <int RL>
struct Cfg {
    static constexpr int AL_STEP = RL * BK * 2;      // LoRA A rows of one k-step
    static constexpr int AL_STAGE = AL_STEP * GK;
    static constexpr int XS = RL <= 32 ? 3 : 2;      // input stages
    static constexpr int R = RL <= 32 ? 3 : 4;       // raw stages
    static_assert(R >= S, "raw ring at least as deep as the A ring (parity-safe waits)");
    static constexpr int SMEM = XS * X_STAGE + XS * AL_STAGE + R * RAW_STAGE + Y_BYTES + BAR_BYTES + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    // a t_s MMA reads 128 rows (16 KB) of A from each k-step's start: the raw
    // ring after the LoRA-A ring keeps every address inside the allocation
    static_assert(R * RAW_STAGE >= 16384, "t_s MMA window");
};

__device__ __forceinline__ int ld_acquire_gpu(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_gpu_add(int *p, int v)
{
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Philox4x64-10 (Salmon et al., SC'11): the noise stream of AQN, keyed by
// (seed, norm index), counter (channel block, step, 0, 0); Box-Muller in FP32.
__device__ __forceinline__ void philox4x64_10(uint64_t c[4], uint64_t k0, uint64_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint64_t a0 = 0xD2E7470EE14C6C93ull * c[0], h0 = __umul64hi(0xD2E7470EE14C6C93ull, c[0]);
        const uint64_t a1 = 0xCA5A826395121157ull * c[2], h1 = __umul64hi(0xCA5A826395121157ull, c[2]);
        c[0] = h1 ^ c[1] ^ k0;
        c[1] = a1;
        c[2] = h0 ^ c[3] ^ k1;
        c[3] = a0;
        k0 += 0x9E3779B97F4A7C15ull;
        k1 += 0xBB67AE8584CAA73Bull;
    }
}
// u1 = ((w0 >> 11) + 1) 2^-53, u2 = (w1 >> 11) 2^-53; ln u1 as log1p(-(1 - u1))
// near 1, where 1 - u1 (formed exactly in integers) would round away in FP32.
__device__ __forceinline__ void box_muller_f32(uint64_t w0, uint64_t w1, float &z0, float &z1)
{
    const uint64_t a = (w0 >> 11) + 1ull;
    const float lnu1 = a > (1ull << 52) ? log1pf(-(float)((1ull << 53) - a) * 0x1p-53f) : logf((float)a * 0x1p-53f);
    const float rad = sqrtf(-2.0f * lnu1);
    float sn, cs;
    sincospif(2.0f * ((float)(w1 >> 11) * 0x1p-53f), &sn, &cs);
    z0 = rad * cs;
    z1 = rad * sn;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

template <int RL, bool PACKED>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    chain_kernel(const __grid_constant__ Plan P, float sigma, unsigned long long seed, unsigned long long step,
                 unsigned int first_layer)
{
    using C = Cfg<RL>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *X_ring = smem;
    uint8_t *AL_ring = X_ring + C::XS * X_STAGE;
    uint8_t *R_ring = AL_ring + C::XS * C::AL_STAGE;
    uint8_t *Ystage = R_ring + C::R * RAW_STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(Ystage + Y_BYTES);
    uint64_t *raw_full = bars;
    uint64_t *raw_empty = raw_full + C::R;
    uint64_t *x_full = raw_empty + C::R;
    uint64_t *x_empty = x_full + C::XS;
    uint64_t *a_full = x_empty + C::XS;
    uint64_t *stage_empty = a_full + S;
    uint64_t *acc_full = stage_empty + S;   // the job's last MMA done
    uint64_t *acc_empty = acc_full + 1;     // the epilogue has read the accumulator
    uint64_t *t_full = acc_empty + 1;       // the job's t_s MMAs done
    uint64_t *t_empty = t_full + 1;         // u_s built from t_s
    uint64_t *drain = t_empty + 1;          // every MMA of the CTA done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *bcast = abort_flag + 1;   // epilogue broadcast word
    float *rs_s = reinterpret_cast<float *>(bars + 64);   // [64] per-token norm factors
    float *red_s = rs_s + BN;                             // [128] epilogue scratch
    float *ns_s = red_s + EPI_THREADS;                    // [128] a tile's next-norm scale
    volatile int *rs_phase = reinterpret_cast<volatile int *>(ns_s + TILE_N);  // phase whose input rs is in rs_s

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int jb = P.job_off[blockIdx.x], je = P.job_off[blockIdx.x + 1];

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::R; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], 4);
        }
        for (int i = 0; i < C::XS; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 1);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(&a_full[i], 4);
            mbar_init(&stage_empty[i], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 1);
        mbar_init(t_full, 1);
        mbar_init(t_empty, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        *rs_phase = -1;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const unsigned long long deadline = globaltimer_ns() + P.timeout_ns;

    auto fail = [&]() {
        *abort_flag = 1;
        latch_error(P.err, QERL_ERR_TIMEOUT);
    };
    // Bounded wait for the phase with this parity; false once the CTA aborts.
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        for (;;) {
            if (*abort_flag) return false;
            if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
            if (globaltimer_ns() > deadline) {
                fail();
                return false;
            }
        }
    };
    // Lane 0 waits, the warp learns the outcome (and is ordered after it).
    auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        const bool ok = __shfl_sync(0xFFFFFFFFu, lane == 0 ? (wait(bar, parity) ? 1 : 0) : 0, 0) != 0;
        __syncwarp();
        return ok;
    };
    // Bounded wait until another phase's counter reaches its total (lane 0).
    auto wait_phase = [&](int ph) -> bool {
        if (ph < 0) return true;
        const int target = P.phase_total[ph];
        for (;;) {
            if (ld_acquire_gpu(&P.phase_cnt[ph]) >= target) return true;
            if (*abort_flag) return false;
            if (globaltimer_ns() > deadline) {
                fail();
                return false;
            }
            __nanosleep(128);
        }
    };
    auto drain_wait = [&](uint64_t *bar, uint32_t parity) {
        const unsigned long long until = globaltimer_ns() + 100000000ull;  // 100 ms
        while (!mbar_try_wait(bar, parity) && globaltimer_ns() < until) {
        }
    };

    if (warp == WARP_RAW) {
        // ------------------------------------------- codes + scales of every job
        const uint64_t pol = policy_evict_first();
        int rj = 0;
        bool ok = true;
        for (int q = jb; q < je && ok; ++q) {
            const Job J = P.jobs[q];
            if (J.type != 0) continue;
            const LinMaps *mp = &P.maps[J.idx];
            for (int kc = J.kc0; kc < J.kc1; ++kc, ++rj) {
                const int slot = rj % C::R;
                const int round = rj / C::R;
                if (round > 0 && !warp_wait(&raw_empty[slot], (uint32_t)(round - 1) & 1u)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    mbar_arrive_expect_tx(&raw_full[slot], RAW_STAGE);
                    uint8_t *dst = R_ring + slot * RAW_STAGE;
                    tma_load_2d_hint(dst, &mp->codes, &raw_full[slot], kc * (KC / 2), J.tile * TILE_N, pol);
                    tma_load_2d_hint(dst + RAW_CODES, &mp->scl, &raw_full[slot], kc * (KC / 16), J.tile * TILE_N, pol);
                }
                __syncwarp();
            }
        }
        if (*abort_flag && lane == 0)  // the copies already issued land before the CTA exits
            for (int i = rj > C::R ? rj - C::R : 0; i < rj; ++i) drain_wait(&raw_full[i % C::R], (uint32_t)(i / C::R) & 1u);
        __syncwarp();
    } else if (warp == WARP_X) {
        // ------------------------------------------- input tiles + LoRA A rows
        const uint64_t pol = policy_evict_last();
        int j = 0, waited = -1, issued = 0;
        bool ok = true;
        for (int q = jb; q < je && ok; ++q) {
            const Job J = P.jobs[q];
            if (J.type != 0) continue;
            const int ph = P.lins[J.idx].phase;
            if (ph - 1 > waited) {  // every unit of the phase before has completed
                ok = __shfl_sync(0xFFFFFFFFu, lane == 0 ? (wait_phase(ph - 1) ? 1 : 0) : 0, 0) != 0;
                if (!ok) break;
                if (lane == 0) fence_proxy_async_global();  // the TMA reads what other CTAs wrote
                __syncwarp();
                waited = ph - 1;
            }
            const LinMaps *mp = &P.maps[J.idx];
            for (int kc = J.kc0; kc < J.kc1; ++kc, ++j) {
                const int slot = j % C::XS;
                const int round = j / C::XS;
                if (round > 0 && !warp_wait(&x_empty[slot], (uint32_t)(round - 1) & 1u)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    // one copy each: the stage's four 64-k blocks of x and of the LoRA A rows
                    mbar_arrive_expect_tx(&x_full[slot], X_STAGE + C::AL_STAGE);
                    tma_load_3d_hint(X_ring + slot * X_STAGE, &mp->x, &x_full[slot], 0, 0, kc * GK, pol);
                    tma_load_3d_hint(AL_ring + slot * C::AL_STAGE, &mp->al, &x_full[slot], 0, 0, kc * GK, pol);
                }
                __syncwarp();
                issued = j + 1;
            }
            ++j;  // the LoRA stage: its slot is filled by the epilogue warps (u_s)
        }
        if (*abort_flag && lane == 0)
            for (int i = issued > C::XS ? issued - C::XS : 0; i < issued; ++i)
                drain_wait(&x_full[i % C::XS], (uint32_t)(i / C::XS) & 1u);
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------- MMA issue (converged warp, elected lane)
        constexpr uint32_t idesc = idesc_bf16_f32(TILE_N, BN);
        const uint64_t bd0 = desc_kmajor_sw128(smem_u32(X_ring));
        int j = 0, ji = 0;
        bool ok = true;
        for (int q = jb; q < je && ok; ++q) {
            const Job J = P.jobs[q];
            if (J.type != 0) continue;
            if (ji > 0) {  // the accumulator and t_s of the previous job are drained
                ok = warp_wait(acc_empty, (uint32_t)(ji - 1) & 1u) && warp_wait(t_empty, (uint32_t)(ji - 1) & 1u);
                if (!ok) break;
            }
            const int nmain = J.kc1 - J.kc0;
            for (int st = 0; st <= nmain && ok; ++st, ++j) {
                const int s = j % S, xs = j % C::XS;
                ok = warp_wait(&a_full[s], (uint32_t)(j / S) & 1u) && warp_wait(&x_full[xs], (uint32_t)(j / C::XS) & 1u);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t at = tmem + (uint32_t)(A_COL0 + s * 32 * GK);
                    const uint64_t bd = bd0 + (uint64_t)((xs * X_STAGE) >> 4);
                    if (st < nmain) {
#pragma unroll
                        for (int sub = 0; sub < GK; ++sub) {
                            const uint64_t ad =
                                desc_kmajor_sw128(smem_u32(AL_ring + xs * C::AL_STAGE + sub * C::AL_STEP));
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk) {
                                const uint32_t acc = (st > 0 || sub > 0 || kk > 0) ? 1u : 0u;
                                const uint64_t b = bd + (uint64_t)((sub * X_STEP) >> 4) + 2u * kk;
                                umma_bf16_ts(tmem + ACC_COL, at + (uint32_t)(sub * 32 + 8 * kk), b, idesc, acc);
                                umma_bf16(tmem + T_COL, ad + 2u * kk, b, idesc, acc);
                            }
                        }
                        umma_commit(&stage_empty[s]);
                        umma_commit(&x_empty[xs]);
                        if (st == nmain - 1) umma_commit(t_full);
                    } else {
                        // LoRA up-projection: B rows (TMEM) x u_s (the stage's input slot)
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            umma_bf16_ts(tmem + ACC_COL, at + (uint32_t)(8 * kk), bd + 2u * kk, idesc, 1u);
                        umma_commit(&stage_empty[s]);
                        umma_commit(&x_empty[xs]);
                        umma_commit(acc_full);
                    }
                }
                __syncwarp();
            }
            ++ji;
        }
        if (elect_one()) umma_commit(drain);  // arrives once every MMA issued above has completed
        __syncwarp();
    } else if (warp < NUM_DQ_WARPS) {
        // ------------------------------------------- dequantize (one weight row per thread)
        const int row = (warp & 3) * 32 + lane;
        const int group = warp >> 2;
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        int j = 0, rj = 0;
        bool ok = true;
        for (int q = jb; q < je && ok; ++q) {
            const Job J = P.jobs[q];
            if (J.type != 0) continue;
            const Lin &L = P.lins[J.idx];
            const int nmain = J.kc1 - J.kc0;
            const float pow2 = pow2f(126 - tc_exponent_offset(*L.ts));
            for (int st = 0; st <= nmain; ++st, ++j) {
                const bool main_stage = st < nmain;
                if (j % DQG == group) {
                    const int s = j % S;
                    const int rs = rj % C::R;
                    if (j >= S && !warp_wait(&stage_empty[s], (uint32_t)(j / S - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    if (main_stage && !warp_wait(&raw_full[rs], (uint32_t)(rj / C::R) & 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t tcol = trow + (uint32_t)(A_COL0 + s * 32 * GK);
                    if (main_stage) {
                        // every code and scale of the row first (all loads in flight); the raw
                        // slot goes back once every loaded word has been used
                        const uint8_t *rb = R_ring + rs * RAW_STAGE;
                        uint4 cw[2 * GK];
#pragma unroll
                        for (int sub = 0; sub < GK; ++sub) {
                            cw[2 * sub] = *reinterpret_cast<const uint4 *>(rb + row * 128 + (((2 * sub) ^ (row & 7)) * 16));
                            cw[2 * sub + 1] =
                                *reinterpret_cast<const uint4 *>(rb + row * 128 + (((2 * sub + 1) ^ (row & 7)) * 16));
                        }
                        const uint4 scv = *reinterpret_cast<const uint4 *>(rb + RAW_CODES + row * 16);
                        const uint32_t scw[GK] = {scv.x, scv.y, scv.z, scv.w};
#pragma unroll
                        for (int sub = 0; sub < GK; ++sub) {
                            uint32_t out[32];
                            const uint32_t sc = scw[sub];
                            const uint32_t f0 = scale_factor_bf16x2(sc << 20, pow2);
                            const uint32_t f1 = scale_factor_bf16x2(sc << 12, pow2);
                            const uint32_t f2 = scale_factor_bf16x2(sc << 4, pow2);
                            const uint32_t f3 = scale_factor_bf16x2(sc >> 4, pow2);
                            const uint4 c0 = cw[2 * sub], c1 = cw[2 * sub + 1];
                            dequant_word<PACKED>(c0.x, f0, out + 0);
                            dequant_word<PACKED>(c0.y, f0, out + 4);
                            dequant_word<PACKED>(c0.z, f1, out + 8);
                            dequant_word<PACKED>(c0.w, f1, out + 12);
                            dequant_word<PACKED>(c1.x, f2, out + 16);
                            dequant_word<PACKED>(c1.y, f2, out + 20);
                            dequant_word<PACKED>(c1.z, f3, out + 24);
                            dequant_word<PACKED>(c1.w, f3, out + 28);
                            tmem_st32(tcol + (uint32_t)(sub * 32), out);
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&raw_empty[rs]);
                    } else {
                        // LoRA up-projection rows B[n, 0..63], zero past r (r % 8 == 0)
                        uint32_t out[32];
                        const __nv_bfloat16 *b = L.B + (size_t)(J.tile * TILE_N + row) * L.r;
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            const uint4 w = (v * 8 < L.r) ? __ldg(reinterpret_cast<const uint4 *>(b) + v)
                                                          : make_uint4(0u, 0u, 0u, 0u);
                            out[4 * v] = w.x;
                            out[4 * v + 1] = w.y;
                            out[4 * v + 2] = w.z;
                            out[4 * v + 3] = w.w;
                        }
                        tmem_st32(tcol, out);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&a_full[s]);
                }
                if (main_stage) ++rj;
            }
        }
    } else {
        // ------------------------------------------- epilogue warps (11-14) and glue
        const int et = threadIdx.x - WARP_EPI * 32;  // 0..127
        const int quad = warp & 3;                   // TMEM lanes 32*quad ..
        const int row = quad * 32 + lane;            // weight row of the tile held by this thread
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        int j = 0, ji = 0;
        bool ok = true;
        for (int q = jb; q < je && ok; ++q) {
            const Job J = P.jobs[q];
            if (J.type == 1) {
                // ------------------------------- glue step unit
                const Glue &G = P.glues[J.idx];
                if (et == 0) *bcast = wait_phase(G.phase - 1) ? 1 : 0;
                named_bar_sync(BAR_EPI, EPI_THREADS);
                ok = *bcast != 0;
                named_bar_sync(BAR_EPI, EPI_THREADS);
                if (!ok) break;
                if (G.kind == GLUE_NOISE) {
                    // Philox block b of norm k: channels 4i .. 4i+3 of that norm
                    const int nb = (G.width + 3) / 4;
                    const int blk = J.tile * EPI_THREADS + et;
                    if (blk < G.n_norms * nb) {
                        const int k = blk / nb, i = blk % nb;
                        uint64_t w[4] = {(uint64_t)i, (uint64_t)step, 0ull, 0ull};
                        philox4x64_10(w, (uint64_t)seed, (uint64_t)(2u * first_layer + (unsigned)k));
                        float z[4];
                        box_muller_f32(w[0], w[1], z[0], z[1]);
                        box_muller_f32(w[2], w[3], z[2], z[3]);
                        const __nv_bfloat16 *gm = G.gammas[k];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = 4 * i + e;
                            if (c < G.width) G.ns[(size_t)k * G.width + c] = bf16f(gm[c]) + sigma * z[e];
                        }
                    }
                } else if (G.kind == GLUE_PRENORM) {
                    // tile J.tile of the first norm's input: xn = bf16(x * ns), sum of squares
                    ns_s[et] = G.ns[J.tile * TILE_N + et];
                    named_bar_sync(BAR_EPI, EPI_THREADS);
                    const int m = et >> 1, cb = (et & 1) * 64;
                    const __nv_bfloat16 *xr = G.a + (size_t)m * G.width + J.tile * TILE_N + cb;
                    uint4 xv[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)  // every load in flight before the math
                        xv[c] = m < P.M ? *reinterpret_cast<const uint4 *>(xr + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
                    float ss = 0.0f;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t xw[4] = {xv[c].x, xv[c].y, xv[c].z, xv[c].w};
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float a0 = bf16lo(xw[e]), a1 = bf16hi(xw[e]);
                            ss = fmaf(a0, a0, ss);
                            ss = fmaf(a1, a1, ss);
                            const __nv_bfloat162 p2 = __floats2bfloat162_rn(a0 * ns_s[cb + 8 * c + 2 * e],
                                                                            a1 * ns_s[cb + 8 * c + 2 * e + 1]);
                            o[e] = *reinterpret_cast<const uint32_t *>(&p2);
                        }
                        if (m < P.M)
                            *reinterpret_cast<uint4 *>(G.out + (size_t)m * G.width + J.tile * TILE_N + cb + 8 * c) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
                    if ((et & 1) == 0) G.sq[J.tile * BN + m] = ss;
                } else {
                    // SwiGLU over columns [unit * cols, +cols)
                    const int c0 = J.tile * G.cols, c1 = min(G.width, c0 + G.cols);
                    const int vecs = (c1 - c0) / 8, items = P.M * vecs;
                    for (int it0 = et; it0 < items; it0 += 4 * EPI_THREADS) {
                        uint4 gv[4], uv[4];
#pragma unroll
                        for (int b = 0; b < 4; ++b) {  // four items' loads in flight at once
                            const int it = it0 + b * EPI_THREADS;
                            const int m = it / vecs, c = c0 + (it % vecs) * 8;
                            gv[b] = it < items ? *reinterpret_cast<const uint4 *>(G.a + (size_t)m * G.width + c)
                                               : make_uint4(0u, 0u, 0u, 0u);
                            uv[b] = it < items ? *reinterpret_cast<const uint4 *>(G.b + (size_t)m * G.width + c)
                                               : make_uint4(0u, 0u, 0u, 0u);
                        }
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            const int it = it0 + b * EPI_THREADS;
                            if (it >= items) break;
                            const int m = it / vecs, c = c0 + (it % vecs) * 8;
                            const uint32_t gw[4] = {gv[b].x, gv[b].y, gv[b].z, gv[b].w};
                            const uint32_t uw[4] = {uv[b].x, uv[b].y, uv[b].z, uv[b].w};
                            uint32_t o[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 p2 = __floats2bfloat162_rn(silu(bf16lo(gw[e])) * bf16lo(uw[e]),
                                                                                silu(bf16hi(gw[e])) * bf16hi(uw[e]));
                                o[e] = *reinterpret_cast<const uint32_t *>(&p2);
                            }
                            *reinterpret_cast<uint4 *>(G.out + (size_t)m * G.width + c) = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                }
                __threadfence();
                fence_proxy_async_global();
                named_bar_sync(BAR_EPI, EPI_THREADS);
                if (et == 0) red_release_gpu_add(&P.phase_cnt[G.phase], 1);
                continue;
            }

            // ----------------------------------- matmul job
            const Lin &L = P.lins[J.idx];
            if (L.kind == LIN_NORMED && *rs_phase != L.phase) {
                // rs = rsqrt(mean h^2 + eps) of the linear's (normed) input, once per
                // input: the partial sums are final once the phase before has completed
                if (et == 0) *bcast = wait_phase(L.phase - 1) ? 1 : 0;
                named_bar_sync(BAR_EPI, EPI_THREADS);
                ok = *bcast != 0;
                if (!ok) break;
                const int m = et & (BN - 1), hf = et / BN;  // token, half of the tiles
                float ss = 0.0f;
                for (int i0 = hf * 16; i0 < L.sq_tiles; i0 += 32) {
                    float sv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) sv[e] = i0 + e < L.sq_tiles ? L.sq_in[(i0 + e) * BN + m] : 0.0f;
#pragma unroll
                    for (int e = 0; e < 16; ++e) ss += sv[e];
                }
                red_s[et] = ss;
                named_bar_sync(BAR_EPI, EPI_THREADS);
                if (et < BN) rs_s[et] = rsqrtf((red_s[et] + red_s[et + BN]) / (float)L.K + P.eps);
                if (et == 0) *rs_phase = L.phase;
                named_bar_sync(BAR_EPI, EPI_THREADS);
            }
            const int nmain = J.kc1 - J.kc0;

            const int jl = j + nmain;  // the job's LoRA stage
            j = jl + 1;
            const float st = *L.ts;
            const float ysc = st * pow2f(tc_exponent_offset(st));
            // u_s = bf16(s t_s / ysc) into the LoRA stage's input slot: token rows of
            // 64 ranks (128 B, the 128-byte swizzle), zeros past r
            bool wok = warp_wait(t_full, (uint32_t)ji & 1u);
            const int xs = jl % C::XS;
            if (wok && jl >= C::XS) wok = warp_wait(&x_empty[xs], (uint32_t)(jl / C::XS - 1) & 1u);
            tc_fence_after();
            if (wok && quad < 2) {
                const int jr = quad * 32 + lane;  // rank
                const float fac = P.lora_scale / ysc;
                uint8_t *dst = X_ring + xs * X_STAGE;
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    uint32_t tr[16];
                    if (quad * 32 < RL) {
                        tmem_ld16(tl + (uint32_t)(T_COL + c0), tr);
                        tmem_wait_ld();
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int m = c0 + e;
                        const bool live = quad * 32 < RL && jr < L.r;
                        const __nv_bfloat16 uv = __float2bfloat16_rn(live ? __uint_as_float(tr[e]) * fac : 0.0f);
                        *reinterpret_cast<__nv_bfloat16 *>(dst + m * 128 + ((((jr >> 3) ^ (m & 7)) << 4) | ((jr & 7) << 1))) =
                            uv;
                    }
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();  // the MMA reads u_s through the async proxy
            wok = named_bar_and(BAR_EPI, EPI_THREADS, wok);
            if (wok && et == 0) {
                mbar_arrive(t_empty);
                mbar_arrive(&x_full[xs]);
            }
            // the accumulator: this thread's weight row, 64 tokens
            wok = wok && warp_wait(acc_full, (uint32_t)ji & 1u);
            tc_fence_after();
            float v[BN];
            if (wok) {
#pragma unroll
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    uint32_t tr[16];
                    tmem_ld16(tl + (uint32_t)(ACC_COL + c0), tr);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[c0 + e] = __uint_as_float(tr[e]);
                }
            }
            tc_fence_before();
            wok = named_bar_and(BAR_EPI, EPI_THREADS, wok);
            if (wok && et == 0) mbar_arrive(acc_empty);
            ++ji;
            if (!wok) {
                ok = false;
                break;
            }
            if (J.nparts > 1) {
                // this part's partial tile [token][row] (a warp's 32 rows of one token
                // are 128 contiguous bytes); the last part of the tile to finish sums them
                float *part = P.partials + (size_t)J.slot * (TILE_N * BN) + row;
#pragma unroll
                for (int c = 0; c < BN; ++c) __stcg(part + (size_t)c * TILE_N, v[c]);
                __threadfence();
                named_bar_sync(BAR_EPI, EPI_THREADS);
                if (et == 0) {
                    const int old = atomicAdd(&P.tile_cnt[L.tile0 + J.tile], 1);
                    *bcast = old == J.nparts - 1 ? 1 : 0;
                }
                named_bar_sync(BAR_EPI, EPI_THREADS);
                const bool last = *bcast != 0;
                named_bar_sync(BAR_EPI, EPI_THREADS);
                if (!last) continue;
                __threadfence();
                const float *p0 = P.partials + (size_t)(J.slot - J.part) * (TILE_N * BN) + row;
#pragma unroll
                for (int c = 0; c < BN; ++c) v[c] = 0.0f;
                for (int pi = 0; pi < J.nparts; ++pi) {  // in part order (deterministic)
                    const float *pp = p0 + (size_t)pi * (TILE_N * BN);
                    float w[BN];  // every load of the part in flight before the adds
#pragma unroll
                    for (int c = 0; c < BN; ++c) w[c] = __ldcg(pp + (size_t)c * TILE_N);
#pragma unroll
                    for (int c = 0; c < BN; ++c) v[c] += w[c];
                }
                if (et == 0) P.tile_cnt[L.tile0 + J.tile] = 0;  // clean for the next launch
            }
            // ----------------------------------- final epilogue of the tile
            const int n0 = J.tile * TILE_N;
            __nv_bfloat16 *Y = reinterpret_cast<__nv_bfloat16 *>(Ystage);
            if (L.kind == LIN_NORMED) {
#pragma unroll
                for (int m = 0; m < BN; ++m) Y[m * TILE_N + row] = __float2bfloat16_rn(v[m] * ysc * rs_s[m]);
                named_bar_sync(BAR_EPI, EPI_THREADS);
                if (L.y) {
                    for (int it = et; it < P.M * (TILE_N / 8); it += EPI_THREADS) {
                        const int m = it / (TILE_N / 8), c = (it % (TILE_N / 8)) * 8;
                        *reinterpret_cast<uint4 *>(L.y + (size_t)m * L.N + n0 + c) =
                            *reinterpret_cast<const uint4 *>(Y + m * TILE_N + c);
                    }
                }
            } else {
                // h_out = bf16(h_in + bf16(v)), xn = bf16(h_out * ns), sum of squares of h_out
#pragma unroll
                for (int m = 0; m < BN; ++m) Y[m * TILE_N + row] = __float2bfloat16_rn(v[m] * ysc);
                if (L.xn_out) ns_s[et] = L.ns_next[n0 + et];
                named_bar_sync(BAR_EPI, EPI_THREADS);
                const int m = et >> 1, cb = (et & 1) * 64;
                float ss = 0.0f;
                if (m < P.M) {
                    uint4 hin[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)  // every load in flight before the math
                        hin[c] = *reinterpret_cast<const uint4 *>(L.h_in + (size_t)m * L.N + n0 + cb + 8 * c);
#pragma unroll
                    for (int ci = 0; ci < 8; ++ci) {
                        const int c = cb + 8 * ci;
                        const uint4 yv = *reinterpret_cast<const uint4 *>(Y + m * TILE_N + c);
                        const uint4 hv = hin[ci];
                        const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w}, hw[4] = {hv.x, hv.y, hv.z, hv.w};
                        uint32_t ho[4], xo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __nv_bfloat162 h2 =
                                __floats2bfloat162_rn(bf16lo(hw[e]) + bf16lo(yw[e]), bf16hi(hw[e]) + bf16hi(yw[e]));
                            ho[e] = *reinterpret_cast<const uint32_t *>(&h2);
                            const float a0 = bf16lo(ho[e]), a1 = bf16hi(ho[e]);
                            ss = fmaf(a0, a0, ss);
                            ss = fmaf(a1, a1, ss);
                            if (L.xn_out) {
                                const __nv_bfloat162 x2 =
                                    __floats2bfloat162_rn(a0 * ns_s[c + 2 * e], a1 * ns_s[c + 2 * e + 1]);
                                xo[e] = *reinterpret_cast<const uint32_t *>(&x2);
                            }
                        }
                        *reinterpret_cast<uint4 *>(L.h_out + (size_t)m * L.N + n0 + c) = make_uint4(ho[0], ho[1], ho[2], ho[3]);
                        if (L.xn_out)
                            *reinterpret_cast<uint4 *>(L.xn_out + (size_t)m * L.N + n0 + c) =
                                make_uint4(xo[0], xo[1], xo[2], xo[3]);
                    }
                }
                ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
                if (L.sq_out && (et & 1) == 0) L.sq_out[J.tile * BN + m] = ss;
            }
            __threadfence();
            fence_proxy_async_global();
            named_bar_sync(BAR_EPI, EPI_THREADS);  // also: Y and rs_s are free again
            if (et == 0) red_release_gpu_add(&P.phase_cnt[L.phase], 1);
        }
    }

    // ------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        if (lane == 0) drain_wait(drain, 0);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    if (threadIdx.x == 0) {
        // The last CTA to leave returns the phase counters to zero for the next launch.
        __threadfence();
        const int old = atomicAdd(P.exit_cnt, 1);
        if (old == P.n_ctas - 1 && !*abort_flag) {
            __threadfence();
            for (int i = 0; i < P.n_phases; ++i) P.phase_cnt[i] = 0;
            *P.exit_cnt = 0;
            __threadfence();
        }
    }
}

}  // namespace
}  // namespace chain
}  // namespace qerl

// ------------------------------------------------------------------ host side

namespace qerl {
namespace chain {
namespace {

struct Layout {
    size_t off_lins = 0, off_maps = 0, off_glues = 0, off_gammas = 0, off_jobs = 0, off_joboff = 0, off_ptotal = 0;
    size_t off_pcnt = 0, off_tcnt = 0, off_exit = 0, off_part = 0;
    size_t off_xn1 = 0, off_xn2 = 0, off_sq1 = 0, off_sq2 = 0, off_hmid = 0, off_hbuf = 0, off_g = 0, off_u = 0;
    size_t off_m = 0, off_ns = 0, off_q = 0, off_k = 0, off_v = 0, total = 0;
    size_t zero_begin = 0, zero_end = 0;
};

struct Sizes {
    int n_lin, n_glue, n_phases, max_jobs, max_tiles, max_parts;
};

// Upper bounds of the tables for L layers on C CTAs.
Sizes table_sizes(const qerl_decoder_dims &d, int L, int C)
{
    Sizes z;
    z.n_lin = 7 * L;
    z.n_glue = 2 + L;
    z.n_phases = 2 + 4 * L;
    const int H = (int)d.hidden;
    const int tiles_qkvo = (int)((2 * d.hidden + 2 * d.kv_dim) / TILE_N);
    const int tiles_gu = (int)(2 * d.intermediate / TILE_N);
    const int tiles_down = H / TILE_N;
    z.max_tiles = std::max(tiles_qkvo, std::max(tiles_gu, tiles_down));
    z.max_parts = z.max_tiles + C;  // a CTA's contiguous range splits at most one extra tile
    // jobs per matmul phase <= tiles + C; SwiGLU units <= C; noise units: one per
    // 128 Philox blocks; first-norm units: one per 128 columns
    const int noise_units = (2 * L * ((H + 3) / 4) + EPI_THREADS - 1) / EPI_THREADS;
    z.max_jobs = L * (3 * (z.max_tiles + C) + C) + noise_units + H / TILE_N;
    return z;
}

Layout layout(const qerl_decoder_dims &d, int L, int C)
{
    const Sizes z = table_sizes(d, L, C);
    Layout o;
    size_t p = 0;
    auto take = [&](size_t bytes, size_t align) {
        p = (p + align - 1) / align * align;
        const size_t at = p;
        p += bytes;
        return at;
    };
    const size_t M = (size_t)d.M, H = (size_t)d.hidden, I = (size_t)d.intermediate;
    o.off_maps = take(sizeof(LinMaps) * z.n_lin, 128);
    o.off_lins = take(sizeof(Lin) * z.n_lin, 256);
    o.off_glues = take(sizeof(Glue) * z.n_glue, 256);
    o.off_gammas = take(sizeof(void *) * 2 * L, 256);
    o.off_jobs = take(sizeof(Job) * z.max_jobs, 256);
    o.off_joboff = take(sizeof(int) * (C + 1), 256);
    o.off_ptotal = take(sizeof(int) * z.n_phases, 256);
    o.zero_begin = p = (p + 255) / 256 * 256;
    o.off_pcnt = take(sizeof(int) * z.n_phases, 256);
    o.off_tcnt = take(sizeof(int) * z.max_tiles * 4, 256);
    o.off_exit = take(sizeof(int), 256);
    o.zero_end = p;
    o.off_part = take((size_t)z.max_parts * TILE_N * BN * sizeof(float), 256);
    o.off_xn1 = take(M * H * 2, 256);
    o.off_xn2 = take(M * H * 2, 256);
    o.off_sq1 = take(H / TILE_N * BN * sizeof(float), 256);
    o.off_sq2 = take(H / TILE_N * BN * sizeof(float), 256);
    o.off_hmid = take(M * H * 2, 256);
    o.off_hbuf = take(2 * M * H * 2, 256);
    o.off_g = take(M * I * 2, 256);
    o.off_u = take(M * I * 2, 256);
    o.off_m = take(M * I * 2, 256);
    o.off_ns = take((size_t)2 * L * H * sizeof(float), 256);
    o.off_q = take(M * (size_t)d.q_dim * 2, 256);
    o.off_k = take(M * (size_t)d.kv_dim * 2, 256);
    o.off_v = take(M * (size_t)d.kv_dim * 2, 256);
    o.total = (p + 255) / 256 * 256;
    return o;
}

template <int RL, bool PACKED>
cudaError_t launch_chain(const Plan &P, int grid, float sigma, uint64_t seed, uint64_t step, unsigned first_layer,
                         cudaStream_t s)
{
    auto kernel = chain_kernel<RL, PACKED>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<RL>::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = Cfg<RL>::SMEM;
    cfg.stream = s;
    // Cooperative: every CTA is resident at once (CTAs wait on one another's phases).
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, P, sigma, (unsigned long long)seed, (unsigned long long)step,
                              first_layer);
}

}  // namespace
}  // namespace chain
}  // namespace qerl

struct qerl_chain {
    qerl::chain::Plan plan;
    int grid = 0, rl = 0, packed = 1, device = 0;
};

using namespace qerl;
using namespace qerl::chain;

namespace {

bool dims_ok(const qerl_decoder_dims *d)
{
    return d && d->M >= 1 && d->M <= BN && d->hidden >= KC && d->hidden % KC == 0 && d->q_dim >= TILE_N &&
           d->q_dim % TILE_N == 0 && d->kv_dim >= TILE_N && d->kv_dim % TILE_N == 0 && d->intermediate >= KC &&
           d->intermediate % KC == 0 && d->hidden <= (1 << 20) && d->intermediate <= (1 << 20) &&
           d->q_dim == d->hidden && d->r >= 8 && d->r <= 64 && d->r % 8 == 0 && d->eps >= 0.0f;
}

int chain_ctas()
{
    int dev = 0;
    cudaGetDevice(&dev);
    int n = num_sms();
    return n > MAX_CTAS ? MAX_CTAS : n;
}

bool lin_ok(const qerl_linear_weights &w)
{
    return w.codes && w.scales && w.tensor_scale && w.A && w.B && aligned16(w.codes) && aligned16(w.scales) &&
           aligned16(w.A) && aligned16(w.B);
}

}  // namespace

extern "C" size_t qerl_decoder_chain_ws_bytes(const qerl_decoder_dims *d, int n_layers)
{
    if (!dims_ok(d) || n_layers < 1 || n_layers > 4096) return 0;
    return layout(*d, n_layers, chain_ctas()).total;
}

extern "C" qerl_status qerl_decoder_chain_plan(const qerl_decoder_layer *layers, int n_layers,
                                               const qerl_decoder_dims *d, const void *x_in, void *x_out, void *ws,
                                               size_t ws_bytes, qerl_chain **out)
{
    if (!out) return QERL_ERR_INVALID_ARG;
    *out = nullptr;
    if (!layers || n_layers < 1 || n_layers > 4096 || !dims_ok(d) || !x_in || !x_out || !ws) return QERL_ERR_INVALID_ARG;
    if (!aligned16(x_in) || !aligned16(x_out) || !aligned16(ws)) return QERL_ERR_ALIGN;
    for (int l = 0; l < n_layers; ++l) {
        const qerl_decoder_layer &Ly = layers[l];
        const qerl_linear_weights *ws7[7] = {&Ly.q, &Ly.k, &Ly.v, &Ly.o, &Ly.gate, &Ly.up, &Ly.down};
        for (auto *w : ws7)
            if (!lin_ok(*w)) return QERL_ERR_INVALID_ARG;
        if (!Ly.gamma_attn || !Ly.gamma_mlp || !Ly.attn || !aligned16(Ly.attn)) return QERL_ERR_INVALID_ARG;
        if ((Ly.q_out && !aligned16(Ly.q_out)) || (Ly.k_out && !aligned16(Ly.k_out)) ||
            (Ly.v_out && !aligned16(Ly.v_out)))
            return QERL_ERR_ALIGN;
    }
    QERL_TRY(check_device());
    const int C = chain_ctas();
    const int L = n_layers;
    const Layout lo = layout(*d, L, C);
    if (ws_bytes < lo.total) return QERL_ERR_WORKSPACE;
    const Sizes z = table_sizes(*d, L, C);
    char *W = static_cast<char *>(ws);
    const int M = (int)d->M, H = (int)d->hidden, I = (int)d->intermediate, NQ = (int)d->q_dim, NKV = (int)d->kv_dim;
    const int r = d->r;
    const int RL = r <= 32 ? 32 : 64;

    auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16 *>(W + off); };
    auto fl = [&](size_t off) { return reinterpret_cast<float *>(W + off); };
    __nv_bfloat16 *hbuf[2] = {bf(lo.off_hbuf), bf(lo.off_hbuf) + (size_t)M * H};
    float *NS = fl(lo.off_ns);

    std::vector<Lin> lins;
    std::vector<LinMaps> maps;
    std::vector<Glue> glues;
    std::vector<int> ptotal;
    std::vector<std::vector<Job>> per(C);

    // phase 0: noise of every norm; phase 1: the first norm's input
    {
        Glue g = {};
        g.kind = GLUE_NOISE;
        g.phase = 0;
        g.width = H;
        g.n_norms = 2 * L;
        g.ns = NS;
        g.gammas = reinterpret_cast<const __nv_bfloat16 *const *>(W + lo.off_gammas);
        const int blocks = 2 * L * ((H + 3) / 4);
        g.units = (blocks + EPI_THREADS - 1) / EPI_THREADS;
        glues.push_back(g);
        for (int u = 0; u < g.units; ++u) per[u % C].push_back(Job{1, 0, u, 0, 0, 0, 1, 0});
        ptotal.push_back(g.units);
    }
    {
        Glue g = {};
        g.kind = GLUE_PRENORM;
        g.phase = 1;
        g.width = H;
        g.a = static_cast<const __nv_bfloat16 *>(x_in);
        g.out = bf(lo.off_xn1);
        g.sq = fl(lo.off_sq1);
        g.ns = NS;  // norm 0
        g.units = H / TILE_N;
        glues.push_back(g);
        for (int u = 0; u < g.units; ++u) per[(u * 7 + 3) % C].push_back(Job{1, 1, u, 0, 0, 0, 1, 0});
        ptotal.push_back(g.units);
    }

    auto add_lin = [&](const qerl_linear_weights &w, int N, int K, int kind, int phase, int tile0, const void *xin,
                       __nv_bfloat16 *y, const float *sq_in, const __nv_bfloat16 *h_in, __nv_bfloat16 *h_out,
                       __nv_bfloat16 *xn_out, const float *ns_next, float *sq_out) -> bool {
        Lin Lr = {};
        Lr.N = N;
        Lr.K = K;
        Lr.r = r;
        Lr.kind = kind;
        Lr.phase = phase;
        Lr.n_tiles = N / TILE_N;
        Lr.sq_tiles = K / TILE_N;
        Lr.tile0 = tile0;
        Lr.codes = w.codes;
        Lr.scales = w.scales;
        Lr.ts = w.tensor_scale;
        Lr.B = static_cast<const __nv_bfloat16 *>(w.B);
        Lr.y = y;
        Lr.sq_in = sq_in;
        Lr.h_in = h_in;
        Lr.h_out = h_out;
        Lr.xn_out = xn_out;
        Lr.ns_next = ns_next;
        Lr.sq_out = sq_out;
        LinMaps mp;
        std::memset(&mp, 0, sizeof(mp));
        if (!make_map_2d(&mp.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.codes, K / 2, N, K / 2, KC / 2, TILE_N,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map_2d(&mp.scl, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.scales, K / 16, N, K / 16, KC / 16, TILE_N,
                         CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_map_kblocks(&mp.al, w.A, K, r, RL, GK) || !make_map_kblocks(&mp.x, xin, K, M, BN, GK))
            return false;
        lins.push_back(Lr);
        maps.push_back(mp);
        return true;
    };

    // A matmul phase: its linears' (tile, 256-k chunk) units divided evenly
    // over the CTAs in (linear, tile, chunk) order; parts numbered per tile.
    auto schedule = [&](int first_lin, int n_lin, int phase) {
        int64_t U = 0;
        for (int i = 0; i < n_lin; ++i) U += (int64_t)lins[first_lin + i].n_tiles * (lins[first_lin + i].K / KC);
        struct Piece {
            int lin, tile, kc0, kc1, cta;
        };
        std::vector<Piece> pieces;
        for (int c = 0; c < C; ++c) {
            int64_t a = U * c / C, b = U * (c + 1) / C;
            int64_t base = 0;
            for (int i = 0; i < n_lin && a < b; ++i) {
                const Lin &Lr = lins[first_lin + i];
                const int nk = Lr.K / KC;
                const int64_t span = (int64_t)Lr.n_tiles * nk;
                if (a < base + span) {
                    while (a < b && a < base + span) {
                        const int64_t off = a - base;
                        const int tile = (int)(off / nk), kc0 = (int)(off % nk);
                        const int64_t end = std::min<int64_t>(b, base + (int64_t)(tile + 1) * nk);
                        pieces.push_back(Piece{first_lin + i, tile, kc0, (int)(kc0 + (end - a)), c});
                        a = end;
                    }
                }
                base += span;
            }
        }
        // parts per tile, in chunk order (pieces are already ordered by cta = chunk order)
        std::sort(pieces.begin(), pieces.end(), [](const Piece &x, const Piece &y) {
            if (x.lin != y.lin) return x.lin < y.lin;
            if (x.tile != y.tile) return x.tile < y.tile;
            return x.kc0 < y.kc0;
        });
        int slot = 0, tiles = 0;
        for (size_t a = 0; a < pieces.size();) {
            size_t b = a;
            while (b < pieces.size() && pieces[b].lin == pieces[a].lin && pieces[b].tile == pieces[a].tile) ++b;
            const int np = (int)(b - a);
            for (size_t k = a; k < b; ++k) {
                const Piece &pc = pieces[k];
                per[pc.cta].push_back(Job{0, pc.lin, pc.tile, pc.kc0, pc.kc1, (int)(k - a), np, np > 1 ? slot + (int)(k - a) : 0});
            }
            if (np > 1) slot += np;
            ++tiles;
            a = b;
        }
        ptotal.push_back(tiles);
        (void)phase;
    };

    // per-CTA job order must follow phases: sort each CTA's list by phase at the end
    std::vector<const __nv_bfloat16 *> gammas(2 * L);
    for (int l = 0; l < L; ++l) {
        const qerl_decoder_layer &Ly = layers[l];
        gammas[2 * l] = static_cast<const __nv_bfloat16 *>(Ly.gamma_attn);
        gammas[2 * l + 1] = static_cast<const __nv_bfloat16 *>(Ly.gamma_mlp);
        const int p0 = 2 + 4 * l;
        const __nv_bfloat16 *h_in = l == 0 ? static_cast<const __nv_bfloat16 *>(x_in) : hbuf[(l - 1) & 1];
        __nv_bfloat16 *h_out = l == L - 1 ? static_cast<__nv_bfloat16 *>(x_out) : hbuf[l & 1];
        __nv_bfloat16 *qo = Ly.q_out ? static_cast<__nv_bfloat16 *>(Ly.q_out) : bf(lo.off_q);
        __nv_bfloat16 *ko = Ly.k_out ? static_cast<__nv_bfloat16 *>(Ly.k_out) : bf(lo.off_k);
        __nv_bfloat16 *vo = Ly.v_out ? static_cast<__nv_bfloat16 *>(Ly.v_out) : bf(lo.off_v);
        // q | k | v | o
        const int first = (int)lins.size();
        int t0 = 0;
        bool okm = add_lin(Ly.q, NQ, H, LIN_NORMED, p0, t0, bf(lo.off_xn1), qo, fl(lo.off_sq1), nullptr, nullptr,
                           nullptr, nullptr, nullptr);
        t0 += NQ / TILE_N;
        okm = okm && add_lin(Ly.k, NKV, H, LIN_NORMED, p0, t0, bf(lo.off_xn1), ko, fl(lo.off_sq1), nullptr, nullptr,
                             nullptr, nullptr, nullptr);
        t0 += NKV / TILE_N;
        okm = okm && add_lin(Ly.v, NKV, H, LIN_NORMED, p0, t0, bf(lo.off_xn1), vo, fl(lo.off_sq1), nullptr, nullptr,
                             nullptr, nullptr, nullptr);
        t0 += NKV / TILE_N;
        okm = okm && add_lin(Ly.o, H, NQ, LIN_RESID, p0, t0, Ly.attn, nullptr, nullptr, h_in, bf(lo.off_hmid),
                             bf(lo.off_xn2), NS + (size_t)(2 * l + 1) * H, fl(lo.off_sq2));
        if (!okm) return QERL_ERR_CUDA;
        schedule(first, 4, p0);
        // gate | up
        const int first2 = (int)lins.size();
        okm = add_lin(Ly.gate, I, H, LIN_NORMED, p0 + 1, 0, bf(lo.off_xn2), bf(lo.off_g), fl(lo.off_sq2), nullptr,
                      nullptr, nullptr, nullptr, nullptr) &&
              add_lin(Ly.up, I, H, LIN_NORMED, p0 + 1, I / TILE_N, bf(lo.off_xn2), bf(lo.off_u), fl(lo.off_sq2),
                      nullptr, nullptr, nullptr, nullptr, nullptr);
        if (!okm) return QERL_ERR_CUDA;
        schedule(first2, 2, p0 + 1);
        // SwiGLU
        {
            Glue g = {};
            g.kind = GLUE_SWIGLU;
            g.phase = p0 + 2;
            g.width = I;
            g.a = bf(lo.off_g);
            g.b = bf(lo.off_u);
            g.out = bf(lo.off_m);
            g.cols = ((I + C - 1) / C + 7) / 8 * 8;
            g.units = (I + g.cols - 1) / g.cols;
            const int gi = (int)glues.size();
            glues.push_back(g);
            for (int u = 0; u < g.units; ++u) per[u % C].push_back(Job{1, gi, u, 0, 0, 0, 1, 0});
            ptotal.push_back(g.units);
        }
        // down (+ residual; the next layer's first norm input)
        const int first3 = (int)lins.size();
        const bool last = l == L - 1;
        okm = add_lin(Ly.down, H, I, LIN_RESID, p0 + 3, 0, bf(lo.off_m), nullptr, nullptr, bf(lo.off_hmid), h_out,
                      last ? nullptr : bf(lo.off_xn1), last ? nullptr : NS + (size_t)(2 * l + 2) * H,
                      last ? nullptr : fl(lo.off_sq1));
        if (!okm) return QERL_ERR_CUDA;
        schedule(first3, 1, p0 + 3);
    }
    // order every CTA's jobs by phase (stable: the order within a phase is kept)
    auto phase_of = [&](const Job &J) { return J.type == 0 ? lins[J.idx].phase : glues[J.idx].phase; };
    std::vector<Job> jobs;
    std::vector<int> joboff(C + 1, 0);
    for (int c = 0; c < C; ++c) {
        std::stable_sort(per[c].begin(), per[c].end(), [&](const Job &a, const Job &b) { return phase_of(a) < phase_of(b); });
        joboff[c] = (int)jobs.size();
        jobs.insert(jobs.end(), per[c].begin(), per[c].end());
    }
    joboff[C] = (int)jobs.size();
    if ((int)lins.size() > z.n_lin || (int)glues.size() > z.n_glue || (int)jobs.size() > z.max_jobs ||
        (int)ptotal.size() != z.n_phases)
        return QERL_ERR_SHAPE;

    // tables to the device (once, synchronously: the plan is built outside any capture)
    if (cudaMemcpy(W + lo.off_maps, maps.data(), sizeof(LinMaps) * maps.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(W + lo.off_lins, lins.data(), sizeof(Lin) * lins.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(W + lo.off_glues, glues.data(), sizeof(Glue) * glues.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(W + lo.off_gammas, gammas.data(), sizeof(void *) * gammas.size(), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemcpy(W + lo.off_jobs, jobs.data(), sizeof(Job) * jobs.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(W + lo.off_joboff, joboff.data(), sizeof(int) * joboff.size(), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemcpy(W + lo.off_ptotal, ptotal.data(), sizeof(int) * ptotal.size(), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemset(W + lo.zero_begin, 0, lo.zero_end - lo.zero_begin) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return QERL_ERR_CUDA;

    qerl_chain *h = new qerl_chain;
    Plan &P = h->plan;
    P.n_ctas = C;
    P.n_lin = (int)lins.size();
    P.n_glue = (int)glues.size();
    P.n_phases = (int)ptotal.size();
    P.M = M;
    P.r_max = r;
    P.lora_scale = d->lora_scale;
    P.eps = d->eps;
    P.lins = reinterpret_cast<const Lin *>(W + lo.off_lins);
    P.maps = reinterpret_cast<const LinMaps *>(W + lo.off_maps);
    P.glues = reinterpret_cast<const Glue *>(W + lo.off_glues);
    P.jobs = reinterpret_cast<const Job *>(W + lo.off_jobs);
    P.job_off = reinterpret_cast<const int *>(W + lo.off_joboff);
    P.phase_total = reinterpret_cast<const int *>(W + lo.off_ptotal);
    P.phase_cnt = reinterpret_cast<int *>(W + lo.off_pcnt);
    P.tile_cnt = reinterpret_cast<int *>(W + lo.off_tcnt);
    P.exit_cnt = reinterpret_cast<int *>(W + lo.off_exit);
    P.partials = fl(lo.off_part);
    P.err = error_word();
    P.timeout_ns = 2000000000ull;
    h->grid = C;
    h->rl = RL;
    cudaGetDevice(&h->device);
    *out = h;
    return QERL_OK;
}

extern "C" qerl_status qerl_decoder_chain_run(const qerl_chain *h, float sigma, uint64_t seed, uint64_t step,
                                              uint32_t first_layer, qerl_stream_t stream)
{
    if (!h) return QERL_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QERL_ERR_CUDA;
    if (dev != h->device) return QERL_ERR_INVALID_ARG;
    if (first_layer > (1u << 30)) return QERL_ERR_INVALID_ARG;
    const cudaError_t e =
        h->rl == 32 ? launch_chain<32, true>(h->plan, h->grid, sigma, seed, step, first_layer, as_cuda(stream))
                    : launch_chain<64, true>(h->plan, h->grid, sigma, seed, step, first_layer, as_cuda(stream));
    return launched(e);
}

extern "C" void qerl_decoder_chain_destroy(qerl_chain *h) { delete h; }
