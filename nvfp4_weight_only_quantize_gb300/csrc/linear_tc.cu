// Tensor-core (tcgen05) path of the NVFP4 LoRA linear, sm_103a.
//
// Swap-AB formulation: the weight is the MMA's 128-row A operand and the
// tokens are its N side, so one kernel serves decode (M = 1..64 tokens, N
// padded to 16) and prefill (M in the thousands, 256-token tiles):
//     D[n, m] = sum_k w''[n, k] * x[m, k] + sum_j B[n, j] * u[m, j]
//     y[m, n] = bf16(ysc * D[n, m]),   ysc = s_t * 2^c
// with w'' = e2m1(code) * e4m3(scale) * 2^-c, exact in bf16, and the LoRA
// down-projection folded in as extra K steps: u = bf16(s * (x A^T) / ysc).
// The exponent offset c is derived from s_t so that w'' and u are normal bf16
// numbers and ysc is finite (see tc_exponent_offset).
//
// Warp roles (one CTA per SM; 352 threads for token tiles up to 128, 608 for
// 256-token tiles):
//   warps 0..4G-1  dequantize, as G = 2 (or 4) groups of four warps taking the
//              stages in turn: packed codes + block scales (smem) -> bf16 A
//              tile in TMEM; warps 0-3 also run the epilogue (TMEM ->
//              registers -> smem -> y, or split-K partials).
//   warp 4G    TMA producer of the packed codes and block scales, 4 k-steps
//              (256 k: 128 code bytes per row, full lines) per raw stage.
//   warp 4G+1  TMA producer of the token tile (x, then u for the LoRA steps).
//   warp 4G+2  allocates TMEM and issues tcgen05.mma and the commits (one
//              elected lane of the converged warp).
// A pipeline stage is SPS k-steps: 4 (one raw stage) for token tiles up to 128,
// 1 for 256-token tiles (their token stages are four times larger, and one
// k-step of 256 tokens is already 512 MMA cycles); each stage costs every role
// mbarrier round trips of ~100+ cycles, so decode stages are made long.
// Every mbarrier wait is bounded by a deadline; on expiry the CTA latches
// QERL_ERR_TIMEOUT, every role leaves its loop, in-flight copies and MMAs are
// drained (bounded), TMEM is freed and the CTA exits.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <mutex>
#include <utility>

#include "dequant.cuh"
#include "linear.cuh"
#include "sm100_ptx.cuh"

namespace qerl {
namespace {

using namespace ptx;

constexpr int BK = 64;          // k per MMA step: one 128-byte swizzle row of bf16
constexpr int GK = 4;           // k-steps per raw stage (256 k)
constexpr int TILE_N = 128;     // weight rows per CTA (MMA M)
constexpr int DQ_GROUP_WARPS = 4; // one warp per 32 weight rows of the tile
constexpr int RAW_CODES = TILE_N * GK * BK / 2;    // 16 KB: 128 rows x 128 code bytes (SW128)
constexpr int RAW_SCALES = TILE_N * GK * BK / 16;  // 2 KB: 128 rows x 16 scale bytes
constexpr int RAW_STAGE = RAW_CODES + RAW_SCALES;  // 18 KB, a multiple of 1024
constexpr int MAX_SPLITS = 8;  // split-K factor cap: bounds the partial traffic

// FUSED: the LoRA down-projection runs inside the kernel (decode tiles, r <= 32,
// no t output): per main k-step one more MMA accumulates t_s^T = A x^T over the
// CTA's k-range in TMEM, and the CTA builds u_s = bf16(s t_s / (s_t 2^c)) in
// shared memory for its own LoRA step (the sum over splits of s t_s B^T is the
// LoRA term).
constexpr int FUSED_R = 32;  // LoRA rows loaded per k-step in fused mode
template <int BN, bool FUSED = false>
struct Cfg {
    // Dequant groups of four warps; group g takes the stages j = g (mod DQG).
    // Two for token tiles up to 128, four for 256-token tiles (one k-step per
    // stage there: every group takes one k-step of each raw stage).
    static constexpr int DQG = BN >= 256 ? 4 : 2;
    static constexpr int NUM_DQ_WARPS = DQG * DQ_GROUP_WARPS;
    static constexpr int WARP_RAW = NUM_DQ_WARPS, WARP_X = NUM_DQ_WARPS + 1, WARP_MMA = NUM_DQ_WARPS + 2;
    static constexpr int NUM_THREADS = (NUM_DQ_WARPS + 3) * 32;
    // k-steps per pipeline stage (1 = 64 k, 4 = 256 k).
    static constexpr int SPS = BN >= 256 ? 1 : 4;
    // A stage holds SPS k-steps of the dequantized weight tile (TMEM); at least
    // DQG of them, so a group never waits on a stage two mbarrier phases ahead
    // of the MMA (parity aliasing).  More stages than groups (where TMEM
    // allows): a group can fill a free stage while the MMA still reads the ones
    // filled before.
    static constexpr int S = SPS == 4 ? 3 : 8;
    static_assert(S >= DQG, "parity waits need at least one stage per dequant group");
    // Token-tile stages (smem), deeper than the A ring: a token slot is reloaded
    // only after the MMA that read it completed, a ~2 us round trip.  256-token
    // tiles take five one-k-step stages (160 KB) beside two raw stages.
    static constexpr int XS = BN >= 256 ? 5 : (FUSED ? 3 : (BN >= 128 ? 2 : 4));
    static constexpr int R = BN >= 256 ? 2 : 4;  // raw (code+scale) stages
    // k-steps of a main stage dequantized into registers before its A slot is
    // free (the rest after): they come off the slot-reuse round trip.
    static constexpr int EARLY = 2;
    static_assert(GK % SPS == 0 && GK / SPS <= DQG, "each group has at most one stage per raw stage");
    static constexpr int RAW_CONSUMERS = (GK / SPS) * DQ_GROUP_WARPS;  // warps that read one raw stage
    static_assert(R * GK >= S * SPS, "raw ring deep enough for parity-safe waits");
    // A group waits for a raw stage before its A slot: the slot's previous raw
    // stage, R raw stages back, was then consumed by this same group.
    static_assert((R * GK / SPS) % DQG == 0, "a raw slot's previous fill belongs to the waiting group");
    static constexpr int X_STEP = BN * BK * 2;
    static constexpr int X_STAGE = X_STEP * SPS;
    // fused: the LoRA A rows of each k-step (FUSED_R x 64 bf16, 128-byte rows)
    static constexpr int AL_STEP = FUSED_R * BK * 2;
    static constexpr int AL_STAGE = FUSED ? AL_STEP * SPS : 0;
    // TMEM: the f32 accumulator (BN columns), then S A stages of 32*SPS columns
    // (128 rows x 64 bf16 per step, two per 32-bit column).
    static constexpr int A_COL0 = BN < 32 ? 32 : BN;
    static constexpr int T_COL = A_COL0 + S * 32 * SPS;  // fused: t_s^T accumulator
    static constexpr int TMEM_NEED = T_COL + (FUSED ? (BN < 32 ? 32 : BN) : 0);
    static constexpr int TMEM_COLS = TMEM_NEED <= 64 ? 64 : (TMEM_NEED <= 128 ? 128 : (TMEM_NEED <= 256 ? 256 : 512));
    static_assert(TMEM_NEED <= 512, "TMEM holds 512 columns");
    static constexpr int BAR_BYTES = 1024;
    // token ring, fused LoRA-A ring (an MMA reads 128 rows = 16 KB from each
    // step's start, so the raw ring must follow it), raw ring, barriers
    static constexpr int SMEM = XS * X_STAGE + XS * AL_STAGE + R * RAW_STAGE + BAR_BYTES + 1024;
    static_assert(!FUSED || R * RAW_STAGE >= 16384, "the LoRA-A MMA window stays inside shared memory");
    static_assert(XS * X_STAGE >= BN * TILE_N * 2, "the y staging tile reuses the token ring");
};

// Up to MAX_GROUPS linears sharing x (and K, r, s): group g owns the weight
// tiles [tile_start[g], tile_start[g + 1]) of the launch.
constexpr int MAX_GROUPS = 3;
struct TcGroups {
    int G;
    int tile_start[MAX_GROUPS + 1];
    int N[MAX_GROUPS];
    const __nv_bfloat16 *Bl[MAX_GROUPS];
    const float *ts[MAX_GROUPS];
    __nv_bfloat16 *y[MAX_GROUPS];
    const float *Bf[MAX_GROUPS];  // FP32 adapters: B as FP32 (lora_parts == 3)
};
// Tensor maps of a launch: per group codes, scales, LoRA A (fused) and u
// (unfused); x is shared.
struct TcMaps {
    CUtensorMap codes[MAX_GROUPS], scl[MAX_GROUPS], al[MAX_GROUPS], u[MAX_GROUPS], x;
};

struct TcFwdParams {
    int M, K;
    int nk;              // K / BK main steps
    int lora_steps;      // lora_parts * ceil(r / BK)
    int lora_parts;      // 1; 3 for FP32 adapters: B_hi u_hi + B_hi u_lo + B_lo u_hi
    int r, r_pad;        // rank, u row length (lora_steps * BK)
    int splits, steps_per_split;
    int n_tiles, m_tiles;  // weight tiles over all groups, token tiles
    TcGroups grp;
    float *partial;
    unsigned int *err;
    unsigned long long timeout_ns;
    int fault;           // test hook: CTA 0 withholds one arrival so its waits time out
    int chain;           // launched chained: token tiles and B wait for the preceding grid
    float lora_scale;    // fused: s
};


// FP32 adapters: one weight row's A-operand values of a LoRA step, B_hi =
// bf16(B) for parts 0 and 1, B_lo = bf16(B - B_hi) for part 2 (the token side
// holds u_hi, u_lo, u_hi), columns jb .. jb + 63 (zero past r), stored to its
// TMEM lane.  Out of line: inlined, its loads raise the register count of the
// dequantizing loop it sits in.
__device__ __noinline__ void lora_rows_f32(const float *brow, int jb, int r, bool row_ok, int part, uint32_t taddr)
{
    uint32_t out[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const int j = jb + 2 * e;
        const float v0 = (row_ok && j < r) ? brow[j] : 0.0f;
        const float v1 = (row_ok && j + 1 < r) ? brow[j + 1] : 0.0f;
        __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
        if (part == 2) h = __floats2bfloat162_rn(v0 - __low2float(h), v1 - __high2float(h));
        out[e] = *reinterpret_cast<const uint32_t *>(&h);
    }
    tmem_st32(taddr, out);
}

// 16 columns of this warp's 32 TMEM lanes of the accumulator, as floats.
__device__ __forceinline__ void acc_load16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    tmem_ld16(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// MX: MXFP4 weights (the E8M0 factor in the dequantizer).  F32AB: FP32
// adapters (B converted to B_hi / B_lo for the three LoRA products).
template <int BN, bool PACKED, bool FUSED, bool MX = false, bool F32AB = false>
__global__ void __launch_bounds__(Cfg<BN, FUSED>::NUM_THREADS, 1)
    tc_fwd_kernel(const __grid_constant__ TcMaps maps, const TcFwdParams p)
{
    using C = Cfg<BN, FUSED>;
    constexpr int SPS = C::SPS;
    constexpr int DQG = C::DQG, NUM_DQ_WARPS = C::NUM_DQ_WARPS;
    constexpr int WARP_RAW = C::WARP_RAW, WARP_X = C::WARP_X, WARP_MMA = C::WARP_MMA;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *X_ring = smem;
    uint8_t *AL_ring = X_ring + C::XS * C::X_STAGE;  // fused: LoRA A rows per k-step
    uint8_t *R_ring = AL_ring + C::XS * C::AL_STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(R_ring + C::R * RAW_STAGE);
    uint64_t *raw_full = bars;
    uint64_t *raw_empty = raw_full + C::R;
    uint64_t *x_full = raw_empty + C::R;
    uint64_t *x_empty = x_full + C::XS;      // MMA of the stage done: frees its token tile
    uint64_t *a_full = x_empty + C::XS;
    uint64_t *stage_empty = a_full + C::S;  // MMA of the stage done: frees its A tile
    uint64_t *acc_full = stage_empty + C::S;
    uint64_t *t_full = acc_full + 1;  // fused: every t_s MMA done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(t_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *ep_ok = abort_flag + 1;  // [4]: epilogue warps' view of acc_full

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // blockIdx.x = (split * m_tiles + m_tile) * n_tiles + n_tile
    const int n_tile = blockIdx.x % p.n_tiles;
    const int m_tile = (blockIdx.x / p.n_tiles) % p.m_tiles;
    const int split = blockIdx.x / (p.n_tiles * p.m_tiles);
    const int tile = m_tile * p.n_tiles + n_tile;
    // the group (linear) this weight tile belongs to
    int g = 0;
#pragma unroll
    for (int i = 1; i < MAX_GROUPS; ++i)
        if (i < p.grp.G && n_tile >= p.grp.tile_start[i]) g = i;
    const int Ng = p.grp.N[g];
    const float *tsg = p.grp.ts[g];
    const __nv_bfloat16 *Blg = p.grp.Bl[g];
    const float *Bfg = p.grp.Bf[g];
    __nv_bfloat16 *yg = p.grp.y[g];
    const CUtensorMap *codes_map = &maps.codes[g], *scl_map = &maps.scl[g], *al_map = &maps.al[g];
    const CUtensorMap *u_map = &maps.u[g], *x_map = &maps.x;
    const int n0 = (n_tile - p.grp.tile_start[g]) * TILE_N, m0 = m_tile * BN;
    const int k_begin = split * p.steps_per_split;  // a multiple of GK
    const int k_end = min(p.nk, k_begin + p.steps_per_split);
    const int n_main = k_end > k_begin ? k_end - k_begin : 0;  // a multiple of GK (K % 256 == 0)
    const int n_groups = n_main / GK;
    // The LoRA steps belong to the last split, or (fused) to every split.
    const int n_steps = n_main + ((FUSED || split == p.splits - 1) ? p.lora_steps : 0);
    const int n_stages = (n_steps + SPS - 1) / SPS;  // the last (LoRA) stage may be partial
    const int main_stages = n_main / SPS;
    // Every CTA walks its k-range from a different raw group, so that the CTAs
    // do not all read the same token tile from L2 at the same time.  The
    // rotation fixes the summation order, hence the result, per weight tile.
    const int grot = n_groups > 0 ? ((n_tile >> 2) * 5 + m_tile * 3) % n_groups : 0;
    // k-step of the CTA's i-th main step.  No division: the producers run on one
    // lane that shares its SM sub-partition with issue-bound dequantizing warps,
    // where every extra dependent instruction costs many cycles.
    auto kstep = [&](int i) {
        int gg = i / GK + grot;  // GK is a power of two
        if (gg >= n_groups) gg -= n_groups;
        return k_begin + gg * GK + i % GK;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::R; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], C::RAW_CONSUMERS);
        }
        for (int i = 0; i < C::XS; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 1);
        }
        for (int i = 0; i < C::S; ++i) {
            mbar_init(&a_full[i], DQ_GROUP_WARPS);
            mbar_init(&stage_empty[i], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(t_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_RAW && lane == 0) {
        prefetch_tensormap(codes_map);
        prefetch_tensormap(scl_map);
    }
    if (warp == WARP_X && lane == 0) {
        prefetch_tensormap(x_map);
        if (FUSED)
            prefetch_tensormap(al_map);
        else
            prefetch_tensormap(u_map);
    }
    if (warp == WARP_MMA) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();  // a chained successor may be scheduled (it waits for this grid before touching memory)
    const unsigned long long deadline = globaltimer_ns() + p.timeout_ns;

    // Bounded wait for the phase with this parity; false once the CTA aborts.
    // A waiting thread is suspended in hardware until the phase completes (or
    // the hint runs out): it takes no issue slots from the dequantizing warps
    // and resumes as soon as the phase completes.
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        for (;;) {
            if (*abort_flag) return false;
            if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
            if (globaltimer_ns() > deadline) {
                *abort_flag = 1;
                latch_error(p.err, QERL_ERR_TIMEOUT);
                return false;
            }
        }
    };
    // Wait used while draining after an abort: ignores the flag, short bound.
    auto drain_wait = [&](uint64_t *bar, uint32_t parity) {
        const unsigned long long until = globaltimer_ns() + 100000000ull;  // 100 ms
        while (!mbar_try_wait(bar, parity) && globaltimer_ns() < until) {
        }
    };

    if (warp == WARP_RAW) {
        // ------------------------------------------- packed codes + block scales
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (int g = 0; g < n_groups; ++g) {
                const int slot = g % C::R;
                const uint32_t round = (uint32_t)(g / C::R);
                if (round > 0 && !wait(&raw_empty[slot], (round - 1) & 1u)) break;
                mbar_arrive_expect_tx(&raw_full[slot], RAW_STAGE);
                const int kk = kstep(g * GK);  // first k-step of the group
                uint8_t *dst = R_ring + slot * RAW_STAGE;
                tma_load_2d_hint(dst, codes_map, &raw_full[slot], kk * (BK / 2), n0, pol);
                tma_load_2d_hint(dst + RAW_CODES, scl_map, &raw_full[slot], kk * (BK / 16), n0, pol);
                issued = g + 1;
            }
            if (*abort_flag)  // let the copies already issued land before the CTA exits
                for (int g = issued > C::R ? issued - C::R : 0; g < issued; ++g)
                    drain_wait(&raw_full[g % C::R], (uint32_t)(g / C::R) & 1u);
        }
        __syncwarp();
        if (FUSED && n_stages > main_stages) {
            // ------------------------------------------- u_s for this CTA's LoRA step
            // Lane j reads row j of t_s^T (TMEM lanes 0-31 belong to this warp)
            // and writes column j of the step's token tile: u_s[m][j] =
            // bf16(s t_s[m][j] / (s_t 2^c)), columns 32..63 zero.
            const int slot = main_stages % C::XS;
            const uint32_t round = (uint32_t)(main_stages / C::XS);
            bool ok = __all_sync(0xFFFFFFFFu, wait(t_full, 0));
            if (ok && round > 0) ok = __all_sync(0xFFFFFFFFu, wait(&x_empty[slot], (round - 1) & 1u));
            if (ok) {
                tc_fence_after();
                const float st = *tsg;
                const float fac = p.lora_scale / (st * pow2f(tc_exponent_offset(st)));
                const uint32_t sdst = smem_u32(X_ring + slot * C::X_STAGE);
                const bool jv = lane < p.r;
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    uint32_t tr[16];
                    tmem_ld16(tmem + (uint32_t)C::T_COL + (uint32_t)c0, tr);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int m = c0 + e;
                        const __nv_bfloat16 uv = __float2bfloat16_rn(jv ? __uint_as_float(tr[e]) * fac : 0.0f);
                        const uint32_t rowb = sdst + (uint32_t)(m * 128);
                        const uint32_t lo = (uint32_t)((((lane >> 3) ^ (m & 7)) << 4) | ((lane & 7) << 1));
                        const uint32_t hi = (uint32_t)(((((lane + 32) >> 3) ^ (m & 7)) << 4) | ((lane & 7) << 1));
                        asm volatile("st.shared.b16 [%0], %1;" ::"r"(rowb + lo), "h"(*reinterpret_cast<const unsigned short *>(&uv))
                                     : "memory");
                        asm volatile("st.shared.b16 [%0], %1;" ::"r"(rowb + hi), "h"((unsigned short)0) : "memory");
                    }
                }
                fence_proxy_async_smem();  // the MMA reads the tile through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(&x_full[slot]);
            }
        }
    } else if (warp == WARP_X) {
        // ------------------------------------------- token tiles (SPS per stage)
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            int issued = 0;
            // Chained: x may come from the work before the down-projection
            // grid, which that grid waited for; wait for it before any x tile.
            if (p.chain) pdl_wait();
            for (int j = 0; j < n_stages; ++j) {
                const int slot = j % C::XS;
                const uint32_t round = (uint32_t)(j / C::XS);
                // u is written by the LoRA down-projection launched just before
                // this kernel, which lets this grid start early (programmatic
                // launch): wait for that grid only before the first u tile.  The
                // token tiles x were complete before that grid was launched.
                if (FUSED && j >= main_stages) break;  // u is built in this CTA
                if (j == main_stages) asm volatile("griddepcontrol.wait;" ::: "memory");
                if (round > 0 && !wait(&x_empty[slot], (round - 1) & 1u)) break;
                const int nsub = min(SPS, n_steps - j * SPS);
                mbar_arrive_expect_tx(&x_full[slot], (uint32_t)((C::X_STEP + (FUSED ? C::AL_STEP : 0)) * nsub));
                uint8_t *dst = X_ring + slot * C::X_STAGE;
                if (FUSED) {  // LoRA A rows 0..31 (zero past r) of each k-step
#pragma unroll
                    for (int sub = 0; sub < SPS; ++sub) {
                        if (sub >= nsub) break;
                        tma_load_2d_hint(AL_ring + slot * C::AL_STAGE + sub * C::AL_STEP, al_map, &x_full[slot],
                                         kstep(j * SPS + sub) * BK, 0, pol);
                    }
                }
#pragma unroll
                for (int sub = 0; sub < SPS; ++sub) {
                    if (sub >= nsub) break;
                    const int i = j * SPS + sub;
                    const CUtensorMap *map = i < n_main ? x_map : u_map;
                    const int kx = i < n_main ? kstep(i) * BK : (i - n_main) * BK;
                    tma_load_2d_hint(dst + sub * C::X_STEP, map, &x_full[slot], kx, m0, pol);
                }
                issued = j + 1;
            }
            if (*abort_flag)
                for (int j = issued > C::XS ? issued - C::XS : 0; j < issued; ++j)
                    drain_wait(&x_full[j % C::XS], (uint32_t)(j / C::XS) & 1u);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------- MMA issue
        // The whole warp runs the loop (stage indices and descriptors stay
        // warp-uniform); one elected lane issues the MMAs and the commit.
        constexpr uint32_t idesc = idesc_bf16_f32(TILE_N, BN);
        const uint64_t bd0 = desc_kmajor_sw128(smem_u32(X_ring));
        const uint32_t at0 = tmem + (uint32_t)C::A_COL0;
        bool ready = n_stages > 0 && __all_sync(0xFFFFFFFFu, wait(&a_full[0], 0) && wait(&x_full[0], 0));
        for (int j = 0; j < n_stages && ready; ++j) {
            const int s = j % C::S, xs = j % C::XS;
            const int nsub = min(SPS, n_steps - j * SPS);
            tc_fence_after();
            if (elect_one()) {
                const uint32_t at = at0 + (uint32_t)(s * 32 * SPS);
                const uint64_t bd = bd0 + (uint64_t)((xs * C::X_STAGE) >> 4);
#pragma unroll
                for (int sub = 0; sub < SPS; ++sub) {
                    if (sub >= nsub) break;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)  // 16 k = 8 TMEM columns of A, 32 bytes of B
                        umma_bf16_ts(tmem, at + (uint32_t)(sub * 32 + 8 * kk),
                                     bd + (uint64_t)((sub * C::X_STEP) >> 4) + 2u * kk, idesc,
                                     (j > 0 || sub > 0 || kk > 0) ? 1u : 0u);
                    if (FUSED && j < main_stages) {
                        // t_s^T += A[0..127 (rows >= 32 unused), k-step] x^T: the same token
                        // tile as B; the LoRA A rows from shared memory as A
                        const uint64_t ad = desc_kmajor_sw128(smem_u32(AL_ring + xs * C::AL_STAGE + sub * C::AL_STEP));
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            umma_bf16(tmem + (uint32_t)C::T_COL, ad + 2u * kk,
                                      bd + (uint64_t)((sub * C::X_STEP) >> 4) + 2u * kk, idesc,
                                      (j > 0 || sub > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                if (FUSED && j == main_stages - 1) umma_commit(t_full);
                umma_commit(&stage_empty[s]);
                umma_commit(&x_empty[xs]);
            }
            __syncwarp();
            if (j + 1 < n_stages) {
                const int s1 = (j + 1) % C::S, xs1 = (j + 1) % C::XS;
                ready = __all_sync(0xFFFFFFFFu, wait(&a_full[s1], (uint32_t)((j + 1) / C::S) & 1u) &&
                                                    wait(&x_full[xs1], (uint32_t)((j + 1) / C::XS) & 1u));
            }
        }
        // Arrives once every MMA issued above has completed (also after an abort).
        if (elect_one()) umma_commit(acc_full);
        __syncwarp();
    } else {
        // ------------------------------------------- dequantize
        // Group g = warp / 4 takes the stages j = g, g + DQG, ...; thread =
        // one weight row of the tile, all 64 k of each of the stage's SPS steps.
        const int row = (warp & 3) * 32 + lane;
        const int group = warp >> 2;
        const int n = n0 + row;
        const bool row_ok = n < Ng;
        const float pow2 = pow2f(126 - tc_exponent_offset(*tsg));
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        for (int j = group; j < n_stages; j += DQG) {
            const int s = j % C::S;
            const uint32_t sround = (uint32_t)(j / C::S);
            const bool main_stage = j < main_stages;
            const int g = (j * SPS) / GK, rs = g % C::R;  // raw stage of a main stage
            // The raw stage first: its codes and scales are read, and the first
            // k-step dequantized, while the MMA may still be reading this A slot.
            // Parity: raw group g - R went through this slot before g, and this
            // group consumed it at its stage j - R * GK / SPS, so that phase has
            // completed and the raw_full parity below cannot alias.
            if (main_stage && !__all_sync(0xFFFFFFFFu, wait(&raw_full[rs], (uint32_t)(g / C::R) & 1u))) break;
            const int nsub = min(SPS, n_steps - j * SPS);
            // A main stage reads all of its codes and scales first (every load in
            // flight at once); the raw slot goes back to the producer once the
            // stage's dequantized values are written (every loaded word used).
            uint4 cw[2 * SPS];
            uint32_t scw[SPS];
            if (main_stage) {
                const uint8_t *rb = R_ring + rs * RAW_STAGE;
                const int q0 = (j * SPS) % GK;
#pragma unroll
                for (int sub = 0; sub < SPS; ++sub) {
                    // codes: row `row`, logical 16-byte chunks 2q and 2q+1 of the
                    // 128-byte row, stored by TMA at chunk ^ (row % 8)
                    const int q = q0 + sub;
                    cw[2 * sub] = *reinterpret_cast<const uint4 *>(rb + row * 128 + (((2 * q) ^ (row & 7)) * 16));
                    cw[2 * sub + 1] =
                        *reinterpret_cast<const uint4 *>(rb + row * 128 + (((2 * q + 1) ^ (row & 7)) * 16));
                    scw[sub] = *reinterpret_cast<const uint32_t *>(rb + RAW_CODES + row * 16 + q * 4);
                }
            }
            // k-step `sub` of a main stage -> 32 bf16 pairs of row `row`
            auto dequant_step = [&](int sub, uint32_t (&out)[32]) {
                const uint4 c0 = cw[2 * sub], c1 = cw[2 * sub + 1];
                const uint32_t sc = scw[sub];
                if (MX) {  // bytes 0, 1 (and 2, 3) hold one 32-block's E8M0 byte twice
                    uint32_t fa0, fb0, fa1, fb1;
                    mx_scale_factors(sc << 20, fa0, fb0);
                    mx_scale_factors(sc << 4, fa1, fb1);
                    dequant_word_mx<PACKED>(c0.x, fa0, fb0, out + 0);
                    dequant_word_mx<PACKED>(c0.y, fa0, fb0, out + 4);
                    dequant_word_mx<PACKED>(c0.z, fa0, fb0, out + 8);
                    dequant_word_mx<PACKED>(c0.w, fa0, fb0, out + 12);
                    dequant_word_mx<PACKED>(c1.x, fa1, fb1, out + 16);
                    dequant_word_mx<PACKED>(c1.y, fa1, fb1, out + 20);
                    dequant_word_mx<PACKED>(c1.z, fa1, fb1, out + 24);
                    dequant_word_mx<PACKED>(c1.w, fa1, fb1, out + 28);
                    return;
                }
                const uint32_t f0 = scale_factor_bf16x2(sc << 20, pow2);
                const uint32_t f1 = scale_factor_bf16x2(sc << 12, pow2);
                const uint32_t f2 = scale_factor_bf16x2(sc << 4, pow2);
                const uint32_t f3 = scale_factor_bf16x2(sc >> 4, pow2);
                dequant_word<PACKED>(c0.x, f0, out + 0);
                dequant_word<PACKED>(c0.y, f0, out + 4);
                dequant_word<PACKED>(c0.z, f1, out + 8);
                dequant_word<PACKED>(c0.w, f1, out + 12);
                dequant_word<PACKED>(c1.x, f2, out + 16);
                dequant_word<PACKED>(c1.y, f2, out + 20);
                dequant_word<PACKED>(c1.z, f3, out + 24);
                dequant_word<PACKED>(c1.w, f3, out + 28);
            };
            constexpr int EARLY = C::EARLY < SPS ? C::EARLY : SPS;
            uint32_t early[EARLY][32];
            if (main_stage) {
#pragma unroll
                for (int e = 0; e < EARLY; ++e) dequant_step(e, early[e]);
            }
            // Then the A slot: free once the MMA is past stage j - S.
            if (sround > 0 && !__all_sync(0xFFFFFFFFu, wait(&stage_empty[s], (sround - 1) & 1u))) break;
#pragma unroll
            for (int sub = 0; sub < SPS; ++sub) {
                if (sub >= nsub) break;
                const int i = j * SPS + sub;
                const uint32_t taddr = trow + (uint32_t)(C::A_COL0 + s * 32 * SPS + sub * 32);
                if (main_stage && sub < EARLY) {
                    tmem_st32(taddr, early[sub]);
                    continue;
                }
                uint32_t out[32];
                if (main_stage) {
                    dequant_step(sub, out);
                } else {
                    // LoRA up-projection rows: B[n, l*64 .. +63], zero past r.
                    // (Chained: B may be written by work before this call.)
                    if (p.chain) pdl_wait();
                    if (F32AB) {  // FP32 adapters: B_hi or B_lo, stored out of line
                        const int L = p.lora_steps / 3, q = i - n_main, part = q / L;
                        lora_rows_f32(Bfg + (size_t)(row_ok ? n : 0) * p.r, (q - part * L) * BK, p.r, row_ok, part,
                                      taddr);
                        continue;
                    }
                    const int j0 = (i - n_main) * BK;
                    const __nv_bfloat16 *b = Blg + (size_t)(row_ok ? n : 0) * p.r + j0;
                    if (row_ok && (p.r & 7) == 0 && j0 + 64 <= p.r) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(b) + q);
                            out[4 * q] = v.x;
                            out[4 * q + 1] = v.y;
                            out[4 * q + 2] = v.z;
                            out[4 * q + 3] = v.w;
                        }
                    } else {
                        const uint16_t *bh = reinterpret_cast<const uint16_t *>(b);
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            const uint32_t lo = (row_ok && j0 + 2 * q < p.r) ? bh[2 * q] : 0u;
                            const uint32_t hi = (row_ok && j0 + 2 * q + 1 < p.r) ? bh[2 * q + 1] : 0u;
                            out[q] = lo | (hi << 16);
                        }
                    }
                }
                // row `row` of the step's A tile: TMEM lane `row`, 32 columns of bf16 pairs
                tmem_st32(taddr, out);
            }
            if (main_stage) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&raw_empty[rs]);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            const bool withhold = p.fault && blockIdx.x == 0 && warp == 0 && j == 0;
            if (lane == 0 && !withhold) mbar_arrive(&a_full[s]);
        }

        // ------------------------------------------- epilogue (warps 0-3)
        if (warp < 4) {
            const bool ok_warp = __all_sync(0xFFFFFFFFu, wait(acc_full, 0));
            if (lane == 0) ep_ok[warp] = ok_warp ? 1 : 0;
            named_bar_sync(1, 128);  // one decision for all four epilogue warps
            const bool ok = ep_ok[0] && ep_ok[1] && ep_ok[2] && ep_ok[3] && !*abort_flag;
            tc_fence_after();
            asm volatile("griddepcontrol.wait;" ::: "memory");  // the workspace and y follow the predecessor
            if (ok) {
                const float st = *tsg;
                const float ysc = st * pow2f(tc_exponent_offset(st));
                const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
                if (p.splits == 1) {
                    // TMEM -> bf16 tile Y[token][row] in the (now idle) token ring,
                    // then 16-byte row-contiguous stores to y.
                    uint8_t *Y = X_ring;
                    for (int c0 = 0; c0 < BN; c0 += 16) {
                        float v[16];
                        acc_load16(taddr + (uint32_t)c0, v);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            reinterpret_cast<__nv_bfloat16 *>(Y)[(c0 + j) * TILE_N + row] = __float2bfloat16_rn(v[j] * ysc);
                    }
                    named_bar_sync(1, 128);
                    const bool vec = (Ng % 8) == 0;
                    for (int v = threadIdx.x; v < BN * (TILE_N / 8); v += 128) {
                        const int m = m0 + v / (TILE_N / 8), nn = n0 + (v % (TILE_N / 8)) * 8;
                        if (m >= p.M || nn >= Ng) continue;
                        const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(Y) +
                                                   (v / (TILE_N / 8)) * TILE_N + (v % (TILE_N / 8)) * 8;
                        __nv_bfloat16 *dst = yg + (size_t)m * Ng + nn;
                        if (vec && nn + 8 <= Ng) {
                            *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
                        } else {
                            for (int e = 0; e < 8 && nn + e < Ng; ++e) dst[e] = src[e];
                        }
                    }
                } else {
                    // this split's FP32 partial tile [token][row]; the chained
                    // split-K reduction kernel sums the splits
                    float *part = p.partial + ((size_t)tile * p.splits + split) * (size_t)(TILE_N * BN);
                    for (int c0 = 0; c0 < BN; c0 += 16) {
                        float v[16];
                        acc_load16(taddr + (uint32_t)c0, v);
#pragma unroll
                        for (int j = 0; j < 16; ++j) __stcg(part + (size_t)(c0 + j) * TILE_N + row, v[j]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        if (lane == 0) drain_wait(acc_full, 0);  // every issued MMA has finished (no-op unless aborted)
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// LoRA down-projection for the tensor-core path: t = x A^T (FP32), written as
// u = bf16(t * s / ysc) into a [M, r_pad] buffer (zeros past r) that the main
// kernel reads as extra K steps, plus t_out when requested.  One CTA computes
// MB token rows x JB adapter rows; its 256 threads stride over K in 8-element
// vectors and the partial sums are reduced in shared memory in a fixed order.
// The main kernel may start (programmatic launch) while this kernel runs.
// AF32 (FP32 adapters): A is FP32 and each u row is [u_hi | u_lo | u_hi]
// (3 r_pad values, u_lo = bf16(t s / ysc - u_hi)) for the three LoRA products.
constexpr int LD_THREADS = 256;

template <int MB, int JB, bool AF32 = false>
__global__ void __launch_bounds__(LD_THREADS)
    lora_down_kernel(const __nv_bfloat16 *__restrict__ x, const void *__restrict__ Av, int M, int K, int r,
                     int r_pad, float s, const float *__restrict__ tensor_scale, float *__restrict__ t_out,
                     __nv_bfloat16 *__restrict__ u)
{
    const __nv_bfloat16 *A = static_cast<const __nv_bfloat16 *>(Av);
    const float *Af = static_cast<const float *>(Av);
    __shared__ float red[LD_THREADS / 32][MB * JB];
    pdl_trigger();  // the main kernel may start streaming its weight now
    pdl_wait();     // chained launch: x and A follow the preceding work
    const int jgroups = r_pad / JB;
    const int m0 = (blockIdx.x / jgroups) * MB, j0 = (blockIdx.x % jgroups) * JB;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float acc[MB][JB];
#pragma unroll
    for (int a = 0; a < MB; ++a)
#pragma unroll
        for (int b = 0; b < JB; ++b) acc[a][b] = 0.0f;
    if (j0 < r) {
#pragma unroll 2
        for (int k = threadIdx.x * 8; k < K; k += LD_THREADS * 8) {
            uint4 xv[MB];
            auto load_x = [&] {
#pragma unroll
                for (int a = 0; a < MB; ++a)
                    xv[a] = (m0 + a < M) ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(m0 + a) * K + k))
                                         : make_uint4(0u, 0u, 0u, 0u);
            };
            if constexpr (AF32) {
                load_x();
                float af[JB][8];  // A[j0 + b, k .. k + 7]
#pragma unroll
                for (int b = 0; b < JB; ++b) {
                    float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
                    if (j0 + b < r) {
                        lo = __ldg(reinterpret_cast<const float4 *>(Af + (size_t)(j0 + b) * K + k));
                        hi = __ldg(reinterpret_cast<const float4 *>(Af + (size_t)(j0 + b) * K + k) + 1);
                    }
                    af[b][0] = lo.x, af[b][1] = lo.y, af[b][2] = lo.z, af[b][3] = lo.w;
                    af[b][4] = hi.x, af[b][5] = hi.y, af[b][6] = hi.z, af[b][7] = hi.w;
                }
#pragma unroll
                for (int a = 0; a < MB; ++a) {
                    const uint32_t xw[4] = {xv[a].x, xv[a].y, xv[a].z, xv[a].w};
#pragma unroll
                    for (int b = 0; b < JB; ++b) {
                        float t = acc[a][b];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            t = fmaf(bf16lo(xw[q]), af[b][2 * q], t);
                            t = fmaf(bf16hi(xw[q]), af[b][2 * q + 1], t);
                        }
                        acc[a][b] = t;
                    }
                }
            } else {
                uint4 av[JB];
#pragma unroll
                for (int b = 0; b < JB; ++b)
                    av[b] = (j0 + b < r) ? __ldg(reinterpret_cast<const uint4 *>(A + (size_t)(j0 + b) * K + k))
                                         : make_uint4(0u, 0u, 0u, 0u);
                load_x();
#pragma unroll
                for (int a = 0; a < MB; ++a) {
                    const uint32_t xw[4] = {xv[a].x, xv[a].y, xv[a].z, xv[a].w};
#pragma unroll
                    for (int b = 0; b < JB; ++b) {
                        const uint32_t aw[4] = {av[b].x, av[b].y, av[b].z, av[b].w};
                        float t = acc[a][b];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            t = fmaf(bf16lo(xw[q]), bf16lo(aw[q]), t);
                            t = fmaf(bf16hi(xw[q]), bf16hi(aw[q]), t);
                        }
                        acc[a][b] = t;
                    }
                }
            }
        }
    }
#pragma unroll
    for (int a = 0; a < MB; ++a)
#pragma unroll
        for (int b = 0; b < JB; ++b) {
            float v = acc[a][b];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
            if (lane == 0) red[warp][a * JB + b] = v;
        }
    __syncthreads();
    if (threadIdx.x < MB * JB) {
        const int a = threadIdx.x / JB, b = threadIdx.x % JB;
        const int m = m0 + a, j = j0 + b;
        if (m < M) {
            float t = 0.0f;
#pragma unroll
            for (int w = 0; w < LD_THREADS / 32; ++w) t += red[w][threadIdx.x];
            if constexpr (AF32) {  // row [u_hi | u_lo | u_hi]
                __nv_bfloat16 uh = __float2bfloat16_rn(0.0f), ul = uh;
                if (j < r) {
                    const float st = *tensor_scale;
                    const float fac = s / (st * pow2f(tc_exponent_offset(st)));
                    if (t_out) t_out[(size_t)m * r + j] = t;
                    uh = __float2bfloat16_rn(t * fac);
                    ul = __float2bfloat16_rn(t * fac - __bfloat162float(uh));
                }
                __nv_bfloat16 *row = u + (size_t)m * 3 * r_pad;
                row[j] = uh;
                row[r_pad + j] = ul;
                row[2 * r_pad + j] = uh;
            } else if (j < r) {
                const float st = *tensor_scale;
                const float fac = s / (st * pow2f(tc_exponent_offset(st)));
                if (t_out) t_out[(size_t)m * r + j] = t;
                u[(size_t)m * r_pad + j] = __float2bfloat16_rn(t * fac);
            } else {
                u[(size_t)m * r_pad + j] = __float2bfloat16_rn(0.0f);
            }
        }
    }
}

// Split-K reduction of the forward: y[m, n] = bf16(s_t 2^c * sum over splits of
// the FP32 partial tiles), the splits summed in order (deterministic).  One
// thread per four rows n of one token m (16-byte partial loads).  Chained
// after the main kernel: it waits for that grid before reading.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *__restrict__ partial, int splits, int n_tiles,
                                                            int m_tiles, int BN, int M, const TcGroups grp)
{
    pdl_trigger();
    pdl_wait();
    const int64_t items = (int64_t)n_tiles * m_tiles * BN * (TILE_N / 4);
    for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < items; it += (int64_t)gridDim.x * blockDim.x) {
        const int rq = (int)(it % (TILE_N / 4)) * 4;
        const int64_t rest = it / (TILE_N / 4);
        const int col = (int)(rest % BN);
        const int64_t tile = rest / BN;  // m_tile * n_tiles + n_tile
        const int n_tile = (int)(tile % n_tiles), m_tile = (int)(tile / n_tiles);
        int g = 0;
#pragma unroll
        for (int i = 1; i < MAX_GROUPS; ++i)
            if (i < grp.G && n_tile >= grp.tile_start[i]) g = i;
        const int N = grp.N[g];
        const int m = m_tile * BN + col, n = (n_tile - grp.tile_start[g]) * TILE_N + rq;
        if (m >= M || n >= N) continue;
        const float st = *grp.ts[g];
        const float ysc = st * pow2f(tc_exponent_offset(st));
        const float *base = partial + (size_t)tile * splits * (size_t)(TILE_N * BN) + (size_t)col * TILE_N + rq;
        float4 v[MAX_SPLITS];  // every load in flight before the (fixed-order) sum
#pragma unroll
        for (int s2 = 0; s2 < MAX_SPLITS; ++s2)
            v[s2] = s2 < splits ? __ldcg(reinterpret_cast<const float4 *>(base + (size_t)s2 * (TILE_N * BN)))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s2 = 0; s2 < MAX_SPLITS; ++s2) {
            a.x += v[s2].x;
            a.y += v[s2].y;
            a.z += v[s2].z;
            a.w += v[s2].w;
        }
        __nv_bfloat16 *dst = grp.y[g] + (size_t)m * N + n;
        const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * ysc, a.y * ysc);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * ysc, a.w * ysc);
        if ((N & 3) == 0 && n + 4 <= N) {
            uint2 w;
            w.x = *reinterpret_cast<const uint32_t *>(&lo);
            w.y = *reinterpret_cast<const uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(dst) = w;
        } else {
            const __nv_bfloat16 v4[4] = {lo.x, lo.y, hi.x, hi.y};
            for (int e = 0; e < 4 && n + e < N; ++e) dst[e] = v4[e];
        }
    }
}

// ------------------------------------------------------------------ host side

struct FwdPlan {
    int BN = 0, n_tiles = 0, m_tiles = 0, splits = 1, sps = 0, nk = 0, lora_steps = 0, r_pad = 0;
    size_t u_bytes = 0, off_u = 0, off_part = 0, off_rows = 0, total = 0;
};

// Launch plan for G linears sharing x: their weight tiles side by side, one
// split factor, one u region per group, the split partials, and (one linear,
// many tokens) the partials of the rows x rank down-projection.  parts = 3
// (FP32 adapters): three LoRA products, u rows of 3 r_pad values.
FwdPlan plan_fwd(int64_t M, const int64_t *N, int G, int64_t K, int r, int parts = 1)
{
    FwdPlan pl;
    pl.BN = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
    pl.n_tiles = 0;
    for (int g = 0; g < G; ++g) pl.n_tiles += (int)((N[g] + TILE_N - 1) / TILE_N);
    pl.m_tiles = (int)((M + pl.BN - 1) / pl.BN);
    pl.nk = (int)(K / BK);
    pl.lora_steps = parts * ((r + BK - 1) / BK);
    pl.r_pad = (r + BK - 1) / BK * BK;
    const int64_t tiles = (int64_t)pl.n_tiles * pl.m_tiles;
    const int sms = num_sms();
    int splits = 1;
    if (tiles < sms) {
        splits = (int)(sms / tiles);
        int max_splits = pl.nk / 2 > 0 ? pl.nk / 2 : 1;  // at least two k-steps per split
        if (max_splits > MAX_SPLITS) max_splits = MAX_SPLITS;
        if (splits > max_splits) splits = max_splits;
        if (splits < 1) splits = 1;
    }
    pl.sps = (pl.nk + splits - 1) / splits;
    pl.sps = (pl.sps + GK - 1) / GK * GK;  // splits start on a raw-stage boundary
    pl.splits = (pl.nk + pl.sps - 1) / pl.sps;  // no empty split
    pl.u_bytes = round256(size_t(M) * pl.r_pad * parts * 2);
    pl.off_u = 0;
    pl.off_part = pl.u_bytes * G;
    pl.off_rows = pl.off_part + (pl.splits > 1 ? size_t(tiles) * pl.splits * TILE_N * pl.BN * 4 : 0);
    // many tokens: the down-projection runs as a split-K rows x rank product
    // (one pass over x for every group)
    pl.total = pl.off_rows +
               (parts == 1 && M > 64 && lora_down_rows_applies(K, r) ? lora_down_rows_ws(M, K, r, G) : 0);
    return pl;
}

bool tc_fwd_applies(int64_t M, int64_t N, int64_t K, int r)
{
    // K % 256: the scale rows (K/16 bytes) must be a multiple of 16 bytes for TMA
    return M >= 1 && N >= 1 && K >= GK * BK && K % (GK * BK) == 0 && r >= 1 && r <= 256 && M <= (1 << 30) &&
           N <= (1 << 30) && K <= (1 << 30);
}

struct Env {
    unsigned long long timeout_ns = 2000000000ull;  // 2 s
    int fault = 0;
    int no_fuse = 0;  // QERL_TC_NO_FUSE = 1: separate down-projection grid always (tests)
    Env()
    {
        const char *nf = std::getenv("QERL_TC_NO_FUSE");
        if (nf && nf[0] == '1') no_fuse = 1;
        const char *f = std::getenv("QERL_TEST_WITHHOLD_ARRIVAL");
        if (f && f[0] == '1') {
            fault = 1;
            timeout_ns = 50000000ull;  // 50 ms
        }
    }
};
const Env &env()
{
    static Env e;
    return e;
}

template <int BN, bool FUSED>
qerl_status launch_fwd(const TcMaps &maps, const TcFwdParams &p0, unsigned grid, bool packed, bool mx, bool f32,
                       bool pdl, cudaStream_t s)
{
    using C = Cfg<BN, FUSED>;
    auto kernel = packed ? tc_fwd_kernel<BN, true, FUSED> : tc_fwd_kernel<BN, false, FUSED>;
    // format variants: standard code layout, separate down-projection
    if ((mx || f32) && (FUSED || packed)) return QERL_ERR_SHAPE;
    if constexpr (!FUSED) {
        if (mx) kernel = tc_fwd_kernel<BN, false, false, true, false>;
        if (f32) kernel = tc_fwd_kernel<BN, false, false, false, true>;
    }
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return QERL_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::NUM_THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    const TcFwdParams p = p0;
    // Programmatic dependent launch: the CTAs may start while the preceding
    // grid still runs and stream their (frozen) weights; the token producer and
    // the epilogue wait for that grid with griddepcontrol.wait.  Every CTA
    // loads its own token tiles.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, maps, p) != cudaSuccess) return QERL_ERR_CUDA;
    return launched();
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 2-D row-major tensor map: `inner` elements per row (contiguous), `outer` rows.
bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_kblocks(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint32_t box_rows,
                      uint32_t kblocks)
{
    auto fn = encode_fn();
    if (!fn || K % 64 != 0) return false;
    // bf16 [rows, K] viewed as (64 k, row, k-block): one box = box_rows rows of
    // kblocks consecutive 64-element k-blocks, landing as kblocks [row][64] tiles
    cuuint64_t dims[3] = {64, rows, K / 64};
    cuuint64_t strides[2] = {K * 2, 128};
    cuuint32_t box[3] = {64, box_rows, kblocks};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t tc_fwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r)
{
    return tc_fwd_applies(M, N, K, r) ? plan_fwd(M, &N, 1, K, r).total : 0;
}

// G linears sharing x, M, K, r, lora_scale and the code layout (G = 1: one
// linear).  Returns QERL_ERR_SHAPE, having launched nothing, when the shapes
// are not covered.
qerl_status tc_fwd_groups(const FwdArgs *ga, int G, char *ws, size_t ws_bytes, cudaStream_t s)
{
    if (G < 1 || G > MAX_GROUPS) return QERL_ERR_SHAPE;
    const FwdArgs &a = ga[0];
    // format variants (one linear): MXFP4 weights, FP32 adapters
    const bool mx = a.mx != 0, f32 = a.Af != nullptr;
    const int parts = f32 ? 3 : 1;
    if ((mx || f32) && (G != 1 || (mx && a.packed) || (f32 && !a.Bf))) return QERL_ERR_SHAPE;
    int64_t Ns[MAX_GROUPS];
    bool any_t = false;
    for (int g = 0; g < G; ++g) {
        if (!tc_fwd_applies(a.M, ga[g].N, a.K, a.r)) return QERL_ERR_SHAPE;
        Ns[g] = ga[g].N;
        any_t = any_t || ga[g].t_out;
    }
    const FwdPlan pl = plan_fwd(a.M, Ns, G, a.K, a.r, parts);
    if (ws_bytes < pl.total) return QERL_ERR_WORKSPACE;
    float *partial = reinterpret_cast<float *>(ws + pl.off_part);
    const int tiles = pl.n_tiles * pl.m_tiles;

    // Fused LoRA down-projection (no separate grid) for decode tiles when t is
    // not requested, for split launches and for groups.  A single unsplit
    // linear keeps the separate grid: it overlaps the long weight stream, while
    // the fused MMAs would load it.
    const bool fused = !any_t && !mx && !f32 && pl.BN <= 64 && a.r <= FUSED_R && (pl.splits > 1 || G > 1) &&
                       !env().no_fuse;
    TcMaps maps = {};
    // codes: 128 rows x 128 bytes (4 k-steps) per box, 128-byte swizzle; scales:
    // 128 rows x 16 bytes (the same 4 k-steps); token tiles: BN rows x 64 bf16;
    // fused: LoRA A rows 0..31 x 64 bf16 (zero past r).
    if (!make_map_2d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, a.K, a.M, a.K * 2, BK, pl.BN,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return QERL_ERR_CUDA;
    for (int g = 0; g < MAX_GROUPS; ++g) {
        const FwdArgs &b = ga[g < G ? g : 0];  // unused slots repeat group 0
        __nv_bfloat16 *u = reinterpret_cast<__nv_bfloat16 *>(ws + pl.off_u + (g < G ? g : 0) * pl.u_bytes);
        if (!make_map_2d(&maps.codes[g], CU_TENSOR_MAP_DATA_TYPE_UINT8, b.codes, a.K / 2, b.N, a.K / 2, GK * BK / 2,
                         TILE_N, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map_2d(&maps.scl[g], CU_TENSOR_MAP_DATA_TYPE_UINT8, b.scales, a.K / 16, b.N, a.K / 16,
                         GK * BK / 16, TILE_N, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_map_2d(&maps.u[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, u, pl.r_pad * parts, a.M,
                         pl.r_pad * parts * 2, BK, pl.BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
            (fused && !make_map_2d(&maps.al[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, b.A, a.K, a.r, a.K * 2, BK, FUSED_R,
                                   CU_TENSOR_MAP_SWIZZLE_128B)))
            return QERL_ERR_CUDA;
    }

    // 1) LoRA down-projection, unless fused.  Chained, it may start before the
    //    preceding work finishes (it waits for it before touching memory), and
    //    the main kernel may then stream and dequantize its (frozen) weight
    //    while that work is still running.
    const bool chain = g_chain.load() != 0;
    const bool rows = !fused && !f32 && a.M > 64 && lora_down_rows_applies(a.K, a.r);
    if (rows) {
        DownRowsGroup dg[MAX_GROUPS];
        for (int g = 0; g < G; ++g)
            dg[g] = DownRowsGroup{ga[g].A, ga[g].tensor_scale, ga[g].t_out,
                                  reinterpret_cast<__nv_bfloat16 *>(ws + pl.off_u + g * pl.u_bytes)};
        QERL_TRY(lora_down_rows(a.x, a.M, a.K, dg, G, a.r, pl.r_pad, a.lora_scale,
                                reinterpret_cast<float *>(ws + pl.off_rows), chain, s));
    }
    for (int g = 0; g < G && !fused && !rows; ++g) {
        const FwdArgs &b = ga[g];
        __nv_bfloat16 *u = reinterpret_cast<__nv_bfloat16 *>(ws + pl.off_u + g * pl.u_bytes);
        const void *Av = f32 ? static_cast<const void *>(b.Af) : static_cast<const void *>(b.A);
        if (a.M <= 64) {  // few registers: its CTAs can share SMs with the main kernel's
            constexpr int MB = 4, JB = 2;
            const unsigned blocks = (unsigned)(((a.M + MB - 1) / MB) * (pl.r_pad / JB));
            auto k = f32 ? lora_down_kernel<MB, JB, true> : lora_down_kernel<MB, JB, false>;
            QERL_TRY(launched(launch_k(k, dim3(blocks), dim3(LD_THREADS), 0, s, chain, a.x, Av, (int)a.M, (int)a.K,
                                       a.r, pl.r_pad, a.lora_scale, b.tensor_scale, b.t_out, u)));
        } else {
            constexpr int MB = 8, JB = 4;
            const unsigned blocks = (unsigned)(((a.M + MB - 1) / MB) * (pl.r_pad / JB));
            auto k = f32 ? lora_down_kernel<MB, JB, true> : lora_down_kernel<MB, JB, false>;
            QERL_TRY(launched(launch_k(k, dim3(blocks), dim3(LD_THREADS), 0, s, chain, a.x, Av, (int)a.M, (int)a.K,
                                       a.r, pl.r_pad, a.lora_scale, b.tensor_scale, b.t_out, u)));
        }
    }

    // 2) main tensor-core kernel
    TcFwdParams p;
    p.M = (int)a.M;
    p.K = (int)a.K;
    p.nk = pl.nk;
    p.lora_steps = pl.lora_steps;
    p.lora_parts = parts;
    p.r = a.r;
    p.r_pad = pl.r_pad;
    p.splits = pl.splits;
    p.steps_per_split = pl.sps;
    p.n_tiles = pl.n_tiles;
    p.m_tiles = pl.m_tiles;
    p.grp.G = G;
    int t0 = 0;
    for (int g = 0; g < MAX_GROUPS; ++g) {
        const FwdArgs &b = ga[g < G ? g : 0];
        p.grp.tile_start[g] = t0;
        if (g < G) t0 += (int)((b.N + TILE_N - 1) / TILE_N);
        p.grp.N[g] = (int)b.N;
        p.grp.Bl[g] = b.B;
        p.grp.ts[g] = b.tensor_scale;
        p.grp.y[g] = b.y;
        p.grp.Bf[g] = b.Bf;
    }
    p.grp.tile_start[MAX_GROUPS] = t0;
    p.partial = partial;
    p.err = error_word();
    p.timeout_ns = env().timeout_ns;
    p.fault = env().fault;
    p.chain = chain ? 1 : 0;
    p.lora_scale = a.lora_scale;
    const unsigned grid = (unsigned)(tiles * pl.splits);
    qerl_status st;
    // The main kernel follows the down-projection grid programmatically; fused,
    // it follows the preceding work when launches are chained.
    const bool pk = a.packed != 0, pdl = fused ? chain : true;
    switch (pl.BN) {
    case 16:
        st = fused ? launch_fwd<16, true>(maps, p, grid, pk, mx, f32, pdl, s)
                   : launch_fwd<16, false>(maps, p, grid, pk, mx, f32, pdl, s);
        break;
    case 32:
        st = fused ? launch_fwd<32, true>(maps, p, grid, pk, mx, f32, pdl, s)
                   : launch_fwd<32, false>(maps, p, grid, pk, mx, f32, pdl, s);
        break;
    case 64:
        st = fused ? launch_fwd<64, true>(maps, p, grid, pk, mx, f32, pdl, s)
                   : launch_fwd<64, false>(maps, p, grid, pk, mx, f32, pdl, s);
        break;
    case 128: st = launch_fwd<128, false>(maps, p, grid, pk, mx, f32, pdl, s); break;
    default: st = launch_fwd<256, false>(maps, p, grid, pk, mx, f32, pdl, s); break;
    }
    if (st != QERL_OK || pl.splits == 1) return st;
    // 3) split-K: sum the partial tiles (chained: waits for the main grid)
    const int64_t items = (int64_t)tiles * pl.BN * (TILE_N / 4);
    int64_t gr = (items + 255) / 256;
    if (gr > 8 * num_sms()) gr = 8 * num_sms();
    return launched(launch_k(splitk_reduce_kernel, dim3((unsigned)gr), dim3(256), 0, s, chain, (const float *)partial,
                             pl.splits, pl.n_tiles, pl.m_tiles, pl.BN, (int)a.M, p.grp));
}

size_t tc_fwd_groups_ws_bytes(int64_t M, const int64_t *N, int G, int64_t K, int r)
{
    if (G < 1 || G > MAX_GROUPS) return 0;
    for (int g = 0; g < G; ++g)
        if (!tc_fwd_applies(M, N[g], K, r)) return 0;
    return plan_fwd(M, N, G, K, r).total;
}

qerl_status lora_down_small(const FwdArgs &a, int r_pad, float *t, __nv_bfloat16 *u, bool chain, cudaStream_t s)
{
    if (a.M < 1 || a.M > 64 || a.K % 8 != 0 || r_pad < a.r || r_pad % 2 != 0) return QERL_ERR_SHAPE;
    constexpr int MB = 4, JB = 2;
    const unsigned blocks = (unsigned)(((a.M + MB - 1) / MB) * (r_pad / JB));
    return launched(launch_k(lora_down_kernel<MB, JB>, dim3(blocks), dim3(LD_THREADS), 0, s, chain, a.x, a.A,
                             (int)a.M, (int)a.K, a.r, r_pad, a.lora_scale, a.tensor_scale, t, u));
}

qerl_status tc_linear_fwd(const FwdArgs &a, char *ws, size_t ws_bytes, cudaStream_t s)
{
    return tc_fwd_groups(&a, 1, ws, ws_bytes, s);
}

namespace {
// MXFP4 scales for the tensor-core path: each E8M0 byte of [N, K/32] written
// twice into [N, K/16] (the per-16 scale layout the raw stages load), and the
// tensor scale 2^-7 (exponent offset 7, output scale 1).  It never triggers
// its dependents early, so the kernels after it may read both before their
// own programmatic wait; it waits for the preceding work before writing (that
// work may still read the workspace).
__global__ void __launch_bounds__(256) mx_expand_scales_kernel(const uint8_t *__restrict__ s32, int64_t n8,
                                                               uint8_t *__restrict__ s16, float *__restrict__ ts)
{
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0) *ts = 0.0078125f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(s32) + i);  // 8 bytes -> 16
        uint4 o;
        o.x = prmt(v.x, 0u, 0x1100u);
        o.y = prmt(v.x, 0u, 0x3322u);
        o.z = prmt(v.y, 0u, 0x1100u);
        o.w = prmt(v.y, 0u, 0x3322u);
        reinterpret_cast<uint4 *>(s16)[i] = o;
    }
}
}  // namespace

size_t tc_fwd_variant_ws_bytes(int64_t M, int64_t N, int64_t K, int r, bool mx, bool f32)
{
    if (!tc_fwd_applies(M, N, K, r)) return 0;
    const size_t lin = plan_fwd(M, &N, 1, K, r, f32 ? 3 : 1).total;
    return mx ? round256(size_t(N) * (K / 16)) + 256 + lin : lin;
}

qerl_status tc_fwd_variant(FwdArgs a, const uint8_t *mx_scales, char *ws, size_t ws_bytes, cudaStream_t s)
{
    const bool mx = mx_scales != nullptr;
    if (!tc_fwd_applies(a.M, a.N, a.K, a.r) || (mx && a.packed)) return QERL_ERR_SHAPE;
    if (ws_bytes < tc_fwd_variant_ws_bytes(a.M, a.N, a.K, a.r, mx, a.Af != nullptr)) return QERL_ERR_WORKSPACE;
    if (mx) {
        const size_t sb = round256(size_t(a.N) * (a.K / 16));
        uint8_t *s16 = reinterpret_cast<uint8_t *>(ws);
        float *ts = reinterpret_cast<float *>(ws + sb);
        const int64_t n8 = a.N * (a.K / 256);  // K % 256 == 0: whole 8-byte groups
        int64_t gr = (n8 + 255) / 256;
        if (gr > 4 * num_sms()) gr = 4 * num_sms();
        QERL_TRY(launched(launch_k(mx_expand_scales_kernel, dim3((unsigned)gr), dim3(256), 0, s, g_chain.load() != 0,
                                   mx_scales, n8, s16, ts)));
        a.scales = s16;
        a.tensor_scale = ts;
        a.mx = 1;
        ws += sb + 256;
        ws_bytes -= sb + 256;
    }
    return tc_fwd_groups(&a, 1, ws, ws_bytes, s);
}

}  // namespace qerl
