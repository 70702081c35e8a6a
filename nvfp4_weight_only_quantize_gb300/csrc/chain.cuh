// Internal tables of the persistent decoder-chain kernel (decode_chain.cu):
// the linears, glue steps, phases and per-CTA job lists of a planned chain of
// decoder layers, as laid out in the plan region of the caller's workspace.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include <cuda_bf16.h>

namespace qerl {
namespace chain {

constexpr int TILE_N = 128;   // weight rows per job tile (MMA M)
constexpr int BN = 64;        // token columns (MMA N): every chain runs M <= 64 tokens
constexpr int KC = 256;       // k per stage (one raw stage: 4 MMA k-steps of 64)
constexpr int MAX_CTAS = 1024;

// Epilogue of a linear's tile (after the split parts are summed, v = D * s_t 2^c):
enum LinKind : int {
    LIN_NORMED = 0,  // y = bf16(v * rs[m]); rs from the input's sum-of-squares partials
    LIN_RESID = 1,   // h_out = bf16(h_in + bf16(v)); next-norm input xn = bf16(h_out * ns),
                     // and the tile's sum of squares of h_out per token
};
// Steps that run on the epilogue warps only.
enum GlueKind : int {
    GLUE_NOISE = 0,    // noisy norm scales ns = gamma + sigma z for every norm of the chain
    GLUE_PRENORM = 1,  // first layer: xn = bf16(x * ns), sum of squares of x per 128-column tile
    GLUE_SWIGLU = 2,   // m = bf16(silu(g) * u)
};

struct Lin {
    int N, K, r, kind;
    int phase;          // phase whose counter this linear's tiles increment
    int n_tiles;        // N / 128
    int sq_tiles;       // normed input: K / 128 sum-of-squares partials per token
    int tile0;          // first tile counter of this linear within its phase
    const uint8_t *codes, *scales;
    const float *ts;                 // tensor scale (device)
    const __nv_bfloat16 *B;          // [N, r]
    __nv_bfloat16 *y;                // LIN_NORMED output [M, N] (may be null)
    const float *sq_in;              // LIN_NORMED: [sq_tiles][64]
    const __nv_bfloat16 *h_in;       // LIN_RESID: [M, N]
    __nv_bfloat16 *h_out;            // LIN_RESID: [M, N]
    __nv_bfloat16 *xn_out;           // LIN_RESID: next-norm input [M, N] (null: none)
    const float *ns_next;            // LIN_RESID: next norm's scale [N]
    float *sq_out;                   // LIN_RESID: [N / 128][64]
};
// TMA maps of a linear, 64-byte aligned: codes, scales, LoRA A rows, input x.
struct LinMaps {
    CUtensorMap codes, scl, al, x;
};

struct Glue {
    int kind, phase;
    int units;          // work units of this step
    int cols;           // GLUE_SWIGLU: columns per unit; GLUE_PRENORM: H
    int width;          // row length of the tensors it touches
    int n_norms;        // GLUE_NOISE: number of norms (2 per layer)
    const __nv_bfloat16 *a, *b;      // SWIGLU: g, u; PRENORM: x
    __nv_bfloat16 *out;              // SWIGLU: m; PRENORM: xn
    float *sq;                       // PRENORM: [H / 128][64]
    float *ns;                       // NOISE: [n_norms][width] out; PRENORM: the first norm's scale
    const __nv_bfloat16 *const *gammas;  // NOISE: [n_norms] device array of gamma pointers
};

// One job of a CTA: a part (k-chunk range) of one tile of a linear, or one unit
// of a glue step.
struct Job {
    int type;           // 0 matmul, 1 glue
    int idx;            // linear or glue index
    int tile;           // matmul: tile; glue: unit
    int kc0, kc1;       // matmul: k-chunk range [kc0, kc1) (256 k each)
    int part, nparts;   // matmul: this part's index within the tile and the tile's part count
    int slot;           // matmul, nparts > 1: partial slot of this part
};

struct Plan {
    int n_ctas, n_lin, n_glue, n_phases;
    int M;              // tokens (<= 64)
    int r_max;
    float lora_scale, eps;
    const Lin *lins;
    const LinMaps *maps;
    const Glue *glues;
    const Job *jobs;
    const int *job_off;        // [n_ctas + 1]
    const int *phase_total;    // [n_phases]: units that complete each phase
    int *phase_cnt;            // [n_phases] (zero between launches)
    int *tile_cnt;             // per phase tile counters (zero between launches)
    int *exit_cnt;             // (zero between launches)
    float *partials;           // [slots][64 tokens][128 rows]
    unsigned int *err;
    unsigned long long timeout_ns;
};

}  // namespace chain
}  // namespace qerl
