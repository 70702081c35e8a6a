// Internal interface between the linear entry points and their kernels.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace qerl {

// Arguments of one forward call, validated by the entry point.
struct FwdArgs {
    const __nv_bfloat16 *x;
    int64_t M, K, N;
    const uint8_t *codes, *scales;
    const float *tensor_scale;
    const __nv_bfloat16 *A, *B;
    int r;
    float lora_scale;
    __nv_bfloat16 *y;
    float *t_out;
    int packed = 0;  // codes in the packed layout (packed_layout.cuh)
    // MXFP4 weight on the tensor-core path: `scales` then holds the E8M0 byte
    // of each block of 32 twice ([N, K/16], tc_fwd_variant) and tensor_scale
    // points to 2^-7, which makes the kernels' exponent offset 7 and their
    // output scale 1 (the E8M0 factor carries the whole scale).
    int mx = 0;
    // FP32 LoRA adapters (A [r, K], B [N, r]) in place of A and B when set.
    const float *Af = nullptr, *Bf = nullptr;
};

struct BwdArgs {
    const __nv_bfloat16 *dy, *x;
    int64_t M, K, N;
    const uint8_t *codes, *scales;
    const float *tensor_scale;
    const __nv_bfloat16 *A, *B;
    int r;
    float lora_scale;
    const float *t_saved;
    __nv_bfloat16 *dx;
    float *dA, *dB;
    int accumulate;
    int packed = 0;
};

size_t linear_fwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r);
size_t linear_bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r);
// QERL_OP_MXFP4_FWD or QERL_OP_LINEAR_FWD_F32AB (qerl_workspace_bytes).
size_t variant_fwd_ws_bytes(int op, int64_t M, int64_t N, int64_t K, int r);

// Tensor-core (tcgen05) path.  Returns QERL_ERR_SHAPE, having launched nothing,
// when it does not cover the call; the caller then runs the CUDA-core path.
size_t tc_fwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r);
qerl_status tc_linear_fwd(const FwdArgs &a, char *ws, size_t ws_bytes, cudaStream_t s);
// G (<= 3) linears sharing x, M, K, r, lora_scale and layout in one launch.
qerl_status tc_fwd_groups(const FwdArgs *ga, int G, char *ws, size_t ws_bytes, cudaStream_t s);
size_t tc_fwd_groups_ws_bytes(int64_t M, const int64_t *N, int G, int64_t K, int r);
// Format variants on the tensor-core path (one linear): an MXFP4 weight
// (mx_scales: E8M0 bytes [N, K/32], 16-byte aligned; a.codes in the standard
// layout) and/or FP32 adapters (a.Af, a.Bf).  Scratch need, 0 when the path
// does not cover the shape; QERL_ERR_SHAPE, having launched nothing, then.
size_t tc_fwd_variant_ws_bytes(int64_t M, int64_t N, int64_t K, int r, bool mx, bool f32);
qerl_status tc_fwd_variant(FwdArgs a, const uint8_t *mx_scales, char *ws, size_t ws_bytes, cudaStream_t s);
// t = x A^T (FP32 [M, r] to `t`) and u = bf16(s t / (s_t 2^c)) ([M, r_pad],
// zero past r; r_pad even) by the CUDA-core down-projection kernel, for
// M <= 64 and K % 8 == 0.
qerl_status lora_down_small(const FwdArgs &a, int r_pad, float *t, __nv_bfloat16 *u, bool chain, cudaStream_t s);

// CUDA-core GEMV path (gemv.cu) for one or two tokens: QERL_ERR_SHAPE, having
// launched nothing, when it does not cover the call (M > 2, K % 32 != 0, r >
// 256, or x too large for shared memory).
bool gemv_applies(int64_t M, int64_t N, int64_t K, int r);
size_t gemv_ws_bytes(int64_t M, int64_t N, int64_t K, int r);
qerl_status gemv_fwd(const FwdArgs &a, char *ws, size_t ws_bytes, cudaStream_t s);

inline size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

// 2-D row-major TMA tensor map: `inner` elements per row (contiguous), `outer`
// rows of `row_bytes`; false if the driver rejects it.
bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);
// 3-D TMA map of a bf16 [rows, K] row-major matrix (K % 64 == 0) whose box is
// box_rows rows x kblocks consecutive 64-element k-blocks, written to shared
// memory as kblocks tiles [box_rows][64] in the 128-byte swizzle (the layout of
// kblocks separate 2-D boxes, in one copy).  Coordinates: (0, row, k / 64).
bool make_map_kblocks(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint32_t box_rows,
                      uint32_t kblocks);

// Rank products on tensor cores (rank_tc.cu), split over the reduction: for g < G,
//   part_g[z][m][j] = sum over k in split z of X[m, k] * W_g[j, k],  j < r_g,
// X [M, Kd] and W_g [r_g, Kd] bf16 row-major, 16-byte aligned, Kd % 8 == 0,
// Kd >= 64, r_g <= 128, and G * rank_tc_pad(max r_g) <= 256 (else QERL_ERR_SHAPE);
// part_g holds rank_tc_part_bytes(M, Kd, r_g) bytes, and the rank_tc_splits(M, Kd)
// partials are summed in split order by the caller.
constexpr int RANK_MAX_G = 3;
inline int rank_tc_pad(int r) { return r <= 32 ? 32 : r <= 64 ? 64 : 128; }
struct RankOut {
    const __nv_bfloat16 *W;
    int r;
    float *part;
};
bool rank_tc_applies(int64_t M, int64_t Kd, int r, const void *X, const void *W);
int rank_tc_splits(int64_t M, int64_t Kd);
size_t rank_tc_part_bytes(int64_t M, int64_t Kd, int r);
qerl_status rank_tc(const __nv_bfloat16 *X, int64_t M, int64_t Kd, const RankOut *outs, int G, bool chain,
                    cudaStream_t s);

// Wide x rank products on tensor cores (rank_tc.cu), split over the tokens:
//   part[z][w][j] (wj) or part[z][j][w] = sum over m in split z of D[m, w] * T[m, j],
// D bf16 [M, Wd] row-major, 16-byte aligned, Wd % 8 == 0, Wd >= 64; T FP32
// [M, r], r <= 64.  tb holds wide_tc_tb_bytes(M, r) bytes of scratch: T as the
// bf16 pair [M][2 RP] (hi = bf16(T), lo = bf16(T - hi), zeros past r; RP =
// rank_tc_pad(r)), written here unless tb_ready.  part holds
// wide_tc_part_bytes(M, Wd, r) bytes; the wide_tc_splits(M, Wd) partials are
// summed in split order by the caller.
bool wide_tc_applies(int64_t M, int64_t Wd, int r, const void *D);
int wide_tc_splits(int64_t M, int64_t Wd);
size_t wide_tc_part_bytes(int64_t M, int64_t Wd, int r);
size_t wide_tc_tb_bytes(int64_t M, int r);
qerl_status wide_tc(const __nv_bfloat16 *D, int64_t M, int64_t Wd, const float *T, int r, bool wj,
                    __nv_bfloat16 *tb, bool tb_ready, float *part, bool chain, cudaStream_t s);

// LoRA down-projection for many tokens, for G (<= 3) linears sharing x (one
// pass over x on tensor cores where rank_tc applies, else CUDA cores group by
// group): t_g = x A_g^T, t_out_g = t_g when given, u_g = bf16(s t_g / (s_t,g
// 2^c_g)) [M, r_pad] (zeros past r).  part holds lora_down_rows_ws(M, K, r, G)
// bytes.  Chained launches when `chain`.
struct DownRowsGroup {
    const __nv_bfloat16 *A;
    const float *tensor_scale;
    float *t_out;
    __nv_bfloat16 *u;
};
bool lora_down_rows_applies(int64_t K, int r);
size_t lora_down_rows_ws(int64_t M, int64_t K, int r, int G);
qerl_status lora_down_rows(const __nv_bfloat16 *x, int64_t M, int64_t K, const DownRowsGroup *grp, int G, int r,
                           int r_pad, float s, float *part, bool chain, cudaStream_t st);

// Tensor-core input gradient dx = dy w_hat + s v A for the shapes it covers
// (K % 256 == 0, N % 64 == 0, r <= 256); v = dy B in FP32 [M, r] is given, and
// vp_ws holds tc_dx_ws_bytes(M, r) bytes of scratch: the LoRA operand
// v' = bf16(s v / (s_t 2^c)) as [M, tc_dx_rpad(r)] (zeros past r), written here
// unless vp_ready.
bool tc_dx_applies(int64_t M, int64_t N, int64_t K, int r);
int tc_dx_rpad(int r);
size_t tc_dx_ws_bytes(int64_t M, int r);
qerl_status tc_dx(const BwdArgs &a, const float *v, char *vp_ws, bool vp_ready, cudaStream_t s);

// Forward with a fixed scratch buffer: validates the arguments like the
// workspace entry point, returns QERL_ERR_TOO_LARGE when the call needs more
// than ws_cap bytes, then asks get_ws for the buffer and runs the same kernels.
qerl_status linear_fwd_fixed_ws(const void *x, int64_t M, int64_t K, int64_t N, const uint8_t *codes,
                                const uint8_t *scales, const float *tensor_scale, const void *A, const void *B, int r,
                                float lora_scale, void *y, float *t_out, size_t ws_cap,
                                qerl_status (*get_ws)(void **), cudaStream_t s);

}  // namespace qerl
