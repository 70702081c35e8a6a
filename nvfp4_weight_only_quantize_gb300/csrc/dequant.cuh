// Register dequantizer of the tensor-core kernels: packed E2M1 codes and E4M3
// block scales -> bf16 pairs w'' = e2m1 * e4m3 * 2^-c (exact in bf16), ready
// to be stored as the 128-row A operand of a tcgen05 MMA.
#pragma once

#include <stdint.h>

#include "sm100_ptx.cuh"

namespace qerl {

// bf16x2 {f, f} with f = e4m3(b) * 2^(126 - c), exact (<= 4 significant bits).
// b20 holds the scale byte b in bits 20..27 (other bits are masked off here).
// As FP32 bits that is e4m3(b) * 2^-120 for every byte < 0x80, subnormal
// bytes included (they land on FP32 subnormals, which the multiply keeps), so
// two exact multiplies by powers of two give f.
__device__ __forceinline__ uint32_t scale_factor_bf16x2(uint32_t b20, float pow2)
{
    const float f = __uint_as_float(b20 & 0x0FF00000u) * __uint_as_float(247u << 23) * pow2;
    const uint32_t u = __float_as_uint(f);
    return ptx::prmt(u, u, 0x3232u);  // {high half, high half}
}

// Eight E2M1 codes (one word, element 2j in the low nibble of byte j) -> four
// bf16x2 words {elem 2j, elem 2j+1}.  The sign goes to bit 15 and the three
// exponent/mantissa bits to bits 8..6, which as a bf16 is e2m1 * 2^-126 (the
// code 0.5 becomes the subnormal 2^-127); one bf16x2 multiply by the block's
// scale factor then gives e2m1 * e4m3 * 2^-c exactly.
template <bool PACKED>
__device__ __forceinline__ void dequant_word(uint32_t q, uint32_t f2, uint32_t *out)
{
    if (PACKED) {
        // Packed layout: pair 0 already in place, pair 1 three bits low, pair 2
        // six bits low with its signs at 13/29, pair 3 three bits high with its
        // signs at 14/30.
        out[0] = ptx::bf16x2_mul(q & 0x81C081C0u, f2);
        out[1] = ptx::bf16x2_mul((q << 3) & 0x81C081C0u, f2);
        out[2] = ptx::bf16x2_mul(((q << 6) & 0x01C001C0u) | ((q << 2) & 0x80008000u), f2);
        out[3] = ptx::bf16x2_mul(((q >> 3) & 0x01C001C0u) | ((q << 1) & 0x80008000u), f2);
        return;
    }
    const uint32_t q4 = q << 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // byte 1 <- byte j of q4 (its high nibble is element 2j), byte 3 <- byte j of q
        const uint32_t u = ptx::prmt(q4, q, 0x4400u + 0x1111u * (uint32_t)j);
        const uint32_t raw = (u & 0x80008000u) | ((u >> 6) & 0x01C001C0u);
        out[j] = ptx::bf16x2_mul(raw, f2);
    }
}

// MXFP4 block scale (OCP MX: E8M0 byte b, scale 2^(b - 127)): bf16x2 factors
// fa, fb with fa * fb = 2^(b - 1), both normal bf16 for every b <= 254 (b = 255,
// the NaN scale, gives fb = NaN).  b20 holds b in bits 20..27.  With the codes
// placed as e2m1 * 2^-126 (dequant_word), (raw * fa) * fb = e2m1 * 2^(b - 127)
// exactly: for b <= 128 the first product is already the value (on the bf16
// subnormal grid at the smallest scales) and fb = 1; above, the first product
// is e2m1 * 2 and fb = 2^(b - 128).
__device__ __forceinline__ void mx_scale_factors(uint32_t b20, uint32_t &fa, uint32_t &fb)
{
    const uint32_t b = (b20 >> 20) & 0xFFu;
    const uint32_t ea = (b < 128u ? b : 128u) + 126u;  // exponent field of 2^(min(b, 128) - 1)
    const uint32_t eb = (b > 128u ? b : 128u) - 1u;    // exponent field of 2^(max(b, 128) - 128)
    fa = (ea << 7) * 0x10001u;
    fb = b == 255u ? 0x7FC07FC0u : (eb << 7) * 0x10001u;
}

// Eight E2M1 codes of an MXFP4 block -> four bf16x2 words e2m1 * 2^(b - 127).
template <bool PACKED>
__device__ __forceinline__ void dequant_word_mx(uint32_t q, uint32_t fa, uint32_t fb, uint32_t *out)
{
    dequant_word<PACKED>(q, fa, out);
#pragma unroll
    for (int j = 0; j < 4; ++j) out[j] = ptx::bf16x2_mul(out[j], fb);
}

}  // namespace qerl
