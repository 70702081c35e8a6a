// The packed code layout read by the tensor-core dequantizer.
//
// Each little-endian 32-bit word holds the eight E2M1 codes of k = 8w .. 8w+7 of
// one weight row, in both layouts.  In the standard layout, element i sits in
// bits 4i .. 4i+3.  In the packed layout, elements 2p (even) and 2p+1 (odd) form
// pair p; its codes are spread so that one shift and one or two masks put them
// where a bf16x2 word wants them: sign at bit 15 (31), and the two exponent
// bits and the mantissa bit at bits 8..6 (24..22), which as bf16 reads
// e2m1 * 2^-126.
//
//   pair p | magnitude bits (m, e0, e1) of the even element | its sign bit
//   -------+-----------------------------------------------+-------------
//     0    |  6, 7, 8                                      |  15
//     1    |  3, 4, 5                                      |  12
//     2    |  0, 1, 2                                      |  13
//     3    |  9, 10, 11                                    |  14
//
// The odd element of each pair uses the same positions plus 16.  The four rows
// plus 16 cover the 32 bits exactly once, so the layout is a bit permutation
// of the word: same size, any K % 8 == 0.
#pragma once

#include <stdint.h>

namespace qerl {

__host__ __device__ constexpr int packed_mag_bit(int p) { return p == 0 ? 6 : p == 1 ? 3 : p == 2 ? 0 : 9; }
__host__ __device__ constexpr int packed_sign_bit(int p) { return p == 0 ? 15 : p == 1 ? 12 : p == 2 ? 13 : 14; }

// Bit position in the packed word of nibble bit b (0 = m, 1 = e0, 2 = e1, 3 = sign) of element i.
__host__ __device__ constexpr int packed_bit(int i, int b)
{
    return (b == 3 ? packed_sign_bit(i >> 1) : packed_mag_bit(i >> 1) + b) + 16 * (i & 1);
}

__host__ __device__ inline uint32_t pack_code_word(uint32_t w)
{
    uint32_t out = 0;
    for (int i = 0; i < 8; ++i)
        for (int b = 0; b < 4; ++b) out |= ((w >> (4 * i + b)) & 1u) << packed_bit(i, b);
    return out;
}

__host__ __device__ inline uint32_t unpack_code_word(uint32_t w)
{
    uint32_t out = 0;
    for (int i = 0; i < 8; ++i)
        for (int b = 0; b < 4; ++b) out |= ((w >> packed_bit(i, b)) & 1u) << (4 * i + b);
    return out;
}

// Code (4 bits) of element i of a packed word.
__host__ __device__ inline uint32_t packed_code(uint32_t w, int i)
{
    const int hi = 16 * (i & 1);
    return ((w >> (packed_mag_bit(i >> 1) + hi)) & 7u) | (((w >> (packed_sign_bit(i >> 1) + hi)) & 1u) << 3);
}

}  // namespace qerl
