// Layout change of the frozen NVFP4 codes: standard packing <-> the packed
// layout of packed_layout.cuh.  A pure bit permutation inside each 32-bit word,
// so it runs in place as well as out of place.  One HBM pass: 8-byte vectors
// (two words; K % 16 == 0 makes every row whole vectors) per thread, grid-stride.
#include "common.cuh"
#include "packed_layout.cuh"

namespace qerl {
namespace {

template <bool TO_PACKED>
__global__ void __launch_bounds__(256) repack_kernel(const uint8_t *in, uint8_t *out,
                                                     int64_t n_vec)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n_vec; v += stride) {
        uint2 w = reinterpret_cast<const uint2 *>(in)[v];
        if (TO_PACKED) {
            w.x = pack_code_word(w.x);
            w.y = pack_code_word(w.y);
        } else {
            w.x = unpack_code_word(w.x);
            w.y = unpack_code_word(w.y);
        }
        reinterpret_cast<uint2 *>(out)[v] = w;
    }
}

template <bool TO_PACKED>
qerl_status repack(const uint8_t *in, int64_t N, int64_t K, uint8_t *out, qerl_stream_t stream)
{
    if (!in || !out || N < 0 || K < 0) return QERL_ERR_INVALID_ARG;
    if (K % 16 != 0) return QERL_ERR_SHAPE;
    if (!aligned16(in) || !aligned16(out)) return QERL_ERR_ALIGN;
    const int64_t bytes = N * (K / 2);  // K % 16 == 0: rows are whole 8-byte vectors
    if (bytes == 0) return QERL_OK;
    // Distinct buffers must not overlap (in place, in == out, is fine).
    if (in != out && in < out + bytes && out < in + bytes) return QERL_ERR_INVALID_ARG;
    QERL_TRY(check_device());
    const int64_t n_vec = bytes / 8;
    int64_t g = (n_vec + 255) / 256;
    if (g > 8 * num_sms()) g = 8 * num_sms();
    repack_kernel<TO_PACKED><<<(unsigned)g, 256, 0, as_cuda(stream)>>>(in, out, n_vec);
    return launched();
}

}  // namespace
}  // namespace qerl

using namespace qerl;

extern "C" qerl_status qerl_nvfp4_pack_codes(const uint8_t *codes, int64_t N, int64_t K, uint8_t *packed,
                                             qerl_stream_t stream)
{
    return repack<true>(codes, N, K, packed, stream);
}

extern "C" qerl_status qerl_nvfp4_unpack_codes(const uint8_t *packed, int64_t N, int64_t K, uint8_t *codes,
                                               qerl_stream_t stream)
{
    return repack<false>(packed, N, K, codes, stream);
}
