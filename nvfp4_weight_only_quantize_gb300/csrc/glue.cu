// Elementwise glue of a Qwen2.5-style decoder layer between its linears: the
// residual add h + y and the SwiGLU product silu(g) * u, each rounded to bf16
// once.  These are not steps of the quantized method itself; they let a
// decoder layer run as a sequence of this library's calls (the decoder-chain
// kernel fuses the same operations).  Both stream bf16 vectors, eight values
// per thread (16-byte accesses) when the pointers and the length allow, and
// are chained launches: they wait for the preceding work before reading.
#include "common.cuh"

namespace qerl {
namespace {

constexpr int kGlueThreads = 256;

// silu(g) * u in FP32, silu(g) = g * sigmoid(g) with the sigmoid formed from
// e = e^-|g| in (0, 1] (expf called): 1 / (1 + e) for g >= 0, e / (1 + e) below,
// so that no intermediate overflows (g / (1 + e^-g) would lose the tiny values
// of very negative g, where e^-g overflows FP32).
__device__ __forceinline__ float swiglu1(float g, float u)
{
    const float e = expf(-fabsf(g));
    const float sig = (g >= 0.0f ? 1.0f : e) / (1.0f + e);
    return g * sig * u;
}

template <bool SWIGLU>
__device__ __forceinline__ float glue1(float a, float b)
{
    return SWIGLU ? swiglu1(a, b) : a + b;
}

// out[i] = bf16(op(a[i], b[i])) for i < n; vec: every pointer 16-byte aligned
// and n % 8 == 0.  out may alias a or b (each element is read before it is
// written, by the same thread).
template <bool SWIGLU>
__global__ void __launch_bounds__(kGlueThreads)
    glue_kernel(const __nv_bfloat16 *a, const __nv_bfloat16 *b, int64_t n, int vec, __nv_bfloat16 *out)
{
    pdl_trigger();
    pdl_wait();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if (vec) {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n / 8; i += stride) {
            const uint4 va = reinterpret_cast<const uint4 *>(a)[i];
            const uint4 vb = reinterpret_cast<const uint4 *>(b)[i];
            const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat162 p = __floats2bfloat162_rn(glue1<SWIGLU>(bf16lo(wa[j]), bf16lo(wb[j])),
                                                               glue1<SWIGLU>(bf16hi(wa[j]), bf16hi(wb[j])));
                o[j] = *reinterpret_cast<const uint32_t *>(&p);
            }
            reinterpret_cast<uint4 *>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    } else {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
            out[i] = __float2bfloat16_rn(glue1<SWIGLU>(bf16f(a[i]), bf16f(b[i])));
    }
}

template <bool SWIGLU>
qerl_status glue(const void *a, const void *b, int64_t n, void *out, qerl_stream_t stream)
{
    if (n < 0) return QERL_ERR_INVALID_ARG;
    if (n == 0) return QERL_OK;
    if (!a || !b || !out) return QERL_ERR_INVALID_ARG;
    QERL_TRY(check_device());
    const bool vec = n % 8 == 0 && aligned16(a) && aligned16(b) && aligned16(out);
    const int64_t items = vec ? n / 8 : n;
    int64_t grid = (items + kGlueThreads - 1) / kGlueThreads;
    if (grid > 8 * num_sms()) grid = 8 * num_sms();
    return launched(launch_k(glue_kernel<SWIGLU>, dim3((unsigned)grid), dim3(kGlueThreads), 0, as_cuda(stream),
                             g_chain.load() != 0, static_cast<const __nv_bfloat16 *>(a),
                             static_cast<const __nv_bfloat16 *>(b), n, vec ? 1 : 0, static_cast<__nv_bfloat16 *>(out)));
}

}  // namespace
}  // namespace qerl

using namespace qerl;

extern "C" qerl_status qerl_residual_add(const void *h, const void *y, int64_t n, void *out, qerl_stream_t stream)
{
    return glue<false>(h, y, n, out, stream);
}

extern "C" qerl_status qerl_swiglu(const void *g, const void *u, int64_t n, void *out, qerl_stream_t stream)
{
    return glue<true>(g, u, n, out, stream);
}
