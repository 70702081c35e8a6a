// qerl_nvfp4_lora_linear_fwd_noalloc: the LoRA linear forward for callers that
// cannot allocate device memory (a host framework that owns every device byte
// through its own pool, or code that must not call cudaMalloc mid-step because
// it can synchronize the device).  Its scratch is a fixed buffer in this
// library's own device memory instead of a caller workspace.
#include <mutex>

#include "linear.cuh"

namespace qerl {
namespace {

// The scratch of the no-allocation forward: the LoRA down-projection u (and
// its split partials for many tokens) and the split-K partial tiles.  Each
// launch writes every scratch element it later reads, so nothing has to start
// at zero.  Every GPU that loads the library holds these
// QERL_NOALLOC_SCRATCH_BYTES until the process exits.  All calls on a device
// share it and keep the previous call's contents; calls that overlap on the
// GPU race.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QERL_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
qerl_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QERL_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return QERL_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return QERL_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return QERL_OK;
}

}  // namespace
}  // namespace qerl

extern "C" qerl_status qerl_nvfp4_lora_linear_fwd_noalloc(const void *x, int64_t M, int64_t K, int64_t N,
                                                          const uint8_t *codes, const uint8_t *scales,
                                                          const float *tensor_scale, const void *A, const void *B,
                                                          int r, float lora_scale, void *y, float *t_out,
                                                          qerl_stream_t stream)
{
    return qerl::linear_fwd_fixed_ws(x, M, K, N, codes, scales, tensor_scale, A, B, r, lora_scale, y, t_out,
                                     QERL_NOALLOC_SCRATCH_BYTES, qerl::scratch_address, qerl::as_cuda(stream));
}
