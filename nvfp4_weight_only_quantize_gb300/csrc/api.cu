// Library-wide entry points: device check, latched errors, workspace sizes,
// status strings, the host-side noise schedule and the launch counter.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "linear.cuh"

namespace qerl {

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_chain{1};

// First error a kernel found on this device (0 = none); cleared by qerl_get_error.
static __device__ unsigned int g_device_error;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_dev_state[kMaxDevices];            // 0 unknown, 1 ok, 2 unsupported
unsigned int *g_err_addr[kMaxDevices];   // device address of g_device_error
}  // namespace

qerl_status check_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QERL_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return QERL_ERR_UNSUPPORTED_DEVICE;
    int st = __atomic_load_n(&g_dev_state[dev], __ATOMIC_ACQUIRE);
    if (st == 1) return QERL_OK;
    if (st == 2) return QERL_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return QERL_ERR_CUDA;
    if (major != 10 || minor != 3) {
        __atomic_store_n(&g_dev_state[dev], 2, __ATOMIC_RELEASE);
        return QERL_ERR_UNSUPPORTED_DEVICE;
    }
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess) return QERL_ERR_CUDA;
    g_err_addr[dev] = static_cast<unsigned int *>(addr);
    __atomic_store_n(&g_dev_state[dev], 1, __ATOMIC_RELEASE);
    return QERL_OK;
}

unsigned int *error_word()
{
    int dev = 0;
    cudaGetDevice(&dev);
    return (dev >= 0 && dev < kMaxDevices) ? g_err_addr[dev] : nullptr;
}

}  // namespace qerl

using namespace qerl;

extern "C" qerl_status qerl_get_error(qerl_stream_t stream)
{
    QERL_TRY(check_device());
    cudaStream_t s = as_cuda(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return QERL_ERR_CUDA;
    unsigned int code = 0;
    unsigned int *w = error_word();
    if (cudaMemcpy(&code, w, sizeof code, cudaMemcpyDeviceToHost) != cudaSuccess) return QERL_ERR_CUDA;
    if (code != 0) {
        unsigned int zero = 0;
        if (cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return QERL_ERR_CUDA;
        return static_cast<qerl_status>(code);
    }
    return cudaPeekAtLastError() == cudaSuccess ? QERL_OK : QERL_ERR_CUDA;
}

extern "C" const char *qerl_status_string(qerl_status s)
{
    switch (s) {
    case QERL_OK: return "ok";
    case QERL_ERR_INVALID_ARG: return "invalid argument";
    case QERL_ERR_SHAPE: return "unsupported shape";
    case QERL_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case QERL_ERR_NONFINITE: return "weight holds Inf or NaN";
    case QERL_ERR_CUDA: return "CUDA runtime error";
    case QERL_ERR_TIMEOUT: return "bounded device wait timed out";
    case QERL_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (GB300)";
    case QERL_ERR_WORKSPACE: return "workspace missing or too small";
    case QERL_ERR_TOO_LARGE: return "problem needs more scratch than the fixed no-allocation buffer holds";
    }
    return "unknown status";
}

extern "C" size_t qerl_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, int r)
{
    auto round256 = [](size_t b) { return (b + 255) & ~size_t(255); };
    if (M < 0 || N < 0 || K < 0 || r < 0) return 0;
    switch (op) {
    case QERL_OP_QUANTIZE: return 4096;  // per-CTA amax partials (<= 1024 words)
    case QERL_OP_AQN_RMSNORM: return round256(size_t(K) * sizeof(float));  // K = H: noisy scale
    case QERL_OP_LINEAR_FWD: return linear_fwd_ws_bytes(M, N, K, r);
    case QERL_OP_LINEAR_BWD: return linear_bwd_ws_bytes(M, N, K, r);
    case QERL_OP_MXFP4_FWD:
    case QERL_OP_LINEAR_FWD_F32AB: return variant_fwd_ws_bytes(op, M, N, K, r);
    }
    return 0;
}

extern "C" float qerl_aqn_sigma(int64_t step, int64_t total_steps, float sigma_start, float sigma_end,
                                int num_stages)
{
    if (num_stages <= 1 || total_steps <= 0 || sigma_start == 0.0f) return sigma_start;
    if (step < 0) step = 0;
    int64_t k = step * num_stages / total_steps;
    if (k > num_stages - 1) k = num_stages - 1;
    double ratio = double(sigma_end) / double(sigma_start);
    return float(double(sigma_start) * pow(ratio, double(k) / double(num_stages - 1)));
}

extern "C" uint64_t qerl_launch_count(void) { return g_launches.load(); }

extern "C" qerl_status qerl_set_launch_chaining(int on)
{
    if (on != 0 && on != 1) return QERL_ERR_INVALID_ARG;
    g_chain.store(on);
    return QERL_OK;
}
