// Shared helpers of the qerl CUDA library (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "qerl.h"

namespace qerl {

// Host-side count of kernel launches made by the library (qerl_launch_count).
extern std::atomic<uint64_t> g_launches;

// QERL_OK when the current device is compute capability 10.3, else
// QERL_ERR_UNSUPPORTED_DEVICE (or QERL_ERR_CUDA).  Cached per device.
qerl_status check_device();

// Device address of this library's latched-error word on the current device
// (a file-scope __device__ variable; resolved once per device).
unsigned int *error_word();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_cuda(qerl_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline int num_sms()
{
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 152;
    if (!cached[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = v > 0 ? v : 152;
    }
    return cached[dev];
}

// After a launch: count it and turn a launch error into QERL_ERR_CUDA.
// Programmatic dependent launch: when `chained`, the kernel may be scheduled
// before the preceding work on the stream has finished; it must execute
// pdl_wait() before it touches memory that preceding work writes or reads.
extern std::atomic<int> g_chain;
template <typename... Params, typename... Args>
cudaError_t launch_k(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool chained,
                     Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = chained ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}
// Wait for the preceding grid (no-op unless launched chained) / let the next
// chained grid be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

inline qerl_status launched()
{
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaPeekAtLastError() == cudaSuccess ? QERL_OK : QERL_ERR_CUDA;
}
inline qerl_status launched(cudaError_t e)
{
    if (e != cudaSuccess) return QERL_ERR_CUDA;
    return launched();
}

#define QERL_TRY(expr)                          \
    do {                                        \
        qerl_status _st = (expr);               \
        if (_st != QERL_OK) return _st;         \
    } while (0)

// ---------------------------------------------------------------- device side

// Latch the first device-detected error (0 = none).
__device__ __forceinline__ void latch_error(unsigned int *err, unsigned int code)
{
    if (err) atomicCAS(err, 0u, code);
}

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(__nv_bfloat16 h) { return __bfloat162float(h); }

// Value of a non-negative E4M3 byte (0..126): exponent bias 7, subnormal m*2^-9.
__device__ __forceinline__ float e4m3_to_float(uint32_t b)
{
    uint32_t e = (b >> 3) & 15u, m = b & 7u;
    return e == 0 ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Value of an E2M1 code (sign bit 3; magnitudes 0,.5,1,1.5,2,3,4,6).
__device__ __forceinline__ float e2m1_to_float(uint32_t c)
{
    uint32_t e = (c >> 1) & 3u, m = c & 1u;
    float v = e == 0 ? 0.5f * (float)m : __uint_as_float(((e + 126u) << 23) | (m << 22));
    return (c & 8u) ? -v : v;
}

// Exponent offset c in [7, 116] with s_t * 2^c in [1, 2) when possible: the
// tensor-core paths carry e2m1 * e4m3 * 2^-c in bf16 (then a normal bf16 range,
// [2^-10-c, 2688 * 2^-c]) and scale by s_t * 2^c once, in FP32.
__device__ __forceinline__ int tc_exponent_offset(float s_t)
{
    int e = 0;
    frexpf(s_t, &e);
    const int c = 1 - e;
    return c < 7 ? 7 : (c > 116 ? 116 : c);
}

// 2^e as a float for e in the normal range (exact, unlike exp2f).
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

}  // namespace qerl
