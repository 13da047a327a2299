// mhcpb_execute_static_scratch: the backward for callers that cannot allocate
// device memory (a host framework that owns the whole device heap, plugin
// code handed only its inputs and outputs).  It runs the same two kernels as
// mhcpb_execute, but the dW partials live in this file's __device__ array
// instead of a caller-allocated workspace, and no plan (which would allocate
// its status word) is involved.  Nothing here calls cudaMalloc or cudaFree.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <functional>
#include <mutex>

#include "mhcpb.h"
#include "mhcpb_internal.h"

using namespace mhcpb;

namespace {

// The scratch: dW partials [S][24][K] FP32 for S * K <= 16 MiB / 96 bytes.
// Part of the module image, so every device that loads it holds it until exit.
constexpr size_t kScratchBytes = MHCPB_STATIC_SCRATCH_BYTES;
__device__ __align__(256) float g_static_scratch[kScratchBytes / sizeof(float)];
// Where the streaming kernel records a device-side wait timeout.
__device__ __align__(256) uint32_t g_static_status[64];

constexpr int kMaxDevices = 64;

// Per-device set-up, done once with that device current: the device
// addresses of the two symbols (in host code the symbol names are host-side
// stand-ins, not device addresses), the kernels' shared-memory limit, the SM
// count and the compute-capability check.
struct DeviceSetup {
    std::once_flag once;
    mhcpb_status_t status = MHCPB_OK;
    float* scratch = nullptr;
    uint32_t* dev_status = nullptr;
    int sms = 0;
};
DeviceSetup g_setup[kMaxDevices];

void setup_device(DeviceSetup& s, int device) {
    int major = 0, minor = 0;
    cudaError_t e;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess) {
        s.status = (mhcpb_status_t)record_cuda_error(e, "cudaDeviceGetAttribute");
        return;
    }
    if (major != 10 || minor != 3) {
        s.status = MHCPB_ERR_UNSUPPORTED_DEVICE;
        return;
    }
    if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.scratch), g_static_scratch)) != cudaSuccess) {
        s.status = (mhcpb_status_t)record_cuda_error(e, "cudaGetSymbolAddress (static scratch)");
        return;
    }
    if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.dev_status), g_static_status)) != cudaSuccess) {
        s.status = (mhcpb_status_t)record_cuda_error(e, "cudaGetSymbolAddress (status word)");
        return;
    }
    if ((e = tc::setup(false)) != cudaSuccess || (e = tc::setup(true)) != cudaSuccess) {
        s.status = (mhcpb_status_t)record_cuda_error(e, "setup (tensor-core kernel)");
        return;
    }
    s.status = MHCPB_OK;
}

bool on_device(const void* ptr, int device) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == device;
}

}  // namespace

extern "C" mhcpb_status_t mhcpb_execute_static_scratch(int64_t T, int64_t K, uint32_t flags,
                                                       const void* x, const float* w,
                                                       const float* grad_proj,
                                                       const float* grad_r, const float* r,
                                                       void* dx, float* dw,
                                                       const void* grad_x_addend, void* stream) {
    if ((flags & MHCPB_ALLOW_TF32) == 0) return MHCPB_ERR_TF32_NOT_ALLOWED;
    if ((flags & ~(uint32_t)(MHCPB_ALLOW_TF32 | MHCPB_HAS_ADDEND | MHCPB_COMPENSATED_DW |
                             MHCPB_ACCUMULATE_DW)) != 0)
        return MHCPB_ERR_INVALID_ARG;
    if (T < 0 || T > MHCPB_MAX_T || K < 8 || K > MHCPB_MAX_K || (K % 8) != 0)
        return MHCPB_ERR_UNSUPPORTED_SHAPE;
    const int chunk = partial_tokens(T);
    const int64_t S = (T + chunk - 1) / chunk;
    const size_t need = (size_t)S * kNProj * (size_t)K * sizeof(float);
    if (need > kScratchBytes) return MHCPB_ERR_SCRATCH_TOO_SMALL;
    const bool add = (flags & MHCPB_HAS_ADDEND) != 0;
    // an operand with no elements (at T = 0: all but W and dW) needs no
    // storage and its pointer is not checked
    const void* all[8] = {x, w, grad_proj, grad_r, r, dx, dw, grad_x_addend};
    const size_t all_sizes[8] = {(size_t)(T * K * 2), (size_t)(kNProj * K * 4), (size_t)(T * kGradProjCols * 4),
                                 (size_t)(T * 4), (size_t)(T * 4), (size_t)(T * K * 2),
                                 (size_t)(kNProj * K * 4), (size_t)(T * K * 2)};
    const void* ptrs[8];
    size_t sizes[8];
    int n = 0;
    for (int i = 0; i < (add ? 8 : 7); ++i) {
        if (all_sizes[i] == 0) continue;
        if (all[i] == nullptr) return MHCPB_ERR_INVALID_ARG;
        ptrs[n] = all[i];
        sizes[n++] = all_sizes[i];
    }
    if (T > 0 && add != (grad_x_addend != nullptr)) return MHCPB_ERR_INVALID_ARG;

    for (int i = 0; i < n; ++i)
        if ((reinterpret_cast<uintptr_t>(ptrs[i]) & 15u) != 0) return MHCPB_ERR_MISALIGNED;
    for (int i = 0; i < n; ++i)
        for (int j = i + 1; j < n; ++j) {
            const uintptr_t a0 = reinterpret_cast<uintptr_t>(ptrs[i]), b0 = reinterpret_cast<uintptr_t>(ptrs[j]);
            if (a0 < b0 + sizes[j] && b0 < a0 + sizes[i]) return MHCPB_ERR_ALIASING;
        }

    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return (mhcpb_status_t)record_cuda_error(e, "cudaGetDevice");
    if (device < 0 || device >= kMaxDevices) return MHCPB_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (!on_device(ptrs[i], device)) return MHCPB_ERR_WRONG_DEVICE;

    DeviceSetup& s = g_setup[device];
    std::call_once(s.once, setup_device, std::ref(s), device);
    if (s.status != MHCPB_OK) return s.status;

    MainParams p{};
    p.T = (int32_t)T;
    p.K = (int32_t)K;
    p.S = (int32_t)S;
    p.chunk = chunk;
    p.n_strips = (int32_t)((K + tc::kStrip - 1) / tc::kStrip);
    p.x = static_cast<const uint16_t*>(x);
    p.w = w;
    p.grad_proj = grad_proj;
    p.grad_r = grad_r;
    p.r = r;
    p.dx = static_cast<uint16_t*>(dx);
    p.addend = static_cast<const uint16_t*>(grad_x_addend);
    p.partial = s.scratch;
    p.status = s.dev_status;
    p.timeout_ns = 1000000000ull;
    p.test_flags = 0;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (T > 0) {   // T = 0: no dX, no partials; the reduction below writes dW = 0 (or dW + 0)
        CUtensorMap m[6];
        if (const char* bad = encode_tc_maps(m, T, K, x, dx, add ? grad_x_addend : x, grad_proj, grad_r, r))
            return (mhcpb_status_t)record_cuda_error(cudaErrorInvalidValue, bad);
        const int64_t items = (int64_t)p.n_strips * p.S;
        p.half_units = tc::use_half_units(items, s.sms) ? 1 : 0;
        const int grid = tc::grid_size(items, s.sms);
        if ((e = tc::launch(p, m[0], m[1], m[2], m[3], m[4], m[5], grid, st)) != cudaSuccess)
            return (mhcpb_status_t)record_cuda_error(e, "launch (tensor-core kernel)");
    }
    if ((e = launch_reduce(p.partial, dw, p.S, (int64_t)kNProj * K,
                           (flags & MHCPB_COMPENSATED_DW) != 0,
                           (flags & MHCPB_ACCUMULATE_DW) != 0, true, st)) != cudaSuccess)
        return (mhcpb_status_t)record_cuda_error(e, "launch (dW reduction)");
    return MHCPB_OK;
}
