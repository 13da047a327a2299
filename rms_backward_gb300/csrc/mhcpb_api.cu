// Host side of the C ABI declared in include/mhcpb.h: plan creation, the
// tensor contract checks of the cuDNN frontend page "DSv4.1 mHC
// projection/RMS backward" ("Requirements and tensor contract"), TMA tensor
// map encoding and the two launches of one execute ("Prepared class API":
// each execute launches the two kernels and allocates no memory).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "mhcpb.h"
#include "mhcpb_check.cuh"
#include "mhcpb_internal.h"

using namespace mhcpb;

struct mhcpb_plan_s {
    int64_t T = 0, K = 0;
    int device = 0;
    uint32_t flags = 0;
    int S = 0;            // dW partials
    int chunk = 0;        // tokens per dW partial
    int half_units = 0;   // tensor-core kernel schedules half items
    int n_strips = 0;     // strips of the streaming kernel in use
    int grid = 0;         // CTAs of the streaming kernel
    size_t ws_bytes = 0;
    size_t smem = 0;
    uint32_t* d_status = nullptr;
    uint64_t timeout_ns = 1000000000ull;  // 1 s bound on every in-kernel wait
    int max_grid = 0;     // default grid of the tensor-core kernel (before any cap)
    uint64_t* d_trace = nullptr;  // timeline stamps (builds with MHCPB_TRACE only)
    size_t trace_bytes = 0;
    int fwd_grid = 0;     // CTAs of the forward's tensor-core kernel
    int fwd_max_grid = 0; // its default (before any cap)
};

namespace {

thread_local char g_cuda_err[256] = "";

mhcpb_status_t cuda_fail(cudaError_t e, const char* what) {
    std::snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", what, cudaGetErrorString(e));
    return MHCPB_ERR_CUDA;
}

// Restores the caller's current device on scope exit.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn get_encode() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

// BF16 [T, K] row-major tensor, boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool encode_bf16_map(CUtensorMap* m, const void* base, int64_t T, int64_t K, uint32_t box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)tc::kBoxCols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP32 tensor maps without swizzle: grad_proj [T, 32] read as boxes of 24
// columns x 128 rows (columns 24..31 are never fetched), and [T] vectors read
// as boxes of 128.
bool encode_f32_map(CUtensorMap* m, const void* base, int64_t T, int cols, uint32_t box_cols,
                    uint32_t box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const cuuint32_t estr[2] = {1, 1};
    if (cols == 0) {
        // a [T] vector as a 2-D {T, 1} tensor (one row; its row stride is never
        // used but must be a multiple of 16 bytes)
        const cuuint64_t dims[2] = {(cuuint64_t)T, 1};
        const cuuint64_t strides[1] = {(cuuint64_t)((T * 4 + 15) / 16 * 16)};
        const cuuint32_t box[2] = {box_rows, 1};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    const cuuint32_t box[2] = {box_cols, box_rows};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encodes the six tensor maps of one execute; on failure names the map.
const char* encode_maps(CUtensorMap (&m)[6], int64_t T, int64_t K, const void* x, const void* dx,
                        const void* add, const void* gp, const void* gr, const void* r) {
    if (!encode_bf16_map(&m[0], x, T, K, tc::kTokenTile)) return "tensor map of x";
    if (!encode_bf16_map(&m[1], dx, T, K, 32)) return "tensor map of dx";
    if (!encode_bf16_map(&m[2], add, T, K, tc::kTokenTile)) return "tensor map of grad_x_addend";
    if (!encode_f32_map(&m[3], gp, T, kGradProjCols, kNProj, tc::kTokenTile))
        return "tensor map of grad_proj";
    if (!encode_f32_map(&m[4], gr, T, 0, 0, tc::kTokenTile)) return "tensor map of grad_r";
    if (!encode_f32_map(&m[5], r, T, 0, 0, tc::kTokenTile)) return "tensor map of r";
    return nullptr;
}

struct Range {
    uintptr_t lo, hi;
};
// an empty range overlaps nothing
bool overlap(const Range& a, const Range& b) {
    return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

mhcpb_status_t check_device_ptr(const void* ptr, int device) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MHCPB_ERR_WRONG_DEVICE;
    }
    if ((a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) || a.device != device)
        return MHCPB_ERR_WRONG_DEVICE;
    return MHCPB_OK;
}

}  // namespace

namespace mhcpb {
const char* encode_tc_maps(CUtensorMap (&m)[6], int64_t T, int64_t K, const void* x,
                           const void* dx, const void* add, const void* gp, const void* gr,
                           const void* r) {
    return encode_maps(m, T, K, x, dx, add, gp, gr, r);
}
int record_cuda_error(cudaError_t e, const char* what) { return (int)cuda_fail(e, what); }
}  // namespace mhcpb

extern "C" {

const char* mhcpb_status_string(mhcpb_status_t s) {
    switch (s) {
        case MHCPB_OK: return "ok";
        case MHCPB_ERR_INVALID_ARG: return "invalid argument";
        case MHCPB_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (T >= 1, K a positive multiple of 8, within limits)";
        case MHCPB_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case MHCPB_ERR_ALIASING: return "operands overlap";
        case MHCPB_ERR_WRONG_DEVICE: return "pointer not in device memory of the plan's device";
        case MHCPB_ERR_TF32_NOT_ALLOWED: return "MHCPB_ALLOW_TF32 is required";
        case MHCPB_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MHCPB_ERR_CUDA: return "CUDA error";
        case MHCPB_ERR_DEVICE_TIMEOUT: return "a wait inside the kernel timed out";
        case MHCPB_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3";
        case MHCPB_ERR_SCRATCH_TOO_SMALL:
            return "shape needs more dW-partial scratch than the built-in 16 MiB buffer";
    }
    return "unknown status";
}

const char* mhcpb_last_cuda_error(void) { return g_cuda_err; }

mhcpb_status_t mhcpb_plan_create(mhcpb_plan_t* out, int64_t T, int64_t K, int device,
                                 uint32_t flags) {
    if (out == nullptr) return MHCPB_ERR_INVALID_ARG;
    if ((flags & MHCPB_ALLOW_TF32) == 0) return MHCPB_ERR_TF32_NOT_ALLOWED;
    if ((flags & ~(uint32_t)(MHCPB_ALLOW_TF32 | MHCPB_HAS_ADDEND | MHCPB_FMA_KERNEL |
                            MHCPB_COMPENSATED_DW | MHCPB_ACCUMULATE_DW |
                            MHCPB_TEST_INJECT_STALL)) != 0)
        return MHCPB_ERR_INVALID_ARG;
    if (T < 0 || T > MHCPB_MAX_T || K < 8 || K > MHCPB_MAX_K || (K % 8) != 0)
        return MHCPB_ERR_UNSUPPORTED_SHAPE;
    if (device < 0) return MHCPB_ERR_INVALID_ARG;

    int ndev = 0;
    cudaError_t e = cudaGetDeviceCount(&ndev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
    if (device >= ndev) return MHCPB_ERR_INVALID_ARG;
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) return MHCPB_ERR_UNSUPPORTED_DEVICE;

    DeviceGuard g(device);
    if (!g.ok) return cuda_fail(cudaErrorInvalidDevice, "cudaSetDevice");

    const bool fma_kernel = (flags & MHCPB_FMA_KERNEL) != 0;
    const bool add = (flags & MHCPB_HAS_ADDEND) != 0;
    if (fma_kernel) {
        if ((e = fma::setup()) != cudaSuccess) return cuda_fail(e, "setup (FMA kernel)");
    } else {
        if (!get_encode()) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled entry point");
    }

    mhcpb_plan_s* p = new mhcpb_plan_s();
    p->T = T;
    p->K = K;
    p->device = device;
    p->flags = flags;
    p->chunk = partial_tokens(T);
    p->S = (int)((T + p->chunk - 1) / p->chunk);
    p->ws_bytes = (size_t)p->S * kNProj * (size_t)K * sizeof(float);
    if (fma_kernel) {
        p->n_strips = (int)((K + fma::kStrip - 1) / fma::kStrip);
        p->grid = p->n_strips * p->S;
        p->smem = fma::smem_bytes();
    } else {
        p->n_strips = (int)((K + tc::kStrip - 1) / tc::kStrip);
        const int64_t items = (int64_t)p->n_strips * p->S;
        p->half_units = tc::use_half_units(items, sms) ? 1 : 0;
        p->grid = tc::grid_size(items, sms);
        p->max_grid = p->grid;
        if ((e = tc::setup(add)) != cudaSuccess) {
            delete p;
            return cuda_fail(e, "setup (tensor-core kernel)");
        }
        p->smem = tc::smem_bytes(add);
    }
    p->fwd_grid = p->fwd_max_grid = fwd::grid_size(T, K, sms);
    if ((e = fwd::setup()) != cudaSuccess) {
        delete p;
        return cuda_fail(e, "setup (forward kernel)");
    }
    if ((e = cudaMalloc(&p->d_status, sizeof(uint32_t))) != cudaSuccess) {
        delete p;
        return cuda_fail(e, "cudaMalloc (status word)");
    }
    if ((e = cudaMemset(p->d_status, 0, sizeof(uint32_t))) != cudaSuccess) {
        cudaFree(p->d_status);
        delete p;
        return cuda_fail(e, "cudaMemset (status word)");
    }
    if (!fma_kernel && T > 0) {
        // The tensor maps depend on the execute's pointers, but their shapes
        // can be checked now: encode them over a real device address (the
        // status word; encoding records the address and reads nothing).
        // T = 0 launches no streaming kernel and needs no map.
        CUtensorMap m[6];
        const void* a = p->d_status;
        if (const char* bad = encode_maps(m, T, K, a, a, a, a, a, a)) {
            cudaFree(p->d_status);
            delete p;
            return cuda_fail(cudaErrorInvalidValue, bad);
        }
#ifdef MHCPB_TRACE
        p->trace_bytes = (size_t)p->grid * kTraceEvents * kTraceTiles * sizeof(uint64_t);
        if (cudaMalloc(&p->d_trace, p->trace_bytes) != cudaSuccess ||
            cudaMemset(p->d_trace, 0, p->trace_bytes) != cudaSuccess) {
            delete p;
            return cuda_fail(cudaErrorMemoryAllocation, "trace buffer");
        }
#endif
    }
    *out = p;
    return MHCPB_OK;
}

mhcpb_status_t mhcpb_workspace_bytes(mhcpb_plan_t plan, size_t* bytes) {
    if (plan == nullptr || bytes == nullptr) return MHCPB_ERR_INVALID_ARG;
    *bytes = plan->ws_bytes;
    return MHCPB_OK;
}

mhcpb_status_t mhcpb_plan_query(mhcpb_plan_t plan, int which, int64_t* value) {
    if (plan == nullptr || value == nullptr) return MHCPB_ERR_INVALID_ARG;
    switch (which) {
        case 0: *value = plan->T; break;
        case 1: *value = plan->K; break;
        case 2: *value = plan->S; break;
        case 3: *value = plan->grid; break;
        case 4: *value = plan->flags; break;
        case 5: *value = (int64_t)plan->smem; break;
        case 6: *value = (plan->flags & MHCPB_FMA_KERNEL) ? plan->chunk : tc::kTokenTile; break;
        case 7: *value = (plan->flags & MHCPB_FMA_KERNEL) ? fma::kStrip : tc::kStrip; break;
        case 8: *value = plan->chunk; break;
        default: return MHCPB_ERR_INVALID_ARG;
    }
    return MHCPB_OK;
}

// What an execute enqueues: kernel 1 (dX and the dW partials), kernel 2 (the
// fixed-order reduction of the partials into dW), or both.
enum : int { kRunStream = 1, kRunReduce = 2, kRunBoth = 3 };

static mhcpb_status_t execute_impl(mhcpb_plan_t plan, int what, const void* x, const float* w,
                                   const float* grad_proj, const float* grad_r, const float* r,
                                   void* dx, float* dw, void* workspace, size_t workspace_bytes,
                                   const void* grad_x_addend, void* stream, void* ev0, void* ev1,
                                   void* ev2) {
    if (plan == nullptr) return MHCPB_ERR_INVALID_ARG;
    const bool run1 = (what & kRunStream) != 0, run2 = (what & kRunReduce) != 0;
    const bool add = (plan->flags & MHCPB_HAS_ADDEND) != 0;
    const int64_t T = plan->T, K = plan->K;
    // operands of the kernels that run: 0..5 kernel 1's inputs and dX, 6 dW,
    // 7 the workspace, 8 the addend.  An operand with no elements (at T = 0:
    // all but W and dW) needs no storage and its pointer is not checked.
    const void* all[9] = {x, w, grad_proj, grad_r, r, dx, dw, workspace, grad_x_addend};
    const size_t all_sizes[9] = {(size_t)(T * K * 2), (size_t)(kNProj * K * 4),
                                 (size_t)(T * kGradProjCols * 4), (size_t)(T * 4), (size_t)(T * 4),
                                 (size_t)(T * K * 2), (size_t)(kNProj * K * 4), plan->ws_bytes,
                                 (size_t)(T * K * 2)};
    const void* ptrs[9];
    size_t sizes[9];
    int n = 0;
    for (int i = 0; i < 9; ++i) {
        const bool used = (i <= 5) ? run1 : (i == 6) ? run2 : (i == 7) ? true : (run1 && add);
        if (!used || all_sizes[i] == 0) continue;
        if (all[i] == nullptr) return MHCPB_ERR_INVALID_ARG;
        ptrs[n] = all[i];
        sizes[n++] = all_sizes[i];
    }
    if (run1 && T > 0 && add != (grad_x_addend != nullptr)) return MHCPB_ERR_INVALID_ARG;
    if (workspace_bytes < plan->ws_bytes) return MHCPB_ERR_WORKSPACE_TOO_SMALL;
    for (int i = 0; i < n; ++i)
        if ((reinterpret_cast<uintptr_t>(ptrs[i]) & 15u) != 0) return MHCPB_ERR_MISALIGNED;
    Range rg[9];
    for (int i = 0; i < n; ++i) {
        rg[i].lo = reinterpret_cast<uintptr_t>(ptrs[i]);
        rg[i].hi = rg[i].lo + sizes[i];
    }
    for (int i = 0; i < n; ++i)
        for (int j = i + 1; j < n; ++j)
            if (overlap(rg[i], rg[j])) return MHCPB_ERR_ALIASING;
    for (int i = 0; i < n; ++i) {
        mhcpb_status_t s = check_device_ptr(ptrs[i], plan->device);
        if (s != MHCPB_OK) return s;
    }

    DeviceGuard g(plan->device);
    if (!g.ok) return cuda_fail(cudaErrorInvalidDevice, "cudaSetDevice");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    cudaError_t e;
    if (ev0 && (e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev0), st)) != cudaSuccess)
        return cuda_fail(e, "cudaEventRecord");
    if (run1 && T > 0) {   // T = 0: no dX, no partials
        MainParams p{};
        p.T = (int32_t)T;
        p.K = (int32_t)K;
        p.S = plan->S;
        p.chunk = plan->chunk;
        p.n_strips = plan->n_strips;
        p.half_units = plan->half_units;
        p.x = static_cast<const uint16_t*>(x);
        p.w = w;
        p.grad_proj = grad_proj;
        p.grad_r = grad_r;
        p.r = r;
        p.dx = static_cast<uint16_t*>(dx);
        p.addend = static_cast<const uint16_t*>(grad_x_addend);
        p.partial = static_cast<float*>(workspace);
        p.status = plan->d_status;
        p.timeout_ns = plan->timeout_ns;
        p.test_flags = (plan->flags & MHCPB_TEST_INJECT_STALL) ? kTestInjectStall : 0u;
        p.trace = plan->d_trace;
        if (plan->flags & MHCPB_FMA_KERNEL) {
            e = fma::launch(p, st);
            if (e != cudaSuccess) return cuda_fail(e, "launch (FMA kernel)");
        } else {
            CUtensorMap m[6];
            if (const char* bad = encode_maps(m, T, K, x, dx, add ? grad_x_addend : x, grad_proj,
                                              grad_r, r))
                return cuda_fail(cudaErrorInvalidValue, bad);
            e = tc::launch(p, m[0], m[1], m[2], m[3], m[4], m[5], plan->grid, st);
            if (e != cudaSuccess) return cuda_fail(e, "launch (tensor-core kernel)");
        }
    }
    if (ev1 && (e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev1), st)) != cudaSuccess)
        return cuda_fail(e, "cudaEventRecord");
    if (run2) {
        // partials written by this same call are dead after the sum (their L2
        // lines may be dropped); a stand-alone reduction leaves them intact.
        // At T = 0 there are none (S = 0): dW = 0, or dW + 0 when accumulating
        e = launch_reduce(static_cast<const float*>(workspace), dw, plan->S, (int64_t)kNProj * K,
                          (plan->flags & MHCPB_COMPENSATED_DW) != 0,
                          (plan->flags & MHCPB_ACCUMULATE_DW) != 0, run1, st);
        if (e != cudaSuccess) return cuda_fail(e, "launch (dW reduction)");
    }
    if (ev2 && (e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev2), st)) != cudaSuccess)
        return cuda_fail(e, "cudaEventRecord");
    return MHCPB_OK;
}

mhcpb_status_t mhcpb_execute(mhcpb_plan_t plan, const void* x, const float* w,
                             const float* grad_proj, const float* grad_r, const float* r, void* dx,
                             float* dw, void* workspace, size_t workspace_bytes,
                             const void* grad_x_addend, void* stream) {
    return execute_impl(plan, kRunBoth, x, w, grad_proj, grad_r, r, dx, dw, workspace,
                        workspace_bytes, grad_x_addend, stream, nullptr, nullptr, nullptr);
}

mhcpb_status_t mhcpb_execute_profiled(mhcpb_plan_t plan, const void* x, const float* w,
                                      const float* grad_proj, const float* grad_r, const float* r,
                                      void* dx, float* dw, void* workspace, size_t workspace_bytes,
                                      const void* grad_x_addend, void* stream, void* ev_before,
                                      void* ev_between, void* ev_after) {
    return execute_impl(plan, kRunBoth, x, w, grad_proj, grad_r, r, dx, dw, workspace,
                        workspace_bytes, grad_x_addend, stream, ev_before, ev_between, ev_after);
}

mhcpb_status_t mhcpb_execute_dx(mhcpb_plan_t plan, const void* x, const float* w,
                                const float* grad_proj, const float* grad_r, const float* r,
                                void* dx, void* workspace, size_t workspace_bytes,
                                const void* grad_x_addend, void* stream) {
    return execute_impl(plan, kRunStream, x, w, grad_proj, grad_r, r, dx, nullptr, workspace,
                        workspace_bytes, grad_x_addend, stream, nullptr, nullptr, nullptr);
}

mhcpb_status_t mhcpb_reduce_dw(mhcpb_plan_t plan, void* workspace, size_t workspace_bytes,
                               float* dw, void* stream) {
    return execute_impl(plan, kRunReduce, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dw,
                        workspace, workspace_bytes, nullptr, stream, nullptr, nullptr, nullptr);
}

mhcpb_status_t mhcpb_forward_workspace_bytes(mhcpb_plan_t plan, size_t* bytes) {
    if (plan == nullptr || bytes == nullptr) return MHCPB_ERR_INVALID_ARG;
    *bytes = fwd::workspace_bytes(plan->T, plan->K);
    return MHCPB_OK;
}

// The forward, and with `gates` (non-null) the gate step fused into its
// reduction.  Operands: 0 x, 1 w, 2 proj, 3 r, 4 workspace (16-byte aligned),
// 5 alpha, 6 bias, 7 h (4-byte aligned, the gate calls' rule).
struct FwdGates {
    const float* alpha;
    const float* bias;
    int n_iter;
    float* h;
};
static mhcpb_status_t forward_impl(mhcpb_plan_t plan, const void* x, const float* w, float eps,
                                   float* proj, float* r, void* workspace, size_t workspace_bytes,
                                   void* stream, void* ev0, void* ev1, void* ev2,
                                   const FwdGates* gates) {
    if (plan == nullptr) return MHCPB_ERR_INVALID_ARG;
    const int64_t T = plan->T, K = plan->K;
    const size_t ws = fwd::workspace_bytes(T, K);
    if (gates != nullptr && (gates->n_iter < 1 || gates->n_iter > MHCPB_GATE_MAX_ITER))
        return MHCPB_ERR_UNSUPPORTED_SHAPE;
    // an operand with no elements (at T = 0: all but W, alpha and bias) needs
    // no storage and its pointer is not checked
    const int n_all = gates != nullptr ? 8 : 5;
    const void* all[8] = {x, w, proj, r, workspace, gates ? gates->alpha : nullptr,
                          gates ? gates->bias : nullptr, gates ? gates->h : nullptr};
    const size_t all_sizes[8] = {(size_t)(T * K * 2), (size_t)(kNProj * K * 4),
                                 (size_t)(T * fwd::kProjCols * 4), (size_t)(T * 4), ws, 3 * 4, kNProj * 4,
                                 (size_t)(T * kNProj * 4)};
    const bool output[8] = {false, false, true, true, true, false, false, true};
    const void* ptrs[8];
    size_t sizes[8];
    uintptr_t align[8];
    bool is_out[8];
    int n = 0;
    for (int i = 0; i < n_all; ++i) {
        if (all_sizes[i] == 0) continue;
        if (all[i] == nullptr) return MHCPB_ERR_INVALID_ARG;
        ptrs[n] = all[i];
        align[n] = i < 5 ? 15u : 3u;
        is_out[n] = output[i];
        sizes[n++] = all_sizes[i];
    }
    if (!(eps >= 0.f) || !(eps < INFINITY)) return MHCPB_ERR_INVALID_ARG;
    if (workspace_bytes < ws) return MHCPB_ERR_WORKSPACE_TOO_SMALL;
    for (int i = 0; i < n; ++i)
        if ((reinterpret_cast<uintptr_t>(ptrs[i]) & align[i]) != 0) return MHCPB_ERR_MISALIGNED;
    Range rg[8];
    for (int i = 0; i < n; ++i) {
        rg[i].lo = reinterpret_cast<uintptr_t>(ptrs[i]);
        rg[i].hi = rg[i].lo + sizes[i];
    }
    // outputs overlap nothing; of the inputs, X and W may not overlap either
    // (the gates' alpha and bias, read-only, may)
    for (int i = 0; i < n; ++i)
        for (int j = i + 1; j < n; ++j)
            if ((is_out[i] || is_out[j] || (ptrs[i] == x && ptrs[j] == w)) && overlap(rg[i], rg[j]))
                return MHCPB_ERR_ALIASING;
    for (int i = 0; i < n; ++i) {
        mhcpb_status_t s = check_device_ptr(ptrs[i], plan->device);
        if (s != MHCPB_OK) return s;
    }
    if (T == 0) return MHCPB_OK;   // no tokens: nothing to write
    if (!get_encode()) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled entry point");
    DeviceGuard g(plan->device);
    if (!g.ok) return cuda_fail(cudaErrorInvalidDevice, "cudaSetDevice");
    CUtensorMap xm, wm;
    if (!encode_bf16_map(&xm, x, T, K, fwd::kTokenTile))
        return cuda_fail(cudaErrorInvalidValue, "tensor map of x");
    if (!encode_f32_map(&wm, w, kNProj, (int)K, fwd::kBox, kNProj))
        return cuda_fail(cudaErrorInvalidValue, "tensor map of w");
    fwd::FwdParams p{};
    p.T = (int32_t)T;
    p.K = (int32_t)K;
    p.n_tt = (int32_t)((T + fwd::kTokenTile - 1) / fwd::kTokenTile);
    p.n_fc = (int32_t)fwd::n_chunks(K);
    p.t_pad = (int32_t)fwd::t_pad(T);
    p.w = w;
    p.partial = static_cast<float*>(workspace);
    p.proj = proj;
    p.r = r;
    p.eps = eps;
    p.status = plan->d_status;
    p.timeout_ns = plan->timeout_ns;
    p.trace = plan->d_trace;
    fwd::GateArgs ga{};
    if (gates != nullptr) ga = fwd::GateArgs{gates->alpha, gates->bias, gates->n_iter, gates->h};
    cudaError_t e = fwd::launch(p, xm, wm, plan->fwd_grid, reinterpret_cast<cudaStream_t>(stream),
                                reinterpret_cast<cudaEvent_t>(ev0), reinterpret_cast<cudaEvent_t>(ev1),
                                reinterpret_cast<cudaEvent_t>(ev2), gates != nullptr ? &ga : nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "launch (forward kernels)");
    return MHCPB_OK;
}

mhcpb_status_t mhcpb_forward(mhcpb_plan_t plan, const void* x, const float* w, float eps,
                             float* proj, float* r, void* workspace, size_t workspace_bytes,
                             void* stream) {
    return forward_impl(plan, x, w, eps, proj, r, workspace, workspace_bytes, stream, nullptr,
                        nullptr, nullptr, nullptr);
}

mhcpb_status_t mhcpb_forward_profiled(mhcpb_plan_t plan, const void* x, const float* w, float eps,
                                      float* proj, float* r, void* workspace,
                                      size_t workspace_bytes, void* stream, void* ev_before,
                                      void* ev_between, void* ev_after) {
    return forward_impl(plan, x, w, eps, proj, r, workspace, workspace_bytes, stream, ev_before,
                        ev_between, ev_after, nullptr);
}

mhcpb_status_t mhcpb_forward_gates(mhcpb_plan_t plan, const void* x, const float* w, float eps,
                                   const float* alpha, const float* bias, int n_iter, float* proj,
                                   float* r, float* h, void* workspace, size_t workspace_bytes,
                                   void* stream) {
    const FwdGates gates{alpha, bias, n_iter, h};
    return forward_impl(plan, x, w, eps, proj, r, workspace, workspace_bytes, stream, nullptr,
                        nullptr, nullptr, &gates);
}

// Shared checks of the two gate calls: shape, pointers (device, alignment,
// overlap of every output with every other operand), per-device set-up.
static mhcpb_status_t gate_checks(int64_t T, int n_iter, const void* const* in, const size_t* in_sz,
                                  int n_in, void* const* out, const size_t* out_sz, int n_out) {
    if (T < 0 || T > MHCPB_MAX_T || n_iter < 1 || n_iter > MHCPB_GATE_MAX_ITER)
        return MHCPB_ERR_UNSUPPORTED_SHAPE;
    // an operand with no elements (at T = 0: all but alpha and bias) needs no
    // storage and its pointer is not checked; its range is empty below
    for (int i = 0; i < n_in; ++i)
        if (in_sz[i] > 0 && in[i] == nullptr) return MHCPB_ERR_INVALID_ARG;
    for (int i = 0; i < n_out; ++i)
        if (out_sz[i] > 0 && out[i] == nullptr) return MHCPB_ERR_INVALID_ARG;
    for (int i = 0; i < n_in; ++i)
        if (in_sz[i] > 0 && (reinterpret_cast<uintptr_t>(in[i]) & 3u) != 0) return MHCPB_ERR_MISALIGNED;
    for (int i = 0; i < n_out; ++i)
        if (out_sz[i] > 0 && (reinterpret_cast<uintptr_t>(out[i]) & 3u) != 0) return MHCPB_ERR_MISALIGNED;
    for (int i = 0; i < n_out; ++i) {
        const Range o{reinterpret_cast<uintptr_t>(out[i]), reinterpret_cast<uintptr_t>(out[i]) + out_sz[i]};
        for (int j = 0; j < n_in; ++j)
            if (overlap(o, Range{reinterpret_cast<uintptr_t>(in[j]), reinterpret_cast<uintptr_t>(in[j]) + in_sz[j]}))
                return MHCPB_ERR_ALIASING;
        for (int j = i + 1; j < n_out; ++j)
            if (overlap(o, Range{reinterpret_cast<uintptr_t>(out[j]), reinterpret_cast<uintptr_t>(out[j]) + out_sz[j]}))
                return MHCPB_ERR_ALIASING;
    }
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    for (int i = 0; i < n_in; ++i) {
        if (in_sz[i] == 0) continue;
        mhcpb_status_t s = check_device_ptr(in[i], device);
        if (s != MHCPB_OK) return s;
    }
    for (int i = 0; i < n_out; ++i) {
        if (out_sz[i] == 0) continue;
        mhcpb_status_t s = check_device_ptr(out[i], device);
        if (s != MHCPB_OK) return s;
    }
    constexpr int kMaxDevices = 64;
    static std::once_flag once[kMaxDevices];
    static mhcpb_status_t setup_status[kMaxDevices];
    if (device < 0 || device >= kMaxDevices) return MHCPB_ERR_INVALID_ARG;
    std::call_once(once[device], [device] {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess) {
            setup_status[device] = cuda_fail(cudaGetLastError(), "cudaDeviceGetAttribute");
            return;
        }
        if (major != 10 || minor != 3) {
            setup_status[device] = MHCPB_ERR_UNSUPPORTED_DEVICE;
            return;
        }
        const cudaError_t se = gates::setup();
        setup_status[device] = se == cudaSuccess ? MHCPB_OK : cuda_fail(se, "setup (gate kernels)");
    });
    return setup_status[device];
}

mhcpb_status_t mhcpb_gate_forward(int64_t T, int n_iter, const float* proj, const float* r,
                                  const float* alpha, const float* bias, float* h, void* stream) {
    if (T < 0 || T > MHCPB_MAX_T) return MHCPB_ERR_UNSUPPORTED_SHAPE;
    const void* in[4] = {proj, r, alpha, bias};
    const size_t in_sz[4] = {(size_t)T * 32 * 4, (size_t)T * 4, 3 * 4, kNProj * 4};
    void* out[1] = {h};
    const size_t out_sz[1] = {(size_t)T * kNProj * 4};
    mhcpb_status_t s = gate_checks(T, n_iter, in, in_sz, 4, out, out_sz, 1);
    if (s != MHCPB_OK || T == 0) return s;   // no tokens: nothing to write
    cudaError_t e = gates::launch_forward(T, n_iter, proj, r, alpha, bias, h,
                                          reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MHCPB_OK : cuda_fail(e, "launch (gate forward)");
}

mhcpb_status_t mhcpb_gate_backward(int64_t T, int n_iter, const float* proj, const float* r,
                                   const float* alpha, const float* bias, const float* grad_h,
                                   float* grad_proj, float* grad_r, float* dlogits, void* stream) {
    if (T < 0 || T > MHCPB_MAX_T) return MHCPB_ERR_UNSUPPORTED_SHAPE;
    const void* in[5] = {proj, r, alpha, bias, grad_h};
    const size_t in_sz[5] = {(size_t)T * 32 * 4, (size_t)T * 4, 3 * 4, kNProj * 4, (size_t)T * kNProj * 4};
    void* out[3] = {grad_proj, grad_r, dlogits};
    const size_t out_sz[3] = {(size_t)T * 32 * 4, (size_t)T * 4, (size_t)T * kNProj * 4};
    mhcpb_status_t s = gate_checks(T, n_iter, in, in_sz, 5, out, out_sz, dlogits ? 3 : 2);
    if (s != MHCPB_OK || T == 0) return s;   // no tokens: nothing to write
    cudaError_t e = gates::launch_backward(T, n_iter, proj, r, alpha, bias, grad_h, grad_proj,
                                           grad_r, dlogits, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MHCPB_OK : cuda_fail(e, "launch (gate backward)");
}

mhcpb_status_t mhcpb_get_device_status(mhcpb_plan_t plan, mhcpb_status_t* status, int clear) {
    if (plan == nullptr || status == nullptr) return MHCPB_ERR_INVALID_ARG;
    DeviceGuard g(plan->device);
    if (!g.ok) return cuda_fail(cudaErrorInvalidDevice, "cudaSetDevice");
    uint32_t v = 0;
    cudaError_t e = cudaMemcpy(&v, plan->d_status, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy (status word)");
    if (clear && v != 0) {
        e = cudaMemset(plan->d_status, 0, sizeof(uint32_t));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset (status word)");
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    }
    *status = static_cast<mhcpb_status_t>(v);
    return MHCPB_OK;
}

mhcpb_status_t mhcpb_plan_set_max_ctas(mhcpb_plan_t plan, int max_ctas) {
    if (plan == nullptr || max_ctas < 0) return MHCPB_ERR_INVALID_ARG;
    plan->fwd_grid = (max_ctas == 0 || max_ctas > plan->fwd_max_grid) ? plan->fwd_max_grid : max_ctas;
    if (plan->flags & MHCPB_FMA_KERNEL) return MHCPB_OK;
    plan->grid = (max_ctas == 0 || max_ctas > plan->max_grid) ? plan->max_grid : max_ctas;
    return MHCPB_OK;
}

mhcpb_status_t mhcpb_plan_set_wait_limit(mhcpb_plan_t plan, uint64_t nanoseconds) {
    if (plan == nullptr) return MHCPB_ERR_INVALID_ARG;
    if (nanoseconds < 1000000ull || nanoseconds > 60000000000ull) return MHCPB_ERR_INVALID_ARG;
    plan->timeout_ns = nanoseconds;
    return MHCPB_OK;
}

mhcpb_status_t mhcpb_destroy(mhcpb_plan_t plan) {
    if (plan == nullptr) return MHCPB_OK;
    if (plan->d_status) {
        DeviceGuard g(plan->device);
        cudaFree(plan->d_status);
        if (plan->d_trace) cudaFree(plan->d_trace);
    }
    delete plan;
    return MHCPB_OK;
}

mhcpb_status_t mhcpb_debug_checked_sites(uint32_t* sites, int* checked) {
    if (sites == nullptr || checked == nullptr) return MHCPB_ERR_INVALID_ARG;
    *checked = check::kEnabled ? 1 : 0;
    cudaError_t e;
    if ((e = tc::checked_site(&sites[0])) != cudaSuccess || (e = fma::checked_site(&sites[1])) != cudaSuccess ||
        (e = reduce_checked_site(&sites[2])) != cudaSuccess || (e = fwd::checked_site(&sites[3])) != cudaSuccess ||
        (e = gates::checked_site(&sites[4])) != cudaSuccess)
        return cuda_fail(e, "checked-build site words");
    return MHCPB_OK;
}

#ifdef MHCPB_TRACE
// Instrumented builds only: copies the last execute's timeline stamps.
mhcpb_status_t mhcpb_debug_trace(mhcpb_plan_t plan, void* host, size_t bytes) {
    if (plan == nullptr || host == nullptr || bytes < plan->trace_bytes) return MHCPB_ERR_INVALID_ARG;
    DeviceGuard g(plan->device);
    cudaError_t e = cudaMemcpy(host, plan->d_trace, plan->trace_bytes, cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? MHCPB_OK : cuda_fail(e, "cudaMemcpy (trace)");
}
#endif

}  // extern "C"
