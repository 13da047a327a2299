// Second kernel of the backward: the fixed-order reduction of the per-chunk
// dW partials (cuDNN frontend page "DSv4.1 mHC projection/RMS backward",
// intro and "Source attribution": partial weight gradients written by
// independent blocks, then reduced in a second kernel, in a fixed order and
// without atomics).
//
//   dW[j,k] = (((partial[0][j][k] + partial[1][j][k]) + partial[2][j][k]) + ...)
//
// One thread owns four consecutive dW elements; the sum runs over s in
// ascending order, so dW depends only on (T, K) and the inputs.
//
// With the plan flag MHCPB_ACCUMULATE_DW the result is added to the dW the
// caller passes (dW_out = dW_in + result, one FP32 addition) instead of
// overwriting it.
//
// Compensated variant (plan flag MHCPB_COMPENSATED_DW): the same order, with
// Knuth's TwoSum at every addition, s + p = s' + e exactly (six FP32
// additions, no branch), the errors e summed beside s and added once at the
// end -- Ogita, Rump and Oishi's Sum2, which is as accurate as the sum in
// twice the working precision rounded once.  FlashInfer's page on
// cake_rmsnorm_det_train_backward describes the same idea for its small-T dw
// column sums.  Launched as a
// programmatic dependent of the streaming kernel: it may be scheduled while
// that kernel drains and waits for its completion before reading.  When the
// same call wrote the partials (nothing reads them again), they are dead once
// read: with a 128-byte-aligned workspace their L2 lines are dropped without
// being written back to HBM.  A stand-alone reduction (the split call) keeps
// them, so it can be repeated on the same workspace.
#include "mhcpb_check.cuh"
#include "mhcpb_internal.h"
#include "ptx.cuh"

namespace mhcpb {

namespace {

constexpr int kReduceThreads = 256;
constexpr int kGroup = 8;   // partials loaded before they are summed

// s + p = s' + e exactly (Knuth's TwoSum; no ordering of |s|, |p| needed).
// Plain IEEE additions: nvcc never reassociates or contracts them.  A
// non-finite sum keeps e = 0, so Inf stays Inf (not Inf - Inf = NaN) and NaN
// stays NaN, as in the plain sum.
__device__ __forceinline__ void two_sum(float& s, float& e_acc, float p) {
    const float t = s + p;
    const float pp = t - s;
    const float e = (s - (t - pp)) + (p - pp);
    s = t;
    e_acc += isfinite(t) ? e : 0.f;
}

template <bool COMP, bool ACC>
__global__ void __launch_bounds__(kReduceThreads) reduce_dw_kernel(const float4* __restrict__ part,
                                                                   float4* __restrict__ dw, int S,
                                                                   int64_t n4, int discard) {
    // the next execute's streaming kernel may be scheduled now; it waits for
    // this grid's completion before it touches global memory
    ptx::grid_launch_dependents();
    ptx::grid_dependency_wait();
    const int64_t i = (int64_t)blockIdx.x * kReduceThreads + threadIdx.x;
    const bool valid = i < n4;   // n4 % 8 == 0: a 128-byte line is all valid or all not
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 c = make_float4(0.f, 0.f, 0.f, 0.f);   // compensation (COMP only)
    for (int s0 = 0; valid && s0 < S; s0 += kGroup) {
        float4 b[kGroup];
#pragma unroll
        for (int g = 0; g < kGroup; ++g)
            if (s0 + g < S && check::in(part + (int64_t)(s0 + g) * n4 + i, 16, part, (size_t)S * n4 * 16, 0))
                b[g] = part[(int64_t)(s0 + g) * n4 + i];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
            if (s0 + g < S) {
                if (s0 + g == 0) {
                    a = b[g];
                } else if (COMP) {
                    two_sum(a.x, c.x, b[g].x);
                    two_sum(a.y, c.y, b[g].y);
                    two_sum(a.z, c.z, b[g].z);
                    two_sum(a.w, c.w, b[g].w);
                } else {
                    a.x += b[g].x; a.y += b[g].y; a.z += b[g].z; a.w += b[g].w;
                }
            }
        }
    }
    if (COMP) {
        a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
    }
    if (valid && check::in(dw + i, 16, dw, (size_t)n4 * 16, 1)) {
        if (ACC) {   // accumulate into the caller's dW: one more FP32 rounding
            const float4 o = dw[i];
            a.x = o.x + a.x; a.y = o.y + a.y; a.z = o.z + a.z; a.w = o.w + a.w;
        }
        dw[i] = a;
    }
    // Every lane of the warp has consumed its loads once the warp has converged
    // here; then the lanes share out the discards of the lines the warp read:
    // 4 per slice (32 float4 = 512 bytes) times S slices.  A line is dropped
    // only if all of it was valid.
    __syncwarp();
    if (discard) {
        const int lane = threadIdx.x & 31;
        const int64_t w0 = i - lane;   // the warp's first float4
        for (int q = lane; q < 4 * S; q += 32) {
            const int64_t f4 = w0 + 8 * (q & 3);
            if (f4 < n4 && check::in(part + (int64_t)(q >> 2) * n4 + f4, 128, part, (size_t)S * n4 * 16, 2))
                ptx::discard_l2_line(part + (int64_t)(q >> 2) * n4 + f4);
        }
    }
}

}  // namespace

cudaError_t reduce_checked_site(uint32_t* site) { return check::read_and_clear(site); }

cudaError_t launch_reduce(const float* partial, float* dw, int S, int64_t n, bool compensated,
                          bool accumulate, bool discard_allowed, cudaStream_t stream) {
    const int64_t n4 = n / 4;
    // discard needs 128-byte-aligned lines: every s-slice starts at a multiple
    // of 96 K bytes (K % 8 == 0, so a multiple of 768) from the base
    const int discard =
        discard_allowed && (reinterpret_cast<uintptr_t>(partial) & 127u) == 0 ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n4 + kReduceThreads - 1) / kReduceThreads));
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float4* part4 = reinterpret_cast<const float4*>(partial);
    float4* dw4 = reinterpret_cast<float4*>(dw);
    if (compensated)
        return accumulate ? cudaLaunchKernelEx(&cfg, reduce_dw_kernel<true, true>, part4, dw4, S, n4, discard)
                          : cudaLaunchKernelEx(&cfg, reduce_dw_kernel<true, false>, part4, dw4, S, n4, discard);
    return accumulate ? cudaLaunchKernelEx(&cfg, reduce_dw_kernel<false, true>, part4, dw4, S, n4, discard)
                      : cudaLaunchKernelEx(&cfg, reduce_dw_kernel<false, false>, part4, dw4, S, n4, discard);
}

}  // namespace mhcpb
