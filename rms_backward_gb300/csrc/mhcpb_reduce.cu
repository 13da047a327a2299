// Second kernel of the backward: the fixed-order reduction of the per-chunk
// dW partials (cuDNN frontend page "DSv4.1 mHC projection/RMS backward",
// intro and "Source attribution": partial weight gradients written by
// independent blocks, then reduced in a second kernel, in a fixed order and
// without atomics).
//
//   dW[j,k] = (((partial[0][j][k] + partial[1][j][k]) + partial[2][j][k]) + ...)
//
// One thread owns four consecutive dW elements; the sum runs over s in
// ascending order, so dW depends only on (T, K) and the inputs.  Launched as a
// programmatic dependent of the streaming kernel: it may be scheduled while
// that kernel drains and waits for its completion before reading.
#include "mhcpb_internal.h"
#include "ptx.cuh"

namespace mhcpb {

namespace {

constexpr int kReduceThreads = 256;

__global__ void __launch_bounds__(kReduceThreads) reduce_dw_kernel(const float4* __restrict__ part,
                                                                   float4* __restrict__ dw, int S,
                                                                   int64_t n4) {
    ptx::grid_dependency_wait();
    const int64_t i = (int64_t)blockIdx.x * kReduceThreads + threadIdx.x;
    if (i >= n4) return;
    float4 a = part[i];
    int s = 1;
    // loads of a group are independent; the additions keep ascending s
    for (; s + 4 <= S; s += 4) {
        const float4 b0 = part[(int64_t)(s + 0) * n4 + i];
        const float4 b1 = part[(int64_t)(s + 1) * n4 + i];
        const float4 b2 = part[(int64_t)(s + 2) * n4 + i];
        const float4 b3 = part[(int64_t)(s + 3) * n4 + i];
        a.x += b0.x; a.y += b0.y; a.z += b0.z; a.w += b0.w;
        a.x += b1.x; a.y += b1.y; a.z += b1.z; a.w += b1.w;
        a.x += b2.x; a.y += b2.y; a.z += b2.z; a.w += b2.w;
        a.x += b3.x; a.y += b3.y; a.z += b3.z; a.w += b3.w;
    }
    for (; s < S; ++s) {
        const float4 b = part[(int64_t)s * n4 + i];
        a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    dw[i] = a;
}

}  // namespace

cudaError_t launch_reduce(const float* partial, float* dw, int S, int64_t n, cudaStream_t stream) {
    const int64_t n4 = n / 4;
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
    return cudaLaunchKernelEx(&cfg, reduce_dw_kernel, reinterpret_cast<const float4*>(partial),
                              reinterpret_cast<float4*>(dw), S, n4);
}

}  // namespace mhcpb
