// FP32-FMA (CUDA-core) streaming kernel for the mHC projection/RMS backward.
//
// Computes, per (64-column strip, token chunk) block (cuDNN frontend page
// "DSv4.1 mHC projection/RMS backward", intro):
//   dX[t,k]            = sum_j P[t,j] W[j,k] + c[t] X[t,k],  c = grad_r / (r K)
//   partial[s][j][k]   = sum_{t in chunk s} P[t,j] X[t,k]
// with P and W rounded to TF32 (round to nearest, ties away) and every sum in
// FP32.  TF32 x BF16 products are exact in FP32, so each FMA rounds only the
// running sum.  Rows are taken in a fixed order inside the block and the eight
// row-groups' dW sums are combined in ascending order, so the partials do not
// depend on scheduling.  This kernel is the measured control for the
// tensor-core kernel: the same arithmetic on the CUDA cores.
#include <cuda_bf16.h>

#include "mhcpb_check.cuh"
#include "mhcpb_internal.h"
#include "ptx.cuh"

namespace mhcpb {
namespace fma {

namespace {

constexpr int kChunk = kMaxTokensPerPartial;   // shared memory is sized for the largest chunk
constexpr int kGroups = kThreads / 32;   // row groups; a warp spans 64 columns

__device__ __forceinline__ float tf32_rna(float v) {
    uint32_t u;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(v));
    return __uint_as_float(u & 0xFFFFE000u);
}

// a read-only global load, bounds-checked in checked builds (0 when outside)
template <class V>
__device__ __forceinline__ V ld_checked(const V* ptr, const void* base, size_t bytes, uint32_t site) {
    return check::in(ptr, sizeof(V), base, bytes, site) ? __ldg(ptr) : V(0);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads) main_fma_kernel(const MainParams p) {
    extern __shared__ float smem[];
    float* sP = smem;                      // [kChunk][24] TF32 P of this chunk
    float* sC = smem + kChunk * kNProj;    // [kChunk] RMS coefficients

    ptx::grid_launch_dependents();

    const int strip = blockIdx.x;
    const int chunk = blockIdx.y;
    const int t0 = chunk * p.chunk;
    const int nt = min(p.T - t0, p.chunk);
    const int K = p.K;
    // buffer extents (bytes) for the checks of a checked build
    const size_t tk_bytes = (size_t)p.T * K * 2, w_bytes = (size_t)kNProj * K * 4,
                 gp_bytes = (size_t)p.T * kGradProjCols * 4, t_bytes = (size_t)p.T * 4,
                 part_bytes = (size_t)p.S * kNProj * K * 4;

    for (int i = threadIdx.x; i < nt * kNProj; i += kThreads) {
        const int tt = i / kNProj, j = i - tt * kNProj;
        sP[i] = tf32_rna(ld_checked(p.grad_proj + (size_t)(t0 + tt) * kGradProjCols + j, p.grad_proj,
                                    gp_bytes, 0));
    }
    for (int i = threadIdx.x; i < nt; i += kThreads)
        sC[i] = ld_checked(p.grad_r + t0 + i, p.grad_r, t_bytes, 1) /
                (ld_checked(p.r + t0 + i, p.r, t_bytes, 2) * static_cast<float>(K));
    __syncthreads();

    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int col = strip * kStrip + 2 * tx;   // K % 8 == 0: col < K implies col+1 < K
    const bool valid = col < K;

    float w0[kNProj], w1[kNProj], a0[kNProj], a1[kNProj];
#pragma unroll
    for (int j = 0; j < kNProj; ++j) {
        w0[j] = valid ? tf32_rna(ld_checked(p.w + (size_t)j * K + col, p.w, w_bytes, 3)) : 0.f;
        w1[j] = valid ? tf32_rna(ld_checked(p.w + (size_t)j * K + col + 1, p.w, w_bytes, 3)) : 0.f;
        a0[j] = 0.f;
        a1[j] = 0.f;
    }

    if (valid) {
        for (int tt = ty; tt < nt; tt += kGroups) {
            const size_t off = (size_t)(t0 + tt) * K + col;
            const uint32_t xv = ld_checked(reinterpret_cast<const uint32_t*>(p.x + off), p.x, tk_bytes, 4);
            const float x0 = __uint_as_float(xv << 16);
            const float x1 = __uint_as_float(xv & 0xFFFF0000u);
            const float* pr = sP + tt * kNProj;
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int j = 0; j < kNProj; ++j) {
                const float pj = pr[j];
                d0 = fmaf(pj, w0[j], d0);
                d1 = fmaf(pj, w1[j], d1);
                a0[j] = fmaf(pj, x0, a0[j]);
                a1[j] = fmaf(pj, x1, a1[j]);
            }
            const float c = sC[tt];
            d0 = fmaf(c, x0, d0);
            d1 = fmaf(c, x1, d1);
            uint32_t out = pack_bf16x2(d0, d1);
            if (p.addend != nullptr) {
                // the value a separate BF16 add gives: bf16(fp32(bf16 core) + fp32(addend))
                const uint32_t av =
                    ld_checked(reinterpret_cast<const uint32_t*>(p.addend + off), p.addend, tk_bytes, 5);
                const float s0 = __uint_as_float(out << 16) + __uint_as_float(av << 16);
                const float s1 =
                    __uint_as_float(out & 0xFFFF0000u) + __uint_as_float(av & 0xFFFF0000u);
                out = pack_bf16x2(s0, s1);
            }
            if (check::in(p.dx + off, 4, p.dx, tk_bytes, 6)) *reinterpret_cast<uint32_t*>(p.dx + off) = out;
        }
    }
    __syncthreads();   // sP is reused below

    // Fixed-order combination of the row groups' dW sums: group 0 + 1 + ... + 7.
    float* sR = smem;  // [kGroups][24][kStrip]
#pragma unroll
    for (int j = 0; j < kNProj; ++j) {
        sR[(ty * kNProj + j) * kStrip + 2 * tx] = a0[j];
        sR[(ty * kNProj + j) * kStrip + 2 * tx + 1] = a1[j];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kNProj * kStrip; i += kThreads) {
        const int j = i / kStrip, cc = i - j * kStrip;
        float s = sR[j * kStrip + cc];
#pragma unroll
        for (int g = 1; g < kGroups; ++g) s += sR[(g * kNProj + j) * kStrip + cc];
        const int c2 = strip * kStrip + cc;
        float* dst = p.partial + ((size_t)chunk * kNProj + j) * K + c2;
        if (c2 < K && check::in(dst, 4, p.partial, part_bytes, 7)) *dst = s;
    }
}

}  // namespace

size_t smem_bytes() {
    // max(P + coefficients, the row-group reduction buffer)
    const size_t a = (size_t)kChunk * kNProj * 4 + (size_t)kChunk * 4;
    const size_t b = (size_t)kGroups * kNProj * kStrip * 4;
    return a > b ? a : b;
}

cudaError_t setup() {
    return cudaFuncSetAttribute(main_fma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes());
}

cudaError_t checked_site(uint32_t* site) { return check::read_and_clear(site); }

cudaError_t launch(const MainParams& p, cudaStream_t stream) {
    dim3 grid(p.n_strips, p.S);
    main_fma_kernel<<<grid, kThreads, smem_bytes(), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace fma
}  // namespace mhcpb
