// Gate/normalisation step of mHC around the projection/RMS stage, forward and
// backward (the backward produces the stage's grad_proj and grad_r).
//
// The cuDNN frontend page "DSv4.1 mHC projection/RMS backward" (intro) feeds
// the stage "the upstream projection and RMS gradients after the gate and
// normalization derivatives"; the prime-kernels PR #15 page ("mhc_projection")
// fuses "gate activations (sigmoid, Sinkhorn)" into the projection.  Neither
// prints the formulas; this file computes the reading stated in mhcpb.h
// (mhcpb_gate_forward): for n = 4 streams the 24 projection columns are the
// 4 pre, 4 post and 16 residual logits
//     l = a_g * proj / r + b,  H_pre = sigmoid(l), H_post = 2 sigmoid(l),
//     H_res = Sinkhorn(exp(l)) (row normalisation then column normalisation,
//     n_iter times)
// and the backward is its exact chain rule.
//
// GB300 layout: a half-warp per token, lane i*4+j owns residual entry (i, j)
// (and lane g < 8 also pre/post gate g), so every row sum is a 2-step and every
// column sum a 2-step shuffle inside the half-warp.  FP32 throughout.
//
// The per-token arithmetic (Sinkhorn iterations, direct with a log-domain
// fallback, and the gates) is in mhcg_math.cuh, shared with the forward's
// fused reduction.  The backward carries the gradient with respect to the logarithms: through
// a column step g <- g - M colsum(g), through a row step g <- g - R rowsum(g),
// starting from G_res * M and ending at dL/dl_res -- the chain rule of the
// normalisations written for log-values, with no division.  It keeps R and M
// (probabilities in [0, 1]) of every iteration in shared memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "mhcg_math.cuh"
#include "mhcpb.h"
#include "mhcpb_check.cuh"
#include "mhcpb_internal.h"

namespace mhcpb {
namespace gates {

namespace {

constexpr int kThreads = 256;            // 16 tokens per block
constexpr int kTokensPerBlock = kThreads / 16;
using gatemath::col_sum;
using gatemath::kFull;
using gatemath::row_sum;

struct Lane {
    int64_t t;       // token
    int l;           // lane within the half-warp: residual entry (l / 4, l % 4)
    bool valid;      // t < T (invalid lanes still take part in the shuffles)
};
__device__ __forceinline__ Lane lane_of(int64_t T) {
    Lane L;
    L.t = (int64_t)blockIdx.x * kTokensPerBlock + (threadIdx.x >> 4);
    L.l = threadIdx.x & 15;
    L.valid = L.t < T;
    return L;
}

__global__ void __launch_bounds__(kThreads) gate_forward_kernel(int64_t T, int n_iter,
                                                                 const float* __restrict__ proj,
                                                                 const float* __restrict__ r,
                                                                 const float* __restrict__ alpha,
                                                                 const float* __restrict__ bias,
                                                                 float* __restrict__ h) {
    const Lane L = lane_of(T);
    // extents (bytes) for the checks of a checked build
    const size_t t4 = (size_t)T * 4, proj_bytes = (size_t)T * 32 * 4, h_bytes = (size_t)T * kNProj * 4;
    const float rv = L.valid && check::in(r + L.t, 4, r, t4, 0) ? r[L.t] : 1.f;
    const float pres = L.valid && check::in(proj + L.t * 32 + 8 + L.l, 4, proj, proj_bytes, 1)
                           ? proj[L.t * 32 + 8 + L.l] : 0.f;
    const float M = gatemath::sinkhorn(gatemath::res_logit(pres, rv, alpha, bias, L.l), n_iter, nullptr,
                                       nullptr, 0);
    if (!L.valid) return;
    if (check::in(h + L.t * kNProj + 8 + L.l, 4, h, h_bytes, 3)) h[L.t * kNProj + 8 + L.l] = M;
    if (L.l < 8) {
        const float pg = check::in(proj + L.t * 32 + L.l, 4, proj, proj_bytes, 1) ? proj[L.t * 32 + L.l] : 0.f;
        const float g = gatemath::pre_post_gate(pg, rv, alpha, bias, L.l);
        if (check::in(h + L.t * kNProj + L.l, 4, h, h_bytes, 3)) h[L.t * kNProj + L.l] = g;
    }
}

__global__ void __launch_bounds__(kThreads) gate_backward_kernel(
    int64_t T, int n_iter, const float* __restrict__ proj, const float* __restrict__ r,
    const float* __restrict__ alpha, const float* __restrict__ bias,
    const float* __restrict__ grad_h, float* __restrict__ grad_proj, float* __restrict__ grad_r,
    float* __restrict__ dlogits) {
    // [n_iter][kThreads] R (after each row step), then [n_iter][kThreads] M
    // (after each column step)
    extern __shared__ float iters[];
    float* Rs = iters;
    float* Ms = iters + (size_t)n_iter * kThreads;
    const Lane L = lane_of(T);
    // extents (bytes) for the checks of a checked build
    const size_t t4 = (size_t)T * 4, proj_bytes = (size_t)T * 32 * 4, h_bytes = (size_t)T * kNProj * 4;
    const float rv = L.valid && check::in(r + L.t, 4, r, t4, 0) ? r[L.t] : 1.f;
    const float a_res = alpha[2];
    const float pres = L.valid && check::in(proj + L.t * 32 + 8 + L.l, 4, proj, proj_bytes, 1)
                           ? proj[L.t * 32 + 8 + L.l] : 0.f;
    const float M = gatemath::sinkhorn(gatemath::res_logit(pres, rv, alpha, bias, L.l), n_iter, Rs, Ms, kThreads);
    // reverse mode on log-values, last iteration first (g = dL/dlog M):
    //   column step log M = log R - LSE_col:  g <- g - M sum_col(g)
    //   row step    log R = log A - LSE_row:  g <- g - R sum_row(g)
    float g = (L.valid && check::in(grad_h + L.t * kNProj + 8 + L.l, 4, grad_h, h_bytes, 4)
                   ? grad_h[L.t * kNProj + 8 + L.l] : 0.f) * M;
    for (int k = n_iter - 1; k >= 0; --k) {
        g = g - Ms[k * kThreads + threadIdx.x] * col_sum(g);
        g = g - Rs[k * kThreads + threadIdx.x] * row_sum(g);
    }
    const float dl_res = g;   // dL / dlog A0 = dL / dlogit
    // pre / post gates: sigmoid'(l) = s (1 - s), times 2 for post
    float dl_g = 0.f, a_g = 0.f, pg = 0.f;
    if (L.l < 8 && L.valid) {
        a_g = L.l < 4 ? alpha[0] : alpha[1];
        pg = check::in(proj + L.t * 32 + L.l, 4, proj, proj_bytes, 1) ? proj[L.t * 32 + L.l] : 0.f;
        const float s = gatemath::sigmoid(a_g * pg / rv + bias[L.l]);
        const float gsc = L.l < 4 ? 1.f : 2.f;
        const float gh = check::in(grad_h + L.t * kNProj + L.l, 4, grad_h, h_bytes, 4) ? grad_h[L.t * kNProj + L.l] : 0.f;
        dl_g = gh * gsc * s * (1.f - s);
    }
    // grad_r = -sum_j dl_j a_j proj_j / r^2 over the token's 24 columns
    float term = dl_res * a_res * pres + dl_g * a_g * pg;
    term += __shfl_xor_sync(kFull, term, 1, 16);
    term += __shfl_xor_sync(kFull, term, 2, 16);
    term += __shfl_xor_sync(kFull, term, 4, 16);
    term += __shfl_xor_sync(kFull, term, 8, 16);
    if (!L.valid) return;
    float* gp = grad_proj + L.t * 32;
    if (check::in(gp + 8 + L.l, 4, grad_proj, proj_bytes, 5)) gp[8 + L.l] = dl_res * a_res / rv;
    if (L.l < 8) {
        if (check::in(gp + L.l, 4, grad_proj, proj_bytes, 5)) gp[L.l] = dl_g * a_g / rv;
    } else if (check::in(gp + 24 + (L.l - 8), 4, grad_proj, proj_bytes, 5)) {
        gp[24 + (L.l - 8)] = 0.f;   // the stored width is 32
    }
    if (L.l == 0 && check::in(grad_r + L.t, 4, grad_r, t4, 6)) grad_r[L.t] = -term / (rv * rv);
    if (dlogits != nullptr) {
        if (check::in(dlogits + L.t * kNProj + 8 + L.l, 4, dlogits, h_bytes, 7)) dlogits[L.t * kNProj + 8 + L.l] = dl_res;
        if (L.l < 8 && check::in(dlogits + L.t * kNProj + L.l, 4, dlogits, h_bytes, 7)) dlogits[L.t * kNProj + L.l] = dl_g;
    }
}

}  // namespace

cudaError_t checked_site(uint32_t* site) { return check::read_and_clear(site); }

size_t backward_smem_bytes(int n_iter) { return (size_t)(2 * n_iter) * kThreads * sizeof(float); }

cudaError_t setup() {
    return cudaFuncSetAttribute(gate_backward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)backward_smem_bytes(kMaxIter));
}

cudaError_t launch_forward(int64_t T, int n_iter, const float* proj, const float* r,
                           const float* alpha, const float* bias, float* h, cudaStream_t stream) {
    const unsigned grid = (unsigned)((T + kTokensPerBlock - 1) / kTokensPerBlock);
    gate_forward_kernel<<<grid, kThreads, 0, stream>>>(T, n_iter, proj, r, alpha, bias, h);
    return cudaGetLastError();
}

cudaError_t launch_backward(int64_t T, int n_iter, const float* proj, const float* r,
                            const float* alpha, const float* bias, const float* grad_h,
                            float* grad_proj, float* grad_r, float* dlogits, cudaStream_t stream) {
    const unsigned grid = (unsigned)((T + kTokensPerBlock - 1) / kTokensPerBlock);
    gate_backward_kernel<<<grid, kThreads, backward_smem_bytes(n_iter), stream>>>(
        T, n_iter, proj, r, alpha, bias, grad_h, grad_proj, grad_r, dlogits);
    return cudaGetLastError();
}

}  // namespace gates
}  // namespace mhcpb
