// Arithmetic of the mHC gate/normalisation step (the reading stated in
// mhcpb.h, mhcpb_gate_forward) for one token held by a half-warp: lane l of
// the 16 owns residual entry (l / 4, l % 4) and, for l < 8, pre/post gate l.
// Shared by the gate kernels and the forward's fused reduction, so that both
// give the same bits from the same projection values.
#pragma once

#include <cuda_runtime.h>

namespace mhcpb {
namespace gatemath {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float row_sum(float v) {   // lanes 4i .. 4i+3 of the half-warp
    v += __shfl_xor_sync(kFull, v, 1, 16);
    v += __shfl_xor_sync(kFull, v, 2, 16);
    return v;
}
__device__ __forceinline__ float col_sum(float v) {   // lanes j, j+4, j+8, j+12
    v += __shfl_xor_sync(kFull, v, 4, 16);
    v += __shfl_xor_sync(kFull, v, 8, 16);
    return v;
}
__device__ __forceinline__ float row_max(float v) {
    v = fmaxf(v, __shfl_xor_sync(kFull, v, 1, 16));
    v = fmaxf(v, __shfl_xor_sync(kFull, v, 2, 16));
    return v;
}
__device__ __forceinline__ float col_max(float v) {
    v = fmaxf(v, __shfl_xor_sync(kFull, v, 4, 16));
    v = fmaxf(v, __shfl_xor_sync(kFull, v, 8, 16));
    return v;
}
__device__ __forceinline__ float sigmoid(float x) { return 1.f / (1.f + expf(-x)); }

// one Sinkhorn iteration on this lane's log-value: returns log M, and log R
// (after the row step) through `lr`
__device__ __forceinline__ float sinkhorn_step_log(float la, float& lr) {
    const float m = row_max(la);
    lr = la - (m + logf(row_sum(expf(la - m))));
    const float m2 = col_max(lr);
    return lr - (m2 + logf(col_sum(expf(lr - m2))));
}
// a sum the direct iterations can divide by: finite and normal with margin
__device__ __forceinline__ bool sum_ok(float v) { return v >= 1e-30f && v <= 1e30f; }

// n_iter Sinkhorn iterations of this lane's residual logit l; stores R and M
// of every iteration at Rs/Ms[k * stride + threadIdx.x] when they are given;
// returns the final M.  Warp-uniform: every lane of the warp calls it.
//
// The iterations first run directly on exp(l - row maximum), dividing by sums
// through their correctly rounded reciprocals.  Where a token's sums leave
// the normal FP32 range (logits ~90 or more apart leave a whole column at 0,
// or the inputs hold NaN), the warp redoes its tokens on logarithms: a row
// normalisation is log R = log A - LSE_row(log A), a column normalisation
// log M = log R - LSE_col(log R), each log-sum-exp taken after subtracting
// the maximum, so no sum can underflow.  Both give the same R and M up to
// rounding.
__device__ __forceinline__ float sinkhorn(float l, int n_iter, float* Rs, float* Ms, int stride) {
    // direct: A = exp(l - row max) in (0, 1]
    float A = expf(l - row_max(l));
    bool ok = true;
    for (int k = 0; k < n_iter; ++k) {
        const float s = row_sum(A);
        const float R = A * __frcp_rn(s);
        const float c = col_sum(R);
        A = R * __frcp_rn(c);
        ok = ok && sum_ok(s) && sum_ok(c);
        if (Rs != nullptr) {
            Rs[k * stride + threadIdx.x] = R;
            Ms[k * stride + threadIdx.x] = A;
        }
    }
    if (!__any_sync(kFull, !ok)) return A;
    // a sum left the safe range somewhere in this warp: redo on logarithms
    float la = l;
    for (int k = 0; k < n_iter; ++k) {
        float lr;
        la = sinkhorn_step_log(la, lr);
        if (Rs != nullptr) {
            Rs[k * stride + threadIdx.x] = expf(lr);
            Ms[k * stride + threadIdx.x] = expf(la);
        }
    }
    return expf(la);
}

// the residual logit of lane l: a_res * proj[8 + l] / r + b[8 + l]
__device__ __forceinline__ float res_logit(float pres, float rv, const float* alpha, const float* bias,
                                           int l) {
    return alpha[2] * pres / rv + bias[8 + l];
}
// pre gate (l < 4: sigmoid) or post gate (4 <= l < 8: 2 sigmoid) of lane l
// from its projection value pg
__device__ __forceinline__ float pre_post_gate(float pg, float rv, const float* alpha, const float* bias,
                                               int l) {
    const float a = l < 4 ? alpha[0] : alpha[1];
    const float s = sigmoid(a * pg / rv + bias[l]);
    return l < 4 ? s : 2.f * s;
}

}  // namespace gatemath
}  // namespace mhcpb
