/* A C program that uses the library through its C ABI alone (no Python):
 * plan and workspace, the backward, the split backward, the forward, the
 * forward with the gates fused in and the gate calls.  The inputs are small
 * integers, so every expected value is exact and checked exactly against
 * plain loops here:
 *     dX[t][k] = sum_j P[t][j] W[j][k]   (grad_r = 0; |dX| <= 96: exact in BF16)
 *     dW[j][k] = sum_t P[t][j] X[t][k]   (|dW| <= 516: exact in FP32)
 *     proj[t][j] = sum_k X[t][k] W[j][k] (|proj| <= 2080: exact in FP32)
 * Built and run by tests/test_c_program_gpu.py; exit status 0 when every
 * check passed. */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "mhcpb.h"

#define CHECK(call)                                                                        \
    do {                                                                                   \
        mhcpb_status_t s_ = (call);                                                        \
        if (s_ != MHCPB_OK) {                                                              \
            fprintf(stderr, "%s: %s %s\n", #call, mhcpb_status_string(s_),                \
                    mhcpb_last_cuda_error());                                              \
            return 1;                                                                      \
        }                                                                                  \
    } while (0)
#define CUDA(call)                                                                         \
    do {                                                                                   \
        cudaError_t e_ = (call);                                                           \
        if (e_ != cudaSuccess) {                                                           \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                    \
            return 1;                                                                      \
        }                                                                                  \
    } while (0)
#define EXPECT(cond, what)                                                                 \
    do {                                                                                   \
        if (!(cond)) {                                                                     \
            fprintf(stderr, "check failed: %s\n", what);                                   \
            return 1;                                                                      \
        }                                                                                  \
    } while (0)

enum { T = 129, K = 520, NP = MHCPB_NPROJ, GP = MHCPB_GRAD_PROJ_COLS };

static uint16_t bf16_of_small_int(int v) {   /* exact for |v| < 256 */
    const float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}
static float f_of_bf16(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}
static int small(unsigned* state) { /* -2 .. 2 from a fixed linear congruential sequence */
    *state = *state * 1664525u + 1013904223u;
    return (int)((*state >> 16) % 5u) - 2;
}

int main(void) {
    static uint16_t x[T * K], dx[T * K], dx2[T * K];
    static float w[NP * K], gp[T * GP], gr[T], r[T], dw[NP * K], dw2[NP * K];
    static float proj[T * GP], rr[T], proj2[T * GP], rr2[T], h[T * NP], h2[T * NP];
    unsigned st = 12345u;
    for (int i = 0; i < T * K; ++i) x[i] = bf16_of_small_int(small(&st));
    for (int i = 0; i < NP * K; ++i) w[i] = (float)small(&st);
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < GP; ++j) gp[t * GP + j] = j < NP ? (float)small(&st) : NAN;   /* 24..31 unread */
        gr[t] = 0.f;
        r[t] = 1.f;
    }
    const float alpha[3] = {1.0f, 0.75f, 0.01f}, bias[NP] = {0};

    void *d_x, *d_w, *d_gp, *d_gr, *d_r, *d_dx, *d_dw, *d_proj, *d_rr, *d_h, *d_h2, *d_a, *d_b;
    CUDA(cudaMalloc(&d_x, sizeof x));
    CUDA(cudaMalloc(&d_w, sizeof w));
    CUDA(cudaMalloc(&d_gp, sizeof gp));
    CUDA(cudaMalloc(&d_gr, sizeof gr));
    CUDA(cudaMalloc(&d_r, sizeof r));
    CUDA(cudaMalloc(&d_dx, sizeof dx));
    CUDA(cudaMalloc(&d_dw, sizeof dw));
    CUDA(cudaMalloc(&d_proj, sizeof proj));
    CUDA(cudaMalloc(&d_rr, sizeof rr));
    CUDA(cudaMalloc(&d_h, sizeof h));
    CUDA(cudaMalloc(&d_h2, sizeof h2));
    CUDA(cudaMalloc(&d_a, sizeof alpha));
    CUDA(cudaMalloc(&d_b, sizeof bias));
    CUDA(cudaMemcpy(d_x, x, sizeof x, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_w, w, sizeof w, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_gp, gp, sizeof gp, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_gr, gr, sizeof gr, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_r, r, sizeof r, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_a, alpha, sizeof alpha, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_b, bias, sizeof bias, cudaMemcpyHostToDevice));
    cudaStream_t stream;
    CUDA(cudaStreamCreate(&stream));

    /* the backward */
    mhcpb_plan_t plan;
    CHECK(mhcpb_plan_create(&plan, T, K, 0, MHCPB_ALLOW_TF32));
    size_t ws_bytes = 0, fws_bytes = 0;
    CHECK(mhcpb_workspace_bytes(plan, &ws_bytes));
    CHECK(mhcpb_forward_workspace_bytes(plan, &fws_bytes));
    void* d_ws;
    CUDA(cudaMalloc(&d_ws, ws_bytes > fws_bytes ? ws_bytes : fws_bytes));
    CHECK(mhcpb_execute(plan, d_x, d_w, d_gp, d_gr, d_r, d_dx, d_dw, d_ws, ws_bytes, NULL, stream));
    CUDA(cudaStreamSynchronize(stream));
    mhcpb_status_t dev = MHCPB_OK;
    CHECK(mhcpb_get_device_status(plan, &dev, 0));
    EXPECT(dev == MHCPB_OK, "device status after the backward");
    CUDA(cudaMemcpy(dx, d_dx, sizeof dx, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(dw, d_dw, sizeof dw, cudaMemcpyDeviceToHost));
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            double s = 0;
            for (int j = 0; j < NP; ++j) s += (double)gp[t * GP + j] * w[j * K + k];
            EXPECT(f_of_bf16(dx[t * K + k]) == (float)s, "dX = P W");
        }
    for (int j = 0; j < NP; ++j)
        for (int k = 0; k < K; ++k) {
            double s = 0;
            for (int t = 0; t < T; ++t) s += (double)gp[t * GP + j] * f_of_bf16(x[t * K + k]);
            EXPECT(dw[j * K + k] == (float)s, "dW = P^T X");
        }

    /* the split backward: the same bits */
    CUDA(cudaMemset(d_dx, 0xFF, sizeof dx));
    CUDA(cudaMemset(d_dw, 0xFF, sizeof dw));
    CHECK(mhcpb_execute_dx(plan, d_x, d_w, d_gp, d_gr, d_r, d_dx, d_ws, ws_bytes, NULL, stream));
    CHECK(mhcpb_reduce_dw(plan, d_ws, ws_bytes, d_dw, stream));
    CUDA(cudaStreamSynchronize(stream));
    CUDA(cudaMemcpy(dx2, d_dx, sizeof dx2, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(dw2, d_dw, sizeof dw2, cudaMemcpyDeviceToHost));
    EXPECT(memcmp(dx, dx2, sizeof dx) == 0 && memcmp(dw, dw2, sizeof dw) == 0, "split backward bits");

    /* the forward */
    const float eps = 1e-6f;
    CHECK(mhcpb_forward(plan, d_x, d_w, eps, (float*)d_proj, (float*)d_rr, d_ws, fws_bytes, stream));
    CUDA(cudaStreamSynchronize(stream));
    CUDA(cudaMemcpy(proj, d_proj, sizeof proj, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(rr, d_rr, sizeof rr, cudaMemcpyDeviceToHost));
    for (int t = 0; t < T; ++t) {
        double ss = 0;
        for (int k = 0; k < K; ++k) ss += (double)f_of_bf16(x[t * K + k]) * f_of_bf16(x[t * K + k]);
        const double want_r = sqrt(ss / K + eps);
        EXPECT(fabs(rr[t] - want_r) <= 1e-6 * want_r, "r = RMS");
        for (int j = 0; j < GP; ++j) {
            double s = 0;
            if (j < NP)
                for (int k = 0; k < K; ++k) s += (double)f_of_bf16(x[t * K + k]) * w[j * K + k];
            EXPECT(proj[t * GP + j] == (float)s, "proj = X W^T (zero pad)");
        }
    }

    /* the forward with the gates fused in: the same bits as the two calls */
    CHECK(mhcpb_forward_gates(plan, d_x, d_w, eps, (const float*)d_a, (const float*)d_b, 20,
                              (float*)d_proj, (float*)d_rr, (float*)d_h, d_ws, fws_bytes, stream));
    CHECK(mhcpb_gate_forward(T, 20, (const float*)d_proj, (const float*)d_rr, (const float*)d_a,
                             (const float*)d_b, (float*)d_h2, stream));
    CUDA(cudaStreamSynchronize(stream));
    CUDA(cudaMemcpy(proj2, d_proj, sizeof proj2, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(rr2, d_rr, sizeof rr2, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(h, d_h, sizeof h, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(h2, d_h2, sizeof h2, cudaMemcpyDeviceToHost));
    EXPECT(memcmp(proj, proj2, sizeof proj) == 0 && memcmp(rr, rr2, sizeof rr) == 0, "fused proj, r");
    EXPECT(memcmp(h, h2, sizeof h) == 0, "fused gates equal the gate call");
    for (int t = 0; t < T; ++t) {   /* every row and column of H_res sums to 1 after the last column step */
        double col[4] = {0, 0, 0, 0};
        for (int i = 0; i < 16; ++i) col[i % 4] += h[t * NP + 8 + i];
        for (int c = 0; c < 4; ++c) EXPECT(fabs(col[c] - 1.0) < 1e-5, "Sinkhorn columns sum to 1");
    }

    /* the gate backward into the backward, then the device status */
    CHECK(mhcpb_gate_backward(T, 20, (const float*)d_proj, (const float*)d_rr, (const float*)d_a,
                              (const float*)d_b, (const float*)d_h, (float*)d_gp, (float*)d_gr, NULL,
                              stream));
    CHECK(mhcpb_execute(plan, d_x, d_w, d_gp, d_gr, d_rr, d_dx, d_dw, d_ws, ws_bytes, NULL, stream));
    CUDA(cudaStreamSynchronize(stream));
    CHECK(mhcpb_get_device_status(plan, &dev, 0));
    EXPECT(dev == MHCPB_OK, "device status at the end");
    CUDA(cudaMemcpy(dw, d_dw, sizeof dw, cudaMemcpyDeviceToHost));
    for (int i = 0; i < NP * K; ++i) EXPECT(isfinite(dw[i]), "dW finite after the chain");

    CHECK(mhcpb_destroy(plan));
    printf("C ABI ok: backward, split, forward, fused gates, gate backward chain\n");
    return 0;
}
