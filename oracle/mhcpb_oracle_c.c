/* CPU oracle of the mHC projection/RMS backward in plain C -- TEST
 * INFRASTRUCTURE ONLY (built beside the library, never linked into it).
 *
 * The same definition as oracle/mhcpb_oracle.py (cuDNN frontend page "DSv4.1
 * mHC projection/RMS backward", intro), evaluated in FP64 over the
 * TF32-rounded product operands and rounded once:
 *
 *     P  = grad_proj[:, :24]                     (TF32, nearest, ties away)
 *     dX = bf16_rne(P @ W + grad_r / (r K) * X)  (W TF32; X BF16 is exact)
 *     dW = fp32_rne(P^T @ X)
 *
 * Plain loops: rows of dX in parallel (OpenMP), dW accumulated per thread over
 * a block of columns, token by token.  The loops use the numpy oracle's
 * order where it fixes one: sum over j first, then add c x.  FP64 sums in
 * another order change at most the last FP64 bits, so the rounded outputs
 * equal the numpy oracle's except at a rounding tie, which random inputs do not
 * produce; tests/test_oracle_c.py checks that.  It is the CPU baseline
 * bench.py times, for a fair measure of host throughput.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define NPROJ 24
#define GP_COLS 32

static double f32_to_f64(float v) { return (double)v; }

/* TF32: keep 10 explicit mantissa bits, round to nearest with ties away from
 * zero (add half of the last kept place to the magnitude's bits, clear the 13
 * dropped bits; a carry into the exponent is the correct result).  Non-finite
 * values pass through. */
static float tf32_rna(float v) {
    if (!isfinite(v)) return v;
    uint32_t u;
    memcpy(&u, &v, 4);
    u = (u + 0x1000u) & 0xFFFFE000u;
    float o;
    memcpy(&o, &u, 4);
    return o;
}

static double bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* FP64 -> BF16 (8 significant bits, FP32's exponent range), nearest-even,
 * with no intermediate FP32 rounding.  The spacing of BF16 values at |v| is
 * 2^(max(e, -126) - 7) for 2^e <= |v| < 2^(e+1); v / spacing is exact and
 * nearbyint rounds half to even in the default rounding mode. */
static uint16_t bf16_rne_from_f64(double v) {
    if (isnan(v)) return 0x7FC0;
    if (isinf(v)) return v > 0 ? 0x7F80 : 0xFF80;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    int e;
    frexp(v, &e);                     /* v = m 2^e, 0.5 <= |m| < 1: binade exponent e - 1 */
    int be = e - 1;
    if (be < -126) be = -126;
    const double ulp = ldexp(1.0, be - 7);
    const double q = nearbyint(v / ulp) * ulp;
    if (fabs(q) >= ldexp(1.0, 128)) return v > 0 ? 0x7F80 : 0xFF80;
    const float qf = (float)q;        /* exact: q is a BF16 value */
    uint32_t u;
    memcpy(&u, &qf, 4);
    return (uint16_t)(u >> 16);
}

/* x BF16 bits [T, K]; w [24, K]; grad_proj [T, 32]; grad_r, r [T];
 * outputs dx BF16 bits [T, K], dw [24, K].  nthreads <= 0: OpenMP's default. */
void mhcpb_oracle_backward(int64_t T, int64_t K, const uint16_t* x, const float* w,
                           const float* grad_proj, const float* grad_r, const float* r,
                           uint16_t* dx, float* dw, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    double* Wt = (double*)malloc(sizeof(double) * NPROJ * (size_t)K);
    double* P = (double*)malloc(sizeof(double) * NPROJ * (size_t)T);
    for (int64_t i = 0; i < NPROJ * K; ++i) Wt[i] = f32_to_f64(tf32_rna(w[i]));
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < NPROJ; ++j) P[t * NPROJ + j] = f32_to_f64(tf32_rna(grad_proj[t * GP_COLS + j]));

    /* dX, one row at a time */
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double c = f32_to_f64(grad_r[t]) / (f32_to_f64(r[t]) * (double)K);
        const double* pt = P + t * NPROJ;
        for (int64_t k = 0; k < K; ++k) {
            double s = 0.0;
            for (int j = 0; j < NPROJ; ++j) s += pt[j] * Wt[(size_t)j * K + k];
            s += c * bf16_to_f64(x[t * K + k]);
            dx[t * K + k] = bf16_rne_from_f64(s);
        }
    }

    /* dW, one block of columns per task: for every token, add P[t, j] x[t, k] */
    const int64_t kb = 256;
    const int64_t nblk = (K + kb - 1) / kb;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t b = 0; b < nblk; ++b) {
        const int64_t k0 = b * kb;
        const int64_t k1 = k0 + kb < K ? k0 + kb : K;
        double acc[NPROJ][256];
        for (int j = 0; j < NPROJ; ++j)
            for (int64_t k = 0; k < k1 - k0; ++k) acc[j][k] = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            const double* pt = P + t * NPROJ;
            const uint16_t* xr = x + t * K;
            for (int j = 0; j < NPROJ; ++j) {
                const double pj = pt[j];
                for (int64_t k = k0; k < k1; ++k) acc[j][k - k0] += pj * bf16_to_f64(xr[k]);
            }
        }
        for (int j = 0; j < NPROJ; ++j)
            for (int64_t k = k0; k < k1; ++k) dw[(size_t)j * K + k] = (float)acc[j][k - k0];
    }
    free(Wt);
    free(P);
}
