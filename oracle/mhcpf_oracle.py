"""CPU oracle for the mHC projection forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this module.  The library never does (no CPU fallback), and nothing
here is shared with the CUDA path.

What the forward computes.  The prime-kernels PR #15 page describes its
``mhc_projection`` as the RMS of the streams and the projection (gate) logits
from a single pass over the streams; the cuDNN frontend page "DSv4.1 mHC
projection/RMS backward" (intro) fixes what the backward of this stage
receives: the gradient of a [T, 32] projection output of which the first 24
columns are used, and the gradient of a per-row RMS r[T].  Its formula,
dX = P @ W + grad_r / (r * K) * X, is exactly the vector-Jacobian product of

    proj[t, j] = sum_k X[t, k] * W[j, k]          (j < 24; TF32 operands, FP32 accumulation)
    r[t]       = sqrt(mean_k X[t, k]^2 + eps)     (eps = 1e-6, the workloads' value)

so these are the forward this oracle defines (the plainest reading; the
pages give no formula for the forward itself).  The output layout mirrors the
backward's input: proj is FP32 [T, 32] with columns 24..31 written as zero,
r is FP32 [T].  The stream collapse that the PR also fuses into its
forward needs the previous sublayer's weights, which the pages do not define;
it is not part of this stage.

Precision: W is rounded to TF32 (nearest, ties away), X is BF16 (exact in
TF32); the oracle evaluates both outputs in FP64 and the tests compare the
GPU's FP32 results within bounds derived from FP32 accumulation
(``check_proj``, ``check_r``).

Pins (tests/test_forward_oracle_pins.py): finite differences of
L(X) = sum P * proj(X) + sum g * r(X) reproduce the backward oracle's dX (which
is pinned to the page's formula), hand-computed values, closed forms (constant
and zero rows, one-hot W, TF32 rounding of W), linearity of proj, and planted
mistakes each caught.
"""
from __future__ import annotations

import numpy as np

from .mhcpb_oracle import bf16_bits_to_f64, tf32_rna

N_PROJ = 24
PROJ_COLS = 32
RMS_EPS = 1e-6


def proj_of(Xd: np.ndarray, w) -> np.ndarray:
    """The projection of FP64 rows Xd [n, K]: Xd @ tf32(W)^T, [n, 24]."""
    Wt = tf32_rna(np.asarray(w, dtype=np.float32)).astype(np.float64)   # [24, K]
    return Xd @ Wt.T


def rms_of(Xd: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """The RMS of FP64 rows Xd [n, K]: sqrt(sum_k X^2 / K + eps), [n]."""
    return np.sqrt(np.sum(Xd * Xd, axis=1) / Xd.shape[1] + eps)


def proj_f64(x_bits, w, rows=None, row_block=1024) -> np.ndarray:
    """proj of the BF16 X in FP64, [T or len(rows), 24]."""
    x_bits = np.asarray(x_bits)
    if rows is not None:
        x_bits = x_bits[np.asarray(rows)]
    out = np.empty((x_bits.shape[0], N_PROJ), dtype=np.float64)
    for t0 in range(0, x_bits.shape[0], row_block):
        out[t0:t0 + row_block] = proj_of(bf16_bits_to_f64(x_bits[t0:t0 + row_block]), w)
    return out


def rms_f64(x_bits, eps: float = RMS_EPS, rows=None, row_block=1024) -> np.ndarray:
    """r of the BF16 X in FP64, [T or len(rows)]."""
    x_bits = np.asarray(x_bits)
    if rows is not None:
        x_bits = x_bits[np.asarray(rows)]
    out = np.empty(x_bits.shape[0], dtype=np.float64)
    for t0 in range(0, x_bits.shape[0], row_block):
        out[t0:t0 + row_block] = rms_of(bf16_bits_to_f64(x_bits[t0:t0 + row_block]), eps)
    return out


def mhc_proj_forward(x_bits, w, eps: float = RMS_EPS, rows=None):
    """(proj [.., 32] FP64 with zero pad columns, r [..] FP64)."""
    p = proj_f64(x_bits, w, rows=rows)
    proj = np.zeros((p.shape[0], PROJ_COLS), dtype=np.float64)
    proj[:, :N_PROJ] = p
    return proj, rms_f64(x_bits, eps, rows=rows)


def proj_abs_bound(x_bits, w, rows=None, row_block=1024) -> np.ndarray:
    """sum_k |X[t,k]| |tf32(W)[j,k]| per proj element."""
    x_bits = np.asarray(x_bits)
    if rows is not None:
        x_bits = x_bits[np.asarray(rows)]
    Wa = np.abs(tf32_rna(np.asarray(w, dtype=np.float32)).astype(np.float64))
    out = np.empty((x_bits.shape[0], N_PROJ), dtype=np.float64)
    for t0 in range(0, x_bits.shape[0], row_block):
        out[t0:t0 + row_block] = np.abs(bf16_bits_to_f64(x_bits[t0:t0 + row_block])) @ Wa.T
    return out


def check_proj(proj, ref, bound, rel=2.0 ** -14):
    """GPU proj (FP32 [.., 32]) against the oracle: columns 0..23 within
    rel * sum_k |X||W| (FP32 accumulation of the products, which are exact:
    the error of n FP32 additions is at most about n * 2**-24 of that sum, and
    the GPU's summation depth is well under 2**10 additions per element);
    columns 24..31 exactly zero.  Returns (ok, stats)."""
    proj = np.asarray(proj, dtype=np.float64)
    err = np.abs(proj[:, :N_PROJ] - ref[:, :N_PROJ])
    tol = rel * bound
    bad = err > tol
    pad_ok = bool(np.all(proj[:, N_PROJ:] == 0.0))
    stats = dict(n=err.size, bad=int(bad.sum()), max_err_over_bound=float(np.max(err / np.maximum(bound, 1e-300))),
                 pad_ok=pad_ok)
    return (not bad.any()) and pad_ok, stats


def check_r(r, ref, rel=2.0 ** -16):
    """GPU r (FP32) against the oracle: relative error within 2**-16 (the sum
    of K exact squares in FP32 in blocks loses at most a few hundred 2**-24,
    halved by the square root, plus the FP32 rounding of r)."""
    r = np.asarray(r, dtype=np.float64)
    err = np.abs(r - ref)
    bad = err > rel * ref
    rel_err = np.where(ref > 0, err / np.where(ref > 0, ref, 1.0), np.where(err > 0, np.inf, 0.0))
    return (not bad.any()), dict(n=err.size, bad=int(bad.sum()), max_rel=float(np.max(rel_err)))
