"""CPU oracle of the mHC gate/normalisation step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this module.  The library never does; nothing here is shared with
the CUDA path.

What the step is (its place in the graph): the cuDNN frontend page "DSv4.1
mHC projection/RMS backward" (intro) takes "the upstream projection and RMS
gradients after the gate and normalization derivatives" and leaves "Sinkhorn,
gate derivatives" to the caller; the prime-kernels PR #15 page ("mhc_projection"
bullet) fuses "gate activations (sigmoid, Sinkhorn)" into the projection.  So
this step maps the forward's projection logits proj = X W^T (24 used columns)
and RMS r to the gates, and its backward turns the gates' upstream gradients
into grad_proj (the backward stage's P) and grad_r.

Neither page writes the gates' formulas.  Declared reading (n = 4 streams; the
24 projection columns are 2n + n^2 = 4 + 4 + 16, the page's 24):

    columns 0..3   pre    logits  l_pre  = a_pre  * proj[:, 0:4]  / r + b[0:4]
    columns 4..7   post   logits  l_post = a_post * proj[:, 4:8]  / r + b[4:8]
    columns 8..23  res    logits  l_res  = a_res  * proj[:, 8:24] / r + b[8:24]
                                  (row-major 4 x 4: column 8 + 4 i + j is entry (i, j))
    H_pre  = sigmoid(l_pre)
    H_post = 2 sigmoid(l_post)
    H_res  = Sinkhorn(exp(l_res)) with n_iter iterations (default 20), each a
             row normalisation (every row divided by its sum) followed by a
             column normalisation (every column divided by its sum)

with r the RMS the forward computes (the projection of the RMS-normalised
streams is proj / r) and a_pre, a_post, a_res, b learnable.  The backward
takes upstream gradients G (the same 24-column layout as H) and returns

    dl         = dL/dlogits (chain rule through sigmoid and the Sinkhorn iterations)
    grad_proj  = dl * a_g / r                         (columns 0..23; 24..31 are 0)
    grad_r     = -sum_j dl_j * a_g(j) * proj_j / r^2

The parameter gradients (of a and b) stay with the caller, as the cuDNN page
says of parameter-gradient accumulation; dl is returned so that they are one
reduction away.

Everything is FP64 from the FP32 inputs.  Parity pins (tests/test_gates_oracle_pins.py):
central finite differences of the forward, hand-derived Sinkhorn values
(tests/golden/sinkhorn_hand.txt), closed forms at zero logits and for rank-1
logits, and planted mistakes.
"""
from __future__ import annotations

import numpy as np

N_STREAMS = 4
N_COLS = 2 * N_STREAMS + N_STREAMS * N_STREAMS   # 24
GROUPS = (slice(0, 4), slice(4, 8), slice(8, 24))


def alpha_per_column(alpha) -> np.ndarray:
    """The three scales (pre, post, res) spread over the 24 columns."""
    a = np.asarray(alpha, dtype=np.float32).astype(np.float64)
    out = np.empty(N_COLS)
    for g, sl in enumerate(GROUPS):
        out[sl] = a[g]
    return out


def logits(proj, r, alpha, bias) -> np.ndarray:
    """l[t, j] = a_g(j) * proj[t, j] / r[t] + b[j] over the 24 used columns."""
    p = np.asarray(proj, dtype=np.float32)[:, :N_COLS].astype(np.float64)
    rr = np.asarray(r, dtype=np.float32).astype(np.float64)
    b = np.asarray(bias, dtype=np.float32).astype(np.float64)
    return alpha_per_column(alpha)[None, :] * p / rr[:, None] + b[None, :]


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def sinkhorn(l_res, n_iter=20):
    """Sinkhorn iteration on exp(l_res) ([T, 4, 4]).  Returns the final matrix
    and, for the backward, every intermediate: A[k] (before the k-th row
    normalisation, k = 0 .. n_iter-1), Rn[k] (after it) and M[k] (after the
    column normalisation that follows)."""
    A = np.exp(np.asarray(l_res, dtype=np.float64))
    As, Rs, Ms = [], [], []
    for _ in range(n_iter):
        As.append(A)
        R = A / A.sum(axis=2, keepdims=True)      # rows sum to 1
        Rs.append(R)
        M = R / R.sum(axis=1, keepdims=True)      # columns sum to 1
        Ms.append(M)
        A = M
    return A, (As, Rs, Ms)


def gate_forward(proj, r, alpha, bias, n_iter=20) -> np.ndarray:
    """H [T, 24]: H_pre (0..3), H_post (4..7), H_res row-major (8..23)."""
    lg = logits(proj, r, alpha, bias)
    T = lg.shape[0]
    h = np.empty((T, N_COLS))
    h[:, 0:4] = sigmoid(lg[:, 0:4])
    h[:, 4:8] = 2.0 * sigmoid(lg[:, 4:8])
    M, _ = sinkhorn(lg[:, 8:24].reshape(T, 4, 4), n_iter)
    h[:, 8:24] = M.reshape(T, 16)
    return h


def sinkhorn_backward(dM, cache):
    """Reverse mode through the iterations: for the column step M = R / c
    (c_j = sum_i R_ij), dR = (dM - sum_i dM_ij M_ij) / c_j; for the row step
    R = A / s (s_i = sum_j A_ij), dA = (dR - sum_j dR_ij R_ij) / s_i; finally
    A0 = exp(l): dl = dA0 * A0."""
    As, Rs, Ms = cache
    d = np.asarray(dM, dtype=np.float64)
    for A, R, M in zip(reversed(As), reversed(Rs), reversed(Ms)):
        c = R.sum(axis=1, keepdims=True)
        dR = (d - (d * M).sum(axis=1, keepdims=True)) / c
        s = A.sum(axis=2, keepdims=True)
        d = (dR - (dR * R).sum(axis=2, keepdims=True)) / s
    return d * As[0]


def gate_backward(proj, r, alpha, bias, grad_h, n_iter=20):
    """Returns (grad_proj [T, 32] with columns 24..31 zero, grad_r [T],
    dl [T, 24]) in FP64."""
    lg = logits(proj, r, alpha, bias)
    G = np.asarray(grad_h, dtype=np.float32)[:, :N_COLS].astype(np.float64)
    T = lg.shape[0]
    dl = np.empty((T, N_COLS))
    s_pre = sigmoid(lg[:, 0:4])
    dl[:, 0:4] = G[:, 0:4] * s_pre * (1.0 - s_pre)
    s_post = sigmoid(lg[:, 4:8])
    dl[:, 4:8] = G[:, 4:8] * 2.0 * s_post * (1.0 - s_post)
    _, cache = sinkhorn(lg[:, 8:24].reshape(T, 4, 4), n_iter)
    dl[:, 8:24] = sinkhorn_backward(G[:, 8:24].reshape(T, 4, 4), cache).reshape(T, 16)
    a = alpha_per_column(alpha)
    p = np.asarray(proj, dtype=np.float32)[:, :N_COLS].astype(np.float64)
    rr = np.asarray(r, dtype=np.float32).astype(np.float64)
    grad_proj = np.zeros((T, 32))
    grad_proj[:, :N_COLS] = dl * a[None, :] / rr[:, None]
    grad_r = -(dl * a[None, :] * p).sum(axis=1) / (rr * rr)
    return grad_proj, grad_r, dl


# --------------------------------------------------------------------------
# Tolerance the CUDA path is held to
# --------------------------------------------------------------------------
def check_rows(got, ref, rel=1e-4, floor=1e-30):
    """Row-wise (per token) acceptance: |got - ref| <= rel * max_j |ref[t, j]|
    + floor, element by element.  FP32 evaluation of the iterations carries a
    relative error of some 1e-6 of the row's magnitudes (tens of FP32 roundings
    through contractive normalisation steps); 1e-4 leaves a wide margin and
    still catches any wrong term.  Non-finite references must match exactly."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if r.ndim == 1:
        g, r = g[:, None], r[:, None]
    scale = np.max(np.abs(np.where(np.isfinite(r), r, 0.0)), axis=1, keepdims=True)
    lim = rel * scale + floor
    fin = np.isfinite(r)
    diff = np.abs(np.subtract(g, r, out=np.zeros_like(g), where=fin))   # 0 where ref is not finite
    ok = np.where(fin, (diff <= lim) & np.isfinite(g), (np.isnan(g) & np.isnan(r)) | (g == r))
    worst = float(np.max(np.where(fin, diff / lim, 0.0))) if r.size else 0.0
    return bool(ok.all()), dict(n=int(r.size), fail=int((~ok).sum()), worst_frac_of_tol=worst)
