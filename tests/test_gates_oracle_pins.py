"""Pins of the gate/normalisation oracle (oracle/mhcg_oracle.py) to facts
other than its own formulas.

The reading the oracle states (2n + n^2 = 24 logits for n = 4 streams, sigmoid
and 2 sigmoid gates, Sinkhorn over exp with row-then-column normalisation) has
no worked example on the pages (cuDNN frontend page "DSv4.1 mHC
projection/RMS backward", intro; prime-kernels PR #15, "mhc_projection"), so the
pins are: central finite differences of the forward for the whole backward,
Sinkhorn values worked by hand in exact fractions (tests/golden/sinkhorn_hand.txt),
closed forms at zero logits and for rank-1 logits, the doubly stochastic
limit, and mistakes planted in copies of the backward.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle.mhcg_oracle as G
from rms_backward_gb300 import workloads as WL


def _loss(proj, r, alpha, bias, gh, n_iter):
    return float(np.sum(np.asarray(gh, np.float64)[:, :24] * G.gate_forward(proj, r, alpha, bias, n_iter)))


def _small(seed=0, T=3):
    wl = WL.make_gates("pin", T=T, seed=seed)
    return wl.proj.astype(np.float64), wl.r.astype(np.float64), wl.alpha, wl.bias, wl.grad_h


def _fd_matches(backward, n_iter=20, seed=0, tol=1e-6):
    """Central differences of sum(G * H) against a backward's grad_proj and grad_r."""
    proj, r, alpha, bias, gh = _small(seed)
    gp, gr, _ = backward(proj, r, alpha, bias, gh, n_iter)
    h = 1e-6
    ok = True
    for t in range(proj.shape[0]):
        for j in range(24):
            e = np.zeros_like(proj)
            e[t, j] = h
            # the oracle reads its inputs as FP32; differences go through FP64 copies
            fd = (_loss64(proj + e, r, alpha, bias, gh, n_iter) - _loss64(proj - e, r, alpha, bias, gh, n_iter)) / (2 * h)
            ok &= abs(gp[t, j] - fd) <= tol * (1 + abs(fd)) * 10
        e = np.zeros_like(r)
        e[t] = h
        fd = (_loss64(proj, r + e, alpha, bias, gh, n_iter) - _loss64(proj, r - e, alpha, bias, gh, n_iter)) / (2 * h)
        ok &= abs(gr[t] - fd) <= tol * (1 + abs(fd)) * 10
    return bool(ok)


def _loss64(proj, r, alpha, bias, gh, n_iter):
    """sum(G * H) with the forward evaluated on FP64 inputs (no FP32 rounding
    of the perturbed operands): the same formulas as the oracle's forward, on
    values that are not rounded to FP32 first."""
    a = G.alpha_per_column(alpha)
    lg = a[None, :] * proj[:, :24] / r[:, None] + np.asarray(bias, np.float64)[None, :]
    T = lg.shape[0]
    hh = np.empty((T, 24))
    hh[:, 0:4] = G.sigmoid(lg[:, 0:4])
    hh[:, 4:8] = 2 * G.sigmoid(lg[:, 4:8])
    M, _ = G.sinkhorn(lg[:, 8:24].reshape(T, 4, 4), n_iter)
    hh[:, 8:24] = M.reshape(T, 16)
    return float(np.sum(np.asarray(gh, np.float64)[:, :24] * hh))


def _backward_fp64(proj, r, alpha, bias, gh, n_iter):
    """The oracle's backward on inputs that are already FP32 values (so that
    its FP32 reading of them changes nothing)."""
    return G.gate_backward(proj.astype(np.float32), r.astype(np.float32), alpha, bias, gh, n_iter)


# ------------------------------------------------------------- finite differences
@pytest.mark.parametrize("n_iter", [1, 3, 20])
def test_backward_matches_central_differences(n_iter):
    proj, r, alpha, bias, gh = _small(seed=n_iter)
    proj, r = proj.astype(np.float32).astype(np.float64), r.astype(np.float32).astype(np.float64)
    gp, gr, dl = G.gate_backward(proj, r, alpha, bias, gh, n_iter)
    h = 1e-6
    for t in range(proj.shape[0]):
        for j in range(24):
            e = np.zeros_like(proj)
            e[t, j] = h
            fd = (_loss64(proj + e, r, alpha, bias, gh, n_iter) - _loss64(proj - e, r, alpha, bias, gh, n_iter)) / (2 * h)
            assert abs(gp[t, j] - fd) <= 1e-7 * (1 + abs(fd)) + 1e-9, (t, j, gp[t, j], fd)
        e = np.zeros_like(r)
        e[t] = h
        fd = (_loss64(proj, r + e, alpha, bias, gh, n_iter) - _loss64(proj, r - e, alpha, bias, gh, n_iter)) / (2 * h)
        assert abs(gr[t] - fd) <= 1e-7 * (1 + abs(fd)) + 1e-9, (t, gr[t], fd)
    assert np.all(gp[:, 24:] == 0)
    # dl is grad_proj undone: dl = grad_proj * r / a
    a = G.alpha_per_column(alpha)
    assert np.allclose(dl, gp[:, :24] * r[:, None] / a[None, :], rtol=1e-12, atol=0)


# --------------------------------------------------------------- hand values
def _hand_fixture():
    path = os.path.join(os.path.dirname(__file__), "golden", "sinkhorn_hand.txt")
    out = {}
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        n, *vals = line.split()
        out[int(n)] = np.array([float(Fraction(v)) for v in vals]).reshape(4, 4)
    return out


def test_sinkhorn_hand_worked_iterations():
    l = np.zeros((1, 4, 4))
    l[0, 3, 3] = np.log(5.0)
    for n_iter, want in _hand_fixture().items():
        M, _ = G.sinkhorn(l, n_iter)
        assert np.allclose(M[0], want, rtol=1e-13, atol=0), (n_iter, M[0], want)


def test_sinkhorn_hand_values_through_the_gate_forward():
    """The same matrix reached through the logits: a_res = 1, r = 1, b = 0."""
    proj = np.zeros((1, 32), np.float32)
    proj[0, 8 + 15] = np.float32(np.log(5.0))
    want = _hand_fixture()[2]
    h = G.gate_forward(proj, np.ones(1, np.float32), np.ones(3, np.float32), np.zeros(24, np.float32), 2)
    # proj[23] is ln 5 rounded to FP32: 1e-7 relative slack
    assert np.allclose(h[0, 8:24].reshape(4, 4), want, rtol=1e-6, atol=0)


# -------------------------------------------------------------- closed forms
def test_zero_logits_closed_form():
    """l = 0: H_pre = 1/2, H_post = 1, H_res = 1/4 everywhere; the sigmoid
    slopes are 1/4 and 2 * 1/4; at the uniform matrix the Sinkhorn backward
    removes each row's and column's mean from G; proj = 0 gives grad_r = 0."""
    T = 2
    proj = np.zeros((T, 32), np.float32)
    r = np.array([2.0, 0.5], np.float32)
    alpha = np.array([1.0, 3.0, 0.5], np.float32)
    gh = np.arange(T * 24, dtype=np.float32).reshape(T, 24) - 20
    h = G.gate_forward(proj, r, alpha, np.zeros(24, np.float32), 5)
    assert np.all(h[:, 0:4] == 0.5) and np.all(h[:, 4:8] == 1.0) and np.all(h[:, 8:24] == 0.25)
    gp, gr, dl = G.gate_backward(proj, r, alpha, np.zeros(24, np.float32), gh, 5)
    assert np.array_equal(dl[:, 0:4], gh[:, 0:4] * 0.25)
    assert np.array_equal(dl[:, 4:8], gh[:, 4:8] * 0.5)
    # at the fixed point (uniform 1/4, every row and column sum 1 after each step):
    # dl = (G - row mean - column mean + grand mean) / 4 -- the projection of G
    # onto matrices with zero row and column sums, times the slope 1/4 of exp-then-normalise
    Gm = gh[:, 8:24].reshape(T, 4, 4).astype(np.float64)
    proj0 = Gm - Gm.mean(2, keepdims=True) - Gm.mean(1, keepdims=True) + Gm.mean((1, 2), keepdims=True)
    assert np.allclose(dl[:, 8:24].reshape(T, 4, 4), proj0 / 4, rtol=0, atol=1e-12)
    assert np.allclose(gp[:, 0:4], dl[:, 0:4] * 1.0 / r[:, None], rtol=1e-15)
    assert np.allclose(gp[:, 4:8], dl[:, 4:8] * 3.0 / r[:, None], rtol=1e-15)
    assert np.allclose(gp[:, 8:24], dl[:, 8:24] * 0.5 / r[:, None], rtol=1e-15)
    assert np.all(gr == 0)


def test_rank_one_logits_give_the_uniform_matrix_in_one_iteration():
    """exp(u_i + v_j) = e^u_i e^v_j: after the row step every row is the same,
    so the column step gives 1/4 everywhere."""
    rng = np.random.default_rng(3)
    u, v = rng.standard_normal(4), rng.standard_normal(4)
    l = (u[:, None] + v[None, :])[None]
    M, _ = G.sinkhorn(l, 1)
    assert np.allclose(M, 0.25, rtol=1e-14, atol=0)


def test_twenty_iterations_are_nearly_doubly_stochastic():
    wl = WL.make_gates("ds", T=200, seed=4)
    h = G.gate_forward(wl.proj, wl.r, wl.alpha, wl.bias, 20)
    M = h[:, 8:24].reshape(-1, 4, 4)
    assert np.allclose(M.sum(1), 1.0, atol=1e-12)          # the last step normalised columns
    assert np.allclose(M.sum(2), 1.0, atol=1e-3)           # rows: converged
    assert np.all(M > 0)
    assert np.all((h[:, 0:4] > 0) & (h[:, 0:4] < 1)) and np.all((h[:, 4:8] > 0) & (h[:, 4:8] < 2))


def test_unused_columns_are_ignored():
    wl = WL.make_gates("ig", T=7, seed=5)
    a = G.gate_backward(wl.proj, wl.r, wl.alpha, wl.bias, wl.grad_h)
    p2 = wl.proj.copy()
    p2[:, 24:] = np.nan
    b = G.gate_backward(p2, wl.r, wl.alpha, wl.bias, wl.grad_h)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ---------------------------------------------------------- planted mistakes
def test_pins_catch_planted_mistakes():
    def col_then_row(proj, r, alpha, bias, gh, n_iter):
        # Sinkhorn with the column step first
        saved = G.sinkhorn

        def swapped(l, n):
            A = np.exp(l)
            As, Rs, Ms = [], [], []
            for _ in range(n):
                As.append(A)
                Rc = A / A.sum(1, keepdims=True)
                Rs.append(Rc)
                A = Rc / Rc.sum(2, keepdims=True)
                Ms.append(A)
            return A, (As, Rs, Ms)
        G.sinkhorn = swapped
        try:
            return G.gate_backward(proj, r, alpha, bias, gh, n_iter)
        finally:
            G.sinkhorn = saved

    def no_factor_two(proj, r, alpha, bias, gh, n_iter):
        gp, gr, dl = G.gate_backward(proj, r, alpha, bias, gh, n_iter)
        gp = gp.copy()
        gp[:, 4:8] /= 2
        return gp, gr, dl

    def grad_r_sign(proj, r, alpha, bias, gh, n_iter):
        gp, gr, dl = G.gate_backward(proj, r, alpha, bias, gh, n_iter)
        return gp, -gr, dl

    def missing_alpha(proj, r, alpha, bias, gh, n_iter):
        return G.gate_backward(proj, r, np.ones(3, np.float32), bias, gh, n_iter)

    def one_iteration_short(proj, r, alpha, bias, gh, n_iter):
        return G.gate_backward(proj, r, alpha, bias, gh, n_iter - 1)

    assert _fd_matches(_backward_fp64, n_iter=4)
    for bad in (col_then_row, no_factor_two, grad_r_sign, missing_alpha, one_iteration_short):
        assert not _fd_matches(bad, n_iter=4), bad.__name__


def test_check_rows_limits():
    ref = np.array([[1.0, -2.0, 0.0], [0.0, 0.0, 0.0]])
    assert G.check_rows(ref + np.array([[1.9e-4, -1.9e-4, 1.9e-4], [0, 0, 0]]), ref)[0]   # 1e-4 of 2
    assert not G.check_rows(ref + np.array([[2.1e-4, 0, 0], [0, 0, 0]]), ref)[0]
    assert not G.check_rows(ref + np.array([[0, 0, 0], [1e-20, 0, 0]]), ref)[0]   # zero row: exact
    assert not G.check_rows(np.array([[np.nan, -2.0, 0.0], [0, 0, 0]]), ref)[0]
