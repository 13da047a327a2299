"""Pins of the forward oracle (oracle/mhcpf_oracle.py) against facts that do
not come from the oracle itself: the backward's formula (the cuDNN frontend
page "DSv4.1 mHC projection/RMS backward", intro) must be the gradient of the
forward's outputs, hand-computed values, closed forms, TF32 rounding of W, and
planted mistakes that each pin catches."""
import numpy as np
import pytest
import torch

import oracle.mhcpb_oracle as O
import oracle.mhcpf_oracle as F


def _bits(X):
    return torch.from_numpy(np.asarray(X, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _dyadic_case(T=3, K=16, seed=0):
    rng = np.random.default_rng(seed)
    P = rng.integers(-64, 65, size=(T, 32)).astype(np.float32) / 64
    W = rng.integers(-64, 65, size=(24, K)).astype(np.float32) / 128
    X = rng.integers(-32, 33, size=(T, K)).astype(np.float32) / 8
    g = rng.integers(-16, 17, size=T).astype(np.float32) / 4
    return P, W, X, g


def _fd_matches_backward(proj_fn, rms_fn, seed=0):
    """Central differences of L(X) = sum P * proj(X) + sum g * r(X), the
    forward under test, against the backward oracle's dX = P W + g/(rK) X."""
    T, K = 3, 16
    P, W, X, g = _dyadic_case(T, K, seed)
    Xd = X.astype(np.float64)
    r = rms_fn(Xd)
    core = O.dx_core_f64(_bits(X), W, P, g, r.astype(np.float32))
    L = lambda Z: float(np.sum(P[:, :24].astype(np.float64) * proj_fn(Z, W)) + np.dot(g, rms_fn(Z)))
    h = 1e-6
    for t in range(T):
        for k in range(K):
            e = np.zeros_like(Xd)
            e[t, k] = h
            fd = (L(Xd + e) - L(Xd - e)) / (2 * h)
            if abs(core[t, k] - fd) > 1e-7 * (1 + abs(fd)):
                return False
    return True


def test_forward_gradient_is_the_backward():
    assert _fd_matches_backward(F.proj_of, F.rms_of, seed=0)
    assert _fd_matches_backward(F.proj_of, F.rms_of, seed=1)


def test_hand_computed_values():
    K = 8
    X = np.array([[1, 2, 3, 4, 5, 6, 7, 8],
                  [-1, 0, 0, 0, 0, 0, 0, 2]], np.float32)
    W = np.zeros((24, K), np.float32)
    W[0, :] = 1.0          # row sums
    W[1, 7] = 0.5          # half of the last column
    W[2, 0] = -2.0
    proj, r = F.mhc_proj_forward(_bits(X), W)
    assert proj[0, 0] == 36 and proj[1, 0] == 1
    assert proj[0, 1] == 4 and proj[1, 1] == 1
    assert proj[0, 2] == -2 and proj[1, 2] == 2
    assert np.all(proj[:, 3:] == 0)
    # sum of squares 204 and 5 over K = 8
    assert r[0] == np.sqrt(204 / 8 + 1e-6) and r[1] == np.sqrt(5 / 8 + 1e-6)


def test_closed_forms_rows_and_one_hot_w():
    K = 64
    X = np.zeros((3, K), np.float32)
    X[0, :] = 0.75          # constant row: r = sqrt(0.75^2 + eps)
    X[2, :] = np.arange(K) / 16
    W = np.zeros((24, K), np.float32)
    for j in range(24):
        W[j, (5 * j) % K] = 1.0     # proj[:, j] picks one column
    proj, r = F.mhc_proj_forward(_bits(X), W)
    assert r[0] == np.sqrt(0.75 ** 2 + 1e-6)
    assert r[1] == np.sqrt(1e-6)    # zero row
    for j in range(24):
        assert np.array_equal(proj[:, j], X[:, (5 * j) % K].astype(np.float64))


def test_w_is_rounded_to_tf32_ties_away():
    K = 16
    X = np.zeros((1, K), np.float32)
    X[0, 0] = 1.0
    W = np.zeros((24, K), np.float32)
    W[0, 0] = 1 + 2 ** -11      # exactly half a TF32 unit above 1: ties away -> 1 + 2**-10
    W[1, 0] = 1 + 2 ** -12      # a quarter unit: rounds down to 1
    W[2, 0] = -(1 + 3 * 2 ** -11)   # 1.5 units: rounds to -(1 + 2 * 2**-10)
    proj, _ = F.mhc_proj_forward(_bits(X), W)
    assert proj[0, 0] == 1 + 2 ** -10
    assert proj[0, 1] == 1.0
    assert proj[0, 2] == -(1 + 2 * 2 ** -10)


def test_projection_is_linear_exactly():
    rng = np.random.default_rng(5)
    K = 32
    W = rng.integers(-64, 65, size=(24, K)).astype(np.float32) / 64
    X1 = rng.integers(-16, 17, size=(4, K)).astype(np.float32) / 4
    X2 = rng.integers(-16, 17, size=(4, K)).astype(np.float32) / 4
    a, b = 3.0, -0.5
    lhs = F.proj_f64(_bits(a * X1 + b * X2), W)
    rhs = a * F.proj_f64(_bits(X1), W) + b * F.proj_f64(_bits(X2), W)
    assert np.array_equal(lhs, rhs)


def test_pins_catch_planted_mistakes():
    def rms_sum_not_mean(Z, eps=1e-6):
        return np.sqrt(np.sum(Z * Z, axis=1) + eps)

    def rms_eps_outside(Z, eps=1e-6):
        return np.sqrt(np.sum(Z * Z, axis=1) / Z.shape[1]) + eps

    def rms_k_plus_one(Z, eps=1e-6):
        return np.sqrt(np.sum(Z * Z, axis=1) / (Z.shape[1] + 1) + eps)

    def proj_reversed_rows(Z, w):
        return F.proj_of(Z, np.ascontiguousarray(np.asarray(w)[::-1]))

    def proj_negated(Z, w):
        return -F.proj_of(Z, w)

    assert _fd_matches_backward(F.proj_of, F.rms_of)
    for p_fn, r_fn in ((F.proj_of, rms_sum_not_mean), (F.proj_of, rms_k_plus_one),
                       (proj_reversed_rows, F.rms_of), (proj_negated, F.rms_of)):
        assert not _fd_matches_backward(p_fn, r_fn), (p_fn.__name__, r_fn.__name__)
    # eps outside the root changes the value, not the gradient: the closed form catches it
    assert rms_eps_outside(np.zeros((1, 8)))[0] != np.sqrt(1e-6)


def test_tolerance_checks_accept_self_and_reject_perturbation():
    from rms_backward_gb300 import workloads as WL
    wl = WL.make("t", T=40, K=256, seed=9)
    proj, r = F.mhc_proj_forward(wl.x, wl.w)
    bound = F.proj_abs_bound(wl.x, wl.w)
    ok, _ = F.check_proj(proj.astype(np.float32), proj, bound)
    assert ok
    bad = proj.astype(np.float32).copy()
    bad[3, 5] += 1e-3 * bound[3, 5]
    assert not F.check_proj(bad, proj, bound)[0]
    bad = proj.astype(np.float32).copy()
    bad[0, 30] = 1e-30
    assert not F.check_proj(bad, proj, bound)[0]
    assert F.check_r(r.astype(np.float32), r)[0]
    assert not F.check_r((r * (1 + 2 ** -12)).astype(np.float32), r)[0]


def test_forward_oracle_reproduces_frozen_fixture():
    """tests/golden/forward_T8_K16.txt holds the forward oracle's output (rounded
    to FP32) on a fixed seeded workload, written by tests/golden/make_golden.py:
    a later change to the oracle's arithmetic shows up here."""
    import os

    from rms_backward_gb300 import workloads as WL
    path = os.path.join(os.path.dirname(__file__), "golden", "forward_T8_K16.txt")
    rec = {}
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        key, *vals = line.split()
        rec[key] = np.array([int(v, 16) for v in vals], dtype=np.uint32)
    wl = WL.make("golden", T=8, K=16, seed=1234, addend=True)
    proj, r = F.mhc_proj_forward(wl.x, wl.w)
    assert np.array_equal(proj.astype(np.float32).view(np.uint32).reshape(-1), rec["proj"])
    assert np.array_equal(r.astype(np.float32).view(np.uint32).reshape(-1), rec["r"])
