"""Pins of the CPU oracle to facts other than its own formula.

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed operand, a wrong K, reading grad_proj's ignored
columns, double rounding) fails at least one of them; ``test_pins_catch_*``
plant such slips in a copy of the oracle and check that they are caught.

Facts used (cuDNN frontend page "DSv4.1 mHC projection/RMS backward", intro and
"Requirements and tensor contract"): the formula's meaning as the gradient of
the projection and of the forward RMS (finite differences), TF32/BF16 number
formats (hand-checked values, torch's BF16 cast), the BF16 add that autograd
performs (torch's CPU BF16 add), closed forms on structured inputs, the
ignored grad_proj columns, and linearity in (grad_proj, grad_r).
"""
import numpy as np
import pytest
import torch

import oracle.mhcpb_oracle as O
from rms_backward_gb300 import workloads as WL


def f32(x):
    return np.float32(x)


# ---------------------------------------------------------------- TF32 ----
@pytest.mark.parametrize("val,expect", [
    (1.0, 1.0),
    (1.0 + 2.0 ** -10, 1.0 + 2.0 ** -10),           # representable
    (1.0 + 2.0 ** -11, 1.0 + 2.0 ** -10),           # exact tie -> away from zero
    (1.0 + 2.0 ** -11 - 2.0 ** -23, 1.0),           # just below the tie
    (-(1.0 + 2.0 ** -11), -(1.0 + 2.0 ** -10)),     # ties away for negatives too
    (2.0 - 2.0 ** -11, 2.0),                        # carry into the exponent
    (1.0 + 3 * 2.0 ** -12, 1.0 + 2.0 ** -10),       # above the tie
    (3.0 * 2.0 ** -140, 0.0),                       # FP32 subnormal below half a TF32 step
    (0.0, 0.0),
])
def test_tf32_rna_hand_values(val, expect):
    got = O.tf32_rna(np.array([val], dtype=np.float32))[0]
    assert got == np.float32(expect), (val, got, expect)


def test_tf32_rna_overflow_and_specials():
    fmax = np.finfo(np.float32).max
    got = O.tf32_rna(np.array([fmax, -fmax, np.inf, -np.inf, np.nan], dtype=np.float32))
    assert np.isposinf(got[0]) and np.isneginf(got[1])
    assert np.isposinf(got[2]) and np.isneginf(got[3]) and np.isnan(got[4])


def test_tf32_rna_properties_random():
    rng = np.random.default_rng(5)
    a = (rng.standard_normal(100000) * 10.0 ** rng.uniform(-20, 20, 100000)).astype(np.float32)
    t = O.tf32_rna(a)
    # low 13 mantissa bits are clear
    assert not np.any(t.view(np.uint32) & np.uint32(0x1FFF))
    # within half a TF32 place (relative 2**-11) of the input, and idempotent
    rel = np.abs(t.astype(np.float64) - a) / np.abs(a.astype(np.float64))
    assert np.all(rel <= 2.0 ** -11 * (1 + 1e-12))
    assert np.array_equal(O.tf32_rna(t).view(np.uint32), t.view(np.uint32))


# ---------------------------------------------------------------- BF16 ----
def test_bf16_from_f32_matches_torch_cast():
    rng = np.random.default_rng(7)
    a = (rng.standard_normal(200000) * 10.0 ** rng.uniform(-38, 38, 200000)).astype(np.float32)
    a[:6] = [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 3.0e38, 2.0 ** -130]
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_rne_from_f32(a), ref)


@pytest.mark.parametrize("val,bits", [
    (1.0 + 2.0 ** -8, 0x3F80),                   # tie -> even (down)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),               # tie -> even (up)
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),      # above the tie: no FP32 double rounding
    (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
    ((2.0 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),    # midpoint above BF16 max -> inf
    ((2.0 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),    # BF16 max
    (2.0 ** -130, 0x0008),                       # subnormal, exact
    (-0.0, 0x8000),
    (0.0, 0x0000),
])
def test_bf16_from_f64_hand_values(val, bits):
    assert int(O.bf16_rne_from_f64(np.array([val]))[0]) == bits


def test_bf16_addend_matches_torch_bf16_add():
    # The fused addend must equal a separate BF16 tensor add (what autograd does).
    rng = np.random.default_rng(11)
    a = O.bf16_rne_from_f64(rng.standard_normal(50000))
    b = O.bf16_rne_from_f64(rng.standard_normal(50000) * 10.0 ** rng.uniform(-6, 2, 50000))
    ta = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    tb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
    ref = (ta + tb).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.add_bf16_like_autograd(a, b), ref)


# ------------------------------------------------- finite-difference VJP ----
def _loss(X, Wm, G, gr, K, eps):
    """Scalar whose gradient the stage is: projections X W^T weighted by the
    upstream projection gradient, plus the forward RMS weighted by grad_r."""
    proj = np.einsum("tk,jk->tj", X, Wm)
    rms = np.sqrt(np.einsum("tk,tk->t", X, X) / K + eps)
    return float(np.sum(G * proj) + np.dot(gr, rms))


def _tf32_exact_case(T=3, K=16, seed=0):
    rng = np.random.default_rng(seed)
    # dyadic values with few bits: exact in TF32 / BF16, so rounding plays no part
    G = rng.integers(-64, 65, size=(T, 32)).astype(np.float32) / 64
    Wm = rng.integers(-64, 65, size=(24, K)).astype(np.float32) / 128
    X = rng.integers(-32, 33, size=(T, K)).astype(np.float32) / 8
    gr = rng.integers(-16, 17, size=T).astype(np.float32) / 4
    xb = torch.from_numpy(X).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    r = np.sqrt((X.astype(np.float64) ** 2).mean(axis=1) + 1e-6)
    return G, Wm, X, gr, xb, r


def test_vjp_matches_finite_differences_dx():
    T, K = 3, 16
    G, Wm, X, gr, xb, r = _tf32_exact_case(T, K)
    core = O.dx_core_f64(xb, Wm, G, gr, r.astype(np.float32))
    Xd = X.astype(np.float64)
    h = 1e-6
    for t in range(T):
        for k in range(K):
            e = np.zeros_like(Xd)
            e[t, k] = h
            fd = (_loss(Xd + e, Wm[:, :].astype(np.float64), G[:, :24].astype(np.float64), gr, K, 1e-6)
                  - _loss(Xd - e, Wm.astype(np.float64), G[:, :24].astype(np.float64), gr, K, 1e-6)) / (2 * h)
            # r passed to the oracle is the forward's RMS rounded to FP32: relative 2**-24 slack
            assert abs(core[t, k] - fd) <= 1e-7 * (1 + abs(fd)), (t, k, core[t, k], fd)


def test_vjp_matches_finite_differences_dw():
    T, K = 3, 16
    G, Wm, X, gr, xb, r = _tf32_exact_case(T, K, seed=1)
    dw = O.dw_f64(xb, G)
    Xd = X.astype(np.float64)
    Wd = Wm.astype(np.float64)
    h = 1e-6
    for j in range(24):
        for k in range(0, K, 3):
            e = np.zeros_like(Wd)
            e[j, k] = h
            fd = (_loss(Xd, Wd + e, G[:, :24].astype(np.float64), gr, K, 1e-6)
                  - _loss(Xd, Wd - e, G[:, :24].astype(np.float64), gr, K, 1e-6)) / (2 * h)
            assert abs(dw[j, k] - fd) <= 1e-7 * (1 + abs(fd)), (j, k, dw[j, k], fd)


# ---------------------------------------------------------- closed forms ----
def test_closed_form_structured_inputs():
    """W[j,k] = 1 where k == j mod K: (P W)[t,k] = sum of P[t,j] over j == k mod K.
    X[t,k] = a[t] b[k]: dW[j,k] = b[k] * sum_t a[t] P[t,j].
    r = 4, K = 16, grad_r = 64 s: the RMS coefficient is exactly s."""
    T, K = 5, 16
    rng = np.random.default_rng(3)
    P = rng.integers(-8, 9, size=(T, 32)).astype(np.float32)
    W = np.zeros((24, K), np.float32)
    for j in range(24):
        W[j, j % K] = 1.0
    a = np.array([1, -2, 3, 0, 1], np.float32)
    b = np.arange(1, K + 1, dtype=np.float32) - 8
    X = np.outer(a, b).astype(np.float32)
    xb = torch.from_numpy(X).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    s = np.array([0.5, -1.0, 0.25, 2.0, 0.0], np.float32)
    r = np.full(T, 4.0, np.float32)
    gr = (64.0 * s).astype(np.float32)
    dx, dw = O.mhc_proj_rms_backward(xb, W, P, gr, r)
    for t in range(T):
        for k in range(K):
            pw = P[t, k] + (P[t, k + 16] if k + 16 < 24 else 0.0)
            expect = pw + s[t] * X[t, k]
            assert O.bf16_bits_to_f64(dx[t, k]) == expect, (t, k)
    for j in range(24):
        for k in range(K):
            assert dw[j, k] == b[k] * float(np.dot(a, P[:, j])), (j, k)


def test_grad_r_zero_reduces_to_matmul():
    wl = WL.make("t", T=33, K=40, seed=21)
    gr0 = np.zeros_like(wl.grad_r)
    core = O.dx_core_f64(wl.x, wl.w, wl.grad_proj, gr0, wl.r)
    Pt = torch.from_numpy(O.tf32_rna(wl.grad_proj[:, :24])).double()
    Wt = torch.from_numpy(O.tf32_rna(wl.w)).double()
    assert np.array_equal(core, (Pt @ Wt).numpy())


def test_p_zero_gives_rms_term_only_and_zero_dw():
    wl = WL.make("t", T=17, K=24, seed=22)
    gp = wl.grad_proj.copy()
    gp[:, :24] = 0
    dx, dw = O.mhc_proj_rms_backward(wl.x, wl.w, gp, wl.grad_r, wl.r)
    assert np.all(dw == 0)
    # each element is one FP64 product of two exact values, rounded once
    X = O.bf16_bits_to_f64(wl.x)
    for t in range(wl.T):
        c = float(wl.grad_r[t]) / (float(wl.r[t]) * wl.K)
        for k in range(wl.K):
            assert int(dx[t, k]) == int(O.bf16_rne_from_f64(np.array([c * X[t, k]]))[0])


def test_dw_cancellation_case_closed_form():
    """The input behind the compensated-reduction pin: the oracle's dW is
    exactly 2**24 + 2 (an FP32 value), its per-chunk sums are exactly 2**24, 1
    and 1, and adding those one FP32 rounding at a time gives 2**24 instead:
    the case separates a once-rounded sum from a sequential FP32 one."""
    wl = WL.make_dw_cancellation(K=16, seed=5)
    dw = O.dw_f64(wl.x, wl.grad_proj)
    assert np.all(dw == 2.0 ** 24 + 2)
    assert np.all(dw.astype(np.float32) == np.float32(16777218.0))
    chunks = [O.dw_f64(wl.x[s * 512:(s + 1) * 512], wl.grad_proj[s * 512:(s + 1) * 512])
              for s in range(3)]
    assert [float(c[0, 0]) for c in chunks] == [2.0 ** 24, 1.0, 1.0]
    seq = np.float32(chunks[0][0, 0])
    for c in chunks[1:]:
        seq = np.float32(seq + np.float32(c[0, 0]))
    assert seq == np.float32(2.0 ** 24)
    # dX is the plain product (grad_r = 0): bf16(P @ W) on the three rows, 0 elsewhere
    dx, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    assert np.all(dx[1:512] == 0) and np.any(dx[0] != 0)


def test_ignored_grad_proj_columns():
    wl = WL.make("t", T=19, K=32, seed=23)
    ref = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    for fill in (1e30, -1e30, np.nan, np.inf):
        gp = wl.grad_proj.copy()
        gp[:, 24:] = fill
        got = O.mhc_proj_rms_backward(wl.x, wl.w, gp, wl.grad_r, wl.r)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_linearity_in_grad_proj_and_grad_r():
    T, K = 6, 16
    G1, Wm, X, g1, xb, r = _tf32_exact_case(T, K, seed=4)
    G2, _, _, g2, _, _ = _tf32_exact_case(T, K, seed=5)
    r = np.full(T, 2.0, np.float32)  # power of two: the coefficient stays exact
    a, b = np.float32(2.0), np.float32(-0.75)
    core12 = O.dx_core_f64(xb, Wm, a * G1 + b * G2, a * g1 + b * g2, r)
    core1 = O.dx_core_f64(xb, Wm, G1, g1, r)
    core2 = O.dx_core_f64(xb, Wm, G2, g2, r)
    assert np.array_equal(core12, float(a) * core1 + float(b) * core2)
    dw12 = O.dw_f64(xb, a * G1 + b * G2)
    assert np.array_equal(dw12, float(a) * O.dw_f64(xb, G1) + float(b) * O.dw_f64(xb, G2))


def test_sampled_rows_and_cols_match_full():
    wl = WL.make("t", T=70, K=48, seed=24)
    dx, dw = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    rows = np.array([0, 5, 69])
    dxs, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, rows=rows)
    assert np.array_equal(dxs, dx[rows])
    cols = np.array([1, 2, 47])
    assert np.array_equal(O.dw_f64(wl.x, wl.grad_proj, cols=cols).astype(np.float32), dw[:, cols])


def test_tolerance_check_accepts_self_and_rejects_one_off():
    wl = WL.make("t", T=16, K=64, seed=25)
    dx, dw = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    bound = O.dx_abs_bound(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    ok, st = O.check_dx(dx, dx, bound)
    assert ok and st["exact"] == dx.size
    bad = dx.copy()
    bad[3, 7] = (int(bad[3, 7]) + 3) & 0xFFFF   # 3 ulps off
    ok, st = O.check_dx(bad, dx, np.zeros_like(bound))
    assert not ok and st["fail"] == 1
    ref = O.dw_f64(wl.x, wl.grad_proj)
    wb = O.dw_abs_bound(wl.x, wl.grad_proj)
    assert O.check_dw(dw, ref, wb)[0]
    dw_bad = dw.copy()
    dw_bad[2, 2] += 2e-3 * wb[2, 2]
    assert not O.check_dw(dw_bad, ref, wb)[0]


# ------------------------------------------- planted mistakes are caught ----
def _fd_dx_ok(core_fn):
    T, K = 3, 16
    G, Wm, X, gr, xb, r = _tf32_exact_case(T, K, seed=9)
    core = core_fn(xb, Wm, G, gr, r.astype(np.float32))
    Xd = X.astype(np.float64)
    h = 1e-6
    for t in range(T):
        for k in range(K):
            e = np.zeros_like(Xd)
            e[t, k] = h
            fd = (_loss(Xd + e, Wm.astype(np.float64), G[:, :24].astype(np.float64), gr, K, 1e-6)
                  - _loss(Xd - e, Wm.astype(np.float64), G[:, :24].astype(np.float64), gr, K, 1e-6)) / (2 * h)
            if abs(core[t, k] - fd) > 1e-7 * (1 + abs(fd)):
                return False
    return True


def test_pins_catch_planted_mistakes():
    def dropped_rms(xb, w, gp, g, r):
        return O.dx_core_f64(xb, w, gp, np.zeros_like(g), r)

    def wrong_sign(xb, w, gp, g, r):
        return O.dx_core_f64(xb, w, gp, -g, r)

    def wrong_k(xb, w, gp, g, r):   # hidden size instead of the full row width
        return O.dx_core_f64(xb, w, gp, g * 4, r)

    def shifted_cols(xb, w, gp, g, r):   # reads grad_proj[:, 8:32]
        return O.dx_core_f64(xb, w, np.ascontiguousarray(gp[:, 8:]), g, r)

    assert _fd_dx_ok(O.dx_core_f64)
    for bad in (dropped_rms, wrong_sign, wrong_k, shifted_cols):
        assert not _fd_dx_ok(bad), bad.__name__


# ------------------------------------------------------- frozen fixture ----
def test_oracle_reproduces_frozen_fixture():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_T8_K16.txt")
    rec = {}
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        key, *vals = line.split()
        rec[key] = np.array([int(v, 16) for v in vals], dtype=np.uint64)
    wl = WL.make("golden", T=8, K=16, seed=1234, addend=True)
    dx, dw = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    dxa, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, addend_bits=wl.addend)
    assert np.array_equal(dx.reshape(-1).astype(np.uint64), rec["dx"])
    assert np.array_equal(dxa.reshape(-1).astype(np.uint64), rec["dx_addend"])
    assert np.array_equal(dw.view(np.uint32).reshape(-1).astype(np.uint64), rec["dw"])
