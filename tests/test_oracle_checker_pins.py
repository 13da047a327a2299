"""Pins of the oracle's acceptance functions: the error bounds
(``dx_abs_bound``, ``dw_abs_bound``) and the checks that use them
(``check_dx``, ``check_dw``, ``check_dx_addend``).

Every parity test rests on these tolerances, so each is pinned to something
other than its own formula: hand-computed values on a structured input, the
identity |sum| = sum of |terms| when every term has the same sign, invariance
of a magnitude bound to the signs of its operands, and hand-placed values just
inside and just outside each acceptance limit.  A bound inflated or shrunk by a
constant, a dropped term, a signed instead of an absolute operand, or a check
with the wrong number of places fails at least one test here.

The limits follow from the precision contract of the cuDNN frontend page
"DSv4.1 mHC projection/RMS backward" (intro: TF32 product operands with FP32
sums, dX stored BF16) and, for the fused addend, from prime-kernels PR #15
("FP8 weight cache, split backward, fused mHC stream gradient": the sum is the
BF16 add autograd would do).
"""
import numpy as np

import oracle.mhcpb_oracle as O
from rms_backward_gb300 import workloads as WL


def _bf16(vals):
    """Exact BF16 bit patterns of values that BF16 represents."""
    a = np.asarray(vals, dtype=np.float64)
    bits = O.bf16_rne_from_f64(a)
    assert np.array_equal(O.bf16_bits_to_f64(bits), a), "test value not representable in BF16"
    return bits


def _structured():
    """T = 2, K = 8, every value a short dyadic (exact in TF32 and BF16).

    P row 0 = (1, -2, 0, ...), row 1 = (0.5, 0, 3, 0, ...); W row 0 = 1,
    W row 1 = (-1)**k, W row 2 = k / 4, other rows 0; r = 2 and grad_r =
    (16, -8), so the RMS coefficient grad_r / (r K) is (1, -0.5)."""
    T, K = 2, 8
    gp = np.zeros((T, 32), np.float32)
    gp[0, 0], gp[0, 1] = 1.0, -2.0
    gp[1, 0], gp[1, 2] = 0.5, 3.0
    gp[:, 24:] = 1e30   # ignored columns: must not reach either bound
    w = np.zeros((24, K), np.float32)
    k = np.arange(K)
    w[0] = 1.0
    w[1] = (-1.0) ** k
    w[2] = k / 4.0
    X = np.array([[1, -1, 2, -2, 0.5, -0.5, 4, 0],
                  [2, 2, 2, 2, -2, -2, -2, -2]], np.float64)
    xb = _bf16(X)
    r = np.full(T, 2.0, np.float32)
    gr = np.array([16.0, -8.0], np.float32)
    return xb, w, gp, gr, r


# hand-computed from the definitions in _structured's docstring
#   core[0, k] = 1 - 2 (-1)^k + X[0, k]        bound[0, k] = 1 + 2 + |X[0, k]|
#   core[1, k] = 0.5 + 0.75 k - 0.5 X[1, k]    bound[1, k] = 0.5 + 0.75 k + 0.5 |X[1, k]|
CORE = np.array([[0, 2, 1, 1, -0.5, 2.5, 3, 3],
                 [-0.5, 0.25, 1, 1.75, 4.5, 5.25, 6, 6.75]])
DX_BOUND = np.array([[4, 4, 5, 5, 3.5, 3.5, 7, 3],
                     [1.5, 2.25, 3, 3.75, 4.5, 5.25, 6, 6.75]])
#   dW[0, k] = X[0, k] + 0.5 X[1, k]   dW[1, k] = -2 X[0, k]   dW[2, k] = 3 X[1, k]
DW = np.array([[2, 0, 3, -1, -0.5, -1.5, 3, -1],
               [-2, 2, -4, 4, -1, 1, -8, 0],
               [6, 6, 6, 6, -6, -6, -6, -6]])
DW_BOUND = np.array([[2, 2, 3, 3, 1.5, 1.5, 5, 1],
                     [2, 2, 4, 4, 1, 1, 8, 0],
                     [6, 6, 6, 6, 6, 6, 6, 6]])


# ------------------------------------------------------------ the bounds ----
def test_bounds_hand_values():
    xb, w, gp, gr, r = _structured()
    assert np.array_equal(O.dx_core_f64(xb, w, gp, gr, r), CORE)
    assert np.array_equal(O.dx_abs_bound(xb, w, gp, gr, r), DX_BOUND)
    dw = O.dw_f64(xb, gp)
    assert np.array_equal(dw[:3], DW) and np.all(dw[3:] == 0)
    wb = O.dw_abs_bound(xb, gp)
    assert np.array_equal(wb[:3], DW_BOUND) and np.all(wb[3:] == 0)
    # sampled rows / columns are the same numbers
    assert np.array_equal(O.dx_abs_bound(xb, w, gp, gr, r, rows=np.array([1])), DX_BOUND[1:])
    assert np.array_equal(O.dw_abs_bound(xb, gp, cols=np.array([6, 2]))[:3], DW_BOUND[:, [6, 2]])


def _same_sign_case(seed):
    """Random inputs whose every term of both sums is >= 0: P, W, X, grad_r
    all non-negative.  Then a sum of magnitudes is the magnitude of the sum."""
    wl = WL.make("t", T=21, K=40, seed=seed)
    gp = np.abs(wl.grad_proj)
    w = np.abs(wl.w)
    xb = wl.x & np.uint16(0x7FFF)           # clear the BF16 sign bits
    gr = np.abs(wl.grad_r)
    return xb, w, gp, gr, wl.r


def test_bounds_equal_the_value_when_every_term_is_nonnegative():
    xb, w, gp, gr, r = _same_sign_case(31)
    core = O.dx_core_f64(xb, w, gp, gr, r)
    bound = O.dx_abs_bound(xb, w, gp, gr, r)
    # the same FP64 terms in the same order of a matrix product: equal up to
    # FP64 rounding of the sums, far below anything the checks resolve
    assert np.allclose(bound, core, rtol=1e-14, atol=0)
    dw = O.dw_f64(xb, gp)
    assert np.allclose(O.dw_abs_bound(xb, gp), dw, rtol=1e-14, atol=0)


def test_bounds_ignore_operand_signs_and_dominate_the_value():
    wl = WL.make("t", T=23, K=48, seed=32)
    rng = np.random.default_rng(33)
    base = O.dx_abs_bound(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    wbase = O.dw_abs_bound(wl.x, wl.grad_proj)
    # flip the sign of random entries of every operand
    sgp = np.where(rng.random(wl.grad_proj.shape) < 0.5, -1, 1).astype(np.float32)
    sw = np.where(rng.random(wl.w.shape) < 0.5, -1, 1).astype(np.float32)
    sx = np.where(rng.random(wl.x.shape) < 0.5, 0x8000, 0).astype(np.uint16)
    sgr = np.where(rng.random(wl.grad_r.shape) < 0.5, -1, 1).astype(np.float32)
    flipped = O.dx_abs_bound(wl.x ^ sx, wl.w * sw, wl.grad_proj * sgp, wl.grad_r * sgr, wl.r)
    assert np.allclose(flipped, base, rtol=1e-14, atol=0)
    assert np.allclose(O.dw_abs_bound(wl.x ^ sx, wl.grad_proj * sgp), wbase, rtol=1e-14, atol=0)
    # and never below the magnitude of the value they bound
    core = O.dx_core_f64(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    assert np.all(base >= np.abs(core) * (1 - 1e-14))
    assert np.all(wbase >= np.abs(O.dw_f64(wl.x, wl.grad_proj)) * (1 - 1e-14))


def test_bound_mutants_are_caught():
    """Plausible slips in a bound, planted in copies of it, each fail one of
    the pins above (hand values or the same-sign identity)."""
    xb, w, gp, gr, r = _structured()

    def inflated(*a):
        return 10.0 * O.dx_abs_bound(*a)

    def signed_w(xb_, w_, gp_, gr_, r_):       # |P| W instead of |P| |W|
        P, Wt, c = O._operands(w_, gp_, gr_, r_, xb_.shape[1])
        return np.abs(P) @ Wt + np.abs(c[:, None] * O.bf16_bits_to_f64(xb_))

    def no_rms_term(xb_, w_, gp_, gr_, r_):
        P, Wt, _ = O._operands(w_, gp_, gr_, r_, xb_.shape[1])
        return np.abs(P) @ np.abs(Wt)

    for bad in (inflated, signed_w, no_rms_term):
        assert not np.array_equal(bad(xb, w, gp, gr, r), DX_BOUND), bad.__name__

    def dw_signed_x(xb_, gp_):
        P = np.abs(O.tf32_rna(gp_[:, :24]).astype(np.float64))
        return P.T @ O.bf16_bits_to_f64(xb_)

    assert not np.array_equal(dw_signed_x(xb, gp)[:3], DW_BOUND)
    assert not np.array_equal(0.5 * O.dw_abs_bound(xb, gp)[:3], DW_BOUND)


# ------------------------------------------------------------ check_dx ----
def test_check_dx_cancellation_limit_is_ulp_plus_scaled_bound():
    """ref = 2**-10 (BF16 place 2**-17), bound = 2**9: the absolute clause
    admits |dx - ref| <= 2**-17 + 2**-16 * 2**9 = 2**-7 + 2**-17 and nothing
    further; the two-place clause alone would admit only 2**-16."""
    ref = _bf16([2.0 ** -10])
    bound = np.array([2.0 ** 9])
    ok_hi = _bf16([2.0 ** -10 + 2.0 ** -7])                  # diff 2**-7
    bad_hi = _bf16([2.0 ** -10 + 2.0 ** -7 + 2.0 ** -14])    # next BF16 value up
    ok_lo = _bf16([2.0 ** -10 - 2.0 ** -7])
    bad_lo = _bf16([2.0 ** -10 - 2.0 ** -7 - 2.0 ** -14])
    assert O.check_dx(ok_hi, ref, bound)[0] and O.check_dx(ok_lo, ref, bound)[0]
    assert not O.check_dx(bad_hi, ref, bound)[0] and not O.check_dx(bad_lo, ref, bound)[0]
    # the bound matters: with a bound ten times smaller the accepted value fails
    assert not O.check_dx(ok_hi, ref, bound / 10)[0]


def test_check_dx_two_places_without_cancellation():
    ref = _bf16([1.5])                      # BF16 place 2**-7 at 1.5
    bound = np.array([1.5])                 # no cancellation: 2**-16 * bound is tiny
    assert O.check_dx(_bf16([1.5 + 2 * 2.0 ** -7]), ref, bound)[0]
    assert not O.check_dx(_bf16([1.5 + 3 * 2.0 ** -7]), ref, bound)[0]
    # non-finite values must match exactly
    assert O.check_dx(_bf16([np.inf]), _bf16([np.inf]), bound)[0]
    assert not O.check_dx(_bf16([-np.inf]), _bf16([np.inf]), bound)[0]
    assert not O.check_dx(_bf16([np.inf]), ref, bound)[0]


def test_check_dw_limit_is_relative_to_the_magnitude_sum():
    ref = np.array([[1.0, -3.0]])
    bound = np.array([[1000.0, 4.0]])       # 1e-3 of it: 1.0 and 0.004
    assert O.check_dw(np.array([[2.0, -3.0039]]), ref, bound)[0]
    assert not O.check_dw(np.array([[2.0 + 1e-9, -3.0]]), ref, bound)[0]
    assert not O.check_dw(np.array([[1.0, -3.0041]]), ref, bound)[0]
    assert not O.check_dw(np.array([[np.nan, -3.0]]), ref, bound)[0]


# ----------------------------------------------------- check_dx_addend ----
def test_check_dx_addend_rejects_three_places_without_cancellation():
    """core 2**-5 plus addend 31/32: the sum 1.0 has BF16 place 2**-7 and the
    core's own place is 2**-12, so the limit is two places of the sum."""
    core = _bf16([2.0 ** -5])
    ref = _bf16([1.0])
    cb = np.array([2.0 ** -5])
    assert O.check_dx_addend(_bf16([1.0 + 2 * 2.0 ** -7]), ref, core, cb)[0]
    assert not O.check_dx_addend(_bf16([1.0 + 3 * 2.0 ** -7]), ref, core, cb)[0]
    assert not O.check_dx_addend(_bf16([1.0 - 5 * 2.0 ** -8]), ref, core, cb)[0]


def test_check_dx_addend_cancellation_limit():
    """core 1.0 (place 2**-7), core bound 2**9, sum 2**-10 (place 2**-17): the
    limit is 2 * 2**-7 + 2**-16 * 2**9 + 2**-17 = 3 * 2**-7 + 2**-17."""
    core = _bf16([1.0])
    ref = _bf16([2.0 ** -10])
    cb = np.array([2.0 ** 9])
    assert O.check_dx_addend(_bf16([2.0 ** -10 + 3 * 2.0 ** -7]), ref, core, cb)[0]
    assert not O.check_dx_addend(_bf16([2.0 ** -10 + 3 * 2.0 ** -7 + 2.0 ** -13]), ref, core, cb)[0]
    assert O.check_dx_addend(_bf16([2.0 ** -10 - 3 * 2.0 ** -7]), ref, core, cb)[0]
    assert not O.check_dx_addend(_bf16([2.0 ** -10 - 3 * 2.0 ** -7 - 2.0 ** -13]), ref, core, cb)[0]
    # one place of the core fewer: a value the limit above admits now fails
    assert not O.check_dx_addend(_bf16([2.0 ** -10 + 3 * 2.0 ** -7]), ref, core, cb, ulps=1.0)[0]


def test_check_dx_addend_on_a_workload():
    """A core off by one BF16 place anywhere, then added like autograd,
    passes; a core off by four places where the addend is small does not."""
    wl = WL.make("t", T=24, K=64, seed=34, addend=True)
    # the addend scaled by 2**-6 (exact in BF16 at these magnitudes), so that
    # it is comparable with the core: some sums cancel, some are core-dominated
    addend = O.bf16_rne_from_f64(O.bf16_bits_to_f64(wl.addend) * 2.0 ** -6)
    ref, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, addend_bits=addend)
    core, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, rows=np.arange(wl.T))
    cb = O.dx_abs_bound(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    assert O.check_dx_addend(ref, ref, core, cb)[0]
    rng = np.random.default_rng(35)
    step = rng.integers(-1, 2, size=core.shape).astype(np.int32)
    near = ((core.astype(np.int32) + step) & 0xFFFF).astype(np.uint16)   # +-1 place (same sign)
    ok, st = O.check_dx_addend(O.add_bf16_like_autograd(near, addend), ref, core, cb)
    assert ok, st
    # an element where the core dominates the sum: |addend| < |core| / 64
    c64 = O.bf16_bits_to_f64(core)
    a64 = O.bf16_bits_to_f64(addend)
    idx = np.argwhere((np.abs(a64) < np.abs(c64) / 64) & (c64 != 0))
    assert len(idx) > 0
    t, k = idx[0]
    far = core.copy()
    far[t, k] = (int(core[t, k]) + 4) & 0xFFFF
    ok, st = O.check_dx_addend(O.add_bf16_like_autograd(far, addend), ref, core, cb)
    assert not ok and st["fail"] == 1
