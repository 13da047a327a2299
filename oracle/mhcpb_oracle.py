"""CPU oracle for the mHC projection/RMS backward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this module.  The library (``rms_backward_gb300``) never does: it
has no CPU fallback.  Nothing here is shared with the CUDA path.

What is computed (cuDNN frontend page "DSv4.1 mHC projection/RMS backward",
intro):

    P  = grad_proj[:, :24]
    dX = P @ W + grad_r / (r * K) * X
    dW = P.T @ X

Precision contract from the same passage: both matrix products take operands
rounded to TF32 with FP32 sums; the RMS term is computed in FP32; dX is
stored BF16 and dW FP32.  The oracle evaluates the exact value of that
definition in FP64 over the TF32-rounded product operands (X is BF16, a subset
of TF32, so it needs no rounding), then rounds once: dX to BF16
(round-to-nearest-even), dW to FP32 (round-to-nearest-even).  FP64 is exact for
every product and far more accurate than FP32 for the sums, so the oracle is
the mathematical target the GPU's FP32 accumulation approximates.

Readings where the page is silent (listed with reasons in the design notes):
  * TF32 conversion rounds to nearest with ties away from zero, keeping 10
    explicit mantissa bits.
  * K in the RMS coefficient is the full row width (n_streams * hidden).
  * With the fused BF16 ``grad_x_addend`` (prime-kernels PR #15, "FP8 weight
    cache, split backward, fused mHC stream gradient": the sum must be the one
    autograd computes), dX = bf16(fp32(bf16(core)) + fp32(addend)): the two
    BF16 tensors are added in FP32 and rounded to BF16, as a separate BF16 add
    would.

Parity pins (tests/test_oracle_pins.py): finite-difference VJP of the scalar
loss whose gradient the formula is, closed forms on structured inputs,
library routines for the BF16 conversion and the BF16 add, hand-checked TF32
and BF16 rounding values, invariance to grad_proj[:, 24:32], linearity.  The
one part with no pin is the exact dW bits of the page's own fixed reduction
order, which no page prints (tolerance parity only).
"""
from __future__ import annotations

import numpy as np

N_PROJ = 24


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------
def tf32_rna(a) -> np.ndarray:
    """Round FP32 values to TF32 (1 sign, 8 exponent, 10 mantissa bits),
    nearest with ties away from zero; result returned as FP32.

    Written from the definition: the 13 dropped mantissa bits are rounded away
    by adding half of the kept last place (0x1000) to the magnitude and
    clearing them; a carry into the exponent field is the correct rounding up
    (to the next binade or to infinity).  NaN and infinity pass through.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32)
    finite = np.isfinite(a)
    out = np.where(finite, (bits + np.uint32(0x1000)) & np.uint32(0xFFFFE000), bits)
    return out.astype(np.uint32).view(np.float32)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> exact FP64 values."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_rne_from_f64(v) -> np.ndarray:
    """Round FP64 values straight to BF16 (8 significant bits, FP32 exponent
    range), nearest-even, with no intermediate FP32 rounding; returns uint16.

    For finite v: the last kept place is ulp = 2**(max(e, -126) - 7) where
    2**e <= |v| < 2**(e+1) (below 2**-126 the spacing stays that of the
    smallest binade: BF16 subnormals).  v / ulp is exact in FP64 (a power-of-2
    scale) and ``np.rint`` rounds half to even.  Results at or above 2**128
    overflow to infinity.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    flat_v = v.reshape(-1)
    flat_o = out.reshape(-1)
    nan = np.isnan(flat_v)
    inf = np.isinf(flat_v)
    fin = ~(nan | inf)
    vf = flat_v[fin]
    mag = np.abs(vf)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
    # guard the log2 floor against its own rounding at binade edges
    e = np.where(np.exp2(e) > mag, e - 1, e)
    e = np.where(np.exp2(e + 1) <= mag, e + 1, e)
    ulp = np.exp2(np.maximum(e, -126.0) - 7.0)
    q = np.rint(vf / ulp) * ulp
    q32 = np.where(np.abs(q) >= 2.0 ** 128, np.copysign(np.inf, vf), q).astype(np.float32)
    # q is now exactly a BF16 value (or inf): its FP32 encoding has 16 zero low bits
    res = (q32.view(np.uint32) >> 16).astype(np.uint16)
    flat_o[fin] = res
    flat_o[inf] = np.where(flat_v[inf] > 0, 0x7F80, 0xFF80).astype(np.uint16)
    flat_o[nan] = 0x7FC0
    return out


def bf16_rne_from_f32(v) -> np.ndarray:
    """FP32 -> BF16 nearest-even (every FP32 value is exact in FP64)."""
    return bf16_rne_from_f64(np.asarray(v, dtype=np.float32).astype(np.float64))


# --------------------------------------------------------------------------
# The stage
# --------------------------------------------------------------------------
def _operands(w, grad_proj, grad_r, r, K):
    """TF32-rounded product operands in FP64 and the FP64 row coefficient.

    Only grad_proj[:, :24] is read: the page states the last 8 columns are
    ignored even when nonzero.
    """
    P = tf32_rna(np.asarray(grad_proj, dtype=np.float32)[:, :N_PROJ]).astype(np.float64)
    Wt = tf32_rna(np.asarray(w, dtype=np.float32)).astype(np.float64)
    c = np.asarray(grad_r, dtype=np.float32).astype(np.float64) / (
        np.asarray(r, dtype=np.float32).astype(np.float64) * float(K))
    return P, Wt, c


def dx_core_f64(x_bits, w, grad_proj, grad_r, r, rows=None) -> np.ndarray:
    """Unrounded dX = P @ W + grad_r / (r K) * X in FP64 (TF32 product operands).

    ``rows`` restricts the computation to those token rows (sampled parity at
    full size).
    """
    x_bits = np.asarray(x_bits)
    K = x_bits.shape[1]
    P, Wt, c = _operands(w, grad_proj, grad_r, r, K)
    if rows is not None:
        rows = np.asarray(rows)
        P, c, x_bits = P[rows], c[rows], x_bits[rows]
    X = bf16_bits_to_f64(x_bits)
    return P @ Wt + c[:, None] * X


def dw_f64(x_bits, grad_proj, cols=None, row_block=2048) -> np.ndarray:
    """Unrounded dW = P.T @ X in FP64 (TF32 P; X exact), summed over every
    token.  ``cols`` restricts to those columns of dW.  Processed in token
    blocks so the FP64 copy of X stays small."""
    x_bits = np.asarray(x_bits)
    T, K = x_bits.shape
    P = tf32_rna(np.asarray(grad_proj, dtype=np.float32)[:, :N_PROJ]).astype(np.float64)
    ncols = K if cols is None else len(cols)
    acc = np.zeros((N_PROJ, ncols), dtype=np.float64)
    for t0 in range(0, T, row_block):
        xb = x_bits[t0:t0 + row_block]
        if cols is not None:
            xb = xb[:, np.asarray(cols)]
        acc += P[t0:t0 + row_block].T @ bf16_bits_to_f64(xb)
    return acc


def add_bf16_like_autograd(core_bits, addend_bits) -> np.ndarray:
    """bf16(fp32(a) + fp32(b)) for two BF16 tensors: what a separate BF16
    tensor add computes (the fused addend must match it bit for bit)."""
    s = bf16_bits_to_f32(core_bits) + bf16_bits_to_f32(addend_bits)  # FP32 add, RNE
    return bf16_rne_from_f32(s)


def mhc_proj_rms_backward(x_bits, w, grad_proj, grad_r, r, addend_bits=None,
                          rows=None):
    """Oracle of the whole stage.

    Returns (dx_bits uint16 [T or len(rows), K], dw float32 [24, K]).
    With ``rows`` given, dX is computed for those rows only and dW is None
    (use :func:`dw_f64` with ``cols`` for sampled dW).
    """
    core = dx_core_f64(x_bits, w, grad_proj, grad_r, r, rows=rows)
    dx = bf16_rne_from_f64(core)
    if addend_bits is not None:
        add = np.asarray(addend_bits)
        if rows is not None:
            add = add[np.asarray(rows)]
        dx = add_bf16_like_autograd(dx, add)
    if rows is not None:
        return dx, None
    dw = dw_f64(x_bits, grad_proj).astype(np.float32)
    return dx, dw


# --------------------------------------------------------------------------
# Tolerances the CUDA path is held to (error bounds of FP32 accumulation)
# --------------------------------------------------------------------------
def bf16_ulp(v) -> np.ndarray:
    """Spacing of BF16 values at |v| (smallest-binade spacing below 2**-126)."""
    mag = np.abs(np.asarray(v, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(mag > 0, mag, 2.0 ** -126)))
    return np.exp2(np.maximum(e, -126.0) - 7.0)


def dx_abs_bound(x_bits, w, grad_proj, grad_r, r, rows=None) -> np.ndarray:
    """Sum of magnitudes sum_j |P||W| + |c x| per dX element: FP32 evaluation
    of dX differs from the exact value by a small multiple of 2**-24 of it."""
    x_bits = np.asarray(x_bits)
    K = x_bits.shape[1]
    P, Wt, c = _operands(w, grad_proj, grad_r, r, K)
    if rows is not None:
        rows = np.asarray(rows)
        P, c, x_bits = P[rows], c[rows], x_bits[rows]
    return np.abs(P) @ np.abs(Wt) + np.abs(c[:, None] * bf16_bits_to_f64(x_bits))


def dw_abs_bound(x_bits, grad_proj, cols=None) -> np.ndarray:
    """sum_t |P[t,j]| |X[t,k]| per dW element."""
    x_bits = np.asarray(x_bits)
    T, K = x_bits.shape
    P = np.abs(tf32_rna(np.asarray(grad_proj, dtype=np.float32)[:, :N_PROJ]).astype(np.float64))
    ncols = K if cols is None else len(cols)
    acc = np.zeros((N_PROJ, ncols), dtype=np.float64)
    for t0 in range(0, T, 2048):
        xb = x_bits[t0:t0 + 2048]
        if cols is not None:
            xb = xb[:, np.asarray(cols)]
        acc += P[t0:t0 + 2048].T @ np.abs(bf16_bits_to_f64(xb))
    return acc


def check_dx(dx_bits, ref_bits, abs_bound, ulps=2.0, rel_abs=2.0 ** -16):
    """Element-wise dX acceptance.

    An element passes when |dx - ref| <= ulps * ulp_bf16(ref), or, where the
    sum cancels, when |dx - ref| <= ulp_bf16(ref) + rel_abs * abs_bound (the
    FP32 accumulation error bound plus the final rounding).  Non-finite
    reference values must match exactly.  Returns (ok, stats dict).
    """
    a = bf16_bits_to_f64(dx_bits)
    b = bf16_bits_to_f64(ref_bits)
    fin = np.isfinite(b)
    same_nonfinite = (~fin) & ((np.isnan(a) & np.isnan(b)) | (a == b))
    diff = np.abs(np.subtract(a, b, out=np.zeros_like(a), where=fin))   # 0 where ref is not finite
    u = bf16_ulp(b)
    pass_ulp = diff <= ulps * u
    pass_abs = diff <= u + rel_abs * np.asarray(abs_bound)
    ok_elem = np.where(fin, (pass_ulp | pass_abs) & np.isfinite(a), same_nonfinite)
    stats = dict(
        n=int(a.size), fail=int((~ok_elem).sum()),
        ulp_pass=int((pass_ulp & fin).sum()),
        abs_only_pass=int((~pass_ulp & pass_abs & fin).sum()),
        exact=int((np.asarray(dx_bits) == np.asarray(ref_bits)).sum()),
        max_ulp=float(np.max(np.where(fin, diff / u, 0.0))) if a.size else 0.0,
    )
    return bool(ok_elem.all()), stats


def check_dw(dw, ref_f64, abs_bound, rel=1e-3):
    """|dw - ref| <= rel * sum_t |P||X| per element (ref in FP64)."""
    dw = np.asarray(dw, dtype=np.float64)
    diff = np.abs(dw - ref_f64)
    lim = rel * np.asarray(abs_bound)
    ok = np.isfinite(dw) & (diff <= lim)
    with np.errstate(divide="ignore", invalid="ignore"):
        worst = float(np.max(np.where(lim > 0, diff / lim, np.where(diff > 0, np.inf, 0.0)))) if dw.size else 0.0
    return bool(ok.all()), dict(n=int(dw.size), fail=int((~ok).sum()), worst_frac_of_tol=worst)


def check_dx_addend(dx_bits, ref_bits, core_ref_bits, core_abs_bound, ulps=2.0,
                    rel_abs=2.0 ** -16):
    """dX acceptance with the fused addend.

    The addend is added after the core is rounded to BF16, so a core that is
    within tolerance of the oracle's core (``ulps`` BF16 places, or the FP32
    accumulation bound under cancellation) moves the sum by at most that much
    plus one rounding of the sum.  An element passes when |dx - ref| is within
    ``ulps`` places of the reference sum, or within
    ulps * ulp(core_ref) + rel_abs * core_abs_bound + ulp(ref).
    """
    a = bf16_bits_to_f64(dx_bits)
    b = bf16_bits_to_f64(ref_bits)
    core = bf16_bits_to_f64(core_ref_bits)
    fin = np.isfinite(b)
    diff = np.abs(np.subtract(a, b, out=np.zeros_like(a), where=fin))   # 0 where ref is not finite
    u = bf16_ulp(b)
    lim = np.maximum(ulps * u, ulps * bf16_ulp(core) + rel_abs * np.asarray(core_abs_bound) + u)
    ok_elem = np.where(fin, (diff <= lim) & np.isfinite(a), (np.isnan(a) & np.isnan(b)) | (a == b))
    within_ulps = diff <= ulps * u
    stats = dict(n=int(a.size), fail=int((~ok_elem).sum()),
                 ulp_pass=int((within_ulps & fin).sum()),
                 abs_only_pass=int((~within_ulps & (diff <= lim) & fin).sum()),
                 exact=int((np.asarray(dx_bits) == np.asarray(ref_bits)).sum()),
                 max_ulp=float(np.max(np.where(fin, diff / u, 0.0))) if a.size else 0.0)
    return bool(ok_elem.all()), stats
