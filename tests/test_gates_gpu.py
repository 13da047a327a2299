"""GPU parity of the gate/normalisation step (mhcpb_gate_forward,
mhcpb_gate_backward) against its FP64 oracle (oracle/mhcg_oracle.py), and the
chain gate backward -> projection/RMS backward.

Tolerance (stated with the oracle): every output within 1e-4 of its token's
largest magnitude of the exact values (FP32 iterations; see check_rows)."""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.mhcg_oracle as G
import oracle.mhcpb_oracle as O
from rms_backward_gb300 import abi, mhc_gate_backward, mhc_gate_forward
from rms_backward_gb300 import workloads as WL

from gpu_helpers import assert_parity_full, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _dev(wl):
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    return dict(proj=f(wl.proj), r=f(wl.r), alpha=f(wl.alpha), bias=f(wl.bias), gh=f(wl.grad_h))


def _fwd(wl, n_iter):
    d = _dev(wl)
    h = torch.full((wl.T, 24), float("nan"), dtype=torch.float32, device=DEV)
    mhc_gate_forward(d["proj"], d["r"], d["alpha"], d["bias"], h, n_iter=n_iter)
    torch.cuda.synchronize()
    return h.cpu().numpy()


def _bwd(wl, n_iter):
    d = _dev(wl)
    gp = torch.full((wl.T, 32), float("nan"), dtype=torch.float32, device=DEV)
    gr = torch.full((wl.T,), float("nan"), dtype=torch.float32, device=DEV)
    dl = torch.full((wl.T, 24), float("nan"), dtype=torch.float32, device=DEV)
    mhc_gate_backward(d["proj"], d["r"], d["alpha"], d["bias"], d["gh"], gp, gr, dl, n_iter=n_iter)
    torch.cuda.synchronize()
    return gp.cpu().numpy(), gr.cpu().numpy(), dl.cpu().numpy()


SHAPES = [(1, 20), (15, 20), (17, 1), (1000, 2), (4096, 20), (4096, 64), (100003, 20)]


@pytest.mark.parametrize("T,n_iter", SHAPES)
def test_gate_forward_matches_oracle(T, n_iter):
    wl = WL.make_gates("gf", T=T, seed=200 + T + n_iter)
    got = _fwd(wl, n_iter)
    ref = G.gate_forward(wl.proj, wl.r, wl.alpha, wl.bias, n_iter)
    ok, st = G.check_rows(got, ref)
    print(f"gate forward T={T} n_iter={n_iter}: {st}")
    assert ok, st


@pytest.mark.parametrize("T,n_iter", SHAPES)
def test_gate_backward_matches_oracle(T, n_iter):
    wl = WL.make_gates("gb", T=T, seed=300 + T + n_iter)
    gp, gr, dl = _bwd(wl, n_iter)
    rgp, rgr, rdl = G.gate_backward(wl.proj, wl.r, wl.alpha, wl.bias, wl.grad_h, n_iter)
    assert np.all(gp[:, 24:] == 0)
    for name, got, ref in (("grad_proj", gp[:, :24], rgp[:, :24]), ("dlogits", dl, rdl)):
        ok, st = G.check_rows(got, ref)
        print(f"gate backward T={T} n_iter={n_iter} {name}: {st}")
        assert ok, (name, st)
    # grad_r: one value per token, a sum of 24 terms of either sign; held to
    # 1e-4 of the sum of the terms' magnitudes
    a = G.alpha_per_column(wl.alpha)
    mag = np.abs(rdl * a[None, :] * wl.proj[:, :24].astype(np.float64)).sum(1) / wl.r.astype(np.float64) ** 2
    assert np.all(np.abs(gr - rgr) <= 1e-4 * mag + 1e-30), np.max(np.abs(gr - rgr) / (mag + 1e-30))


def test_gate_forward_hand_worked_sinkhorn():
    path = os.path.join(os.path.dirname(__file__), "golden", "sinkhorn_hand.txt")
    proj = np.zeros((1, 32), np.float32)
    proj[0, 8 + 15] = np.float32(np.log(5.0))
    wl = WL.GateWorkload("hand", 1, 0, proj, np.ones(1, np.float32), np.ones(3, np.float32),
                         np.zeros(24, np.float32), np.zeros((1, 24), np.float32))
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        n, *vals = line.split()
        want = np.array([float(Fraction(v)) for v in vals])
        got = _fwd(wl, int(n))[0, 8:24]
        assert np.allclose(got, want, rtol=2e-6, atol=0), (n, got, want)
        assert np.all(_fwd(wl, int(n))[0, 0:4] == 0.5) and np.all(_fwd(wl, int(n))[0, 4:8] == 1.0)


def test_gate_backward_bitwise_reproducible_and_unused_columns_ignored():
    wl = WL.make_gates("rep", T=5000, seed=7)
    a = _bwd(wl, 20)
    wl.proj[:, 24:] = np.nan
    b = _bwd(wl, 20)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def test_gate_rejections_write_nothing():
    wl = WL.make_gates("rej", T=64, seed=8)
    d = _dev(wl)
    gp = torch.full((64, 32), 7.0, device=DEV)
    gr = torch.full((64,), 7.0, device=DEV)
    st = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()  # noqa: E731
    host = torch.zeros(64, 32)
    cases = [
        (lambda: abi.mhcpb_gate_backward(64, 0, P(d["proj"]), P(d["r"]), P(d["alpha"]), P(d["bias"]),
                                         P(d["gh"]), P(gp), P(gr), None, st), abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
        (lambda: abi.mhcpb_gate_backward(64, 65, P(d["proj"]), P(d["r"]), P(d["alpha"]), P(d["bias"]),
                                         P(d["gh"]), P(gp), P(gr), None, st), abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
        (lambda: abi.mhcpb_gate_backward(-1, 20, P(d["proj"]), P(d["r"]), P(d["alpha"]), P(d["bias"]),
                                         P(d["gh"]), P(gp), P(gr), None, st), abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
        (lambda: abi.mhcpb_gate_backward(64, 20, P(d["proj"]) + 2, P(d["r"]), P(d["alpha"]), P(d["bias"]),
                                         P(d["gh"]), P(gp), P(gr), None, st), abi.MHCPB_ERR_MISALIGNED),
        (lambda: abi.mhcpb_gate_backward(64, 20, P(d["proj"]), P(d["r"]), P(d["alpha"]), P(d["bias"]),
                                         P(d["gh"]), P(d["proj"]), P(gr), None, st), abi.MHCPB_ERR_ALIASING),
        (lambda: abi.mhcpb_gate_backward(64, 20, P(d["proj"]), P(d["r"]), P(d["alpha"]), P(d["bias"]),
                                         P(d["gh"]), P(gp), P(gp) + 4, None, st), abi.MHCPB_ERR_ALIASING),
        (lambda: abi.mhcpb_gate_backward(64, 20, P(host), P(d["r"]), P(d["alpha"]), P(d["bias"]),
                                         P(d["gh"]), P(gp), P(gr), None, st), abi.MHCPB_ERR_WRONG_DEVICE),
        (lambda: abi.mhcpb_gate_forward(64, 20, P(d["proj"]), P(d["r"]), P(d["alpha"]), P(d["bias"]),
                                        0, st), abi.MHCPB_ERR_INVALID_ARG),
    ]
    for call, status in cases:
        with pytest.raises(abi.MhcpbError) as ei:
            call()
        assert ei.value.status == status
    torch.cuda.synchronize()
    assert bool((gp == 7.0).all()) and bool((gr == 7.0).all())


def test_chain_gate_backward_into_projection_backward():
    """The gate backward's outputs are the projection/RMS backward's inputs as
    they are ([T, 32] grad_proj, [T] grad_r): run both on the GPU and check
    the second against the oracle on the first's outputs, and the first
    against its own oracle."""
    T, K = 1100, 2056
    gw = WL.make_gates("chain", T=T, seed=9)
    gp, gr, _ = _bwd(gw, 20)
    rgp, rgr, _ = G.gate_backward(gw.proj, gw.r, gw.alpha, gw.bias, gw.grad_h, 20)
    assert G.check_rows(gp[:, :24], rgp[:, :24])[0]
    wl = WL.make("chain", T=T, K=K, seed=10)
    wl.grad_proj = gp.astype(np.float32)
    wl.grad_r = gr.astype(np.float32)
    dx, dw = run_gpu(wl)
    st = assert_parity_full(wl, dx, dw, "chain")
    print(f"chain: dX {st[0]} dW {st[1]}")


@pytest.mark.parametrize("scale", [5.0, 20.0, 60.0])
def test_gates_large_logits(scale):
    """Logits far apart (x5: |l| up to 35; x20: 138; x60: 414): exp of the raw
    logits leaves whole columns at 0 in FP32 beyond ~90 apart, which the
    log-domain iterations avoid -- the forward matches the oracle at every
    scale.  The backward through 20 unrolled iterations amplifies FP32
    rounding once the logits span ~100 (an FP32 model of the same steps is off
    by 1e-3 at x10 and completely at x20, while the FP64 map barely moves when
    its inputs are rounded to FP32), so its parity is checked at x5 and only
    its finiteness beyond."""
    wl = WL.make_gates("big", T=999, seed=12)
    wl.proj = (wl.proj * scale).astype(np.float32)
    got = _fwd(wl, 20)
    ok, st = G.check_rows(got, G.gate_forward(wl.proj, wl.r, wl.alpha, wl.bias, 20))
    assert ok, st
    gp, gr, dl = _bwd(wl, 20)
    assert np.all(np.isfinite(gp)) and np.all(np.isfinite(gr)) and np.all(np.isfinite(dl))
    if scale <= 5.0:
        rgp, rgr, rdl = G.gate_backward(wl.proj, wl.r, wl.alpha, wl.bias, wl.grad_h, 20)
        ok, st = G.check_rows(gp[:, :24], rgp[:, :24])
        print(f"large logits x{scale}: grad_proj {st}")
        assert ok, st


def test_gates_nan_stays_in_its_token():
    """A NaN logit poisons its own token's outputs (as in the oracle) and no
    other token's."""
    wl = WL.make_gates("nan", T=64, seed=13)
    wl.proj[5, 10] = np.nan
    got = _fwd(wl, 20)
    ref = G.gate_forward(wl.proj, wl.r, wl.alpha, wl.bias, 20)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    others = np.ones(64, bool)
    others[5] = False
    assert not np.any(np.isnan(got[others]))
    ok, _ = G.check_rows(got[others], ref[others])
    assert ok
