"""The forward with the gate step fused into its reduction (mhcpb_forward_gates;
the prime-kernels PR #15 page's mhc_projection fuses the gate activations,
sigmoid and Sinkhorn, into the projection).  Its proj and r are bitwise those
of mhcpb_forward and its h bitwise that of mhcpb_gate_forward on them, at
every T (past the one-wave point too, where the plain forward takes its other
reduction layout), for n_iter from 1 to the maximum, and where the logits are
far enough apart to take the log-domain iterations; h also against the
oracles (the forward's, then the gates')."""
import numpy as np
import pytest
import torch

import oracle.mhcg_oracle as G
import oracle.mhcpf_oracle as F
from rms_backward_gb300 import Plan, abi, mhc_gate_forward
from rms_backward_gb300 import workloads as WL

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _params(seed, scale=1.0):
    rng = np.random.default_rng(seed)
    alpha = (rng.uniform(0.5, 1.5, 3) * scale).astype(np.float32)
    bias = rng.normal(0, 0.5, 24).astype(np.float32)
    return alpha, bias


def _run(wl, alpha, bias, n_iter, eps=1e-6):
    """(fused proj, r, h) and (separate proj, r, h) as numpy."""
    T, K = wl.T, wl.K
    plan = Plan(T, K, 0)
    x = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).to(DEV)
    w = torch.from_numpy(wl.w).to(DEV)
    a, b = torch.from_numpy(alpha).to(DEV), torch.from_numpy(bias).to(DEV)
    ws = torch.empty(plan.forward_workspace_bytes, dtype=torch.uint8, device=DEV)
    nan = lambda *s: torch.full(s, float("nan"), device=DEV)  # noqa: E731
    p1, r1, h1 = nan(T, 32), nan(T), nan(T, 24)
    plan.forward_gates(x, w, a, b, p1, r1, h1, ws, eps=eps, n_iter=n_iter)
    p2, r2, h2 = nan(T, 32), nan(T), nan(T, 24)
    plan.forward(x, w, p2, r2, ws, eps=eps)
    mhc_gate_forward(p2, r2, a, b, h2, n_iter=n_iter)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    plan.close()
    c = lambda t: t.cpu().numpy()  # noqa: E731
    return (c(p1), c(r1), c(h1)), (c(p2), c(r2), c(h2))


def _bits_equal(fused, sep, label):
    for name, u, v in zip(("proj", "r", "h"), fused, sep):
        assert np.array_equal(u.view(np.uint32), v.view(np.uint32)), f"{label}: {name} differs"


@pytest.mark.parametrize("T,K,n_iter", [(1, 8, 20), (17, 72, 1), (129, 520, 20), (1537, 5128, 64),
                                        (4096, 20480, 20), (5000, 2056, 20), (16384, 1024, 7)])
def test_fused_equals_forward_then_gates_bitwise(T, K, n_iter):
    wl = WL.make("fg", T=T, K=K, seed=100 + T)
    alpha, bias = _params(T)
    fused, sep = _run(wl, alpha, bias, n_iter)
    _bits_equal(fused, sep, f"T={T} K={K} n_iter={n_iter}")


@pytest.mark.parametrize("scale", [5.0, 60.0])
def test_fused_equals_separate_with_far_apart_logits(scale):
    """Large alphas spread the logits far enough that some warps take the
    log-domain iterations: the warp-wide choice is the same in both paths."""
    wl = WL.make("fg_far", T=1000, K=2056, seed=7)
    alpha, bias = _params(3, scale)
    fused, sep = _run(wl, alpha, bias, 20)
    _bits_equal(fused, sep, f"alpha x{scale}")


def test_fused_with_a_nan_row():
    """A NaN in one token's X row makes that token's proj, r and gates NaN;
    every other token, including its warp partner, matches the separate path."""
    wl = WL.make("fg_nan", T=300, K=520, seed=8)
    wl.x[37, 5] = 0x7FC0   # BF16 NaN
    alpha, bias = _params(4)
    fused, sep = _run(wl, alpha, bias, 20)
    _bits_equal(fused, sep, "NaN row")
    assert np.isnan(fused[2][37]).all() and not np.isnan(np.delete(fused[2], 37, axis=0)).any()


def test_fused_gates_against_the_oracles():
    wl = WL.make("fg_or", T=777, K=2056, seed=9)
    alpha, bias = _params(5)
    (proj, r, h), _ = _run(wl, alpha, bias, 20)
    ref_p, ref_r = F.mhc_proj_forward(wl.x, wl.w)
    assert F.check_proj(proj, ref_p, F.proj_abs_bound(wl.x, wl.w))[0]
    assert F.check_r(r, ref_r)[0]
    ref_h = G.gate_forward(ref_p.astype(np.float32), ref_r.astype(np.float32), alpha, bias, 20)
    ok, st = G.check_rows(h, ref_h)
    assert ok, st


def test_rejections_write_nothing():
    wl = WL.make("fg_rej", T=64, K=512, seed=10)
    plan = Plan(wl.T, wl.K, 0)
    x = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).to(DEV)
    w = torch.from_numpy(wl.w).to(DEV)
    alpha, bias = (torch.from_numpy(v).to(DEV) for v in _params(6))
    proj = torch.full((64, 32), 7.0, device=DEV)
    r = torch.full((64,), 7.0, device=DEV)
    h = torch.full((64, 24), 7.0, device=DEV)
    ws = torch.empty(plan.forward_workspace_bytes, dtype=torch.uint8, device=DEV)
    st = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()  # noqa: E731
    args = lambda **kw: dict(dict(x=P(x), w=P(w), alpha=P(alpha), bias=P(bias), n_iter=20, proj=P(proj),  # noqa: E731
                                  r=P(r), h=P(h)), **kw)
    cases = [(args(n_iter=0), abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
             (args(n_iter=abi.MHCPB_GATE_MAX_ITER + 1), abi.MHCPB_ERR_UNSUPPORTED_SHAPE),
             (args(alpha=0), abi.MHCPB_ERR_INVALID_ARG),
             (args(h=0), abi.MHCPB_ERR_INVALID_ARG),
             (args(h=P(h) + 2), abi.MHCPB_ERR_MISALIGNED),
             (args(h=P(proj)), abi.MHCPB_ERR_ALIASING),
             (args(bias=P(h) + 4), abi.MHCPB_ERR_ALIASING)]
    for a, status in cases:
        with pytest.raises(abi.MhcpbError) as ei:
            abi.mhcpb_forward_gates(plan.handle, a["x"], a["w"], 1e-6, a["alpha"], a["bias"], a["n_iter"],
                                    a["proj"], a["r"], a["h"], P(ws), plan.forward_workspace_bytes, st)
        assert ei.value.status == status, (a, ei.value.status)
    torch.cuda.synchronize()
    assert bool((proj == 7).all()) and bool((r == 7).all()) and bool((h == 7).all())
    plan.close()


def test_empty_batch():
    plan = Plan(0, 512, 0)
    w = torch.ones((24, 512), device=DEV)
    alpha, bias = (torch.from_numpy(v).to(DEV) for v in _params(11))
    abi.mhcpb_forward_gates(plan.handle, 0, w.data_ptr(), 1e-6, alpha.data_ptr(), bias.data_ptr(), 20,
                            0, 0, 0, 0, 0, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    plan.close()


def test_graph_capture_and_replay_with_new_inputs():
    """Captured once in a CUDA graph, the fused call replays with new input
    values in the same buffers and still equals the two calls bitwise."""
    T, K = 1000, 1032
    wl1, wl2 = WL.make("fg_g1", T=T, K=K, seed=21), WL.make("fg_g2", T=T, K=K, seed=22)
    alpha, bias = (torch.from_numpy(v).to(DEV) for v in _params(12))
    plan = Plan(T, K, 0)
    x = torch.from_numpy(wl1.x.view(np.int16)).view(torch.bfloat16).to(DEV)
    w = torch.from_numpy(wl1.w).to(DEV)
    proj, r, h = torch.empty((T, 32), device=DEV), torch.empty(T, device=DEV), torch.empty((T, 24), device=DEV)
    ws = torch.empty(plan.forward_workspace_bytes, dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.forward_gates(x, w, alpha, bias, proj, r, h, ws, stream=s)   # warm-up outside capture
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            plan.forward_gates(x, w, alpha, bias, proj, r, h, ws, stream=s)
    for wl in (wl2, wl1):
        x.copy_(torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16))
        w.copy_(torch.from_numpy(wl.w))
        g.replay()
        torch.cuda.synchronize()
        a, b = alpha.cpu().numpy(), bias.cpu().numpy()
        _, sep = _run(wl, a, b, 20)
        _bits_equal((proj.cpu().numpy(), r.cpu().numpy(), h.cpu().numpy()), sep, f"graph replay {wl.name}")
    assert plan.device_status() == 0
    plan.close()
