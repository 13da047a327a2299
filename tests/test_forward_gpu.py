"""The forward of the stage (mhcpb_forward) against the forward oracle
(oracle/mhcpf_oracle.py): proj = X W^T over TF32 W and r = sqrt(mean X^2 +
eps), the two outputs whose gradients the backward receives (cuDNN frontend
page "DSv4.1 mHC projection/RMS backward", intro; the prime-kernels PR #15
page's mhc_projection computes both from a single pass over X)."""
import numpy as np
import pytest
import torch

import oracle.mhcpf_oracle as F
import oracle.mhcpb_oracle as O
from rms_backward_gb300 import Plan, abi
from rms_backward_gb300 import workloads as WL

from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_forward(wl, eps=1e-6, cap=0, plan=None):
    own = plan is None
    if own:
        plan = Plan(wl.T, wl.K, 0)
    if cap:
        plan.set_max_ctas(cap)
    x = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).to(DEV)
    w = torch.from_numpy(wl.w).to(DEV)
    proj = torch.full((wl.T, 32), float("nan"), device=DEV)
    r = torch.full((wl.T,), float("nan"), device=DEV)
    ws = torch.full((plan.forward_workspace_bytes // 4,), float("nan"), device=DEV)
    plan.forward(x, w, proj, r, ws, eps=eps)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    if own:
        plan.close()
    return proj.cpu().numpy(), r.cpu().numpy()


def assert_forward_parity(wl, proj, r, rows=None, eps=1e-6, label=""):
    ref_p, ref_r = F.mhc_proj_forward(wl.x, wl.w, eps=eps, rows=rows)
    bound = F.proj_abs_bound(wl.x, wl.w, rows=rows)
    sel = slice(None) if rows is None else np.asarray(rows)
    ok, st = F.check_proj(proj[sel], ref_p, bound)
    assert ok, f"{label} proj: {st}"
    okr, str_ = F.check_r(r[sel], ref_r)
    assert okr, f"{label} r: {str_}"


def test_tiny_config():
    wl = WL.config("tiny")
    assert_forward_parity(wl, *run_forward(wl), label="tiny")


@pytest.mark.parametrize("T,K", [(1, 8), (129, 72), (300, 520), (1000, 1032), (777, 2056), (2048, 4096)])
def test_small_and_ragged_shapes(T, K):
    wl = WL.make("f", T=T, K=K, seed=70 + T)
    assert_forward_parity(wl, *run_forward(wl), label=f"T={T} K={K}")


def test_edge_rows_six_decades():
    wl = WL.make("f", T=1000, K=2048, seed=71, edge="rows")
    assert_forward_parity(wl, *run_forward(wl), label="edge rows")


@pytest.mark.parametrize("name", ["training_profile", "long_sublayer"])
def test_full_size_every_row(name):
    """Every element of proj and r at the full sizes (the oracle works in
    blocks of 1024 rows), with the launch configuration the bench times."""
    wl = WL.config(name)
    proj, r = run_forward(wl)
    assert_forward_parity(wl, proj, r, label=name)
    assert np.all(proj[:, 24:] == 0)


def test_exact_integer_inputs_bitwise():
    """Integer X and dyadic W with few bits: every product and partial sum is
    exact in FP32, so proj must equal the oracle exactly; the squares sum
    exactly too, so r differs from the once-rounded oracle by at most the
    rounding of the FP32 '+ eps' (one ulp)."""
    T, K = 260, 2048
    rng = np.random.default_rng(72)
    X = rng.integers(-8, 9, size=(T, K)).astype(np.float32)
    W = rng.integers(-64, 65, size=(24, K)).astype(np.float32) / 64
    wl = WL.make("f", T=T, K=K, seed=72)
    wl.x = torch.from_numpy(X).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    wl.w = W
    proj, r = run_forward(wl)
    ref_p, ref_r = F.mhc_proj_forward(wl.x, wl.w)
    assert np.array_equal(proj[:, :24], ref_p[:, :24].astype(np.float32))
    ulp = np.spacing(ref_r.astype(np.float32))
    assert np.all(np.abs(r.astype(np.float64) - ref_r) <= ulp)


def test_zero_rows_and_eps():
    wl = WL.make("f", T=200, K=512, seed=73)
    wl.x = wl.x.copy()
    wl.x[5:9] = 0
    for eps in (1e-6, 0.0, 0.25):
        proj, r = run_forward(wl, eps=eps)
        assert np.all(r[5:9] == np.sqrt(np.float32(eps)))
        assert np.all(proj[5:9] == 0)
        assert_forward_parity(wl, proj, r, eps=eps, label=f"eps={eps}")


def test_bitwise_repeatable_and_grid_independent():
    """Kernel 1's unit boundaries depend only on (T, K), and the reduction's
    two layouts sum in the same order: T = 1537 makes 49 blocks of 32 tokens,
    so caps 1 and 5 run the output-thread reduction and caps 77 and none the
    line reduction; every result has the same bits."""
    wl = WL.make("f", T=1537, K=5128, seed=74)
    outs = [run_forward(wl, cap=c) for c in (0, 1, 5, 77, 0)]
    for p, r in outs[1:]:
        assert np.array_equal(p.view(np.uint32), outs[0][0].view(np.uint32))
        assert np.array_equal(r.view(np.uint32), outs[0][1].view(np.uint32))


def test_forward_feeds_the_backward():
    """The forward's r as the backward's input: the backward then matches the
    oracle evaluated with that r (the stages compose)."""
    wl = WL.make("f", T=640, K=1024, seed=75)
    _, r = run_forward(wl)
    wl.r = r.astype(np.float32)
    from gpu_helpers import assert_parity_full, run_gpu
    dx, dw = run_gpu(wl)
    assert_parity_full(wl, dx, dw, "backward on the forward's r")


def test_forward_rejections_write_nothing():
    wl = WL.make("f", T=300, K=520, seed=76)
    plan = Plan(wl.T, wl.K, 0)
    i = to_dev(wl)
    proj = torch.full((wl.T, 32), 7.0, device=DEV)
    r = torch.full((wl.T,), 7.0, device=DEV)
    ws = torch.empty(plan.forward_workspace_bytes // 4, device=DEV)
    h, st = plan.handle, torch.cuda.current_stream().cuda_stream
    x, w = i["x"].data_ptr(), i["w"].data_ptr()
    big = torch.empty(wl.T * wl.K + 64, dtype=torch.bfloat16, device=DEV)
    cases = [
        (dict(eps=float("nan")), abi.MHCPB_ERR_INVALID_ARG),
        (dict(eps=-1.0), abi.MHCPB_ERR_INVALID_ARG),
        (dict(x=big.data_ptr() + 2), abi.MHCPB_ERR_MISALIGNED),
        (dict(proj=x), abi.MHCPB_ERR_ALIASING),
        (dict(wsb=plan.forward_workspace_bytes - 4), abi.MHCPB_ERR_WORKSPACE_TOO_SMALL),
        (dict(r=None), abi.MHCPB_ERR_INVALID_ARG),
    ]
    for over, status in cases:
        a = dict(x=x, w=w, eps=1e-6, proj=proj.data_ptr(), r=r.data_ptr(), ws=ws.data_ptr(),
                 wsb=plan.forward_workspace_bytes)
        a.update(over)
        with pytest.raises(abi.MhcpbError) as ei:
            abi.mhcpb_forward(h, a["x"], a["w"], a["eps"], a["proj"], a["r"], a["ws"], a["wsb"], st)
        assert ei.value.status == status, over
    torch.cuda.synchronize()
    assert bool((proj == 7.0).all()) and bool((r == 7.0).all())
    plan.close()


def test_graph_capture_replay_and_new_inputs():
    """Captured once into a CUDA graph on a side stream, the forward replays
    with the same bits, and picks up new contents of the captured buffers."""
    wl = WL.make("fg", T=1000, K=1032, seed=77)
    wl2 = WL.make("fg2", T=1000, K=1032, seed=78)
    ref_p, ref_r = run_forward(wl)
    ref2_p, ref2_r = run_forward(wl2)
    plan = Plan(wl.T, wl.K, 0)
    x = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).to(DEV)
    w = torch.from_numpy(wl.w).to(DEV)
    proj = torch.full((wl.T, 32), float("nan"), device=DEV)
    r = torch.full((wl.T,), float("nan"), device=DEV)
    ws = torch.full((plan.forward_workspace_bytes // 4,), float("nan"), device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            plan.forward(x, w, proj, r, ws, stream=s)
    torch.cuda.synchronize()
    for _ in range(3):
        proj.fill_(float("nan"))
        r.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(proj.cpu().numpy().view(np.uint32), ref_p.view(np.uint32))
        assert np.array_equal(r.cpu().numpy().view(np.uint32), ref_r.view(np.uint32))
    x.copy_(torch.from_numpy(wl2.x.view(np.int16)).view(torch.bfloat16))
    w.copy_(torch.from_numpy(wl2.w))
    g.replay()
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert np.array_equal(proj.cpu().numpy().view(np.uint32), ref2_p.view(np.uint32))
    assert np.array_equal(r.cpu().numpy().view(np.uint32), ref2_r.view(np.uint32))
    plan.close()
