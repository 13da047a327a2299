"""Split backward (mhcpb_execute_dx + mhcpb_reduce_dw) and accumulation of dW
into the caller's buffer (MHCPB_ACCUMULATE_DW).

The split follows the split backward of the prime-kernels PR #15 (the input
gradient is produced before the weight gradients); the accumulation follows
its option of adding weight gradients into an FP32 buffer the caller owns.  Both must
leave the arithmetic unchanged: the split gives mhcpb_execute's bits, and an
accumulating execute gives exactly fp32(dW_in + D) with D the bits the
non-accumulating execute writes.
"""
import numpy as np
import pytest
import torch

from rms_backward_gb300 import Plan, abi
from rms_backward_gb300 import workloads as WL

from gpu_helpers import assert_parity_full, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _bufs(wl, plan, fill=float("nan")):
    dx = torch.full((wl.T, wl.K), fill, dtype=torch.bfloat16, device=DEV)
    dw = torch.full((24, wl.K), fill, dtype=torch.float32, device=DEV)
    ws = torch.full((plan.workspace_bytes // 4,), fill, dtype=torch.float32, device=DEV)
    return dx, dw, ws


def _fused(wl, i, **flags):
    plan = Plan(wl.T, wl.K, 0, addend=wl.has_addend, **flags)
    dx, dw, ws = _bufs(wl, plan)
    plan.execute(i["x"], i["w"], i["grad_proj"], i["grad_r"], i["r"], dx, dw, ws, addend=i["addend"])
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    plan.close()
    return dx, dw


@pytest.mark.parametrize("fma", [False, True], ids=["tcgen05", "fma"])
@pytest.mark.parametrize("addend", [False, True])
def test_split_equals_fused(fma, addend):
    wl = WL.make("split", T=1100, K=1032, seed=60, addend=addend)
    i = to_dev(wl)
    ref_dx, ref_dw = _fused(wl, i, fma_kernel=fma)
    plan = Plan(wl.T, wl.K, 0, addend=addend, fma_kernel=fma)
    dx, dw, ws = _bufs(wl, plan)
    plan.execute_dx(i["x"], i["w"], i["grad_proj"], i["grad_r"], i["r"], dx, ws, addend=i["addend"])
    torch.cuda.synchronize()
    assert torch.isnan(dw).all()          # nothing has touched dW yet
    assert torch.equal(dx.view(torch.int16), ref_dx.view(torch.int16))
    plan.reduce_dw(ws, dw)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert torch.equal(dw.view(torch.int32), ref_dw.view(torch.int32))
    # and against the oracle, every element of both outputs
    st = assert_parity_full(wl, dx.view(torch.int16).cpu().numpy().view(np.uint16), dw.cpu().numpy(),
                            "split")
    print(f"split fma={fma} addend={addend}: dX {st[0]} dW {st[1]}")
    plan.close()


@pytest.mark.parametrize("accumulate", [False, True])
def test_reduce_dw_twice_on_one_workspace(accumulate):
    """mhcpb_reduce_dw only reads the partials: a second call on the same
    workspace sums the same values again (the same bits, or with
    MHCPB_ACCUMULATE_DW the same D added a second time)."""
    wl = WL.make("twice", T=1600, K=776, seed=65)
    i = to_dev(wl)
    _, d = _fused(wl, i)
    dn = d.cpu().numpy()
    plan = Plan(wl.T, wl.K, 0, accumulate_dw=accumulate)
    dx, dw, ws = _bufs(wl, plan)
    plan.execute_dx(i["x"], i["w"], i["grad_proj"], i["grad_r"], i["r"], dx, ws)
    rng = np.random.default_rng(8)
    dw_in = (rng.standard_normal((24, wl.K)) * 2).astype(np.float32)
    if accumulate:
        dw.copy_(torch.from_numpy(dw_in))
    plan.reduce_dw(ws, dw)
    torch.cuda.synchronize()
    first = dw.cpu().numpy().copy()
    plan.reduce_dw(ws, dw)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    second = dw.cpu().numpy()
    if accumulate:
        want1 = (dw_in + dn).astype(np.float32)
        assert np.array_equal(first.view(np.uint32), want1.view(np.uint32))
        assert np.array_equal(second.view(np.uint32), (want1 + dn).astype(np.float32).view(np.uint32))
    else:
        assert np.array_equal(first.view(np.uint32), dn.view(np.uint32))
        assert np.array_equal(second.view(np.uint32), dn.view(np.uint32))
    plan.close()


def test_split_with_other_work_and_another_stream_between():
    """dX is consumed on the stream (a reduction over it) before the weight
    gradient is reduced on a second stream ordered by an event."""
    wl = WL.make("split", T=2048, K=2048, seed=61)
    i = to_dev(wl)
    ref_dx, ref_dw = _fused(wl, i)
    plan = Plan(wl.T, wl.K, 0)
    dx, dw, ws = _bufs(wl, plan)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        plan.execute_dx(i["x"], i["w"], i["grad_proj"], i["grad_r"], i["r"], dx, ws, stream=s1)
        dx_sum = dx.float().sum()
        done = torch.cuda.Event()
        done.record(s1)
    s2.wait_event(done)
    plan.reduce_dw(ws, dw, stream=s2)
    torch.cuda.synchronize()
    assert torch.equal(dw.view(torch.int32), ref_dw.view(torch.int32))
    assert float(dx_sum) == float(ref_dx.float().sum())
    plan.close()


@pytest.mark.parametrize("compensated", [False, True])
def test_accumulate_adds_exactly_once_rounded(compensated):
    wl = WL.make("acc", T=1500, K=520, seed=62)
    i = to_dev(wl)
    _, d = _fused(wl, i, compensated_dw=compensated)
    d = d.cpu().numpy()
    rng = np.random.default_rng(7)
    dw_in = (rng.standard_normal((24, wl.K)) * 3).astype(np.float32)
    plan = Plan(wl.T, wl.K, 0, compensated_dw=compensated, accumulate_dw=True)
    dx, _, ws = _bufs(wl, plan)
    dw = torch.from_numpy(dw_in.copy()).to(DEV)
    plan.execute(i["x"], i["w"], i["grad_proj"], i["grad_r"], i["r"], dx, dw, ws)
    torch.cuda.synchronize()
    got = dw.cpu().numpy()
    want = (dw_in + d).astype(np.float32)          # numpy float32 add: one IEEE rounding
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # a second accumulating execute adds D again
    plan.execute(i["x"], i["w"], i["grad_proj"], i["grad_r"], i["r"], dx, dw, ws)
    torch.cuda.synchronize()
    assert np.array_equal(dw.cpu().numpy().view(np.uint32), (want + d).astype(np.float32).view(np.uint32))
    # dX does not depend on the flag
    assert_parity_full(wl, dx.view(torch.int16).cpu().numpy().view(np.uint16), d, "accumulate")
    plan.close()


def test_accumulate_through_split_calls_and_graph_replay():
    wl = WL.make("acc", T=777, K=1024, seed=63)
    i = to_dev(wl)
    _, d = _fused(wl, i)
    plan = Plan(wl.T, wl.K, 0, accumulate_dw=True)
    dx, _, ws = _bufs(wl, plan)
    dw = torch.zeros((24, wl.K), dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            plan.execute_dx(i["x"], i["w"], i["grad_proj"], i["grad_r"], i["r"], dx, ws, stream=s)
            plan.reduce_dw(ws, dw, stream=s)
    torch.cuda.synchronize()
    dw.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    dn = d.cpu().numpy()
    want = np.zeros_like(dn)
    for _ in range(3):
        want = (want + dn).astype(np.float32)
    assert np.array_equal(dw.cpu().numpy().view(np.uint32), want.view(np.uint32))
    plan.close()


def test_split_rejections_enqueue_nothing():
    wl = WL.make("rej", T=300, K=520, seed=64)
    i = to_dev(wl)
    plan = Plan(wl.T, wl.K, 0)
    dx, dw, ws = _bufs(wl, plan, fill=7.0)
    h, st = plan.handle, torch.cuda.current_stream().cuda_stream
    cases = [
        (lambda: abi.mhcpb_reduce_dw(h, ws.data_ptr(), plan.workspace_bytes - 16, dw.data_ptr(), st),
         abi.MHCPB_ERR_WORKSPACE_TOO_SMALL),
        (lambda: abi.mhcpb_reduce_dw(h, dw.data_ptr(), plan.workspace_bytes, dw.data_ptr(), st),
         abi.MHCPB_ERR_ALIASING),
        (lambda: abi.mhcpb_reduce_dw(h, ws.data_ptr() + 4, plan.workspace_bytes, dw.data_ptr(), st),
         abi.MHCPB_ERR_MISALIGNED),
        (lambda: abi.mhcpb_execute_dx(h, i["x"].data_ptr(), i["w"].data_ptr(), i["grad_proj"].data_ptr(),
                                      i["grad_r"].data_ptr(), i["r"].data_ptr(), dx.data_ptr(),
                                      ws.data_ptr(), plan.workspace_bytes, i["x"].data_ptr(), st),
         abi.MHCPB_ERR_INVALID_ARG),       # an addend the plan does not expect
        (lambda: abi.mhcpb_execute_dx(h, i["x"].data_ptr(), i["w"].data_ptr(), i["grad_proj"].data_ptr(),
                                      i["grad_r"].data_ptr(), i["r"].data_ptr(), i["x"].data_ptr(),
                                      ws.data_ptr(), plan.workspace_bytes, None, st),
         abi.MHCPB_ERR_ALIASING),          # dx over x
    ]
    for call, status in cases:
        with pytest.raises(abi.MhcpbError) as ei:
            call()
        assert ei.value.status == status
    torch.cuda.synchronize()
    assert bool((dx == 7.0).all()) and bool((dw == 7.0).all())
    plan.close()
