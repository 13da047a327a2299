"""The tensor contract on a GPU (cuDNN frontend page "DSv4.1 mHC
projection/RMS backward", "Requirements and tensor contract"): operands on one
device, disjoint, 16-byte aligned, enough workspace; anything else is rejected
with a status and nothing is enqueued."""
import numpy as np
import pytest
import torch

from rms_backward_gb300 import abi, Plan

pytestmark = pytest.mark.gpu

T, K = 300, 520


def _bufs(addend=False):
    dev = "cuda:0"
    b = dict(
        x=torch.randn(T, K, device=dev).to(torch.bfloat16),
        w=torch.randn(24, K, device=dev),
        gp=torch.randn(T, 32, device=dev),
        gr=torch.randn(T, device=dev),
        r=torch.rand(T, device=dev) + 0.5,
        dx=torch.full((T, K), 7.0, device=dev, dtype=torch.bfloat16),
        dw=torch.full((24, K), 7.0, device=dev),
    )
    b["add"] = torch.randn(T, K, device=dev).to(torch.bfloat16) if addend else None
    return b


def _exec(plan, b, wsbuf, **over):
    args = dict(x=b["x"].data_ptr(), w=b["w"].data_ptr(), gp=b["gp"].data_ptr(),
                gr=b["gr"].data_ptr(), r=b["r"].data_ptr(), dx=b["dx"].data_ptr(),
                dw=b["dw"].data_ptr(), ws=wsbuf.data_ptr(), wsb=wsbuf.numel(),
                add=None if b["add"] is None else b["add"].data_ptr())
    args.update(over)
    abi.mhcpb_execute(plan.handle, args["x"], args["w"], args["gp"], args["gr"], args["r"],
                      args["dx"], args["dw"], args["ws"], args["wsb"], args["add"],
                      torch.cuda.current_stream().cuda_stream)


def _untouched(b):
    torch.cuda.synchronize()
    return bool((b["dx"] == 7.0).all()) and bool((b["dw"] == 7.0).all())


@pytest.mark.parametrize("case,status", [
    ("misaligned_x", abi.MHCPB_ERR_MISALIGNED),
    ("misaligned_dw", abi.MHCPB_ERR_MISALIGNED),
    ("alias_dx_x", abi.MHCPB_ERR_ALIASING),
    ("alias_ws_dw", abi.MHCPB_ERR_ALIASING),
    ("host_pointer", abi.MHCPB_ERR_WRONG_DEVICE),
    ("small_workspace", abi.MHCPB_ERR_WORKSPACE_TOO_SMALL),
    ("unexpected_addend", abi.MHCPB_ERR_INVALID_ARG),
    ("null_x", abi.MHCPB_ERR_INVALID_ARG),
])
def test_rejections_enqueue_nothing(case, status):
    plan = Plan(T, K)
    b = _bufs()
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda:0")
    big = torch.zeros(T * K * 4 + 64, dtype=torch.uint8, device="cuda:0")
    host = torch.zeros(T * K * 2, dtype=torch.uint8).pin_memory()
    over = {
        "misaligned_x": dict(x=big.data_ptr() + 2),
        "misaligned_dw": dict(dw=b["dw"].data_ptr() + 4),
        "alias_dx_x": dict(dx=b["x"].data_ptr()),
        "alias_ws_dw": dict(ws=b["dw"].data_ptr()),
        "host_pointer": dict(x=host.data_ptr()),
        "small_workspace": dict(wsb=plan.workspace_bytes - 16),
        "unexpected_addend": dict(add=big.data_ptr()),
        "null_x": dict(x=None),
    }[case]
    with pytest.raises(abi.MhcpbError) as ei:
        _exec(plan, b, ws, **over)
    assert ei.value.status == status
    assert _untouched(b)
    plan.close()


def test_missing_addend_rejected():
    plan = Plan(T, K, addend=True)
    b = _bufs(addend=False)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda:0")
    with pytest.raises(abi.MhcpbError) as ei:
        _exec(plan, b, ws)
    assert ei.value.status == abi.MHCPB_ERR_INVALID_ARG
    assert _untouched(b)
    plan.close()


def test_plan_facts():
    plan = Plan(4096, 20480)
    assert plan.workspace_bytes == 15_728_640
    assert plan.query("S") == 8
    assert plan.query("partial_tokens") == 512
    assert plan.query("grid") == min(torch.cuda.get_device_properties(0).multi_processor_count,
                                     160 * 8)
    assert plan.query("smem") <= 232448
    plan.close()
    plan = Plan(16384, 20480)
    assert plan.query("S") == 32 and plan.query("partial_tokens") == 512
    plan.close()


def test_device_status_clear_after_good_runs():
    plan = Plan(T, K)
    b = _bufs()
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda:0")
    _exec(plan, b, ws)
    assert plan.device_status(clear=True) == abi.MHCPB_OK
    plan.close()
