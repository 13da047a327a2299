"""Failure detection without a GPU fault.

Every wait inside the tensor-core kernel is bounded; when one runs out the
kernel records MHCPB_ERR_DEVICE_TIMEOUT in the plan's status word, drains its
own copies and MMAs, frees TMEM and returns.  The test makes a wait run out on
purpose (the MMA issuer waits on a barrier that nothing completes, under a
20 ms limit), reads the status on the host, and checks that the CUDA context
is still usable for a correct backward afterwards.
"""
import numpy as np
import pytest
import torch

from rms_backward_gb300 import Plan, abi
from rms_backward_gb300 import workloads as WL

from gpu_helpers import assert_parity_full, run_gpu, to_dev

pytestmark = pytest.mark.gpu


def test_wait_limit_range_checked():
    plan = Plan(64, 512)
    for bad in (0, 999_999, 60_000_000_001):
        with pytest.raises(abi.MhcpbError) as ei:
            plan.set_wait_limit(bad)
        assert ei.value.status == abi.MHCPB_ERR_INVALID_ARG
    plan.set_wait_limit(5_000_000)
    plan.close()


def test_device_timeout_reported_and_context_survives():
    wl = WL.make("stall", T=700, K=1024, seed=40)
    i = to_dev(wl)
    plan = Plan(wl.T, wl.K, 0, test_inject_stall=True)
    plan.set_wait_limit(20_000_000)
    dx = torch.zeros((wl.T, wl.K), dtype=torch.bfloat16, device="cuda:0")
    dw = torch.zeros((24, wl.K), dtype=torch.float32, device="cuda:0")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda:0")
    plan.execute(i["x"], i["w"], i["grad_proj"], i["grad_r"], i["r"], dx, dw, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == abi.MHCPB_ERR_DEVICE_TIMEOUT
    assert plan.device_status(clear=True) == abi.MHCPB_ERR_DEVICE_TIMEOUT
    assert plan.device_status() == abi.MHCPB_OK
    # a second stalled execute reports again, on the same context
    plan.execute(i["x"], i["w"], i["grad_proj"], i["grad_r"], i["r"], dx, dw, ws)
    torch.cuda.synchronize()
    assert plan.device_status(clear=True) == abi.MHCPB_ERR_DEVICE_TIMEOUT
    plan.close()
    # the context is still good: a normal plan gives the oracle's answer
    dx2, dw2 = run_gpu(wl)
    assert_parity_full(wl, dx2, dw2, "after timeout")
    assert np.isfinite(dw2).all()
