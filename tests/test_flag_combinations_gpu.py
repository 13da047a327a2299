"""Every combination of the plan flags that change the arithmetic (fused
addend, compensated dW reduction, accumulating dW), on both kernels, at a
ragged shape: dX against the oracle element by element (the cuDNN frontend
page "DSv4.1 mHC projection/RMS backward", intro, with the addend folded in
as a separate BF16 add would fold it, prime-kernels PR #15), dW against the
oracle, and the accumulating call equal to fp32(dW_in + D) bit for bit, D
being the same plan's result without accumulation."""
import itertools

import numpy as np
import pytest
import torch

from gpu_helpers import DEV, assert_parity_full, to_dev
from rms_backward_gb300 import Plan
from rms_backward_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

CASES = list(itertools.product([False, True], [False, True], [False, True]))


def _run(wl, inp, dw_in, *, fma, addend, compensated, accumulate):
    plan = Plan(wl.T, wl.K, 0, addend=addend, fma_kernel=fma, compensated_dw=compensated,
                accumulate_dw=accumulate)
    dx = torch.full((wl.T, wl.K), float("nan"), dtype=torch.bfloat16, device=DEV)
    dw = torch.from_numpy(dw_in.copy()).to(DEV)
    ws = torch.full((plan.workspace_bytes // 4,), float("nan"), device=DEV)
    plan.execute(inp["x"], inp["w"], inp["grad_proj"], inp["grad_r"], inp["r"], dx, dw, ws,
                 addend=inp["addend"])
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    plan.close()
    return dx.view(torch.int16).cpu().numpy().view(np.uint16), dw.cpu().numpy()


@pytest.mark.parametrize("fma", [False, True], ids=["tcgen05", "fma"])
@pytest.mark.parametrize("addend,compensated,accumulate", CASES,
                         ids=[f"add{int(a)}-comp{int(c)}-acc{int(u)}" for a, c, u in CASES])
def test_flag_combination(fma, addend, compensated, accumulate):
    wl = WL.make("flags", T=300, K=520, seed=81, addend=addend)
    inp = to_dev(wl)
    nan = np.full((24, wl.K), np.nan, np.float32)
    dx_d, d = _run(wl, inp, nan, fma=fma, addend=addend, compensated=compensated, accumulate=False)
    label = f"fma={fma} addend={addend} compensated={compensated}"
    assert_parity_full(wl, dx_d, d, label)
    if not accumulate:
        return
    dw_in = (np.random.default_rng(5).standard_normal((24, wl.K)) * 2).astype(np.float32)
    dx_a, dw_out = _run(wl, inp, dw_in, fma=fma, addend=addend, compensated=compensated, accumulate=True)
    assert np.array_equal(dx_a, dx_d), f"{label}: dX depends on the accumulate flag"
    want = (dw_in + d).astype(np.float32)   # one IEEE FP32 rounding
    assert np.array_equal(dw_out.view(np.uint32), want.view(np.uint32)), label
