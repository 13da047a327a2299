"""An empty batch (T = 0) through every entry point (include/mhcpb.h, shape
limits): dW, the sum over no tokens, is written as zeros, or left as dW + 0
when accumulating, which is what the oracle gives for T = 0 (the cuDNN frontend
page "DSv4.1 mHC projection/RMS backward", intro: dW = P^T X); dX, proj, r
and the gate outputs are empty and nothing else is written.  Operands with no
elements may be NULL (an empty torch tensor's data_ptr() is 0)."""
import numpy as np
import pytest
import torch

import oracle.mhcpb_oracle as O
from rms_backward_gb300 import Plan, abi, mhc_gate_backward, mhc_gate_forward
from rms_backward_gb300 import workloads as WL

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
K = 520   # not a multiple of the strip width: the reduction's tail is covered too


def _empty_operands(with_addend=False):
    e = dict(x=torch.empty((0, K), dtype=torch.bfloat16, device=DEV),
             grad_proj=torch.empty((0, 32), device=DEV), grad_r=torch.empty(0, device=DEV),
             r=torch.empty(0, device=DEV), dx=torch.empty((0, K), dtype=torch.bfloat16, device=DEV))
    if with_addend:
        e["addend"] = torch.empty((0, K), dtype=torch.bfloat16, device=DEV)
    return e


def _w():
    return torch.from_numpy(WL.make("empty_w", T=1, K=K, seed=5).w).to(DEV)


def _oracle_dw(w):
    x = np.zeros((0, K), np.uint16)
    _, dw = O.mhc_proj_rms_backward(x, w.cpu().numpy(), np.zeros((0, 32), np.float32),
                                    np.zeros(0, np.float32), np.zeros(0, np.float32))
    return dw


@pytest.mark.parametrize("flags", [{}, {"compensated_dw": True}, {"fma_kernel": True}, {"addend": True}],
                         ids=["plain", "compensated", "fma", "addend"])
def test_execute_writes_zero_dw(flags):
    plan = Plan(0, K, 0, **flags)
    assert plan.workspace_bytes == 0
    e = _empty_operands(with_addend=flags.get("addend", False))
    w = _w()
    dw = torch.full((24, K), float("nan"), device=DEV)
    ws = torch.empty(0, dtype=torch.uint8, device=DEV)
    plan.execute(e["x"], w, e["grad_proj"], e["grad_r"], e["r"], e["dx"], dw, ws, addend=e.get("addend"))
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    got = dw.cpu().numpy()
    assert np.array_equal(got, _oracle_dw(w)) and not np.signbit(got).any()   # +0 everywhere
    plan.close()


def test_accumulate_leaves_dw_unchanged():
    plan = Plan(0, K, 0, accumulate_dw=True)
    e = _empty_operands()
    before = torch.randn((24, K), device=DEV)
    dw = before.clone()
    plan.execute(e["x"], _w(), e["grad_proj"], e["grad_r"], e["r"], e["dx"], dw,
                 torch.empty(0, dtype=torch.uint8, device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(dw, before)   # dW + 0: the same bits for every nonzero value
    plan.close()


def test_split_and_static_scratch():
    e = _empty_operands()
    w = _w()
    plan = Plan(0, K, 0)
    ws = torch.empty(0, dtype=torch.uint8, device=DEV)
    plan.execute_dx(e["x"], w, e["grad_proj"], e["grad_r"], e["r"], e["dx"], ws)
    dw = torch.full((24, K), float("nan"), device=DEV)
    plan.reduce_dw(ws, dw)
    dw2 = torch.full((24, K), float("nan"), device=DEV)
    abi.mhcpb_execute_static_scratch(0, K, abi.MHCPB_ALLOW_TF32, 0, w.data_ptr(), 0, 0, 0, 0,
                                     dw2.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    zeros = np.zeros((24, K), np.float32)
    assert np.array_equal(dw.cpu().numpy(), zeros) and np.array_equal(dw2.cpu().numpy(), zeros)
    plan.close()


def test_non_empty_operands_still_checked():
    """NULL for every empty operand is accepted; W and dW are not empty at
    T = 0, and a NULL there is still rejected."""
    plan = Plan(0, K, 0)
    stream = torch.cuda.current_stream().cuda_stream
    w = _w()
    dw = torch.full((24, K), 7.0, device=DEV)
    abi.mhcpb_execute(plan.handle, 0, w.data_ptr(), 0, 0, 0, 0, dw.data_ptr(), 0, 0, None, stream)
    torch.cuda.synchronize()
    assert not dw.any()
    with pytest.raises(abi.MhcpbError) as ei:
        abi.mhcpb_execute(plan.handle, 0, 0, 0, 0, 0, 0, dw.data_ptr(), 0, 0, None, stream)
    assert ei.value.status == abi.MHCPB_ERR_INVALID_ARG   # W is NULL
    with pytest.raises(abi.MhcpbError) as ei:
        abi.mhcpb_execute(plan.handle, 0, w.data_ptr(), 0, 0, 0, 0, 0, 0, 0, None, stream)
    assert ei.value.status == abi.MHCPB_ERR_INVALID_ARG   # dW is NULL
    plan.close()


def test_forward_and_gates_do_nothing():
    plan = Plan(0, K, 0)
    assert plan.forward_workspace_bytes == 0
    e = _empty_operands()
    proj, r = torch.empty((0, 32), device=DEV), torch.empty(0, device=DEV)
    plan.forward(e["x"], _w(), proj, r, torch.empty(0, dtype=torch.uint8, device=DEV))
    alpha = torch.ones(3, device=DEV)
    bias = torch.zeros(24, device=DEV)
    h, gh = torch.empty((0, 24), device=DEV), torch.empty((0, 24), device=DEV)
    gp, gr = torch.empty((0, 32), device=DEV), torch.empty(0, device=DEV)
    mhc_gate_forward(proj, r, alpha, bias, h)
    mhc_gate_backward(proj, r, alpha, bias, gh, gp, gr)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    # alpha and bias are not empty: NULL is still rejected
    with pytest.raises(abi.MhcpbError) as ei:
        abi.mhcpb_gate_forward(0, 20, 0, 0, 0, bias.data_ptr(), 0, torch.cuda.current_stream().cuda_stream)
    assert ei.value.status == abi.MHCPB_ERR_INVALID_ARG
    plan.close()
