"""Shapes at the limits of the contract (include/mhcpb.h: T <= 2**24, K <= 2**20,
K a multiple of 8): the widest K with a handful of tokens, and the longest T
with the narrowest K (S = 32768 dW partials, 131072 token tiles).  Backward
(both kernels for the wide case) and forward against the oracles; above the
limits the host rejects the shape (tests/test_abi_host.py)."""
import numpy as np
import pytest
import torch

import oracle.mhcpf_oracle as F
import oracle.mhcpb_oracle as O
from rms_backward_gb300 import Plan
from rms_backward_gb300 import workloads as WL

from gpu_helpers import assert_parity_full, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _forward(wl):
    plan = Plan(wl.T, wl.K, 0)
    x = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).to(DEV)
    w = torch.from_numpy(wl.w).to(DEV)
    proj = torch.full((wl.T, 32), float("nan"), device=DEV)
    r = torch.full((wl.T,), float("nan"), device=DEV)
    ws = torch.empty(plan.forward_workspace_bytes // 4, device=DEV)
    plan.forward(x, w, proj, r, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    plan.close()
    return proj.cpu().numpy(), r.cpu().numpy()


@pytest.fixture(scope="module")
def widest():
    return WL.make("widest", T=3, K=1 << 20, seed=90)


@pytest.mark.parametrize("fma", [False, True], ids=["tcgen05", "fma"])
def test_backward_widest_k(widest, fma):
    dx, dw = run_gpu(widest, fma_kernel=fma)
    assert_parity_full(widest, dx, dw, "K = 2**20")


def test_forward_widest_k(widest):
    proj, r = _forward(widest)
    ref_p, ref_r = F.mhc_proj_forward(widest.x, widest.w)
    ok, st = F.check_proj(proj, ref_p, F.proj_abs_bound(widest.x, widest.w))
    assert ok, st
    okr, str_ = F.check_r(r, ref_r)
    assert okr, str_


@pytest.fixture(scope="module")
def longest():
    return WL.make("longest", T=1 << 24, K=8, seed=91)


def test_backward_longest_t(longest):
    wl = longest
    dx, dw = run_gpu(wl)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, 511, 512, wl.T - 8, wl.T - 1], rng.integers(0, wl.T, 200)]))
    ref_dx, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, rows=rows)
    bound = O.dx_abs_bound(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, rows=rows)
    ok, st = O.check_dx(dx[rows], ref_dx, bound)
    assert ok, st
    okw, stw = O.check_dw(dw, O.dw_f64(wl.x, wl.grad_proj), O.dw_abs_bound(wl.x, wl.grad_proj))
    assert okw, stw


def test_forward_longest_t(longest):
    wl = longest
    proj, r = _forward(wl)
    rng = np.random.default_rng(6)
    rows = np.unique(np.concatenate([[0, 127, 128, wl.T - 1], rng.integers(0, wl.T, 300)]))
    ref_p, ref_r = F.mhc_proj_forward(wl.x, wl.w, rows=rows)
    ok, st = F.check_proj(proj[rows], ref_p, F.proj_abs_bound(wl.x, wl.w, rows=rows))
    assert ok, st
    okr, str_ = F.check_r(r[rows], ref_r)
    assert okr, str_
