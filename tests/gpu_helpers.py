"""Helpers for the GPU tests: upload a seeded workload, run the CUDA path
through the C ABI, bring the results back as numpy, and compare with the
CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle.mhcpb_oracle as O
from rms_backward_gb300 import Plan

DEV = "cuda:0"


def to_dev(wl):
    """Device copies of a workload's inputs (BF16 as torch.bfloat16)."""
    d = dict(
        x=torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).to(DEV),
        w=torch.from_numpy(wl.w).to(DEV),
        grad_proj=torch.from_numpy(wl.grad_proj).to(DEV),
        grad_r=torch.from_numpy(wl.grad_r).to(DEV),
        r=torch.from_numpy(wl.r).to(DEV),
    )
    d["addend"] = None if wl.addend is None else \
        torch.from_numpy(wl.addend.view(np.int16)).view(torch.bfloat16).to(DEV)
    return d


class Runner:
    """A plan plus output/workspace buffers for one workload shape."""

    def __init__(self, wl, fma_kernel=False, fill=float("nan"), compensated_dw=False):
        self.wl = wl
        self.plan = Plan(wl.T, wl.K, 0, addend=wl.has_addend, fma_kernel=fma_kernel,
                         compensated_dw=compensated_dw)
        self.inp = to_dev(wl)
        self.dx = torch.full((wl.T, wl.K), fill, dtype=torch.bfloat16, device=DEV)
        self.dw = torch.full((24, wl.K), fill, dtype=torch.float32, device=DEV)
        self.ws = torch.full((self.plan.workspace_bytes // 4,), fill, dtype=torch.float32, device=DEV)

    def run(self, stream=None):
        i = self.inp
        self.plan.execute(i["x"], i["w"], i["grad_proj"], i["grad_r"], i["r"], self.dx, self.dw,
                          self.ws, addend=i["addend"], stream=stream)

    def results(self):
        torch.cuda.synchronize()
        assert self.plan.device_status() == 0, "device-side wait timed out"
        dx = self.dx.view(torch.int16).cpu().numpy().view(np.uint16)
        dw = self.dw.cpu().numpy()
        return dx, dw


def run_gpu(wl, fma_kernel=False, compensated_dw=False):
    r = Runner(wl, fma_kernel=fma_kernel, compensated_dw=compensated_dw)
    r.run()
    out = r.results()
    r.plan.close()
    return out


def assert_parity_full(wl, dx, dw, label=""):
    """Every element of dX and dW against the oracle."""
    ref_dx, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r,
                                        addend_bits=wl.addend)
    bound = O.dx_abs_bound(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    if wl.addend is not None:
        core, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, rows=np.arange(wl.T))
        ok, st = O.check_dx_addend(dx, ref_dx, core, bound)
    else:
        ok, st = O.check_dx(dx, ref_dx, bound)
    assert ok, f"{label} dX mismatch: {st}"
    ref_dw = O.dw_f64(wl.x, wl.grad_proj)
    okw, stw = O.check_dw(dw, ref_dw, O.dw_abs_bound(wl.x, wl.grad_proj))
    assert okw, f"{label} dW mismatch: {stw}"
    return st, stw


def assert_parity_all_rows(wl, dx, dw, label="", block=256):
    """Every element of dX and dW against the oracle at any size: the oracle
    computes dX one block of rows at a time (its own row selection) so its
    FP64 arrays stay small, and dW over all columns.  Returns the merged
    check statistics."""
    T = wl.T
    tot = dict(n=0, fail=0, exact=0, max_ulp=0.0, abs_only_pass=0)
    for r0 in range(0, T, block):
        rows = np.arange(r0, min(T, r0 + block))
        ref_dx, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r,
                                            addend_bits=wl.addend, rows=rows)
        bound = O.dx_abs_bound(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, rows=rows)
        if wl.addend is not None:
            core, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, rows=rows)
            ok, st = O.check_dx_addend(dx[rows], ref_dx, core, bound)
        else:
            ok, st = O.check_dx(dx[rows], ref_dx, bound)
        assert ok, f"{label} dX mismatch in rows {r0}..{rows[-1]}: {st}"
        for k in ("n", "fail", "exact", "abs_only_pass"):
            tot[k] += st.get(k, 0)
        tot["max_ulp"] = max(tot["max_ulp"], st["max_ulp"])
    ref_dw = O.dw_f64(wl.x, wl.grad_proj)
    okw, stw = O.check_dw(dw, ref_dw, O.dw_abs_bound(wl.x, wl.grad_proj))
    assert okw, f"{label} dW mismatch: {stw}"
    return tot, stw


def sample_rows(T, n=48, seed=0):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 511, 512, T - 1, T - 2, T // 2]
    rows = set(x for x in fixed if 0 <= x < T)
    rows.update(rng.integers(0, T, size=n).tolist())
    return np.array(sorted(rows))


def sample_cols(K, n=48, seed=1):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 63, 64, 127, 128, K - 1, K - 8, K // 2]
    cols = set(x for x in fixed if 0 <= x < K)
    cols.update(rng.integers(0, K, size=n).tolist())
    return np.array(sorted(cols))


def assert_parity_sampled(wl, dx, dw, rows, cols, label=""):
    """Sampled rows of dX and sampled columns of dW against the oracle, which
    computes them one by one (full-size workloads)."""
    ref_dx, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r,
                                        addend_bits=wl.addend, rows=rows)
    bound = O.dx_abs_bound(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, rows=rows)
    if wl.addend is not None:
        core, _ = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, rows=rows)
        ok, st = O.check_dx_addend(dx[rows], ref_dx, core, bound)
    else:
        ok, st = O.check_dx(dx[rows], ref_dx, bound)
    assert ok, f"{label} dX mismatch on sampled rows: {st}"
    ref_dw = O.dw_f64(wl.x, wl.grad_proj, cols=cols)
    okw, stw = O.check_dw(dw[:, cols], ref_dw, O.dw_abs_bound(wl.x, wl.grad_proj, cols=cols))
    assert okw, f"{label} dW mismatch on sampled cols: {stw}"
    return st, stw
