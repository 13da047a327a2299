"""The allocation-free entry point, mhcpb_execute_static_scratch.

It serves callers that cannot allocate device memory at all (a framework that
owns the whole device heap, plugin code handed only its buffers): no plan, no
workspace, the dW partials in the library's own 16 MiB __device__ buffer.  It
launches the same kernels with the same partition as the workspace entry
point, mhcpb_execute, so its results must be the same bits; they are also held
to the oracle's own check.  Two calls in a row (different shapes, the second
with the fused addend) check that sharing the one buffer is harmless.
This file is collected last so a run stopping at its first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.mhcpb_oracle as O
from rms_backward_gb300 import abi
from rms_backward_gb300 import workloads as WL

from gpu_helpers import assert_parity_full, assert_parity_sampled, sample_rows


def _lib():
    import os
    if not os.path.exists(abi.LIB_PATH):
        from rms_backward_gb300 import build
        build.build()
    return abi.load()


def test_oversized_shapes_rejected_before_any_cuda_call():
    lib = _lib()
    nul = [None] * 9
    # S * 24 * K * 4 bytes of partials must fit the 16 MiB buffer
    assert lib.mhcpb_execute_static_scratch(16384, 20480, abi.MHCPB_ALLOW_TF32, *nul) == \
        abi.MHCPB_ERR_SCRATCH_TOO_SMALL
    # at K = 20480: 8 partials (T <= 4096) fit, 9 do not
    assert lib.mhcpb_execute_static_scratch(4097, 20480, abi.MHCPB_ALLOW_TF32, *nul) == \
        abi.MHCPB_ERR_SCRATCH_TOO_SMALL
    for T in (4000, 4096):   # fit: with null pointers the next check rejects them
        assert lib.mhcpb_execute_static_scratch(T, 20480, abi.MHCPB_ALLOW_TF32, *nul) == \
            abi.MHCPB_ERR_INVALID_ARG
    assert lib.mhcpb_execute_static_scratch(64, 512, 0, *nul) == abi.MHCPB_ERR_TF32_NOT_ALLOWED
    assert lib.mhcpb_execute_static_scratch(64, 512, abi.MHCPB_ALLOW_TF32 | abi.MHCPB_FMA_KERNEL,
                                            *nul) == abi.MHCPB_ERR_INVALID_ARG


def _dev(wl):
    d = dict(
        x=torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).cuda(),
        w=torch.from_numpy(wl.w).cuda(),
        gp=torch.from_numpy(wl.grad_proj).cuda(),
        gr=torch.from_numpy(wl.grad_r).cuda(),
        r=torch.from_numpy(wl.r).cuda(),
    )
    d["add"] = None if wl.addend is None else \
        torch.from_numpy(wl.addend.view(np.int16)).view(torch.bfloat16).cuda()
    return d


def _outputs(wl):
    dx = torch.full((wl.T, wl.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    dw = torch.full((24, wl.K), float("nan"), dtype=torch.float32, device="cuda")
    return dx, dw


def _with_workspace(wl, d):
    """The reference: the existing entry point with a caller-allocated workspace."""
    flags = abi.MHCPB_ALLOW_TF32 | (abi.MHCPB_HAS_ADDEND if wl.has_addend else 0)
    plan = abi.mhcpb_plan_create(wl.T, wl.K, 0, flags)
    ws = torch.empty(abi.mhcpb_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    dx, dw = _outputs(wl)
    abi.mhcpb_execute(plan, d["x"].data_ptr(), d["w"].data_ptr(), d["gp"].data_ptr(),
                      d["gr"].data_ptr(), d["r"].data_ptr(), dx.data_ptr(), dw.data_ptr(),
                      ws.data_ptr(), ws.numel(), None if d["add"] is None else d["add"].data_ptr(),
                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert abi.mhcpb_get_device_status(plan) == abi.MHCPB_OK
    abi.mhcpb_destroy(plan)
    return dx, dw


def _static_scratch(wl, d):
    flags = abi.MHCPB_ALLOW_TF32 | (abi.MHCPB_HAS_ADDEND if wl.has_addend else 0)
    dx, dw = _outputs(wl)
    abi.mhcpb_execute_static_scratch(
        wl.T, wl.K, flags, d["x"].data_ptr(), d["w"].data_ptr(), d["gp"].data_ptr(),
        d["gr"].data_ptr(), d["r"].data_ptr(), dx.data_ptr(), dw.data_ptr(),
        None if d["add"] is None else d["add"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return dx, dw


def _bits(dx, dw):
    return dx.view(torch.int16).cpu().numpy().view(np.uint16), dw.cpu().numpy()


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_twice():
    # first call: the largest shape the buffer holds (training profile, 15 MiB
    # of partials); second call right after: another shape with the addend
    calls = [WL.config("training_profile"),
             WL.make("no_alloc_addend", T=777, K=2056, seed=51, addend=True)]
    for wl in calls:
        d = _dev(wl)
        ref_dx, ref_dw = _bits(*_with_workspace(wl, d))
        got_dx, got_dw = _bits(*_static_scratch(wl, d))
        # the same kernels with the same partition: the same bits
        assert np.array_equal(got_dx, ref_dx), f"T={wl.T} K={wl.K}: dX differs from mhcpb_execute"
        assert np.array_equal(got_dw.view(np.uint32), ref_dw.view(np.uint32)), \
            f"T={wl.T} K={wl.K}: dW differs from mhcpb_execute"
        # and the oracle's own check, unwidened
        if wl.has_addend:
            st = assert_parity_full(wl, got_dx, got_dw, "static scratch")
        else:
            rows = np.unique(np.concatenate([sample_rows(wl.T, n=200), np.arange(0, wl.T, 97)]))
            st = assert_parity_sampled(wl, got_dx, got_dw, rows, np.arange(wl.K), "static scratch")
        print(f"static scratch T={wl.T} K={wl.K}: dX {st[0]} dW {st[1]}")
        del d


@pytest.mark.gpu
def test_static_scratch_compensated_dw_once_rounded():
    """MHCPB_COMPENSATED_DW through the allocation-free entry point: the
    cancellation input's exact dW, 2**24 + 2, comes back bit for bit."""
    wl = WL.make_dw_cancellation(K=256, seed=52)
    d = _dev(wl)
    dx, dw = _outputs(wl)
    abi.mhcpb_execute_static_scratch(
        wl.T, wl.K, abi.MHCPB_ALLOW_TF32 | abi.MHCPB_COMPENSATED_DW, d["x"].data_ptr(),
        d["w"].data_ptr(), d["gp"].data_ptr(), d["gr"].data_ptr(), d["r"].data_ptr(),
        dx.data_ptr(), dw.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.all(dw.cpu().numpy() == np.float32(16777218.0))
