"""The compensated dW reduction (plan flag MHCPB_COMPENSATED_DW).

The second kernel sums each dW element's chunk partials in the usual fixed
order but with TwoSum at every addition and one final FP32 rounding (the
compensated, once-rounded dw sums described on FlashInfer's
cake_rmsnorm_det_train_backward page, applied to the cross-chunk sum).

Pin: an input whose per-chunk sums are exact (2**24, 1, 1) and whose exact dW
(2**24 + 2) is an FP32 value.  The compensated reduction must return the
oracle's once-rounded dW bit for bit; the plain sequential reduction returns
2**24 there, which the test also checks, so the case cannot pass by accident.
"""
import numpy as np
import pytest
import torch

import oracle.mhcpb_oracle as O
from rms_backward_gb300 import Plan, abi
from rms_backward_gb300 import workloads as WL

from gpu_helpers import Runner, assert_parity_full, run_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fma", [False, True], ids=["tcgen05", "fma"])
@pytest.mark.parametrize("K", [128, 520])
def test_cancellation_once_rounded_bitwise(fma, K):
    wl = WL.make_dw_cancellation(K=K, seed=50)
    ref = O.dw_f64(wl.x, wl.grad_proj).astype(np.float32)
    assert np.all(ref == np.float32(16777218.0))
    _, dw_c = run_gpu(wl, fma_kernel=fma, compensated_dw=True)
    assert np.array_equal(dw_c.view(np.uint32), ref.view(np.uint32))
    dx_p, dw_p = run_gpu(wl, fma_kernel=fma, compensated_dw=False)
    assert np.all(dw_p == np.float32(2.0 ** 24))
    assert_parity_full(wl, dx_p, dw_p, "plain")


@pytest.mark.parametrize("fma", [False, True], ids=["tcgen05", "fma"])
@pytest.mark.parametrize("T,K", [(64, 512), (1000, 520), (1537, 264)])
def test_compensated_parity(fma, T, K):
    wl = WL.make("c", T=T, K=K, seed=51 + T)
    dx, dw = run_gpu(wl, fma_kernel=fma, compensated_dw=True)
    assert_parity_full(wl, dx, dw, "compensated")


def test_compensated_edge_rows_and_addend():
    wl = WL.make("c", T=1100, K=1024, seed=53, edge="rows")
    dx, dw = run_gpu(wl, compensated_dw=True)
    assert_parity_full(wl, dx, dw, "compensated edge")
    wl = WL.make("c", T=700, K=512, seed=54, addend=True)
    dx, dw = run_gpu(wl, compensated_dw=True)
    assert_parity_full(wl, dx, dw, "compensated addend")


def test_compensated_only_changes_dw():
    """dX does not depend on the flag.  The two reductions of the same S = 8
    partials differ by at most the plain one's rounding error, which is below
    (S - 1) * 2**-24 * sum_s |partial_s| <= 7 * 2**-24 * sum_t |P||X|."""
    wl = WL.make("c", T=4096, K=1024, seed=55)
    dx_p, dw_p = run_gpu(wl)
    dx_c, dw_c = run_gpu(wl, compensated_dw=True)
    assert np.array_equal(dx_p, dx_c)
    bound = O.dw_abs_bound(wl.x, wl.grad_proj)
    diff = np.abs(dw_c.astype(np.float64) - dw_p.astype(np.float64))
    assert np.all(diff <= 8 * 2.0 ** -24 * bound)
    assert np.any(diff > 0)   # the flag does change the rounding somewhere


def test_compensated_bitwise_repeatable_and_grid_independent():
    wl = WL.make("c", T=2600, K=1288, seed=56)
    outs = []
    for cap in (0, 1, 7, 64, 0):
        r = Runner(wl, compensated_dw=True)
        if cap:
            r.plan.set_max_ctas(cap)
        r.run()
        outs.append(r.results())
        r.plan.close()
    for dx, dw in outs[1:]:
        assert np.array_equal(dx, outs[0][0])
        assert np.array_equal(dw.view(np.uint32), outs[0][1].view(np.uint32))


def test_compensated_keeps_inf():
    """An overflowing dW element stays +-Inf (TwoSum's error term would be
    Inf - Inf = NaN if it were not guarded)."""
    wl = WL.make("c", T=1024, K=128, seed=57)
    x = np.zeros_like(wl.x)
    x[0, :] = 0x7F00    # BF16 1.7e38
    x[600, :] = 0x7F00
    gp = np.zeros_like(wl.grad_proj)
    gp[0, :24] = 4.0
    gp[600, :24] = 4.0
    wl.x, wl.grad_proj = x, gp
    wl.r = WL.rms_from_x(x)
    _, dw = run_gpu(wl, compensated_dw=True)
    assert np.all(np.isposinf(dw))
