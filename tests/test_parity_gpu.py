"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerances (stated for the stage): dX within 2 BF16 places of the oracle
(or, where the sum cancels, within the FP32 accumulation bound
2**-16 * (sum_j |P||W| + |c x|) plus one place); dW within 1e-3 of
sum_t |P||X| per element.  Small shapes are compared element by element and
span several tiles with ragged tails; the full-size workloads are compared
element by element too (the oracle works through dX a block of rows at a
time), in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle.mhcpb_oracle as O
from rms_backward_gb300 import workloads as WL

from gpu_helpers import Runner, assert_parity_all_rows, assert_parity_full, run_gpu

pytestmark = pytest.mark.gpu

KERNELS = [pytest.param(False, id="tcgen05"), pytest.param(True, id="fma")]

SMALL_SHAPES = [
    (64, 512),      # the tiny workload's shape
    (1, 8),         # smallest legal shape
    (129, 136),     # one token past a tile; a strip with a 8-column tail
    (513, 264),     # a second chunk holding one token; 2 strips + tail
    (1000, 1024),   # several chunks, ragged last tile
    (700, 20480),   # full row width of the training profile
    (2048, 640),    # four chunks of full tiles
]


@pytest.mark.parametrize("fma", KERNELS)
def test_tiny_config(fma):
    wl = WL.config("tiny")
    dx, dw = run_gpu(wl, fma_kernel=fma)
    assert_parity_full(wl, dx, dw, "tiny")


@pytest.mark.parametrize("fma", KERNELS)
@pytest.mark.parametrize("T,K", SMALL_SHAPES)
def test_small_shapes(fma, T, K):
    wl = WL.make("small", T=T, K=K, seed=100 + T + K)
    dx, dw = run_gpu(wl, fma_kernel=fma)
    assert_parity_full(wl, dx, dw, f"T={T} K={K}")


@pytest.mark.parametrize("fma", KERNELS)
@pytest.mark.parametrize("edge", ["rows", "rows_nan", "grad_r0", "p0"])
def test_edge_recipes_small(fma, edge):
    wl = WL.make("edge_small", T=300, K=1032, seed=7, edge=edge)
    dx, dw = run_gpu(wl, fma_kernel=fma)
    assert_parity_full(wl, dx, dw, edge)
    if edge == "p0":
        assert np.all(dw == 0)


@pytest.mark.parametrize("fma", KERNELS)
def test_fused_addend_small(fma):
    wl = WL.make("add_small", T=777, K=2056, seed=9, addend=True)
    dx, dw = run_gpu(wl, fma_kernel=fma)
    assert_parity_full(wl, dx, dw, "addend")


@pytest.mark.parametrize("fma", KERNELS)
def test_fused_addend_equals_separate_bf16_add(fma):
    """The fused sum is bit for bit what adding the addend to the unfused dX
    as a BF16 tensor add gives."""
    wl = WL.make("add_exact", T=515, K=1024, seed=10, addend=True)
    dx_add, dw_add = run_gpu(wl, fma_kernel=fma)
    plain = WL.make("add_exact", T=515, K=1024, seed=10, addend=True)
    plain.addend = None
    dx0, dw0 = run_gpu(plain, fma_kernel=fma)
    t0 = torch.from_numpy(dx0.view(np.int16)).view(torch.bfloat16)
    ta = torch.from_numpy(wl.addend.view(np.int16)).view(torch.bfloat16)
    ref = (t0 + ta).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(dx_add, ref)
    assert np.array_equal(dw_add.view(np.uint32), dw0.view(np.uint32))


@pytest.mark.parametrize("fma", KERNELS)
def test_rms_term_visible(fma):
    """grad_r large and P small, so the RMS term is comparable to P@W and a
    wrong coefficient would show."""
    wl = WL.make("rms", T=256, K=1024, seed=12)
    wl.grad_r = (wl.grad_r * 1e4).astype(np.float32)
    wl.grad_proj = (wl.grad_proj * 1e-2).astype(np.float32)
    dx, dw = run_gpu(wl, fma_kernel=fma)
    assert_parity_full(wl, dx, dw, "rms-visible")
    core = O.dx_core_f64(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    pw = O.dx_core_f64(wl.x, wl.w, wl.grad_proj, np.zeros_like(wl.grad_r), wl.r)
    assert np.median(np.abs(core - pw)) > np.median(np.abs(pw))


@pytest.mark.parametrize("fma", KERNELS)
def test_exact_integer_inputs_bitwise(fma):
    """Inputs whose every product and partial sum is exact in FP32: the GPU
    result must equal the oracle bit for bit, whatever the summation order."""
    T, K = 1100, 384
    rng = np.random.default_rng(13)
    wl = WL.make("exact", T=T, K=K, seed=13)
    X = rng.integers(-8, 9, size=(T, K)).astype(np.float32)
    wl.x = torch.from_numpy(X).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    wl.w = (rng.integers(-64, 65, size=(24, K)) / 64).astype(np.float32)
    gp = (rng.integers(-64, 65, size=(T, 32)) / 64).astype(np.float32)
    gp[:, 24:] = 1e30
    wl.grad_proj = gp
    wl.grad_r = np.zeros(T, np.float32)
    wl.r = np.ones(T, np.float32)
    dx, dw = run_gpu(wl, fma_kernel=fma)
    ref_dx, ref_dw = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    assert np.array_equal(dw.view(np.uint32), ref_dw.view(np.uint32))
    assert np.array_equal(dx, ref_dx)


@pytest.mark.parametrize("fma", KERNELS)
def test_outputs_overwritten_not_accumulated(fma):
    wl = WL.make("ow", T=300, K=520, seed=14)
    r = Runner(wl, fma_kernel=fma, fill=float("nan"))
    r.run()
    dx1, dw1 = r.results()
    assert not np.any(np.isnan(O.bf16_bits_to_f64(dx1))) and not np.any(np.isnan(dw1))
    r.dx.fill_(1234.0)
    r.dw.fill_(-77.0)
    r.run()
    dx2, dw2 = r.results()
    assert np.array_equal(dx1, dx2) and np.array_equal(dw1.view(np.uint32), dw2.view(np.uint32))
    r.plan.close()


# ---------------------------------------------------------------- full size ----
FULL = ["training_profile", "long_sublayer", "edge", "fused_addend"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_element(name):
    """The named full-size workloads in the benchmark's launch configuration,
    every element of dX and of dW against the oracle."""
    wl = WL.config(name)
    dx, dw = run_gpu(wl)
    st, stw = assert_parity_all_rows(wl, dx, dw, name)
    print(f"{name} T={wl.T} K={wl.K}: dX {st}; dW {stw}")


@pytest.mark.parametrize("edge", ["rows_nan", "grad_r0", "p0"])
def test_full_size_edge_subcases(edge):
    wl = WL.make("edge", T=1000, K=20480, seed=3, edge=edge)
    dx, dw = run_gpu(wl)
    st, stw = assert_parity_all_rows(wl, dx, dw, edge)
    print(f"edge {edge}: dX {st}; dW {stw}")
    if edge == "p0":
        assert np.all(dw == 0)
