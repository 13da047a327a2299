"""The seeded input generator shared by the CUDA path and the oracle (CPU).

Pins the input recipe (shapes, distributions, draw determinism, edge-case
sub-recipes), the five named workloads, and the algorithmic byte counts that
the bench divides by time.  The byte counts are re-derived here from the
sizes of the arrays each step reads and writes."""
import numpy as np
import pytest
import torch

from rms_backward_gb300 import workloads as WL


def _f64(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def test_same_seed_same_bits_other_seed_other_bits():
    a = WL.make("a", T=48, K=64, seed=7, addend=True)
    b = WL.make("b", T=48, K=64, seed=7, addend=True)
    c = WL.make("c", T=48, K=64, seed=8, addend=True)
    for f in ("x", "w", "grad_proj", "grad_r", "r", "addend"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
        assert not np.array_equal(getattr(a, f), getattr(c, f)), f


def test_shapes_dtypes_and_distributions():
    T, K = 512, 1024
    wl = WL.make("s", T=T, K=K, seed=3, addend=True)
    assert wl.x.shape == (T, K) and wl.x.dtype == np.uint16
    assert wl.w.shape == (24, K) and wl.w.dtype == np.float32
    assert wl.grad_proj.shape == (T, 32) and wl.grad_proj.dtype == np.float32
    assert wl.grad_r.shape == (T,) and wl.r.shape == (T,) and wl.r.dtype == np.float32
    assert wl.addend.shape == (T, K) and wl.addend.dtype == np.uint16
    # N(0, sigma) draws: sample standard deviations within a few percent
    for arr, sigma in ((_f64(wl.x), 1.0), (wl.w, 0.02), (wl.grad_proj, 1e-2),
                       (wl.grad_r, 1e-3), (_f64(wl.addend), 1e-2)):
        a = np.asarray(arr, dtype=np.float64)
        assert abs(a.std() / sigma - 1.0) < 0.05
        assert abs(a.mean()) < 0.05 * sigma


def test_r_is_the_rms_of_the_bf16_rows():
    wl = WL.make("r", T=40, K=72, seed=11)
    x = _f64(wl.x)
    want = np.sqrt((x * x).sum(axis=1) / wl.K + 1e-6).astype(np.float32)
    assert np.array_equal(wl.r, want)


def test_edge_recipes():
    T, K = 400, 64
    rows = WL.make("e", T=T, K=K, seed=5, edge="rows")
    rms = rows.r.astype(np.float64)
    assert np.log10(rms.max() / rms.min()) > 4.5          # 10^U(-3,3) row scales
    assert np.all(np.abs(rows.grad_proj[:, 24:]) == np.float32(1e30))
    nan = WL.make("e", T=T, K=K, seed=5, edge="rows_nan")
    tail = nan.grad_proj[:, 24:]
    assert np.isnan(tail).any() and np.isinf(tail).any() and not np.isfinite(tail).any()
    assert np.array_equal(nan.x, rows.x)                   # same draws before the tail
    g0 = WL.make("e", T=T, K=K, seed=5, edge="grad_r0")
    assert not g0.grad_r.any() and np.array_equal(g0.x, rows.x)
    p0 = WL.make("e", T=T, K=K, seed=5, edge="p0")
    assert not p0.grad_proj[:, :24].any()
    assert np.array_equal(p0.grad_proj[:, 24:], rows.grad_proj[:, 24:])
    with pytest.raises(ValueError):
        WL.make("e", T=4, K=8, seed=5, edge="bogus")


def test_named_workloads():
    assert WL.CONFIGS == {
        "tiny": dict(T=64, K=512, seed=0),
        "training_profile": dict(T=4096, K=20480, seed=1),
        "long_sublayer": dict(T=16384, K=20480, seed=2),
        "edge": dict(T=1000, K=20480, seed=3, edge="rows"),
        "fused_addend": dict(T=4096, K=20480, seed=4, addend=True),
    }
    tiny = WL.config("tiny")
    assert (tiny.T, tiny.K, tiny.seed) == (64, 512, 0)


@pytest.mark.parametrize("addend", [False, True])
def test_algorithmic_bytes_from_the_arrays(addend):
    T, K = 96, 128
    wl = WL.make("b", T=T, K=K, seed=2, addend=addend)
    read = wl.x.nbytes + wl.w.nbytes + wl.grad_proj[:, :24].nbytes + wl.r.nbytes + wl.grad_r.nbytes
    read += wl.addend.nbytes if addend else 0
    write = wl.x.nbytes + wl.w.nbytes            # dX like X, dW like W
    assert WL.algorithmic_bytes(T, K, addend) == read + write


def test_algorithmic_bytes_at_the_profile():
    assert WL.algorithmic_bytes(4096, 20480) == 339_902_464
    assert WL.algorithmic_bytes(4096, 20480, addend=True) == 507_674_624
    assert WL.algorithmic_bytes(16384, 20480) == 1_347_813_376
    # forward: read X and W, write proj [T, 32] FP32 and r
    T, K = 4096, 20480
    assert WL.algorithmic_bytes_forward(T, K) == 2 * T * K + 24 * K * 4 + T * 32 * 4 + T * 4


def test_dw_cancellation_fixture():
    wl = WL.make_dw_cancellation(K=16, seed=5)
    x = _f64(wl.x)
    p = wl.grad_proj[:, :24].astype(np.float64)
    dw = p.T @ x                                   # exact: all values are small integers or 2^24
    assert np.all(dw == 2.0 ** 24 + 2) and wl.notes["exact_dw"] == 2.0 ** 24 + 2
    chunks = [p[i * 512:(i + 1) * 512].T @ x[i * 512:(i + 1) * 512] for i in range(3)]
    seq = np.float32(chunks[0][0, 0])
    for c in chunks[1:]:
        seq = np.float32(seq + np.float32(c[0, 0]))
    assert seq == np.float32(2.0 ** 24)            # one FP32 rounding per chunk loses the 2
