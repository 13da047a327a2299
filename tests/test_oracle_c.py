"""The C oracle (the CPU baseline bench.py times) against the pinned numpy
oracle: the same definition, so the same bits.  The two sum in different
orders in FP64; the outputs round the same unless an FP64 sum sits within
its own rounding error of a BF16 or FP32 tie, which these inputs do not hit."""
import numpy as np
import pytest

import oracle.mhcpb_oracle as O
from rms_backward_gb300 import workloads as WL


@pytest.fixture(scope="module")
def C():
    import shutil
    if shutil.which("gcc") is None and shutil.which("cc") is None:
        pytest.skip("no C compiler")
    import oracle.mhcpb_oracle_c as C
    C.load()
    return C


@pytest.mark.parametrize("T,K,edge,threads", [
    (64, 512, None, 1), (129, 136, None, 4), (513, 264, "rows", 0), (300, 1032, "rows_nan", 3),
    (200, 2048, "grad_r0", 2), (37, 48, "p0", 1), (700, 20480, None, 0)])
def test_c_oracle_equals_numpy_oracle(C, T, K, edge, threads):
    wl = WL.make("c", T=T, K=K, seed=T + K, edge=edge)
    dx, dw = C.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r, nthreads=threads)
    ref_dx, ref_dw = O.mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    assert np.array_equal(dx, ref_dx)
    assert np.array_equal(dw.view(np.uint32), ref_dw.view(np.uint32))


def test_c_oracle_structured_closed_form(C):
    """The closed form of the numpy oracle's pin: one-hot W, rank-one X,
    power-of-two coefficient (every value exact)."""
    import torch
    T, K = 5, 16
    rng = np.random.default_rng(3)
    P = rng.integers(-8, 9, size=(T, 32)).astype(np.float32)
    W = np.zeros((24, K), np.float32)
    for j in range(24):
        W[j, j % K] = 1.0
    a = np.array([1, -2, 3, 0, 1], np.float32)
    b = np.arange(1, K + 1, dtype=np.float32) - 8
    X = np.outer(a, b).astype(np.float32)
    xb = torch.from_numpy(X).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    s = np.array([0.5, -1.0, 0.25, 2.0, 0.0], np.float32)
    dx, dw = C.mhc_proj_rms_backward(xb, W, P, (64.0 * s).astype(np.float32), np.full(T, 4.0, np.float32))
    for t in range(T):
        for k in range(K):
            pw = P[t, k] + (P[t, k + 16] if k + 16 < 24 else 0.0)
            assert O.bf16_bits_to_f64(dx[t, k]) == pw + s[t] * X[t, k]
    for j in range(24):
        for k in range(K):
            assert dw[j, k] == b[k] * float(np.dot(a, P[:, j]))
