"""Seeded synthetic inputs for the mHC projection/RMS backward.

This module only *draws* inputs; it holds none of the backward's arithmetic.
Both the CUDA path (tests, bench, smoke) and the CPU oracle consume the same
host arrays made here, so a parity test compares the two on identical bits.

Shapes and distributions follow the workloads stated for the stage
("DSv4.1 mHC projection/RMS backward", cuDNN frontend page, intro: the training
profile is 4 residual streams x hidden 5120 = K 20480 and 4096 tokens per rank):

  X          BF16 [T, K]   ~ N(0, 1)
  W          FP32 [24, K]  ~ N(0, 0.02)
  grad_proj  FP32 [T, 32]  ~ N(0, 1e-2)   (only columns 0..23 are read)
  grad_r     FP32 [T]      ~ N(0, 1e-3)
  r          FP32 [T]      = sqrt(mean_k X^2 + 1e-6), the forward's RMS,
                             computed in FP64 from the BF16 X, rounded to FP32
  addend     BF16 [T, K]   ~ N(0, 1e-2)   (only for the fused-addend workload)

Draw order from one CPU ``torch.Generator`` seeded per workload: X, W,
grad_proj, grad_r, then (when present) the addend, then any edge-case extras.
All arrays are returned as numpy (BF16 as raw uint16 bit patterns).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

N_PROJ = 24          # columns of grad_proj that the stage uses (P = grad_proj[:, :24])
GRAD_PROJ_COLS = 32  # stored width of grad_proj
RMS_EPS = 1e-6


@dataclass
class Workload:
    name: str
    T: int
    K: int
    seed: int
    x: np.ndarray            # uint16 [T, K]  BF16 bits
    w: np.ndarray            # float32 [24, K]
    grad_proj: np.ndarray    # float32 [T, 32]
    grad_r: np.ndarray       # float32 [T]
    r: np.ndarray            # float32 [T]
    addend: Optional[np.ndarray] = None   # uint16 [T, K] BF16 bits or None
    notes: dict = field(default_factory=dict)

    @property
    def has_addend(self) -> bool:
        return self.addend is not None


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rms_from_x(x_bits: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """The forward's per-row RMS of the BF16 X, in FP64, rounded to FP32.

    Processed in row blocks so a [4096, 20480] input does not need an FP64 copy.
    """
    T = x_bits.shape[0]
    out = np.empty(T, dtype=np.float32)
    step = max(1, (1 << 22) // max(1, x_bits.shape[1]))
    for t0 in range(0, T, step):
        xd = _bits_to_f64(x_bits[t0:t0 + step])
        out[t0:t0 + step] = np.sqrt(np.mean(xd * xd, axis=1) + eps).astype(np.float32)
    return out


def make(name: str, T: int, K: int, seed: int, *, addend: bool = False,
         edge: Optional[str] = None) -> Workload:
    """Draw one workload.

    ``edge`` selects the edge-case recipe:
      * "rows"   X rows scaled by 10**U(-3, 3) (r spans six decades) and
                 grad_proj[:, 24:32] = +-1e30 (must be ignored);
      * "rows_nan"  as "rows" but grad_proj[:, 24:32] = NaN / +-Inf;
      * "grad_r0"   as "rows" with grad_r = 0;
      * "p0"        as "rows" with grad_proj[:, :24] = 0.
    """
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, K, generator=g, dtype=torch.float32)
    w = torch.randn(N_PROJ, K, generator=g, dtype=torch.float32) * 0.02
    gp = torch.randn(T, GRAD_PROJ_COLS, generator=g, dtype=torch.float32) * 1e-2
    gr = torch.randn(T, generator=g, dtype=torch.float32) * 1e-3
    add = None
    if addend:
        add = torch.randn(T, K, generator=g, dtype=torch.float32) * 1e-2
    notes = {}
    if edge is not None:
        scale = torch.pow(10.0, torch.rand(T, 1, generator=g, dtype=torch.float64) * 6.0 - 3.0)
        x = (x.double() * scale).float()
        sign = torch.where(torch.rand(T, 8, generator=g) < 0.5, -1.0, 1.0)
        if edge == "rows_nan":
            tail = torch.full((T, 8), float("nan"))
            tail[:, 1::3] = float("inf") * sign[:, 1::3]
        else:
            tail = 1e30 * sign
        gp[:, N_PROJ:] = tail
        if edge == "grad_r0":
            gr.zero_()
        elif edge == "p0":
            gp[:, :N_PROJ] = 0.0
        elif edge not in ("rows", "rows_nan"):
            raise ValueError(f"unknown edge recipe {edge!r}")
        notes["edge"] = edge
    x_bits = _bf16_bits(x)
    return Workload(
        name=name, T=T, K=K, seed=seed, x=x_bits,
        w=w.numpy().astype(np.float32, copy=False),
        grad_proj=gp.numpy().astype(np.float32, copy=False),
        grad_r=gr.numpy().astype(np.float32, copy=False),
        r=rms_from_x(x_bits),
        addend=None if add is None else _bf16_bits(add),
        notes=notes,
    )


@dataclass
class GateWorkload:
    """Inputs of the gate/normalisation step (draws only; see make_gates)."""
    name: str
    T: int
    seed: int
    proj: np.ndarray     # float32 [T, 32]: projection logits (columns 24..31 unused)
    r: np.ndarray        # float32 [T]: RMS of each row
    alpha: np.ndarray    # float32 [3]: scales of the pre, post and res logits
    bias: np.ndarray     # float32 [24]
    grad_h: np.ndarray   # float32 [T, 24]: upstream gradients of H_pre, H_post, H_res


def make_gates(name: str, T: int, seed: int) -> GateWorkload:
    """Draw the gate step's inputs at the training profile's scale: proj has
    the spread of X W^T for X ~ N(0, 1) and W ~ N(0, 0.02) over K = 20480
    (standard deviation 0.02 sqrt(20480) = 2.86), r the RMS of such rows
    (about 1, here U(0.9, 1.1)), alpha = 0.5 U(0.5, 1.5) each, bias ~ N(0, 0.5),
    grad_h ~ N(0, 1e-2); proj[:, 24:32] = +-1e30 (never read).  Draw order:
    proj, r, alpha, bias, grad_h, signs of the unused columns."""
    g = torch.Generator().manual_seed(seed)
    proj = torch.randn(T, GRAD_PROJ_COLS, generator=g, dtype=torch.float32) * 2.862
    r = 0.9 + 0.2 * torch.rand(T, generator=g, dtype=torch.float32)
    alpha = 0.5 * (0.5 + torch.rand(3, generator=g, dtype=torch.float32))
    bias = torch.randn(N_PROJ, generator=g, dtype=torch.float32) * 0.5
    gh = torch.randn(T, N_PROJ, generator=g, dtype=torch.float32) * 1e-2
    sign = torch.where(torch.rand(T, 8, generator=g) < 0.5, -1.0, 1.0)
    proj[:, N_PROJ:] = 1e30 * sign
    return GateWorkload(name=name, T=T, seed=seed, proj=proj.numpy(), r=r.numpy(),
                        alpha=alpha.numpy(), bias=bias.numpy(), grad_h=gh.numpy())


def make_dw_cancellation(K: int, seed: int, chunk: int = 512) -> Workload:
    """Three chunks of ``chunk`` tokens whose dW contributions are 2**24, 1 and
    1 for every (j, k): X is zero except X[0, :] = 2**24, X[chunk, :] = 1 and
    X[2 * chunk, :] = 1 (all exact in BF16), grad_proj[:, :24] is zero except
    1.0 on those three rows, grad_r = 0.  Every product and every per-chunk
    sum is exact, and the exact dW = 2**24 + 2 is an FP32 value, but adding
    the three chunk sums one FP32 rounding at a time gives 2**24 (2**24 + 1 is
    a tie that rounds to even).  W is drawn from ``seed``."""
    T = 3 * chunk
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(N_PROJ, K, generator=g, dtype=torch.float32) * 0.02
    x = torch.zeros(T, K, dtype=torch.float32)
    x[0, :] = 2.0 ** 24
    x[chunk, :] = 1.0
    x[2 * chunk, :] = 1.0
    gp = torch.zeros(T, GRAD_PROJ_COLS, dtype=torch.float32)
    gp[[0, chunk, 2 * chunk], :N_PROJ] = 1.0
    x_bits = _bf16_bits(x)
    return Workload(
        name="dw_cancellation", T=T, K=K, seed=seed, x=x_bits,
        w=w.numpy().astype(np.float32, copy=False),
        grad_proj=gp.numpy(), grad_r=np.zeros(T, dtype=np.float32), r=rms_from_x(x_bits),
        notes={"exact_dw": float(2 ** 24 + 2)},
    )


# The five named workloads: (T, K, seed, addend, edge).  K = n_streams * hidden.
CONFIGS = {
    "tiny": dict(T=64, K=4 * 128, seed=0),
    "training_profile": dict(T=4096, K=4 * 5120, seed=1),
    "long_sublayer": dict(T=16384, K=4 * 5120, seed=2),
    "edge": dict(T=1000, K=4 * 5120, seed=3, edge="rows"),
    "fused_addend": dict(T=4096, K=4 * 5120, seed=4, addend=True),
}


def config(name: str, **override) -> Workload:
    kw = dict(CONFIGS[name])
    kw.update(override)
    return make(name, **kw)


def algorithmic_bytes(T: int, K: int, addend: bool = False) -> int:
    """Compulsory HBM bytes of one backward: read X and write dX (2TK each),
    read W and write dW (96K each), read the 24 used grad_proj columns (96T),
    read r and grad_r (8T), plus a read of the BF16 addend (2TK) when fused."""
    b = 2 * T * K + 2 * T * K + 96 * K + 96 * K + 96 * T + 8 * T
    if addend:
        b += 2 * T * K
    return b


def algorithmic_bytes_forward(T: int, K: int) -> int:
    """Compulsory HBM bytes of one forward: read X (2TK) and W (96K), write
    proj [T, 32] FP32 (128T) and r (4T)."""
    return 2 * T * K + 96 * K + 128 * T + 4 * T


def algorithmic_flops(T: int, K: int) -> int:
    """Two rank-24 contractions (2*24 FMAs per X element) plus the RMS term."""
    return 4 * T * N_PROJ * K + 2 * T * K
