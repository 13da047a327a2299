"""Writes tests/golden/oracle_T8_K16.txt (the backward) and
tests/golden/forward_T8_K16.txt (the forward) from the CPU oracles only.

The fixture freezes the oracle's output on one small seeded workload so that a
later change to the oracle's arithmetic shows up as a diff (and must then be
justified by the passage it follows).  Run from the repository root:

    python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from oracle import mhc_proj_rms_backward  # noqa: E402
from oracle.mhcpf_oracle import mhc_proj_forward  # noqa: E402
from rms_backward_gb300 import workloads  # noqa: E402


def main():
    wl = workloads.make("golden", T=8, K=16, seed=1234, addend=True)
    dx, dw = mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    dxa, _ = mhc_proj_rms_backward(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r,
                                   addend_bits=wl.addend)
    lines = ["# oracle output on workloads.make('golden', T=8, K=16, seed=1234, addend=True)",
             "# written by tests/golden/make_golden.py (calls only oracle/ and the input generator)",
             "# dx: BF16 bits row-major [8,16]; dx_addend: same with the fused addend;",
             "# dw: FP32 bits row-major [24,16]"]
    lines.append("dx " + " ".join(f"{int(v):04x}" for v in dx.reshape(-1)))
    lines.append("dx_addend " + " ".join(f"{int(v):04x}" for v in dxa.reshape(-1)))
    lines.append("dw " + " ".join(f"{int(v):08x}" for v in dw.view(np.uint32).reshape(-1)))
    with open(os.path.join(HERE, "oracle_T8_K16.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")

    proj, r = mhc_proj_forward(wl.x, wl.w)
    lines = ["# forward oracle output on workloads.make('golden', T=8, K=16, seed=1234, addend=True)",
             "# written by tests/golden/make_golden.py (calls only oracle/ and the input generator)",
             "# the FP64 results rounded to FP32 (the forward's stored precision; robust to",
             "# the summation order of the host's FP64 matrix product):",
             "# proj: FP32 bits row-major [8,32] (columns 24..31 zero); r: FP32 bits [8]"]
    p32 = proj.astype(np.float32).view(np.uint32).reshape(-1)
    r32 = r.astype(np.float32).view(np.uint32).reshape(-1)
    lines.append("proj " + " ".join(f"{int(v):08x}" for v in p32))
    lines.append("r " + " ".join(f"{int(v):08x}" for v in r32))
    with open(os.path.join(HERE, "forward_T8_K16.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
