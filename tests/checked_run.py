"""Child process of tests/test_checked_build_gpu.py (not a test module).

Builds the bounds-checked library (-DMHCPB_CHECKED) beside the product one,
loads it before anything else (so every binding of the package calls it),
runs every entry point over the tests' edge shapes, and checks that (a) no
kernel found an access outside its buffer (mhcpb_debug_checked_sites) and
(b) the results still match the oracles.  Exits non-zero on any failure."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

from rms_backward_gb300 import abi  # noqa: E402
from rms_backward_gb300 import build as B  # noqa: E402

LIB = B.build(extra_flags=["-DMHCPB_CHECKED"], out_dir=os.path.join(B.BUILD, "checked"))
abi.load(LIB)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle.mhcg_oracle as G  # noqa: E402
import oracle.mhcpf_oracle as F  # noqa: E402
from gpu_helpers import DEV, assert_parity_all_rows, assert_parity_full, run_gpu, to_dev  # noqa: E402
from rms_backward_gb300 import Plan, mhc_gate_backward, mhc_gate_forward  # noqa: E402
from rms_backward_gb300 import workloads as WL  # noqa: E402


def no_sites(label):
    torch.cuda.synchronize()
    checked, sites = abi.mhcpb_debug_checked_sites()
    assert checked, "the loaded library is not a checked build"
    bad = {k: v for k, v in sites.items() if v}
    assert not bad, f"{label}: out-of-range accesses (family: 1 + site) {bad}"


def backward():
    shapes = [(1, 8, {}), (129, 72, {}), (300, 520, {"addend": True}), (1000, 1032, {}),
              (1537, 5128, {}), (700, 20480, {}), (4096, 20480, {})]
    for T, K, kw in shapes:
        wl = WL.make("chk", T=T, K=K, seed=3 + T, **kw)
        for fma in (False, True):
            for comp in (False, True):
                dx, dw = run_gpu(wl, fma_kernel=fma, compensated_dw=comp)
                label = f"backward T={T} K={K} fma={fma} compensated={comp}"
                no_sites(label)
                if T * K <= 2 * 1024 * 1024:
                    assert_parity_full(wl, dx, dw, label)
                else:
                    assert_parity_all_rows(wl, dx, dw, label)


def backward_caps_split_accumulate():
    wl = WL.make("chk_cap", T=1537, K=5128, seed=9)
    i = to_dev(wl)
    ref = None
    for cap in (0, 1, 5, 77):
        plan = Plan(wl.T, wl.K, 0, accumulate_dw=True)
        plan.set_max_ctas(cap)
        dx = torch.empty((wl.T, wl.K), dtype=torch.bfloat16, device=DEV)
        dw = torch.zeros((24, wl.K), device=DEV)
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=DEV)
        plan.execute_dx(i["x"], i["w"], i["grad_proj"], i["grad_r"], i["r"], dx, ws)
        plan.reduce_dw(ws, dw)
        plan.reduce_dw(ws, dw)   # the partials survive a stand-alone reduction
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        plan.close()
        got = (dx.view(torch.int16).cpu().numpy(), dw.cpu().numpy())
        if ref is None:
            ref = got
            d_once = run_gpu(wl)[1]
            assert np.array_equal(got[1], (d_once + d_once).astype(np.float32))
        else:
            assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1].view(np.uint32), ref[1].view(np.uint32))
    no_sites("split, accumulate, grid caps")


def static_scratch():
    wl = WL.make("chk_static", T=700, K=20480, seed=12)
    i = to_dev(wl)
    dx = torch.empty((wl.T, wl.K), dtype=torch.bfloat16, device=DEV)
    dw = torch.empty((24, wl.K), device=DEV)
    abi.mhcpb_execute_static_scratch(wl.T, wl.K, abi.MHCPB_ALLOW_TF32, i["x"].data_ptr(), i["w"].data_ptr(),
                                     i["grad_proj"].data_ptr(), i["grad_r"].data_ptr(), i["r"].data_ptr(),
                                     dx.data_ptr(), dw.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    no_sites("static scratch")
    assert_parity_full(wl, dx.view(torch.int16).cpu().numpy().view(np.uint16), dw.cpu().numpy(), "static scratch")


def forward():
    # caps 1 and 5 at T = 1537 take the output-thread reduction, 0 and 77 the line one;
    # T = 5000 takes the output-thread one on every grid
    for T, K, caps in [(1, 8, (0,)), (129, 72, (0,)), (1537, 5128, (0, 1, 5, 77)), (5000, 2056, (0,)),
                       (4096, 20480, (0,))]:
        wl = WL.make("chk_f", T=T, K=K, seed=30 + T)
        x = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).to(DEV)
        w = torch.from_numpy(wl.w).to(DEV)
        ref_p, ref_r = F.mhc_proj_forward(wl.x, wl.w)
        bound = F.proj_abs_bound(wl.x, wl.w)
        for cap in caps:
            plan = Plan(T, K, 0)
            plan.set_max_ctas(cap)
            proj = torch.full((T, 32), float("nan"), device=DEV)
            r = torch.full((T,), float("nan"), device=DEV)
            ws = torch.empty(plan.forward_workspace_bytes, dtype=torch.uint8, device=DEV)
            plan.forward(x, w, proj, r, ws)
            torch.cuda.synchronize()
            assert plan.device_status() == 0
            plan.close()
            no_sites(f"forward T={T} K={K} cap={cap}")
            ok, st = F.check_proj(proj.cpu().numpy(), ref_p, bound)
            okr, str_ = F.check_r(r.cpu().numpy(), ref_r)
            assert ok and okr, f"forward T={T} cap={cap}: {st} {str_}"
        # the gate step fused into the reduction: the same bits as the gate call on proj and r
        plan = Plan(T, K, 0)
        alpha = torch.tensor([1.0, 0.75, 1.25], device=DEV)
        bias = torch.linspace(-0.5, 0.5, 24, device=DEV)
        p1, r1, h1 = (torch.empty(s_, device=DEV) for s_ in ((T, 32), (T,), (T, 24)))
        h2 = torch.empty((T, 24), device=DEV)
        ws = torch.empty(plan.forward_workspace_bytes, dtype=torch.uint8, device=DEV)
        plan.forward_gates(x, w, alpha, bias, p1, r1, h1, ws)
        mhc_gate_forward(p1, r1, alpha, bias, h2)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        plan.close()
        no_sites(f"forward with gates T={T} K={K}")
        assert torch.equal(h1.view(torch.int32), h2.view(torch.int32)), f"fused gates T={T}"


def gates():
    for T in (1, 17, 5000):
        wl = WL.make_gates("chk_g", T=T, seed=40 + T)
        f = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
        proj, r, al, b, gh = f(wl.proj), f(wl.r), f(wl.alpha), f(wl.bias), f(wl.grad_h)
        h = torch.full((T, 24), float("nan"), device=DEV)
        gp = torch.full((T, 32), float("nan"), device=DEV)
        gr = torch.full((T,), float("nan"), device=DEV)
        dl = torch.full((T, 24), float("nan"), device=DEV)
        mhc_gate_forward(proj, r, al, b, h)
        mhc_gate_backward(proj, r, al, b, gh, gp, gr, dl)
        no_sites(f"gates T={T}")
        okh, sth = G.check_rows(h.cpu().numpy(), G.gate_forward(wl.proj, wl.r, wl.alpha, wl.bias))
        ref_gp, ref_gr, ref_dl = G.gate_backward(wl.proj, wl.r, wl.alpha, wl.bias, wl.grad_h)
        okg, stg = G.check_rows(gp.cpu().numpy(), ref_gp)
        okd, std = G.check_rows(dl.cpu().numpy(), ref_dl)
        # grad_r, a sum of 24 terms of either sign: 1e-4 of the terms' magnitudes
        # (the tolerance of tests/test_gates_gpu.py)
        a = G.alpha_per_column(wl.alpha)
        mag = np.abs(ref_dl * a[None, :] * wl.proj[:, :24].astype(np.float64)).sum(1) / wl.r.astype(np.float64) ** 2
        err = np.abs(gr.cpu().numpy() - ref_gr)
        okr = bool(np.all(err <= 1e-4 * mag + 1e-30))
        assert okh and okg and okr and okd, f"gates T={T}: {sth} {stg} grad_r ok={okr} {std}"


def empty():
    plan = Plan(0, 520, 0)
    w = torch.ones((24, 520), device=DEV)
    dw = torch.full((24, 520), 3.0, device=DEV)
    abi.mhcpb_execute(plan.handle, 0, w.data_ptr(), 0, 0, 0, 0, dw.data_ptr(), 0, 0, None,
                      torch.cuda.current_stream().cuda_stream)
    no_sites("empty batch")
    assert not dw.any()
    plan.close()


if __name__ == "__main__":
    for step in (backward, backward_caps_split_accumulate, static_scratch, forward, gates, empty):
        step()
        print(f"{step.__name__}: no out-of-range access, parity holds", flush=True)
    print("checked build ok")
