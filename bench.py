#!/usr/bin/env python3
"""Benchmark of the mHC projection/RMS backward on GB300.

One step = one backward (both kernels) over the training-profile workload
(T=4096 tokens, K = 4 streams x hidden 5120 = 20480), synthetic seeded inputs
already resident in HBM.  The metric is achieved HBM bandwidth: algorithmic
bytes (read X, write dX, read W, write dW, read the 24 used grad_proj columns,
read r and grad_r) divided by the step time measured with CUDA events on the
launching stream.  Every timed step is preceded by an L2 flush (a 256 MiB
write, outside the events) and has its own pair of events; the step time is
the median over the timed steps.  Also reported: the median of a separate run
of at least 200 flushed steps, the same steps back to back between one pair of
events (`block`: allowed because the inputs are larger than L2), each kernel
alone, the end-to-end call with host buffers, the stage's forward, and the
oracle on the host cores.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 (launched by torch.distributed.run) every rank runs an independent
replica on its own GPU: the stage has no exchange step (the per-rank dW is
the caller's to combine), so there is no collective on the data path; ranks
only meet at barriers and for the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rms_backward_gb300 import workloads as WL  # noqa: E402

METRIC = "mHC proj-bwd µs and achieved HBM GB/s (% of GB300 peak) at T=4096, K=20480"
WORKLOAD = "training_profile"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--kernel", choices=["tcgen05", "fma"], default="tcgen05")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["training_profile", "long_sublayer", "edge", "fused_addend"],
                    help="the headline is the training profile; the others are extra lines")
    ap.add_argument("--stage", choices=["backward", "forward", "gates"], default="backward",
                    help="backward (the headline), the stage's forward (proj and r), or the "
                         "gate/normalisation step's backward (grad_proj and grad_r from the "
                         "gates' gradients) at the workload's T")
    ap.add_argument("--compensated-dw", action="store_true",
                    help="plan flag MHCPB_COMPENSATED_DW (TwoSum dW reduction, one rounding)")
    ap.add_argument("--timing", choices=["block", "flushed"], default="flushed",
                    help="flushed (the headline): L2 flushed before every step, events "
                         "around each step, median over the steps; block: the K steps back "
                         "to back between two events, no L2 flush (only when the step's "
                         "inputs are larger than L2)")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: the oracle's time budget for warm-up plus timed "
                         "steps, which sets the tokens each step processes")
    ap.add_argument("--quick", action="store_true",
                    help="warm-up and timed steps only (for profiler runs); prints a short line")
    ap.add_argument("--no-forward", action="store_true",
                    help="skip the forward side measurement of the backward line")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the long-sublayer (T=16384) side measurement of the backward line")
    ap.add_argument("--cpu-worker", default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


def _dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def _max_over_ranks(x: float, world: int) -> float:
    """The largest of the ranks' values (all ranks get it); x itself at N = 1."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _replica_seed(seed: int, rank: int) -> int:
    """Every replica draws its own inputs."""
    return seed + 97 * rank


def _aggregate_gbs(bytes_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: the bytes all ranks moved over the slowest rank's time."""
    return world * bytes_per_rank / (max_ms * 1e-3) / 1e9


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ oracle timing
class _CpuClock:
    """Wall time and process CPU time (all threads) over the timed oracle calls;
    their ratio is the number of cores the oracle actually kept busy."""

    def __init__(self):
        self.wall = 0.0
        self.cpu = 0.0

    def __enter__(self):
        self._w, self._c = time.perf_counter(), time.process_time()
        return self

    def __exit__(self, *exc):
        self.wall += time.perf_counter() - self._w
        self.cpu += time.process_time() - self._c

    def cores(self):
        return round(self.cpu / self.wall, 1) if self.wall > 0 else 1.0


def _cpu_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        blas = [d["num_threads"] for d in info if d.get("user_api") == "blas"]
        if blas:
            return int(max(blas))
    except Exception:
        pass
    return None   # not known without threadpoolctl


def run_reference(args):
    """The oracle as the reference arm: each step runs it on a bounded slice of
    the training-profile workload, sized so the whole run stays within a few
    minutes."""
    rank, world, _ = _dist_env()
    if rank != 0:
        return 0
    run_oracle, impl = _oracle_impl()
    T, K = WL.CONFIGS[WORKLOAD]["T"], WL.CONFIGS[WORKLOAD]["K"]
    # calibrate tokens per step against the time budget for warmup + steps
    probe = WL.make("ref_probe", T=64, K=K, seed=77)
    run_oracle(probe.x, probe.w, probe.grad_proj, probe.grad_r, probe.r)   # first call: set-up
    t0 = time.perf_counter()
    run_oracle(probe.x, probe.w, probe.grad_proj, probe.grad_r, probe.r)
    per_token = (time.perf_counter() - t0) / 64
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    tok = int(max(1, min(T, budget / max(per_token, 1e-9))))
    wl = WL.make("ref_step", T=tok, K=K, seed=78)
    for _ in range(args.warmup):
        run_oracle(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    clock = _CpuClock()
    with clock:
        for _ in range(args.steps):
            run_oracle(wl.x, wl.w, wl.grad_proj, wl.grad_r, wl.r)
    secs = clock.wall
    gbs = WL.algorithmic_bytes(tok, K) * args.steps / secs / 1e9
    cores = clock.cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"training profile T={T} K={K} (4 streams x hidden 5120)",
                   "T": T, "K": K, "sample_tokens_per_step": tok},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "impl": impl,
                         "cores_available": os.cpu_count(), "blas_threads": _cpu_threads(),
                         "sample": f"{tok} tokens x K={K} of the training profile per step"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
# the sources the streaming (tensor-core) kernel is compiled from
_STREAMING_KERNEL_SOURCES = ("mhcpb_check.cuh", "mhcpb_internal.h", "mhcpb_tc.cu", "mhcpb_wait.cuh", "ptx.cuh")


def _l2_bytes(dev):
    import torch
    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (132 << 20))


def _timing_mode(args, input_bytes, dev):
    """Timing rule: between timed steps either flush L2 or use inputs larger
    than L2.  The headline flushes; block timing (K steps back to back between
    two events) needs inputs larger than L2."""
    big = input_bytes > _l2_bytes(dev)
    if args.timing == "block" and not big:
        raise SystemExit("--timing block needs inputs larger than L2")
    return args.timing


def _step_times(step, flush, steps, mode, stream):
    """Per-step times in ms.  flushed: L2 flushed before every step (outside
    the events), a pair of events around each step, one time per step.  block:
    one pair of events around `steps` back-to-back steps, one mean time."""
    import torch
    if mode == "block":
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) / steps]
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush.fill_(float(i & 7))
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def _timed_steps(step, flush, steps, mode, stream):
    """ms per step: the median of the flushed steps' times, or the block mean."""
    return float(np.median(_step_times(step, flush, steps, mode, stream)))


def _stats_us(times_ms):
    t = np.asarray(times_ms, dtype=np.float64) * 1e3
    return {"reps": int(t.size), "median_us": float(np.median(t)), "mean_us": float(np.mean(t)),
            "p10_us": float(np.percentile(t, 10)), "p90_us": float(np.percentile(t, 90)),
            "min_us": float(np.min(t))}


def _l2_note(mode, input_bytes, dev):
    if mode == "block":
        return (f"not flushed: the step's inputs ({input_bytes / 1e6:.0f} MB) are larger than L2 "
                f"({_l2_bytes(dev) / 1e6:.0f} MB); the K steps run back to back between two events")
    return ("flushed before every timed step (256 MiB write, outside the events); "
            "median of the per-step times")


def _kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rms_backward_gb300", "csrc")
    for name in _STREAMING_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def _ncu_traffic(kernel):
    """DRAM bytes per launch of the streaming kernel from the committed ncu
    summary, if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel)
        if ent and ent.get("source_hash") == _kernel_source_hash():
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def _ncu_l2_writes(kernel):
    """L2 write bytes per launch of the streaming kernel (ncu lts write
    sectors x 32) from the committed summary, if taken on the current sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel)
        if ent and ent.get("source_hash") == _kernel_source_hash() and "l2_write_bytes_per_launch" in ent:
            return float(ent["l2_write_bytes_per_launch"])
    except Exception:
        pass
    return None


def _forward_side(plan, x, w, flush, stream, T, K, peak, reps=100):
    """The stage's forward on the same X and W: flushed per-call median, and
    each of its two kernels alone (events between them)."""
    import torch
    from rms_backward_gb300 import abi
    lib = abi.load()
    proj = torch.empty((T, 32), dtype=torch.float32, device=x.device)
    r = torch.empty((T,), dtype=torch.float32, device=x.device)
    wsb = plan.forward_workspace_bytes
    ws = torch.empty(wsb, dtype=torch.uint8, device=x.device)
    sh = stream.cuda_stream
    eps = 1e-6

    def call():
        abi.mhcpb_forward(plan.handle, x.data_ptr(), w.data_ptr(), eps, proj.data_ptr(),
                          r.data_ptr(), ws.data_ptr(), wsb, sh)

    for _ in range(5):
        flush.fill_(1.0)
        call()
    times = _step_times(call, flush, reps, "flushed", stream)
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    k1, k2 = [], []
    for _ in range(reps):
        flush.fill_(1.0)
        e0.record(stream)
        e1.record(stream)
        e2.record(stream)
        st = lib.mhcpb_forward_profiled(plan.handle, x.data_ptr(), w.data_ptr(), eps,
                                        proj.data_ptr(), r.data_ptr(), ws.data_ptr(), wsb, sh,
                                        e0.cuda_event, e1.cuda_event, e2.cuda_event)
        if st != 0:
            raise RuntimeError(f"mhcpb_forward_profiled: {abi.status_string(st)}")
        e2.synchronize()
        k1.append(e0.elapsed_time(e1))
        k2.append(e1.elapsed_time(e2))
    if plan.device_status() != 0:
        raise RuntimeError("device-side timeout in the forward")
    # the gate step after it: fused into the forward's reduction, and as the
    # separate gate call after the plain forward (flushed before each pair)
    rng = np.random.default_rng(0)
    alpha = torch.from_numpy(rng.uniform(0.5, 1.5, 3).astype(np.float32)).to(x.device)
    bias = torch.from_numpy(rng.normal(0, 0.5, 24).astype(np.float32)).to(x.device)
    h = torch.empty((T, 24), dtype=torch.float32, device=x.device)
    from rms_backward_gb300 import mhc_gate_forward

    def fused():
        abi.mhcpb_forward_gates(plan.handle, x.data_ptr(), w.data_ptr(), eps, alpha.data_ptr(),
                                bias.data_ptr(), 20, proj.data_ptr(), r.data_ptr(), h.data_ptr(),
                                ws.data_ptr(), wsb, sh)

    def separate():
        call()
        mhc_gate_forward(proj, r, alpha, bias, h, n_iter=20, stream=sh)

    for _ in range(3):
        flush.fill_(1.0)
        fused()
        separate()
    t_fused = _step_times(fused, flush, reps, "flushed", stream)
    t_sep = _step_times(separate, flush, reps, "flushed", stream)
    if plan.device_status() != 0:
        raise RuntimeError("device-side timeout in the forward")
    alg = WL.algorithmic_bytes_forward(T, K)
    med = float(np.median(times))
    k1_bytes = 2 * T * K + 96 * K
    k1_mean = float(np.mean(k1))
    return {"metric": "forward (proj = X W^T over TF32 W, r = RMS) achieved HBM GB/s",
            "flushed": _stats_us(times), "value": alg / (med * 1e-3) / 1e9,
            "pct_of_hbm_peak": 100.0 * alg / (med * 1e-3) / 1e9 / peak,
            "algorithmic_bytes_per_step": alg,
            "kernel_us": k1_mean * 1e3, "kernel_median_us": float(np.median(k1)) * 1e3,
            "reduce_us": float(np.mean(k2)) * 1e3,
            "kernel_frac": k1_bytes / (k1_mean * 1e-3) / 1e9 / peak,
            "kernel_algorithmic_bytes": k1_bytes,
            "with_gates": {"fused_flushed": _stats_us(t_fused), "separate_flushed": _stats_us(t_sep),
                           "n_iter": 20,
                           "how": "mhcpb_forward_gates against mhcpb_forward then mhcpb_gate_forward, "
                                  "L2 flushed before each call or pair; median of the per-call times"}}


def _gates_side(T, flush, stream, peak, reps=100, n_iter=20):
    """The gate/normalisation step at T tokens (its own seeded inputs): the
    backward (grad_proj and grad_r from the gates' gradients) and the forward,
    flushed per-call medians."""
    import torch
    from rms_backward_gb300 import mhc_gate_backward, mhc_gate_forward
    g = WL.make_gates("bench_gates", T=T, seed=11)
    dev = flush.device
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    proj, r, al, b, gh = f(g.proj), f(g.r), f(g.alpha), f(g.bias), f(g.grad_h)
    gp = torch.empty((T, 32), dtype=torch.float32, device=dev)
    gr = torch.empty((T,), dtype=torch.float32, device=dev)
    h = torch.empty((T, 24), dtype=torch.float32, device=dev)
    out = {}
    for name, call, nbytes in (
            ("backward", lambda: mhc_gate_backward(proj, r, al, b, gh, gp, gr, n_iter=n_iter, stream=stream),
             T * (96 + 4 + 96 + 128 + 4)),
            ("forward", lambda: mhc_gate_forward(proj, r, al, b, h, n_iter=n_iter, stream=stream),
             T * (96 + 4 + 96))):
        for _ in range(5):
            call()
        st = _stats_us(_step_times(call, flush, reps, "flushed", stream))
        gbs = nbytes / (st["median_us"] * 1e-6) / 1e9
        out[name] = dict(st, algorithmic_bytes=nbytes, achieved_gbs=gbs, frac_of_hbm_peak=gbs / peak)
    out["config"] = {"T": T, "n_iter": n_iter, "threads_per_token": 16}
    return out


def _oracle_impl():
    """The oracle the CPU baseline times: the C one (FP64 loops, OpenMP over
    rows; bit-equal to the numpy oracle) when it is built, else numpy."""
    try:
        import oracle.mhcpb_oracle_c as OC
        OC.load()
        return OC.mhc_proj_rms_backward, "C (FP64 loops, OpenMP over rows)"
    except Exception:
        import oracle.mhcpb_oracle as O
        return (lambda x, w, gp, gr, r: O.mhc_proj_rms_backward(x, w, gp, gr, r)), "numpy (FP64)"


def _long_side(lib_abi, flush, stream, peak, reps=50):
    """The same backward at the long sublayer (T=16384, K=20480): flushed
    per-step median.  Its fixed per-step costs (launch, ramp-up, drain, the
    reduction) weigh four times less than at the training profile."""
    import torch
    from rms_backward_gb300 import Plan
    cfg = dict(WL.CONFIGS["long_sublayer"])
    T, K = cfg["T"], cfg["K"]
    wl = WL.make("long_sublayer", **cfg)
    dev = flush.device
    x = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).to(dev)
    w, gp = torch.from_numpy(wl.w).to(dev), torch.from_numpy(wl.grad_proj).to(dev)
    gr, r = torch.from_numpy(wl.grad_r).to(dev), torch.from_numpy(wl.r).to(dev)
    del wl
    plan = Plan(T, K, dev.index or 0)
    dx = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((24, K), dtype=torch.float32, device=dev)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    sh = stream.cuda_stream

    def step():
        lib_abi.mhcpb_execute(plan.handle, x.data_ptr(), w.data_ptr(), gp.data_ptr(), gr.data_ptr(),
                              r.data_ptr(), dx.data_ptr(), dw.data_ptr(), ws.data_ptr(),
                              plan.workspace_bytes, None, sh)

    for _ in range(5):
        flush.fill_(1.0)
        step()
    st = _stats_us(_step_times(step, flush, reps, "flushed", stream))
    chain = _sublayer_chain(plan, x, w, r, dx, dw, ws, flush, stream, reps)
    if plan.device_status() != 0:
        raise RuntimeError("device-side timeout at the long sublayer")
    plan.close()
    alg = WL.algorithmic_bytes(T, K)
    gbs = alg / (st["median_us"] * 1e-6) / 1e9
    return dict(st, T=T, K=K, value=gbs, unit="GB/s", pct_of_hbm_peak=100.0 * gbs / peak,
                how=_l2_note("flushed", 2 * T * K, None), chain=chain)


def _sublayer_chain(plan, x, w, r, dx, dw, ws, flush, stream, reps):
    """The parts of an mHC sublayer's forward and backward this library
    covers, in order, at the long sublayer: the forward with the gates fused
    in, the gate backward, then this stage's backward fed by it.  Flushed
    medians of the chain and of each part alone.  Context beside the pages'
    per-sublayer figure at 16k tokens, which covers more (the stream collapse
    and the rest of the layer)."""
    import torch
    from rms_backward_gb300 import mhc_gate_backward
    T, K = plan.T, plan.K
    dev = x.device
    rng = np.random.default_rng(1)
    alpha = torch.from_numpy(rng.uniform(0.5, 1.5, 3).astype(np.float32)).to(dev)
    bias = torch.from_numpy(rng.normal(0, 0.5, 24).astype(np.float32)).to(dev)
    gh = torch.from_numpy(rng.normal(0, 1e-2, (T, 24)).astype(np.float32)).to(dev)
    proj = torch.empty((T, 32), dtype=torch.float32, device=dev)
    rr = torch.empty((T,), dtype=torch.float32, device=dev)
    h = torch.empty((T, 24), dtype=torch.float32, device=dev)
    gp = torch.empty((T, 32), dtype=torch.float32, device=dev)
    gr = torch.empty((T,), dtype=torch.float32, device=dev)
    fws = torch.empty(plan.forward_workspace_bytes, dtype=torch.uint8, device=dev)
    sh = stream.cuda_stream

    def fwd():
        plan.forward_gates(x, w, alpha, bias, proj, rr, h, fws, stream=sh)

    def gbwd():
        mhc_gate_backward(proj, rr, alpha, bias, gh, gp, gr, stream=sh)

    def bwd():
        plan.execute(x, w, gp, gr, rr, dx, dw, ws, stream=sh)

    def chain():
        fwd()
        gbwd()
        bwd()

    for _ in range(3):
        flush.fill_(1.0)
        chain()
    out = {"total": _stats_us(_step_times(chain, flush, reps, "flushed", stream))}
    for name, fn in (("forward_gates", fwd), ("gate_backward", gbwd), ("backward", bwd)):
        out[name + "_median_us"] = _stats_us(_step_times(fn, flush, reps, "flushed", stream))["median_us"]
    out["how"] = ("mhcpb_forward_gates, mhcpb_gate_backward, mhcpb_execute in sequence at T=16384, "
                  "K=20480, 20 Sinkhorn iterations, L2 flushed before each chain or part; the parts "
                  "of an mHC sublayer this library covers, not the whole sublayer")
    return out


def _cpu_worker(spec):
    """Child process of the CPU baseline: times the oracle on one config with
    the cores the parent left it; prints one JSON line."""
    run_oracle, impl = _oracle_impl()
    cfg = json.loads(spec)
    reps, seconds = int(cfg["reps"]), float(cfg["seconds"])
    if cfg["config"] == "tiny":
        wl = WL.config("tiny")
        pieces = [wl]
        T_full, K = wl.T, wl.K
    else:
        T_full, K = WL.CONFIGS[WORKLOAD]["T"], WL.CONFIGS[WORKLOAD]["K"]
        pieces = [WL.make("cpu_sample", T=512, K=K, seed=1 + 1000 * i) for i in range(8)]
    rates, cores, toks = [], [], []
    for _ in range(reps):
        clock = _CpuClock()
        nbytes, done, i = 0, 0, 0
        while clock.wall < seconds or i == 0:
            pc = pieces[i % len(pieces)]
            with clock:
                run_oracle(pc.x, pc.w, pc.grad_proj, pc.grad_r, pc.r)
            nbytes += WL.algorithmic_bytes(pc.T, pc.K)
            done += pc.T
            i += 1
        rates.append(nbytes / clock.wall / 1e9)
        cores.append(clock.cores())
        toks.append(done)
    print(json.dumps({"gbs": rates, "cores": cores, "tokens": toks, "T_full": T_full, "K": K,
                      "impl": impl}), flush=True)
    return 0


def _cpu_baseline_protocol(T, K, reps=3):
    """The oracle on the host cores, as the CPU baseline: the training profile
    and the tiny config, each on every core and on one core, median of `reps`
    bounded runs.  Each setting runs in a child process, so the BLAS thread
    count is fixed before numpy loads (one core: affinity to one CPU and one
    BLAS thread)."""
    nproc = os.cpu_count()
    out = {}
    for cores_mode in ("all", "one"):
        env = dict(os.environ)
        pre = None
        if cores_mode == "one":
            for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                      "BLIS_NUM_THREADS"):
                env[v] = "1"
            first = sorted(os.sched_getaffinity(0))[0]
            pre = lambda: os.sched_setaffinity(0, {first})  # noqa: E731
        for cfg, secs in (("training", 3.0), ("tiny", 0.5)):
            spec = json.dumps({"config": cfg, "reps": reps, "seconds": secs})
            res = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", spec],
                                 env=env, preexec_fn=pre, capture_output=True, text=True,
                                 timeout=600)
            try:
                d = json.loads(res.stdout.strip().splitlines()[-1])
            except Exception:
                out[f"{cfg}_{cores_mode}"] = {"error": (res.stderr or res.stdout)[-300:]}
                continue
            out[f"{cfg}_{cores_mode}"] = {
                "impl": d.get("impl"),
                "median_gbs": float(np.median(d["gbs"])), "runs_gbs": d["gbs"],
                "cores_busy": float(np.median(d["cores"])), "tokens_per_run": d["tokens"],
                "seconds_per_run": secs}
    head = out.get("training_all", {})
    return {"value": head.get("median_gbs"), "unit": "GB/s", "cores": head.get("cores_busy"),
            "kind": "oracle", "impl": head.get("impl"), "nproc": nproc,
            "sample": (f"median of {reps} runs of about 3 s each over 512-token slices of the "
                       f"training profile (T={T}, K={K}), on all {nproc} host cores"),
            "protocol": out}


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = _dist_env()
    if world != args.gpus:
        if rank == 0:
            print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from rms_backward_gb300 import Plan, abi

    cfg = dict(WL.CONFIGS[args.workload])
    T, K = cfg["T"], cfg["K"]
    cfg["seed"] = _replica_seed(cfg["seed"], rank)
    wl = WL.make(args.workload, **cfg)
    has_add = wl.has_addend
    plan = Plan(T, K, local, addend=has_add, fma_kernel=(args.kernel == "fma"),
                compensated_dw=args.compensated_dw)

    pin = lambda a: torch.from_numpy(a).pin_memory()  # noqa: E731
    h_x = pin(wl.x.view(np.int16)).view(torch.bfloat16)
    h_w, h_gp, h_gr, h_r = pin(wl.w), pin(wl.grad_proj), pin(wl.grad_r), pin(wl.r)
    x = h_x.to(dev)
    w, gp, gr, r = h_w.to(dev), h_gp.to(dev), h_gr.to(dev), h_r.to(dev)
    h_add = pin(wl.addend.view(np.int16)).view(torch.bfloat16) if has_add else None
    add = h_add.to(dev) if has_add else None
    add_ptr = add.data_ptr() if has_add else None
    dx = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((24, K), dtype=torch.float32, device=dev)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def step():
        abi.mhcpb_execute(plan.handle, x.data_ptr(), w.data_ptr(), gp.data_ptr(), gr.data_ptr(),
                          r.data_ptr(), dx.data_ptr(), dw.data_ptr(), ws.data_ptr(),
                          plan.workspace_bytes, add_ptr, sh)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if plan.device_status() != 0:
        raise RuntimeError("device-side timeout during warm-up")

    if args.quick:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / max(1, args.steps)
        if rank == 0:
            print(json.dumps({"quick": True, "kernel": args.kernel, "steps": args.steps,
                              "ms_per_step_no_flush": ms}), flush=True)
        status = plan.device_status()
        plan.close()
        return 0 if status == 0 else 1

    input_bytes = 2 * T * K * (2 if has_add else 1)   # X (and the addend)
    mode = _timing_mode(args, input_bytes, dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    times = _step_times(step, flush, args.steps, mode, stream)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    if plan.device_status() != 0:
        raise RuntimeError("device-side timeout during the timed steps")
    step_ms = float(np.median(times))
    step_ms_max = _max_over_ranks(step_ms, world)

    alg = WL.algorithmic_bytes(T, K, addend=has_add)
    value = _aggregate_gbs(alg, world, step_ms_max)
    peak, peak_kind = _peaks()
    # side measurements (same rank set, max over ranks of each median):
    # a longer flushed run (>= 200 steps) and the block timing
    long_n = max(200, args.steps)
    long_f = _step_times(step, flush, long_n, "flushed", stream)
    lf_ms = _max_over_ranks(float(np.median(long_f)), world)
    flushed = dict(_stats_us(long_f), value=_aggregate_gbs(alg, world, lf_ms),
                   pct_of_hbm_peak=100.0 * (_aggregate_gbs(alg, world, lf_ms) / world) / peak,
                   how=_l2_note("flushed", input_bytes, dev))
    block = None
    if input_bytes > _l2_bytes(dev):
        b_ms = _max_over_ranks(_timed_steps(step, flush, long_n, "block", stream), world)
        b_val = _aggregate_gbs(alg, world, b_ms)
        block = {"us_per_step": b_ms * 1e3, "steps": long_n, "value": b_val,
                 "pct_of_hbm_peak": 100.0 * (b_val / world) / peak,
                 "how": _l2_note("block", input_bytes, dev)}

    # dominant kernel (the streaming kernel) timed alone: events around each kernel
    lib = abi.load()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    k1, k2 = [], []
    for i in range(200):
        flush.fill_(1.0)
        # torch only knows an event was recorded if it recorded it itself; the
        # library then re-records the same handles at the kernel boundaries
        e0.record(stream)
        e1.record(stream)
        e2.record(stream)
        st = lib.mhcpb_execute_profiled(
            plan.handle, x.data_ptr(), w.data_ptr(), gp.data_ptr(), gr.data_ptr(), r.data_ptr(),
            dx.data_ptr(), dw.data_ptr(), ws.data_ptr(), plan.workspace_bytes, add_ptr, sh,
            e0.cuda_event, e1.cuda_event, e2.cuda_event)
        if st != 0:
            raise RuntimeError(f"mhcpb_execute_profiled: {abi.status_string(st)}")
        e2.synchronize()
        k1.append(e0.elapsed_time(e1))
        k2.append(e1.elapsed_time(e2))
    k1_ms, k2_ms = float(np.mean(k1)), float(np.mean(k2))
    k1_med_ms = float(np.median(k1))
    k1_bytes = alg - 96 * K          # everything but the dW write, which kernel 2 does
    k1_gbs = k1_bytes / (k1_ms * 1e-3) / 1e9

    # end to end through the public call with host buffers: every step copies
    # its inputs in from pinned host memory, runs the backward and reads dX and
    # dW back.  Steps are pipelined over three streams with two device buffer
    # sets: step i's inputs go in while step i-1 computes and step i-2's
    # results come out (each set is reused only after its previous step's
    # results are out).
    h_dx = [torch.empty((T, K), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h_dw = [torch.empty((24, K), dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = x.numel() * 2 + w.numel() * 4 + gp.numel() * 4 + gr.numel() * 4 + r.numel() * 4
    h2d += add.numel() * 2 if has_add else 0
    d2h = dx.numel() * 2 + dw.numel() * 4
    sets = [dict(x=x, w=w, gp=gp, gr=gr, r=r, add=add, dx=dx, dw=dw)]
    sets.append(dict(x=torch.empty_like(x), w=torch.empty_like(w), gp=torch.empty_like(gp),
                     gr=torch.empty_like(gr), r=torch.empty_like(r),
                     add=torch.empty_like(add) if has_add else None,
                     dx=torch.empty_like(dx), dw=torch.empty_like(dw)))
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_steps(n):
        comp_done, out_done = [], []
        for i in range(n):
            b = sets[i % 2]
            ev_in = torch.cuda.Event()
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])   # step i-2 has read this set's inputs
                b["x"].copy_(h_x, non_blocking=True)
                b["w"].copy_(h_w, non_blocking=True)
                b["gp"].copy_(h_gp, non_blocking=True)
                b["gr"].copy_(h_gr, non_blocking=True)
                b["r"].copy_(h_r, non_blocking=True)
                if has_add:
                    b["add"].copy_(h_add, non_blocking=True)
                ev_in.record(s_in)
            s_comp.wait_event(ev_in)
            if i >= 2:
                s_comp.wait_event(out_done[i - 2])      # step i-2's results are out of this set
            abi.mhcpb_execute(plan.handle, b["x"].data_ptr(), b["w"].data_ptr(), b["gp"].data_ptr(),
                              b["gr"].data_ptr(), b["r"].data_ptr(), b["dx"].data_ptr(),
                              b["dw"].data_ptr(), ws.data_ptr(), plan.workspace_bytes,
                              b["add"].data_ptr() if has_add else None, s_comp.cuda_stream)
            ev_c = torch.cuda.Event()
            ev_c.record(s_comp)
            comp_done.append(ev_c)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c)
                h_dx[i % 2].copy_(b["dx"], non_blocking=True)
                h_dw[i % 2].copy_(b["dw"], non_blocking=True)
                ev_o = torch.cuda.Event()
                ev_o.record(s_out)
                out_done.append(ev_o)

    e2e_steps(4)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(s_in)
    s_comp.wait_event(ea)
    s_out.wait_event(ea)
    e2e_steps(args.e2e_steps)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_comp)
    eb.record(s_out)
    torch.cuda.synchronize()
    if plan.device_status() != 0:
        raise RuntimeError("device-side timeout in the end-to-end steps")
    e2e_ms = _max_over_ranks(ea.elapsed_time(eb) / args.e2e_steps, world)
    e2e_value = _aggregate_gbs(alg, world, e2e_ms)
    # the same loop one step at a time (no overlap between steps), for comparison
    n_serial = max(5, args.e2e_steps // 3)
    eo, ef = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    eo.record(stream)
    for _ in range(n_serial):
        x.copy_(h_x, non_blocking=True)
        w.copy_(h_w, non_blocking=True)
        gp.copy_(h_gp, non_blocking=True)
        gr.copy_(h_gr, non_blocking=True)
        r.copy_(h_r, non_blocking=True)
        if has_add:
            add.copy_(h_add, non_blocking=True)
        step()
        h_dx[0].copy_(dx, non_blocking=True)
        h_dw[0].copy_(dw, non_blocking=True)
    ef.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = eo.elapsed_time(ef) / n_serial

    fwd = None
    gates = None
    if not args.no_forward and not has_add:
        fwd = _forward_side(plan, x, w, flush, stream, T, K, peak)
        gates = _gates_side(T, flush, stream, peak)
    long_sub = None
    if not args.no_long and args.workload == WORKLOAD and args.kernel == "tcgen05" and rank == 0 \
            and world == 1:
        long_sub = _long_side(abi, flush, stream, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == WORKLOAD:
        cpu = _cpu_baseline_protocol(T, K)

    metric = METRIC if args.workload == WORKLOAD else \
        f"mHC proj-bwd achieved HBM GB/s at T={T}, K={K} ({args.workload})"
    desc = {"training_profile": "training profile", "long_sublayer": "long sublayer",
            "edge": "edge (rows scaled 10^U(-3,3), grad_proj[:, 24:] = +-1e30)",
            "fused_addend": "training profile with the fused BF16 addend"}[args.workload]
    if rank == 0:
        line = {
            "metric": metric, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": step_ms_max, "us_per_step": step_ms_max * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "tf32", "data": "synthetic",
            "precision": ("products exact in TF32 (each TF32 operand split into BF16 hi + lo on "
                          "BF16 tensor cores), FP32 accumulation; X and dX BF16, W, grad_proj, "
                          "dW FP32") if args.kernel == "tcgen05" else
                         "TF32-rounded operands, FP32 FMA on CUDA cores; X and dX BF16, dW FP32",
            "config": {"workload": f"{desc} T={T} K={K} (4 streams x hidden 5120)",
                       "T": T, "K": K, "kernel": args.kernel, "addend": has_add,
                       "dw_reduction": "compensated" if args.compensated_dw else "plain",
                       "parallelism": f"replicas{world}" if world > 1 else "single",
                       "timing": mode, "l2": _l2_note(mode, input_bytes, dev),
                       "algorithmic_bytes_per_step": alg,
                       "pct_of_hbm_peak": 100.0 * (value / world) / peak,
                       "target_pct_of_hbm_peak": 75.0,
                       "wall_s_timed_region": wall},
            "flushed": flushed,
            "block": block,
            "roofline": {"bound": "hbm", "achieved": k1_gbs, "peak": peak, "unit": "GB/s",
                         "frac": k1_gbs / peak, "traffic": _ncu_traffic(args.kernel),
                         "l2_write_bytes": _ncu_l2_writes(args.kernel),
                         "kernel": "streaming kernel (dX + dW partials)",
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "kernel_us": k1_ms * 1e3, "kernel_median_us": k1_med_ms * 1e3,
                         "reduce_us": k2_ms * 1e3,
                         "algorithmic_bytes_per_launch": k1_bytes},
            "forward": fwd,
            "gates": gates,
            "long_sublayer": long_sub,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "how": "pinned host inputs copied in and dX, dW copied out every step; steps "
                           "pipelined over three streams with two device buffer sets",
                    "serial_ms_per_step": e2e_serial_ms,
                    "serial_value": _aggregate_gbs(alg, world, e2e_serial_ms)},
            "gpu_launches": 2 * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    plan.close()
    return 0


def run_forward(args):
    """The stage's forward (mhcpb_forward): proj = X W^T and r = RMS(X) on the
    workload's X and W, same timing rules as the backward."""
    import torch
    import torch.distributed as dist

    rank, world, local = _dist_env()
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from rms_backward_gb300 import Plan, abi

    cfg = dict(WL.CONFIGS[args.workload])
    cfg.pop("addend", None)
    T, K = cfg["T"], cfg["K"]
    cfg["seed"] = _replica_seed(cfg["seed"], rank)
    wl = WL.make(args.workload, **cfg)
    plan = Plan(T, K, local)
    pin = lambda a: torch.from_numpy(a).pin_memory()  # noqa: E731
    h_x = pin(wl.x.view(np.int16)).view(torch.bfloat16)
    h_w = pin(wl.w)
    x, w = h_x.to(dev), h_w.to(dev)
    proj = torch.empty((T, 32), dtype=torch.float32, device=dev)
    r = torch.empty((T,), dtype=torch.float32, device=dev)
    wsb = plan.forward_workspace_bytes
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    eps = 1e-6

    def step():
        abi.mhcpb_forward(plan.handle, x.data_ptr(), w.data_ptr(), eps, proj.data_ptr(),
                          r.data_ptr(), ws.data_ptr(), wsb, sh)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if plan.device_status() != 0:
        raise RuntimeError("device-side timeout during warm-up")
    if args.quick:
        for _ in range(args.steps):
            flush.fill_(1.0)
            step()
        torch.cuda.synchronize()
        status = plan.device_status()
        if rank == 0:
            print(json.dumps({"quick": True, "stage": "forward", "steps": args.steps,
                              "status": status}), flush=True)
        plan.close()
        return 0 if status == 0 else 1
    input_bytes = 2 * T * K   # X
    mode = _timing_mode(args, input_bytes, dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    mean_ms = _timed_steps(step, flush, args.steps, mode, stream)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    if plan.device_status() != 0:
        raise RuntimeError("device-side timeout during the timed steps")
    mean_ms = _max_over_ranks(mean_ms, world)
    alg = WL.algorithmic_bytes_forward(T, K)
    value = _aggregate_gbs(alg, world, mean_ms)
    peak, peak_kind = _peaks()
    long_n = max(200, args.steps)
    long_f = _step_times(step, flush, long_n, "flushed", stream)
    lf_ms = _max_over_ranks(float(np.median(long_f)), world)
    flushed = dict(_stats_us(long_f), value=_aggregate_gbs(alg, world, lf_ms),
                   pct_of_hbm_peak=100.0 * (_aggregate_gbs(alg, world, lf_ms) / world) / peak,
                   how=_l2_note("flushed", input_bytes, dev))
    block = None
    if input_bytes > _l2_bytes(dev):
        b_ms = _max_over_ranks(_timed_steps(step, flush, long_n, "block", stream), world)
        b_val = _aggregate_gbs(alg, world, b_ms)
        block = {"us_per_step": b_ms * 1e3, "steps": long_n, "value": b_val,
                 "pct_of_hbm_peak": 100.0 * (b_val / world) / peak,
                 "how": _l2_note("block", input_bytes, dev)}

    lib = abi.load()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    k1, k2 = [], []
    for i in range(min(200, args.steps)):
        flush.fill_(1.0)
        e0.record(stream)
        e1.record(stream)
        e2.record(stream)
        st = lib.mhcpb_forward_profiled(plan.handle, x.data_ptr(), w.data_ptr(), eps,
                                        proj.data_ptr(), r.data_ptr(), ws.data_ptr(), wsb, sh,
                                        e0.cuda_event, e1.cuda_event, e2.cuda_event)
        if st != 0:
            raise RuntimeError(f"mhcpb_forward_profiled: {abi.status_string(st)}")
        e2.synchronize()
        k1.append(e0.elapsed_time(e1))
        k2.append(e1.elapsed_time(e2))
    k1_ms, k2_ms = float(np.mean(k1)), float(np.mean(k2))
    k1_bytes = 2 * T * K + 96 * K    # kernel 1 reads X and W; kernel 2 writes proj and r
    k1_gbs = k1_bytes / (k1_ms * 1e-3) / 1e9

    h_proj = torch.empty((T, 32), dtype=torch.float32).pin_memory()
    h_r = torch.empty((T,), dtype=torch.float32).pin_memory()
    h2d, d2h = x.numel() * 2 + w.numel() * 4, proj.numel() * 4 + r.numel() * 4
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(args.e2e_steps):
        x.copy_(h_x, non_blocking=True)
        w.copy_(h_w, non_blocking=True)
        step()
        h_proj.copy_(proj, non_blocking=True)
        h_r.copy_(r, non_blocking=True)
    eb.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e2e_ms = _max_over_ranks(ea.elapsed_time(eb) / args.e2e_steps, world)
    e2e_value = _aggregate_gbs(alg, world, e2e_ms)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle.mhcpf_oracle as F
        done, nbytes, i = 0, 0, 0
        clock = _CpuClock()
        while clock.wall < 10.0 and done < T:
            piece = WL.make("cpu_sample", T=256, K=K, seed=cfg["seed"] + 1000 * i)
            with clock:
                F.mhc_proj_forward(piece.x, piece.w)
            done += 256
            nbytes += WL.algorithmic_bytes_forward(256, K)
            i += 1
        secs = clock.wall
        cpu = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": clock.cores(), "kind": "oracle",
               "cores_available": os.cpu_count(), "blas_threads": _cpu_threads(),
               "sample": f"{done} of {T} tokens x K={K} (256-token slices, {secs:.1f} s)"}

    if rank == 0:
        line = {
            "metric": f"mHC proj-fwd achieved HBM GB/s at T={T}, K={K} ({args.workload})",
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": mean_ms, "us_per_step": mean_ms * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "tf32", "data": "synthetic",
            "precision": ("products exact in TF32 (W split into BF16 hi + lo on BF16 tensor "
                          "cores), FP32 accumulation; X BF16, proj and r FP32"),
            "config": {"workload": f"forward, {args.workload} T={T} K={K} (4 streams x hidden 5120)",
                       "T": T, "K": K, "eps": eps,
                       "parallelism": f"replicas{world}" if world > 1 else "single",
                       "timing": mode, "l2": _l2_note(mode, input_bytes, dev),
                       "algorithmic_bytes_per_step": alg,
                       "pct_of_hbm_peak": 100.0 * (value / world) / peak,
                       "wall_s_timed_region": wall},
            "flushed": flushed,
            "block": block,
            "roofline": {"bound": "hbm", "achieved": k1_gbs, "peak": peak, "unit": "GB/s",
                         "frac": k1_gbs / peak, "traffic": None,
                         "kernel": "forward streaming kernel (projection + squares, partials)",
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "kernel_us": k1_ms * 1e3, "reduce_us": k2_ms * 1e3,
                         "algorithmic_bytes_per_launch": k1_bytes},
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": 2 * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    plan.close()
    return 0


def run_gates(args):
    """The gate/normalisation step's backward at the workload's T (one GPU):
    flushed per-call median over the K timed calls; --quick runs the calls
    only (for profiler captures)."""
    import torch
    from rms_backward_gb300 import mhc_gate_backward
    rank, world, local = _dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    T = WL.CONFIGS[args.workload]["T"]
    g = WL.make_gates("bench_gates", T=T, seed=_replica_seed(11, rank))
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    proj, r, al, b, gh = f(g.proj), f(g.r), f(g.alpha), f(g.bias), f(g.grad_h)
    gp = torch.empty((T, 32), dtype=torch.float32, device=dev)
    gr = torch.empty((T,), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        mhc_gate_backward(proj, r, al, b, gh, gp, gr, n_iter=20, stream=stream)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1.0)
        call()
    torch.cuda.synchronize()
    if args.quick:
        for _ in range(args.steps):
            flush.fill_(1.0)
            call()
        torch.cuda.synchronize()
        if rank == 0:
            print(json.dumps({"quick": True, "stage": "gates", "steps": args.steps}), flush=True)
        return 0
    times = _step_times(call, flush, args.steps, "flushed", stream)
    st = _stats_us(times)
    nbytes = T * (96 + 4 + 96 + 128 + 4)
    peak, peak_kind = _peaks()
    gbs = nbytes / (st["median_us"] * 1e-6) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": f"mHC gate/normalisation backward (grad_proj, grad_r) at T={T}, 20 Sinkhorn iterations",
            "value": st["median_us"], "unit": "us", "higher_is_better": False, "n_gpus": 1,
            "steps": args.steps, "warmup": max(3, args.warmup), "dtype": "f32", "data": "synthetic",
            "flushed": st,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "traffic": None, "peak_source": f"{peak_kind} hbm_gbs",
                         "algorithmic_bytes_per_launch": nbytes,
                         "note": "latency-bound: a serial chain of shuffle reductions per token"},
            "config": {"workload": f"gates, T={T}", "T": T, "n_iter": 20}}), flush=True)
    return 0


def main():
    args = _args()
    if args.cpu_worker is not None:
        return _cpu_worker(args.cpu_worker)
    if args.impl == "reference":
        return run_reference(args)
    if args.stage == "forward":
        return run_forward(args)
    if args.stage == "gates":
        return run_gates(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
