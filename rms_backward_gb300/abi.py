"""ctypes binding of the C ABI in ``include/mhcpb.h`` (argument marshalling only).

Every function keeps its C name.  Pointers are plain integers (device
addresses, e.g. ``tensor.data_ptr()``); streams are raw ``cudaStream_t``
handles (``torch.cuda.Stream.cuda_stream``).  A non-OK status raises
:class:`MhcpbError`.  There is no fallback: if ``libmhcpb.so`` has not been
built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB as LIB_PATH

MHCPB_OK = 0
MHCPB_ERR_INVALID_ARG = 1
MHCPB_ERR_UNSUPPORTED_SHAPE = 2
MHCPB_ERR_MISALIGNED = 3
MHCPB_ERR_ALIASING = 4
MHCPB_ERR_WRONG_DEVICE = 5
MHCPB_ERR_TF32_NOT_ALLOWED = 6
MHCPB_ERR_WORKSPACE_TOO_SMALL = 7
MHCPB_ERR_CUDA = 8
MHCPB_ERR_DEVICE_TIMEOUT = 9
MHCPB_ERR_UNSUPPORTED_DEVICE = 10
MHCPB_ERR_SCRATCH_TOO_SMALL = 11

MHCPB_ALLOW_TF32 = 1
MHCPB_HAS_ADDEND = 2
MHCPB_FMA_KERNEL = 4
MHCPB_COMPENSATED_DW = 8
MHCPB_ACCUMULATE_DW = 16
MHCPB_TEST_INJECT_STALL = 1 << 30

MHCPB_NPROJ = 24
MHCPB_GRAD_PROJ_COLS = 32
def MHCPB_PARTIAL_TOKENS(T: int) -> int:
    """Tokens per dW partial (fixed: never a function of the GPU)."""
    return 512

MHCPB_STATIC_SCRATCH_BYTES = 16 << 20
MHCPB_GATE_MAX_ITER = 64

QUERY = {"T": 0, "K": 1, "S": 2, "grid": 3, "flags": 4, "smem": 5, "token_tile": 6, "strip": 7,
         "partial_tokens": 8}

EXPORTED = ("mhcpb_plan_create", "mhcpb_workspace_bytes", "mhcpb_execute", "mhcpb_execute_profiled",
            "mhcpb_get_device_status", "mhcpb_plan_query", "mhcpb_plan_set_wait_limit",
            "mhcpb_destroy", "mhcpb_status_string", "mhcpb_last_cuda_error",
            "mhcpb_execute_static_scratch", "mhcpb_plan_set_max_ctas", "mhcpb_execute_dx",
            "mhcpb_reduce_dw", "mhcpb_forward_workspace_bytes", "mhcpb_forward",
            "mhcpb_forward_profiled", "mhcpb_gate_forward", "mhcpb_gate_backward",
            "mhcpb_debug_checked_sites", "mhcpb_forward_gates")


class MhcpbError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: status {status} ({status_string(status)})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libmhcpb.so (once) and declares the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P, I64, U32, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32, ctypes.c_int, ctypes.c_size_t
    lib.mhcpb_plan_create.argtypes = [ctypes.POINTER(P), I64, I64, I32, U32]
    lib.mhcpb_workspace_bytes.argtypes = [P, ctypes.POINTER(SZ)]
    lib.mhcpb_execute.argtypes = [P, P, P, P, P, P, P, P, P, SZ, P, P]
    lib.mhcpb_execute_profiled.argtypes = [P, P, P, P, P, P, P, P, P, SZ, P, P, P, P, P]
    lib.mhcpb_get_device_status.argtypes = [P, ctypes.POINTER(I32), I32]
    lib.mhcpb_plan_query.argtypes = [P, I32, ctypes.POINTER(I64)]
    lib.mhcpb_plan_set_wait_limit.argtypes = [P, ctypes.c_uint64]
    lib.mhcpb_plan_set_max_ctas.argtypes = [P, I32]
    lib.mhcpb_execute_static_scratch.argtypes = [I64, I64, U32, P, P, P, P, P, P, P, P, P]
    lib.mhcpb_execute_dx.argtypes = [P, P, P, P, P, P, P, P, SZ, P, P]
    lib.mhcpb_reduce_dw.argtypes = [P, P, SZ, P, P]
    lib.mhcpb_forward_workspace_bytes.argtypes = [P, ctypes.POINTER(SZ)]
    lib.mhcpb_forward.argtypes = [P, P, P, ctypes.c_float, P, P, P, SZ, P]
    lib.mhcpb_forward_profiled.argtypes = [P, P, P, ctypes.c_float, P, P, P, SZ, P, P, P, P]
    lib.mhcpb_forward_gates.argtypes = [P, P, P, ctypes.c_float, P, P, I32, P, P, P, P, SZ, P]
    lib.mhcpb_gate_forward.argtypes = [I64, I32, P, P, P, P, P, P]
    lib.mhcpb_gate_backward.argtypes = [I64, I32, P, P, P, P, P, P, P, P, P]
    lib.mhcpb_debug_checked_sites.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(I32)]
    lib.mhcpb_destroy.argtypes = [P]
    lib.mhcpb_status_string.argtypes = [I32]
    lib.mhcpb_status_string.restype = ctypes.c_char_p
    lib.mhcpb_last_cuda_error.argtypes = []
    lib.mhcpb_last_cuda_error.restype = ctypes.c_char_p
    for name in ("mhcpb_plan_create", "mhcpb_workspace_bytes", "mhcpb_execute",
                 "mhcpb_execute_profiled", "mhcpb_get_device_status", "mhcpb_plan_query",
                 "mhcpb_plan_set_wait_limit", "mhcpb_destroy", "mhcpb_execute_static_scratch",
                 "mhcpb_plan_set_max_ctas", "mhcpb_execute_dx", "mhcpb_reduce_dw",
                 "mhcpb_forward_workspace_bytes", "mhcpb_forward", "mhcpb_forward_profiled",
                 "mhcpb_gate_forward", "mhcpb_gate_backward", "mhcpb_debug_checked_sites",
                 "mhcpb_forward_gates"):
        getattr(lib, name).restype = I32
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().mhcpb_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != MHCPB_OK:
        detail = load().mhcpb_last_cuda_error().decode() if status == MHCPB_ERR_CUDA else ""
        raise MhcpbError(status, where, detail)


def mhcpb_plan_create(T: int, K: int, device: int = 0, flags: int = MHCPB_ALLOW_TF32) -> int:
    h = ctypes.c_void_p()
    _check(load().mhcpb_plan_create(ctypes.byref(h), int(T), int(K), int(device), int(flags)),
           "mhcpb_plan_create")
    return h.value


def mhcpb_workspace_bytes(plan: int) -> int:
    n = ctypes.c_size_t()
    _check(load().mhcpb_workspace_bytes(plan, ctypes.byref(n)), "mhcpb_workspace_bytes")
    return n.value


def mhcpb_execute(plan: int, x: int, w: int, grad_proj: int, grad_r: int, r: int, dx: int,
                  dw: int, workspace: int, workspace_bytes: int, grad_x_addend: int | None,
                  stream: int | None) -> None:
    _check(load().mhcpb_execute(plan, x, w, grad_proj, grad_r, r, dx, dw, workspace,
                                int(workspace_bytes), grad_x_addend or None, stream or None),
           "mhcpb_execute")


def mhcpb_execute_dx(plan: int, x: int, w: int, grad_proj: int, grad_r: int, r: int, dx: int,
                     workspace: int, workspace_bytes: int, grad_x_addend: int | None,
                     stream: int | None) -> None:
    _check(load().mhcpb_execute_dx(plan, x, w, grad_proj, grad_r, r, dx, workspace,
                                   int(workspace_bytes), grad_x_addend or None, stream or None),
           "mhcpb_execute_dx")


def mhcpb_reduce_dw(plan: int, workspace: int, workspace_bytes: int, dw: int,
                    stream: int | None) -> None:
    _check(load().mhcpb_reduce_dw(plan, workspace, int(workspace_bytes), dw, stream or None),
           "mhcpb_reduce_dw")


def mhcpb_forward_workspace_bytes(plan: int) -> int:
    n = ctypes.c_size_t()
    _check(load().mhcpb_forward_workspace_bytes(plan, ctypes.byref(n)), "mhcpb_forward_workspace_bytes")
    return n.value


def mhcpb_forward(plan: int, x: int, w: int, eps: float, proj: int, r: int, workspace: int,
                  workspace_bytes: int, stream: int | None) -> None:
    _check(load().mhcpb_forward(plan, x, w, float(eps), proj, r, workspace, int(workspace_bytes),
                                stream or None), "mhcpb_forward")


def mhcpb_forward_gates(plan: int, x: int, w: int, eps: float, alpha: int, bias: int, n_iter: int,
                        proj: int, r: int, h: int, workspace: int, workspace_bytes: int,
                        stream: int | None) -> None:
    """The forward with the gate step fused into its reduction: proj, r and h."""
    _check(load().mhcpb_forward_gates(plan, x, w, float(eps), alpha, bias, int(n_iter), proj, r, h,
                                      workspace, int(workspace_bytes), stream or None),
           "mhcpb_forward_gates")


def mhcpb_get_device_status(plan: int, clear: bool = False) -> int:
    s = ctypes.c_int()
    _check(load().mhcpb_get_device_status(plan, ctypes.byref(s), 1 if clear else 0),
           "mhcpb_get_device_status")
    return s.value


def mhcpb_plan_query(plan: int, which) -> int:
    v = ctypes.c_int64()
    code = QUERY[which] if isinstance(which, str) else int(which)
    _check(load().mhcpb_plan_query(plan, code, ctypes.byref(v)), "mhcpb_plan_query")
    return v.value


def mhcpb_plan_set_wait_limit(plan: int, nanoseconds: int) -> None:
    _check(load().mhcpb_plan_set_wait_limit(plan, int(nanoseconds)), "mhcpb_plan_set_wait_limit")


def mhcpb_plan_set_max_ctas(plan: int, max_ctas: int) -> None:
    _check(load().mhcpb_plan_set_max_ctas(plan, int(max_ctas)), "mhcpb_plan_set_max_ctas")


def mhcpb_destroy(plan: int) -> None:
    _check(load().mhcpb_destroy(plan), "mhcpb_destroy")


def mhcpb_status_string(status: int) -> str:
    return status_string(status)


def mhcpb_last_cuda_error() -> str:
    return load().mhcpb_last_cuda_error().decode()


def mhcpb_execute_static_scratch(T: int, K: int, flags: int, x: int, w: int, grad_proj: int,
                                 grad_r: int, r: int, dx: int, dw: int,
                                 grad_x_addend: int | None, stream: int | None) -> None:
    """The backward without plan or workspace: dW partials in the library's
    built-in 16 MiB device buffer (for callers that cannot allocate)."""
    _check(load().mhcpb_execute_static_scratch(int(T), int(K), int(flags), x, w, grad_proj, grad_r,
                                               r, dx, dw, grad_x_addend or None, stream or None),
           "mhcpb_execute_static_scratch")


def mhcpb_gate_forward(T: int, n_iter: int, proj: int, r: int, alpha: int, bias: int, h: int,
                       stream: int | None) -> None:
    """Gates from the projection logits and r: H_pre, H_post, H_res [T, 24]."""
    _check(load().mhcpb_gate_forward(int(T), int(n_iter), proj, r, alpha, bias, h, stream or None),
           "mhcpb_gate_forward")


def mhcpb_gate_backward(T: int, n_iter: int, proj: int, r: int, alpha: int, bias: int,
                        grad_h: int, grad_proj: int, grad_r: int, dlogits: int | None,
                        stream: int | None) -> None:
    """grad_proj [T, 32] and grad_r [T] (and optionally dL/dlogits [T, 24])
    from the gates' upstream gradients."""
    _check(load().mhcpb_gate_backward(int(T), int(n_iter), proj, r, alpha, bias, grad_h, grad_proj,
                                      grad_r, dlogits or None, stream or None),
           "mhcpb_gate_backward")


CHECKED_FAMILIES = ("tensor-core backward", "FMA backward", "dW reduction", "forward", "gate kernels")


def mhcpb_debug_checked_sites():
    """(checked, sites): whether the loaded library is a bounds-checked build,
    and per kernel family the first out-of-range site recorded since the last
    call (0: none; else 1 + the site), which the call clears."""
    sites = (ctypes.c_uint32 * 5)()
    checked = ctypes.c_int()
    _check(load().mhcpb_debug_checked_sites(sites, ctypes.byref(checked)), "mhcpb_debug_checked_sites")
    return bool(checked.value), dict(zip(CHECKED_FAMILIES, list(sites)))
