"""GB300-native mHC projection/RMS backward.

    P  = grad_proj[:, :24]
    dX = P @ W + grad_r / (r * K) * X        (BF16)
    dW = P.T @ X                              (FP32, fixed-order reduction)

The computation runs in two sm_103a CUDA kernels behind the C ABI of
``include/mhcpb.h`` (``libmhcpb.so``).  This package is the Python side:
``abi`` binds the C functions by name; :class:`Plan` and
:func:`mhc_projection_backward` marshal torch CUDA tensors into them (torch
supplies device memory and streams only).
"""
from __future__ import annotations

from . import abi
from .abi import (  # noqa: F401
    MHCPB_ACCUMULATE_DW, MHCPB_ALLOW_TF32, MHCPB_COMPENSATED_DW, MHCPB_FMA_KERNEL,
    MHCPB_HAS_ADDEND, MhcpbError, mhcpb_destroy, mhcpb_execute_dx, mhcpb_forward,
    mhcpb_forward_workspace_bytes, mhcpb_reduce_dw,
    mhcpb_execute, mhcpb_get_device_status, mhcpb_last_cuda_error, mhcpb_plan_create,
    mhcpb_plan_query, mhcpb_plan_set_max_ctas, mhcpb_plan_set_wait_limit, mhcpb_status_string,
    mhcpb_workspace_bytes,
)


class Plan:
    """A prepared backward for one (T, K) on one device (owns a C plan handle)."""

    def __init__(self, T: int, K: int, device: int = 0, *, addend: bool = False,
                 fma_kernel: bool = False, compensated_dw: bool = False,
                 accumulate_dw: bool = False, test_inject_stall: bool = False):
        flags = abi.MHCPB_ALLOW_TF32
        if compensated_dw:
            flags |= abi.MHCPB_COMPENSATED_DW
        if accumulate_dw:
            flags |= abi.MHCPB_ACCUMULATE_DW
        if test_inject_stall:
            flags |= abi.MHCPB_TEST_INJECT_STALL
        if addend:
            flags |= abi.MHCPB_HAS_ADDEND
        if fma_kernel:
            flags |= abi.MHCPB_FMA_KERNEL
        self.T, self.K, self.device, self.flags = int(T), int(K), int(device), flags
        self.handle = mhcpb_plan_create(T, K, device, flags)
        self.workspace_bytes = mhcpb_workspace_bytes(self.handle)

    def set_wait_limit(self, nanoseconds: int) -> None:
        mhcpb_plan_set_wait_limit(self.handle, nanoseconds)

    def set_max_ctas(self, max_ctas: int) -> None:
        mhcpb_plan_set_max_ctas(self.handle, max_ctas)

    def query(self, which: str) -> int:
        return mhcpb_plan_query(self.handle, which)

    def execute(self, x, w, grad_proj, grad_r, r, dx, dw, workspace, addend=None, stream=None):
        """Enqueue on ``stream`` (a torch.cuda.Stream, a raw handle, or None for
        the device's current stream)."""
        if stream is None:
            import torch
            stream = torch.cuda.current_stream(x.device).cuda_stream
        elif hasattr(stream, "cuda_stream"):
            stream = stream.cuda_stream
        mhcpb_execute(self.handle, x.data_ptr(), w.data_ptr(), grad_proj.data_ptr(),
                      grad_r.data_ptr(), r.data_ptr(), dx.data_ptr(), dw.data_ptr(),
                      workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                      None if addend is None else addend.data_ptr(), stream)

    @staticmethod
    def _stream(stream, like):
        if stream is None:
            import torch
            return torch.cuda.current_stream(like.device).cuda_stream
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream

    def execute_dx(self, x, w, grad_proj, grad_r, r, dx, workspace, addend=None, stream=None):
        """First half of the split backward: dX, and the dW partials in
        ``workspace`` (see ``mhcpb_execute_dx``)."""
        mhcpb_execute_dx(self.handle, x.data_ptr(), w.data_ptr(), grad_proj.data_ptr(),
                         grad_r.data_ptr(), r.data_ptr(), dx.data_ptr(), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(),
                         None if addend is None else addend.data_ptr(), self._stream(stream, x))

    def reduce_dw(self, workspace, dw, stream=None):
        """Second half: dW from the partials in ``workspace``."""
        mhcpb_reduce_dw(self.handle, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                        dw.data_ptr(), self._stream(stream, dw))

    @property
    def forward_workspace_bytes(self) -> int:
        return mhcpb_forward_workspace_bytes(self.handle)

    def forward(self, x, w, proj, r, workspace, eps: float = 1e-6, stream=None):
        """The stage's forward: proj [T, 32] = X W^T (columns 24..31 zero) and
        r [T] = sqrt(mean X^2 + eps) (see ``mhcpb_forward``)."""
        mhcpb_forward(self.handle, x.data_ptr(), w.data_ptr(), eps, proj.data_ptr(), r.data_ptr(),
                      workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                      self._stream(stream, x))

    def forward_gates(self, x, w, alpha, bias, proj, r, h, workspace, eps: float = 1e-6,
                      n_iter: int = 20, stream=None):
        """The forward with the gate step fused in: proj and r as ``forward``,
        and h [T, 24] as ``mhc_gate_forward`` gives from them (see
        ``mhcpb_forward_gates``)."""
        abi.mhcpb_forward_gates(self.handle, x.data_ptr(), w.data_ptr(), eps, alpha.data_ptr(),
                                bias.data_ptr(), n_iter, proj.data_ptr(), r.data_ptr(), h.data_ptr(),
                                workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                self._stream(stream, x))

    def device_status(self, clear: bool = False) -> int:
        return mhcpb_get_device_status(self.handle, clear)

    def close(self):
        if getattr(self, "handle", None):
            mhcpb_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mhc_projection_backward(x, weight, grad_proj, grad_r, r, addend=None, *, stream=None,
                            fma_kernel: bool = False, compensated_dw: bool = False):
    """Allocating convenience call: returns (dx BF16 [T,K], dw FP32 [24,K]).

    Outputs and workspace are allocated by torch on the tensors' device.  The
    call waits for the stream before it returns (it owns a temporary plan).
    """
    import torch
    T, K = x.shape
    plan = Plan(T, K, x.device.index or 0, addend=addend is not None, fma_kernel=fma_kernel,
                compensated_dw=compensated_dw)
    dx = torch.empty((T, K), dtype=torch.bfloat16, device=x.device)
    dw = torch.empty((24, K), dtype=torch.float32, device=x.device)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=x.device)
    plan.execute(x, weight, grad_proj, grad_r, r, dx, dw, ws, addend=addend, stream=stream)
    # the plan (its status word) and the workspace must outlive the enqueued work
    if stream is None:
        torch.cuda.current_stream(x.device).synchronize()
    elif hasattr(stream, "synchronize"):
        stream.synchronize()
    else:
        torch.cuda.synchronize(x.device)
    plan.close()
    return dx, dw


def _stream_handle(stream, like):
    import torch
    if stream is None:
        return torch.cuda.current_stream(like.device).cuda_stream
    return getattr(stream, "cuda_stream", stream)


def mhc_gate_forward(proj, r, alpha, bias, h, *, n_iter: int = 20, stream=None):
    """Gates H [T, 24] (H_pre, H_post, H_res row-major) from the projection
    logits proj [T, 32] and r [T] (FP32 CUDA tensors); writes h."""
    from . import abi
    abi.mhcpb_gate_forward(proj.shape[0], n_iter, proj.data_ptr(), r.data_ptr(), alpha.data_ptr(),
                           bias.data_ptr(), h.data_ptr(), _stream_handle(stream, proj))


def mhc_gate_backward(proj, r, alpha, bias, grad_h, grad_proj, grad_r, dlogits=None, *,
                      n_iter: int = 20, stream=None):
    """grad_proj [T, 32] and grad_r [T] (the projection/RMS backward's inputs)
    from the gates' upstream gradients grad_h [T, 24]; dlogits [T, 24] if given."""
    from . import abi
    abi.mhcpb_gate_backward(proj.shape[0], n_iter, proj.data_ptr(), r.data_ptr(), alpha.data_ptr(),
                            bias.data_ptr(), grad_h.data_ptr(), grad_proj.data_ptr(),
                            grad_r.data_ptr(), None if dlogits is None else dlogits.data_ptr(),
                            _stream_handle(stream, proj))
