"""Anchor-attention forward H = A Delta^{-1} A^T V on GB300 (sm_103a).

Thin ctypes binding over the C ABI in include/anchor_attn.h (libanchor_attn.so, built
in-tree by ``_build.build()``).  This module only marshals arguments: every step of the
forward runs in the library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  There is no CPU fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = [
    "LIB_PATH", "load", "forward", "anchor_attn_forward", "anchor_attn_forward_f32",
    "anchor_attn_forward_ptr", "anchor_attn_forward_f32_ptr", "anchor_attn_forward_static_scratch_ptr",
    "static_scratch_bytes", "device_error", "query_plan", "status_string", "anchor_attn_test_forward_ptr",
    "AnchorAttnError", "STATUS", "VARIANTS", "backward", "anchor_attn_backward_ptr", "anchor_attn_backward_f32_ptr",
    "full_forward", "relative_error", "causal_forward", "block_forward", "anchor_attn_block_forward_ptr",
    "forward_host", "anchor_attn_forward_host_ptr", "anchor_attn_forward_host_f32_ptr",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libanchor_attn.so")

STATUS = {0: "OK", 1: "ERR_INVALID_ARG", 2: "ERR_UNSUPPORTED", 3: "ERR_ALIAS", 4: "ERR_ALLOC", 5: "ERR_CUDA",
          6: "ERR_SCRATCH_LIMIT"}
VARIANTS = {0: "empty", 1: "simt_slice", 2: "simt_split", 3: "umma", 4: "stream", 5: "split_tc", 6: "short_tc"}

_lock = threading.Lock()
_lib = None


class AnchorAttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"anchor_attn: {STATUS.get(status, status)}: {msg}")
        self.status = status


class _Plan(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("kernels_per_call", ctypes.c_int), ("splits", ctypes.c_int),
                ("flags", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t)]


PLAN_STORED_A = 1


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"anchor_attn CUDA library not built ({p}); run __graft_entry__.build()")
        lib = ctypes.CDLL(p)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        for name in ("anchor_attn_forward", "anchor_attn_forward_f32", "anchor_attn_forward_static_scratch",
                     "anchor_attn_forward_host", "anchor_attn_forward_host_f32"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp]
            fn.restype = ctypes.c_int
        for name in ("anchor_attn_backward", "anchor_attn_backward_f32"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
            fn.restype = ctypes.c_int
        for name in ("anchor_attn_causal_forward", "anchor_attn_causal_forward_f32"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp]
            fn.restype = ctypes.c_int
        for name in ("anchor_attn_full_forward", "anchor_attn_full_forward_f32"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, vp, vp, i, i, i, i, f, vp]
            fn.restype = ctypes.c_int
        lib.anchor_attn_block_forward.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
        lib.anchor_attn_block_forward.restype = ctypes.c_int
        lib.anchor_attn_relative_error.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
        lib.anchor_attn_relative_error.restype = ctypes.c_int
        lib.anchor_attn_test_forward.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, i, ctypes.c_ulonglong, i, vp]
        lib.anchor_attn_test_forward.restype = ctypes.c_int
        lib.anchor_attn_query_plan.argtypes = [i, i, i, i, i, i, ctypes.POINTER(_Plan)]
        lib.anchor_attn_query_plan.restype = ctypes.c_int
        lib.anchor_attn_static_scratch_bytes.argtypes = []
        lib.anchor_attn_static_scratch_bytes.restype = ctypes.c_size_t
        lib.anchor_attn_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.anchor_attn_device_error.restype = ctypes.c_int
        lib.anchor_attn_status_string.argtypes = [ctypes.c_int]
        lib.anchor_attn_status_string.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().anchor_attn_status_string(int(status)).decode()


def _raise(st: int, what: str) -> None:
    if st != 0:
        raise AnchorAttnError(st, f"{what}: {status_string(st)}")


def anchor_attn_forward_ptr(Q: int, U: int, V: int, H: int, B: int, heads: int, n: int, m: int, d: int,
                            scale: float, stream: int = 0) -> int:
    """Raw C-ABI call (bf16 device pointers as integers); returns the status code."""
    return load().anchor_attn_forward(Q, U, V, H, B, heads, n, m, d, float(scale), stream)


def anchor_attn_forward_f32_ptr(Q: int, U: int, V: int, H: int, B: int, heads: int, n: int, m: int,
                                d: int, scale: float, stream: int = 0) -> int:
    """Raw C-ABI call (fp32 device pointers as integers); returns the status code."""
    return load().anchor_attn_forward_f32(Q, U, V, H, B, heads, n, m, d, float(scale), stream)


def anchor_attn_forward_host_ptr(Q: int, U: int, V: int, H: int, B: int, heads: int, n: int, m: int, d: int,
                                 scale: float, stream: int = 0) -> int:
    """Raw C-ABI call of the host-buffer forward (bf16 host pointers as integers); returns the
    status code.  Asynchronous on `stream` (a CUDA stream handle)."""
    return load().anchor_attn_forward_host(Q, U, V, H, B, heads, n, m, d, float(scale), stream)


def anchor_attn_forward_host_f32_ptr(Q: int, U: int, V: int, H: int, B: int, heads: int, n: int, m: int,
                                     d: int, scale: float, stream: int = 0) -> int:
    """Raw C-ABI call of the fp32 host-buffer forward; returns the status code."""
    return load().anchor_attn_forward_host_f32(Q, U, V, H, B, heads, n, m, d, float(scale), stream)


def anchor_attn_forward_static_scratch_ptr(Q: int, U: int, V: int, H: int, B: int, heads: int, n: int,
                                           m: int, d: int, scale: float, stream: int = 0) -> int:
    """Raw C-ABI call of the allocation-free variant (bf16 device pointers); returns the status."""
    return load().anchor_attn_forward_static_scratch(Q, U, V, H, B, heads, n, m, d, float(scale), stream)


def anchor_attn_test_forward_ptr(Q: int, U: int, V: int, H: int, B: int, heads: int, n: int, m: int, d: int,
                                 scale: float, hold_slice: int = -1, wait_ns: int = 2_000_000_000,
                                 force_recompute: bool = False, stream: int = 0) -> int:
    """Raw call of the failure-detection test entry (tests only); returns the status code."""
    return load().anchor_attn_test_forward(Q, U, V, H, B, heads, n, m, d, float(scale), int(hold_slice),
                                           int(wait_ns), 1 if force_recompute else 0, stream)


def anchor_attn_backward_ptr(Q: int, U: int, V: int, dH: int, dQ: int, dU: int, dV: int, B: int, heads: int,
                             n: int, m: int, d: int, scale: float, stream: int = 0) -> int:
    """Raw C-ABI call of the bf16 backward (device pointers as integers); returns the status."""
    return load().anchor_attn_backward(Q, U, V, dH, dQ, dU, dV, B, heads, n, m, d, float(scale), stream)


def anchor_attn_backward_f32_ptr(Q: int, U: int, V: int, dH: int, dQ: int, dU: int, dV: int, B: int, heads: int,
                                 n: int, m: int, d: int, scale: float, stream: int = 0) -> int:
    """Raw C-ABI call of the fp32 backward (device pointers as integers); returns the status."""
    return load().anchor_attn_backward_f32(Q, U, V, dH, dQ, dU, dV, B, heads, n, m, d, float(scale), stream)


def static_scratch_bytes() -> int:
    return int(load().anchor_attn_static_scratch_bytes())


def device_error() -> int:
    """Synchronise and return (and clear) the tensor-core kernel's device error word."""
    code = ctypes.c_uint(0)
    _raise(load().anchor_attn_device_error(ctypes.byref(code)), "device_error")
    return int(code.value)


def query_plan(dtype: str, B: int, heads: int, n: int, m: int, d: int) -> dict:
    """What one call launches: variant, kernels per call, splits, workspace bytes."""
    pl = _Plan()
    st = load().anchor_attn_query_plan(1 if dtype == "f32" else 0, B, heads, n, m, d, ctypes.byref(pl))
    _raise(st, "query_plan")
    return {"variant": VARIANTS.get(pl.variant, pl.variant), "kernels_per_call": pl.kernels_per_call,
            "splits": pl.splits, "workspace_bytes": pl.workspace_bytes,
            "stored_a": bool(pl.flags & PLAN_STORED_A)}


def _check_tensors(Q, U, V, H, dtype):
    import torch
    for name, t in (("Q", Q), ("U", U), ("V", V), ("H", H)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if Q.dim() != 4 or U.dim() != 3:
        raise ValueError("Q, V, H are [B, heads, n, d]; U is [heads, m, d]")
    if V.shape != Q.shape or H.shape != Q.shape:
        raise ValueError("V and H must have Q's shape")
    if U.shape[0] != Q.shape[1] or U.shape[2] != Q.shape[3]:
        raise ValueError("U must be [heads, m, d] matching Q")


def forward(Q, U, V, H=None, scale: float | None = None, stream=None):
    """H = A Delta^{-1} A^T V for torch CUDA tensors (bf16 or fp32).

    Q, V: [B, heads, n, d]; U: [heads, m, d].  scale defaults to 1/sqrt(d).  Runs on
    ``stream`` (a torch.cuda.Stream) or the current stream; asynchronous.
    """
    import torch
    if H is None:
        H = torch.empty_like(Q)
    _check_tensors(Q, U, V, H, Q.dtype)
    B, heads, n, d = Q.shape
    m = U.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    s = stream if stream is not None else torch.cuda.current_stream(Q.device)
    with torch.cuda.device(Q.device):
        if Q.dtype == torch.bfloat16:
            st = anchor_attn_forward_ptr(Q.data_ptr(), U.data_ptr(), V.data_ptr(), H.data_ptr(), B, heads, n, m,
                                         d, scale, s.cuda_stream)
        elif Q.dtype == torch.float32:
            st = anchor_attn_forward_f32_ptr(Q.data_ptr(), U.data_ptr(), V.data_ptr(), H.data_ptr(), B, heads,
                                             n, m, d, scale, s.cuda_stream)
        else:
            raise TypeError("Q must be bfloat16 or float32")
    _raise(st, "forward")
    return H


def forward_host(Q, U, V, H=None, scale: float | None = None, stream=None, device=None):
    """The forward on host (CPU) torch tensors (bf16 or fp32; pinned memory for asynchronous
    copies): the library copies chunks of the batch to the device, runs the forward and copies
    H back, overlapping the three.  Q, V: [B, heads, n, d]; U: [heads, m, d].  Runs on
    ``stream`` (a torch.cuda.Stream of ``device``, default the current device's current
    stream); asynchronous: H is complete once the stream reaches this point."""
    import torch
    if H is None:
        H = torch.empty(Q.shape, dtype=Q.dtype).pin_memory() if Q.is_pinned() else torch.empty_like(Q)
    for name, t in (("Q", Q), ("U", U), ("V", V), ("H", H)):
        if not isinstance(t, torch.Tensor) or t.is_cuda:
            raise TypeError(f"{name} must be a host (CPU) torch.Tensor")
        if t.dtype != Q.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous and of Q's dtype")
    if Q.dim() != 4 or U.dim() != 3 or V.shape != Q.shape or H.shape != Q.shape:
        raise ValueError("Q, V, H are [B, heads, n, d]; U is [heads, m, d]")
    if U.shape[0] != Q.shape[1] or U.shape[2] != Q.shape[3]:
        raise ValueError("U must be [heads, m, d] matching Q")
    B, heads, n, d = Q.shape
    m = U.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        if Q.dtype == torch.bfloat16:
            st = anchor_attn_forward_host_ptr(Q.data_ptr(), U.data_ptr(), V.data_ptr(), H.data_ptr(), B, heads, n,
                                              m, d, scale, s.cuda_stream)
        elif Q.dtype == torch.float32:
            st = anchor_attn_forward_host_f32_ptr(Q.data_ptr(), U.data_ptr(), V.data_ptr(), H.data_ptr(), B, heads,
                                                  n, m, d, scale, s.cuda_stream)
        else:
            raise TypeError("Q must be bfloat16 or float32")
    _raise(st, "forward_host")
    return H


def anchor_attn_forward(Q, U, V, H=None, scale=None, stream=None):
    """bf16 entry point (see ``forward``)."""
    import torch
    if Q.dtype != torch.bfloat16:
        raise TypeError("anchor_attn_forward takes bfloat16 tensors")
    return forward(Q, U, V, H, scale, stream)


def anchor_attn_forward_f32(Q, U, V, H=None, scale=None, stream=None):
    """fp32 entry point (see ``forward``)."""
    import torch
    if Q.dtype != torch.float32:
        raise TypeError("anchor_attn_forward_f32 takes float32 tensors")
    return forward(Q, U, V, H, scale, stream)


def backward(Q, U, V, dH, scale: float | None = None, stream=None):
    """(dQ, dU, dV) for torch CUDA tensors (bf16 or fp32): the gradients of a loss with
    upstream gradient dH = dL/dH of H = forward(Q, U, V).  dU sums the batch entries (they
    share the anchors).  scale defaults to 1/sqrt(d).  Asynchronous on ``stream`` or the
    current stream."""
    import torch
    _check_tensors(Q, U, V, dH, Q.dtype)
    B, heads, n, d = Q.shape
    m = U.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dQ, dU, dV = torch.empty_like(Q), torch.empty_like(U), torch.empty_like(V)
    s = stream if stream is not None else torch.cuda.current_stream(Q.device)
    ptrs = (Q.data_ptr(), U.data_ptr(), V.data_ptr(), dH.data_ptr(), dQ.data_ptr(), dU.data_ptr(), dV.data_ptr())
    with torch.cuda.device(Q.device):
        if Q.dtype == torch.bfloat16:
            st = anchor_attn_backward_ptr(*ptrs, B, heads, n, m, d, scale, s.cuda_stream)
        elif Q.dtype == torch.float32:
            st = anchor_attn_backward_f32_ptr(*ptrs, B, heads, n, m, d, scale, s.cuda_stream)
        else:
            raise TypeError("Q must be bfloat16 or float32")
    _raise(st, "backward")
    return dQ, dU, dV


def full_forward(Q, K, V, H=None, scale: float | None = None, stream=None):
    """Full softmax attention softmax(scale Q K^T) V for torch CUDA tensors (bf16 or fp32):
    Q, V [B, heads, n, d], K [heads, n, d] (one key matrix per head).  The reference of the
    approximation-error diagnostic."""
    import torch
    if H is None:
        H = torch.empty_like(Q)
    _check_tensors(Q, K, V, H, Q.dtype)
    B, heads, n, d = Q.shape
    if K.shape[1] != n:
        raise ValueError("K must be [heads, n, d]: one key per token of the slice")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    s = stream if stream is not None else torch.cuda.current_stream(Q.device)
    lib = load()
    fn = lib.anchor_attn_full_forward if Q.dtype == torch.bfloat16 else lib.anchor_attn_full_forward_f32
    with torch.cuda.device(Q.device):
        st = fn(Q.data_ptr(), K.data_ptr(), V.data_ptr(), H.data_ptr(), B, heads, n, d, float(scale), s.cuda_stream)
    _raise(st, "full_forward")
    return H


def relative_error(Href, H, stream=None):
    """Per (batch, head) slice ||Href - H||_F / ||Href||_F as a float32 CUDA tensor [B, heads]."""
    import torch
    if Href.shape != H.shape or Href.dtype != H.dtype or Href.dim() != 4:
        raise ValueError("Href and H must be [B, heads, n, d] of one dtype")
    B, heads, n, d = Href.shape
    err = torch.empty((B, heads), dtype=torch.float32, device=Href.device)
    s = stream if stream is not None else torch.cuda.current_stream(Href.device)
    with torch.cuda.device(Href.device):
        st = load().anchor_attn_relative_error(Href.data_ptr(), H.data_ptr(), err.data_ptr(), B, heads, n, d,
                                               1 if Href.dtype == torch.float32 else 0, s.cuda_stream)
    _raise(st, "relative_error")
    return err


def causal_forward(Q, U, V, H=None, scale: float | None = None, stream=None):
    """The masked (causal) variant: token i's anchor summaries use tokens j <= i only.  Same
    tensors as ``forward`` (bf16 or fp32)."""
    import torch
    if H is None:
        H = torch.empty_like(Q)
    _check_tensors(Q, U, V, H, Q.dtype)
    B, heads, n, d = Q.shape
    m = U.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    s = stream if stream is not None else torch.cuda.current_stream(Q.device)
    lib = load()
    fn = lib.anchor_attn_causal_forward if Q.dtype == torch.bfloat16 else lib.anchor_attn_causal_forward_f32
    with torch.cuda.device(Q.device):
        st = fn(Q.data_ptr(), U.data_ptr(), V.data_ptr(), H.data_ptr(), B, heads, n, m, d, float(scale), s.cuda_stream)
    _raise(st, "causal_forward")
    return H


def anchor_attn_block_forward_ptr(X: int, Wq: int, Wv: int, U: int, H: int, B: int, heads: int, n: int, m: int,
                                  d: int, dm: int, scale: float, stream: int = 0) -> int:
    """Raw C-ABI call of the block front end (bf16 device pointers); returns the status code."""
    return load().anchor_attn_block_forward(X, Wq, Wv, U, H, B, heads, n, m, d, dm, float(scale), stream)


def block_forward(X, Wq, Wv, U, H=None, scale: float | None = None, stream=None):
    """The block front end for bf16 torch CUDA tensors: Q = X Wq^T and V = X Wv^T per head,
    then the forward, in one kernel.  X [B, n, dm]; Wq, Wv [heads, d, dm]; U [heads, m, d];
    returns H [B, heads, n, d]."""
    import torch
    if X.dim() != 3 or Wq.dim() != 3 or Wv.shape != Wq.shape or U.dim() != 3:
        raise ValueError("X must be [B, n, dm], Wq and Wv [heads, d, dm], U [heads, m, d]")
    B, n, dm = X.shape
    heads, d, _ = Wq.shape
    m = U.shape[1]
    if Wq.shape[2] != dm or U.shape[0] != heads or U.shape[2] != d:
        raise ValueError("inconsistent shapes")
    for t in (X, Wq, Wv, U):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous bfloat16 CUDA tensors")
    if H is None:
        H = torch.empty((B, heads, n, d), dtype=torch.bfloat16, device=X.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    s = stream if stream is not None else torch.cuda.current_stream(X.device)
    with torch.cuda.device(X.device):
        st = anchor_attn_block_forward_ptr(X.data_ptr(), Wq.data_ptr(), Wv.data_ptr(), U.data_ptr(), H.data_ptr(),
                                           B, heads, n, m, d, dm, scale, s.cuda_stream)
    _raise(st, "block_forward")
    return H
