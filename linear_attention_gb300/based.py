"""ctypes binding of the C ABI in ``include/based.h`` (argument marshalling only).

Every step of the Based forward pass runs in the CUDA kernels of ``libbased_gb300.so``; this module
only checks tensor metadata, passes device pointers, sizes and the current CUDA stream, and turns
return codes into exceptions. It has no fallback: if the library is missing it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB_PATH

_lib = None


class BasedError(RuntimeError):
    pass


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise BasedError(
            f"CUDA library not built: {LIB_PATH} is missing (run linear_attention_gb300.build.build())")
    L = ctypes.CDLL(LIB_PATH)
    u16p = ctypes.c_void_p
    i = ctypes.c_int
    L.based_fwd.argtypes = [u16p, u16p, u16p, i, i, i, i, i, ctypes.c_float, ctypes.c_void_p,
                            ctypes.c_void_p]
    L.based_fwd.restype = i
    L.based_fwd_ws.argtypes = [u16p, u16p, u16p, i, i, i, i, i, ctypes.c_float, ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    L.based_fwd_ws.restype = i
    L.based_fwd_noalloc.argtypes = [u16p, u16p, u16p, i, i, i, i, i, ctypes.c_float,
                                    ctypes.c_void_p, ctypes.c_void_p]
    L.based_fwd_noalloc.restype = i
    L.based_fwd_timed.argtypes = [u16p, u16p, u16p, i, i, i, i, i, ctypes.c_float,
                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p]
    L.based_fwd_timed.restype = i
    L.based_fwd_bf16_out.argtypes = [u16p, u16p, u16p, i, i, i, i, i, ctypes.c_float, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p]
    L.based_fwd_bf16_out.restype = i
    L.based_fwd_kernel_count.argtypes = [i, i, i, i, i]
    L.based_fwd_kernel_count.restype = i
    L.based_fwd_workspace_size.argtypes = [i, i, i, i, i]
    L.based_fwd_workspace_size.restype = ctypes.c_size_t
    L.based_fwd_host.argtypes = [u16p, u16p, u16p, i, i, i, i, i, ctypes.c_float, ctypes.c_void_p,
                                 ctypes.c_void_p]
    L.based_fwd_host.restype = i
    L.based_device_status.argtypes = [i, ctypes.POINTER(ctypes.c_uint), i]
    L.based_device_status.restype = i
    L.based_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong]
    L.based_selftest_wait_timeout.restype = i
    L.based_fwd_strerror.argtypes = [i]
    L.based_fwd_strerror.restype = ctypes.c_char_p
    L.based_strerror.argtypes = [i]
    L.based_strerror.restype = ctypes.c_char_p
    L.based_last_cuda_error.argtypes = []
    L.based_last_cuda_error.restype = ctypes.c_char_p
    L.based_abi_version.argtypes = []
    L.based_abi_version.restype = i
    _lib = L
    return L


def library():
    """The loaded ctypes library (raises if it was not built)."""
    return _load()


def _check(rc: int, what: str):
    if rc != 0:
        L = _load()
        msg = L.based_fwd_strerror(rc).decode()
        cuda = L.based_last_cuda_error().decode()
        raise BasedError(f"{what} failed: {msg} ({rc})" + (f": {cuda}" if cuda else ""))


def _on_device(dev: torch.device, fn, *args) -> int:
    # fn(*args) with dev as the current CUDA device; the switch (a context manager, a few
    # microseconds per call) only when it is not current already
    if dev.index is None or dev.index == torch.cuda.current_device():
        return fn(*args)
    with torch.cuda.device(dev):
        return fn(*args)


def _stream_ptr(dev: torch.device, stream: Optional[torch.cuda.Stream]) -> int:
    return (stream if stream is not None else torch.cuda.current_stream(dev)).cuda_stream


def _scale_arg(scale: Optional[float]) -> float:
    # None (or a non-positive value) lets the library use its default K ** -0.5
    return -1.0 if scale is None else float(scale)


def _shapes(q, k, v):
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("expected q, k of shape (B,T,H,K) and v of shape (B,T,H,V)")
    for t in (q, k, v):
        if t.dtype != torch.bfloat16:
            raise TypeError("q, k, v must be bfloat16")
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    B, T, H, K = q.shape
    return B, T, H, K, v.shape[-1]


def based_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
              out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
              workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Based causal forward on CUDA tensors: q, k (B,T,H,K) bf16, v (B,T,H,V) bf16 -> o fp32.

    Launches on ``stream`` (default: the current stream of q's device). With ``workspace`` (a
    CUDA byte tensor of at least ``workspace_size(...)`` bytes) the caller-owned workspace entry
    point is used; otherwise the library's own.
    """
    L = _load()
    B, T, H, K, V = _shapes(q, k, v)
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("based_fwd takes CUDA tensors; use based_fwd_host for host tensors")
    if out is None:
        out = torch.empty(B, T, H, V, dtype=torch.float32, device=q.device)
    elif out.dtype != torch.float32 or tuple(out.shape) != (B, T, H, V) or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor of shape (B,T,H,V)")
    dev = q.device
    st = _stream_ptr(dev, stream)
    if workspace is None:
        rc = _on_device(dev, L.based_fwd, q.data_ptr(), k.data_ptr(), v.data_ptr(), B, T, H, K, V,
                        _scale_arg(scale), out.data_ptr(), st)
    else:
        rc = _on_device(dev, L.based_fwd_ws, q.data_ptr(), k.data_ptr(), v.data_ptr(), B, T, H, K, V,
                        _scale_arg(scale), out.data_ptr(), workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), st)
    _check(rc, "based_fwd")
    return out


def based_fwd_bf16_out(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
                       out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
                       workspace: Optional[torch.Tensor] = None,
                       events: Optional[tuple] = None) -> torch.Tensor:
    """based_fwd with a bf16 output: o (B,T,H,V) bf16, each element the fp32 result rounded to
    nearest even. ``workspace`` as for based_fwd; ``events`` = (ev_begin, ev_end), already-recorded
    torch CUDA events, brackets the forward kernel as in based_fwd_timed."""
    L = _load()
    B, T, H, K, V = _shapes(q, k, v)
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("based_fwd_bf16_out takes CUDA tensors")
    if out is None:
        out = torch.empty(B, T, H, V, dtype=torch.bfloat16, device=q.device)
    elif out.dtype != torch.bfloat16 or tuple(out.shape) != (B, T, H, V) or not out.is_contiguous():
        raise ValueError("out must be a contiguous bfloat16 tensor of shape (B,T,H,V)")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (
        workspace.data_ptr(), workspace.numel() * workspace.element_size())
    eb, ee = (None, None) if events is None else (events[0].cuda_event, events[1].cuda_event)
    dev = q.device
    rc = _on_device(dev, L.based_fwd_bf16_out, q.data_ptr(), k.data_ptr(), v.data_ptr(), B, T, H, K, V,
                    _scale_arg(scale), out.data_ptr(), ws_ptr, ws_bytes, _stream_ptr(dev, stream), eb, ee)
    _check(rc, "based_fwd_bf16_out")
    return out


def based_fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                      scale: Optional[float] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """based_fwd for callers that may not allocate device memory while they run: the library's
    scratch is a fixed array of its device image and the caller passes the output buffer. Calls
    on one device share that array, so calls that overlap on the GPU race; order them."""
    L = _load()
    B, T, H, K, V = _shapes(q, k, v)
    if not (q.is_cuda and k.is_cuda and v.is_cuda and out.is_cuda):
        raise ValueError("based_fwd_noalloc takes CUDA tensors")
    if out.dtype != torch.float32 or tuple(out.shape) != (B, T, H, V) or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor of shape (B,T,H,V)")
    dev = q.device
    rc = _on_device(dev, L.based_fwd_noalloc, q.data_ptr(), k.data_ptr(), v.data_ptr(), B, T, H, K, V,
                    _scale_arg(scale), out.data_ptr(), _stream_ptr(dev, stream))
    _check(rc, "based_fwd_noalloc")
    return out


def based_fwd_timed(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                    ev_begin: torch.cuda.Event, ev_end: torch.cuda.Event,
                    scale: Optional[float] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """based_fwd that records ev_begin / ev_end (already-recorded torch CUDA events, so that their
    handles exist) on the stream right before and after the forward kernel."""
    L = _load()
    B, T, H, K, V = _shapes(q, k, v)
    if not (q.is_cuda and k.is_cuda and v.is_cuda and out.is_cuda):
        raise ValueError("based_fwd_timed takes CUDA tensors")
    dev = q.device
    rc = _on_device(dev, L.based_fwd_timed, q.data_ptr(), k.data_ptr(), v.data_ptr(), B, T, H, K, V,
                    _scale_arg(scale), out.data_ptr(), _stream_ptr(dev, stream), ev_begin.cuda_event,
                    ev_end.cuda_event)
    _check(rc, "based_fwd_timed")
    return out


def kernel_count(B: int, T: int, H: int, K: int, V: int, device=None) -> int:
    L = _load()
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(L.based_fwd_kernel_count(B, T, H, K, V))


def workspace_size(B: int, T: int, H: int, K: int, V: int, device=None) -> int:
    L = _load()
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(L.based_fwd_workspace_size(B, T, H, K, V))


def based_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
                   out: Optional[torch.Tensor] = None, device=None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """End-to-end call on host (CPU) tensors: copies in, computes on the GPU, copies out, waits."""
    L = _load()
    B, T, H, K, V = _shapes(q, k, v)
    if q.is_cuda or k.is_cuda or v.is_cuda:
        raise ValueError("based_fwd_host takes host tensors")
    if out is None:
        out = torch.empty(B, T, H, V, dtype=torch.float32, pin_memory=q.is_pinned())
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = stream if stream is not None else torch.cuda.current_stream(dev)
        rc = L.based_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, T, H, K, V,
                              _scale_arg(scale), out.data_ptr(), st.cuda_stream)
    _check(rc, "based_fwd_host")
    return out


def device_status(device: int = 0, clear: bool = False) -> int:
    L = _load()
    s = ctypes.c_uint(0)
    _check(L.based_device_status(device, ctypes.byref(s), 1 if clear else 0), "based_device_status")
    return int(s.value)


def selftest_wait_timeout(limit_ns: int = 20_000_000) -> None:
    """Runs the bounded-wait self-test; the device status word is left reporting its timeout
    (site 255) until it is cleared with device_status(dev, clear=True)."""
    L = _load()
    _check(L.based_selftest_wait_timeout(limit_ns), "based_selftest_wait_timeout")
