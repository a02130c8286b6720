"""Exact tiled attention forward for GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libfa.so`` (C ABI in ``include/fa.h``).  It only
marshals arguments: torch supplies device memory and the current stream,
every step of the computation runs in the library's CUDA kernels.  There is no
CPU fallback: if the shared library is missing or a call fails, an exception
is raised.

    import exact_attention_90_gb300 as fa
    o, lse = fa.fwd(q, k, v, causal=True)          # q [B,Hq,T,d], k/v [B,Hkv,T,d]

The operation (yelogs.com Flash Attention2/Triton tutorial, section "核心
Kernel 實現"; "Flash Attention Memory Optimization Explained", section "What is
Flash Attention?"): O = softmax(scale * Q K^T (+ causal mask)) V per
(batch, head), and the row log-sum-exp L = m + ln l of the scaled, masked
scores; query head h reads KV head h // (Hq // Hkv).
"""

from __future__ import annotations

import ctypes
import math
import os

__all__ = [
    "FaError", "load_library", "library_path", "fwd", "fa_fwd", "fa_fwd_simt",
    "fa_status_string", "fa_version", "fa_debug_sync_check", "fa_last_cuda_error",
    "fa_unit_tma", "fa_unit_qk", "fa_unit_pv", "fa_unit_timeout", "fa_unit_pipe_rate",
    "fa_fwd_window", "fa_fwd_split",
    "fa_fwd_split_static",
    "fa_fwd_split_workspace_size", "fa_fwd_split_heuristic", "fa_bwd", "fa_bwd_workspace_size",
    "fa_fwd_local_global", "fa_fwd_local_global_workspace_size",
    "fa_fwd_local_global_packed_workspace_size", "fa_bwd_local_global",
    "fa_bwd_local_global_workspace_size", "fa_fwd_host", "fa_fwd_host_workspace_size", "fwd_host",
    "fa_bwd_host", "fa_bwd_host_workspace_size", "bwd_host",
    "bwd", "FA_DTYPE_F32",
    "FA_DTYPE_BF16", "FA_DTYPE_F16",
]

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5
FA_ERR_WORKSPACE = 6
FA_DTYPE_F32 = 0
FA_DTYPE_BF16 = 1
FA_DTYPE_F16 = 2

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB = None

# (name, restype, argtypes) of every exported symbol (include/fa.h, include/fa_unit.h)
_P, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
EXPORTS = [
    ("fa_fwd", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    ("fa_status_string", ctypes.c_char_p, [_I]),
    ("fa_version", _I, []),
    ("fa_debug_sync_check", _I, [_P]),
    ("fa_last_cuda_error", _I, []),
    ("fa_unit_tma", _I, [_P, _P, _I, _P]),
    ("fa_unit_qk", _I, [_P, _P, _P, _I, _P]),
    ("fa_unit_pv", _I, [_P, _P, _P, _P, _I, _I, ctypes.c_uint, ctypes.c_uint, _P]),
    ("fa_unit_timeout", _I, [ctypes.c_longlong, _P, _P]),
    ("fa_unit_pipe_rate", _I, [_I, _I, _I, _P, _P, _P]),
    ("fa_fwd_window", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P]),
    ("fa_fwd_split", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P,
                          ctypes.c_ulonglong, _P]),
    ("fa_fwd_split_static", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P]),
    ("fa_fwd_split_workspace_size", ctypes.c_ulonglong, [_I, _I, _I, _I, _I]),
    ("fa_fwd_split_heuristic", _I, [_I, _I, _I, _I, _I, _I]),
    ("fa_fwd_simt", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    ("fa_bwd", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I, _I,
                    _P, ctypes.c_ulonglong, _P]),
    ("fa_bwd_workspace_size", ctypes.c_ulonglong, [_I, _I, _I]),
    ("fa_fwd_local_global", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _I, _I,
                                 _P, ctypes.c_ulonglong, _P]),
    ("fa_fwd_local_global_workspace_size", ctypes.c_ulonglong, [_I]),
    ("fa_fwd_local_global_packed_workspace_size", ctypes.c_ulonglong, [_I, _I, _I, _I, _I, _I]),
    ("fa_bwd_local_global", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I,
                                 _I, _P, _I, _I, _P, ctypes.c_ulonglong, _P]),
    ("fa_bwd_local_global_workspace_size", ctypes.c_ulonglong, [_I, _I, _I]),
    ("fa_fwd_host", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P,
                         ctypes.c_ulonglong, _P]),
    ("fa_fwd_host_workspace_size", ctypes.c_ulonglong, [_I, _I, _I, _I, _I, _I, _I]),
    ("fa_bwd_host", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I,
                         _I, _I, _P, ctypes.c_ulonglong, _P]),
    ("fa_bwd_host_workspace_size", ctypes.c_ulonglong, [_I, _I, _I, _I, _I, _I, _I]),
]


class FaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = _status_text(status)
        if status == FA_ERR_CUDA and _LIB is not None:
            msg += f" (cuda error {_LIB.fa_last_cuda_error()})"
        super().__init__(f"{what}: {msg}" if what else msg)


def library_path() -> str:
    return os.path.join(_PKG, "libfa.so")


def load_library():
    """Loads libfa.so (built in-tree by ``build.py``); raises if it is absent."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m exact_attention_90_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, res, args in EXPORTS:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _status_text(s: int) -> str:
    if _LIB is not None:
        return _LIB.fa_status_string(int(s)).decode()
    return f"status {s}"


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != FA_OK:
        raise FaError(status, what)


# ------------------------------------------------------------------ raw C ABI
def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, dtype, stream=None) -> int:
    """The C function fa_fwd with the same arguments (tensors or raw device
    pointers); returns the status code."""
    lib = load_library()
    return lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv),
                      int(T), int(d), float(scale), int(causal), int(dtype), _stream(stream))


def fa_fwd_simt(q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, dtype, stream=None) -> int:
    lib = load_library()
    return lib.fa_fwd_simt(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                           int(Hkv), int(T), int(d), float(scale), int(causal), int(dtype),
                           _stream(stream))


def fa_fwd_window(q, k, v, o, lse, B, Hq, Hkv, T, d, scale, window_left, window_right, dtype,
                  stream=None) -> int:
    """The C function fa_fwd_window (band / sliding-window mask)."""
    lib = load_library()
    return lib.fa_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                             int(Hkv), int(T), int(d), float(scale), int(window_left),
                             int(window_right), int(dtype), _stream(stream))


def fa_fwd_split(q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, dtype, num_splits,
                 workspace, workspace_bytes, stream=None) -> int:
    """The C function fa_fwd_split (split-KV forward into a caller workspace)."""
    lib = load_library()
    return lib.fa_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                            int(Hkv), int(T), int(d), float(scale), int(causal), int(dtype),
                            int(num_splits), _ptr(workspace), int(workspace_bytes),
                            _stream(stream))


def fa_fwd_split_static(q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, dtype, num_splits,
                        stream=None) -> int:
    """The C function fa_fwd_split_static: split-KV forward for callers that
    cannot allocate device memory (a host application's own memory pool, or a
    path that cannot afford cudaMalloc's synchronisation); its scratch is a
    fixed 64 MiB array inside the library."""
    lib = load_library()
    return lib.fa_fwd_split_static(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                   int(Hq), int(Hkv), int(T), int(d), float(scale), int(causal),
                                   int(dtype), int(num_splits), _stream(stream))


def fa_fwd_split_workspace_size(B, Hq, T, d, num_splits) -> int:
    return load_library().fa_fwd_split_workspace_size(int(B), int(Hq), int(T), int(d),
                                                      int(num_splits))


def fa_fwd_split_heuristic(B, Hq, Hkv, T, d, causal) -> int:
    return load_library().fa_fwd_split_heuristic(int(B), int(Hq), int(Hkv), int(T), int(d),
                                                 int(causal))


def fa_bwd(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, T, d, scale, causal, window_left,
           window_right, dtype, workspace, workspace_bytes, stream=None) -> int:
    """The C function fa_bwd (gradients of the forward for an upstream dO)."""
    lib = load_library()
    return lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o), _ptr(dq),
                      _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv), int(T), int(d), float(scale),
                      int(causal), int(window_left), int(window_right), int(dtype),
                      _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_fwd_local_global(q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, local_window,
                        global_tokens, num_global, dtype, workspace, workspace_bytes,
                        stream=None) -> int:
    """The C function fa_fwd_local_global (band OR global keys)."""
    lib = load_library()
    return lib.fa_fwd_local_global(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                   int(Hq), int(Hkv), int(T), int(d), float(scale), int(causal),
                                   int(local_window), _ptr(global_tokens), int(num_global),
                                   int(dtype), _ptr(workspace), int(workspace_bytes),
                                   _stream(stream))


def fa_fwd_local_global_workspace_size(T) -> int:
    return load_library().fa_fwd_local_global_workspace_size(int(T))


def fa_fwd_local_global_packed_workspace_size(B, Hkv, T, d, dtype, num_global) -> int:
    return load_library().fa_fwd_local_global_packed_workspace_size(
        int(B), int(Hkv), int(T), int(d), int(dtype), int(num_global))


def fa_bwd_local_global(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, T, d, scale, causal,
                        local_window, global_tokens, num_global, dtype, workspace,
                        workspace_bytes, stream=None) -> int:
    """The C function fa_bwd_local_global."""
    lib = load_library()
    return lib.fa_bwd_local_global(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o),
                                   _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv), int(T),
                                   int(d), float(scale), int(causal), int(local_window),
                                   _ptr(global_tokens), int(num_global), int(dtype),
                                   _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_local_global_workspace_size(B, Hq, T) -> int:
    return load_library().fa_bwd_local_global_workspace_size(int(B), int(Hq), int(T))


def fa_fwd_host(q, k, v, o, lse, B, Hq, Hkv, T, d, scale, causal, dtype, chunks, workspace,
                workspace_bytes, stream=None) -> int:
    """The C function fa_fwd_host (host buffers in and out, chunks pipelined)."""
    lib = load_library()
    return lib.fa_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                           int(Hkv), int(T), int(d), float(scale), int(causal), int(dtype),
                           int(chunks), _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_fwd_host_workspace_size(B, Hq, Hkv, T, d, dtype, chunks) -> int:
    return load_library().fa_fwd_host_workspace_size(int(B), int(Hq), int(Hkv), int(T), int(d),
                                                     int(dtype), int(chunks))


def fa_bwd_host(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, T, d, scale, causal, window_left,
                window_right, dtype, chunks, workspace, workspace_bytes, stream=None) -> int:
    """The C function fa_bwd_host (host buffers in and out, chunks pipelined)."""
    lib = load_library()
    return lib.fa_bwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o), _ptr(dq),
                           _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv), int(T), int(d),
                           float(scale), int(causal), int(window_left), int(window_right),
                           int(dtype), int(chunks), _ptr(workspace), int(workspace_bytes),
                           _stream(stream))


def fa_bwd_host_workspace_size(B, Hq, Hkv, T, d, dtype, chunks) -> int:
    return load_library().fa_bwd_host_workspace_size(int(B), int(Hq), int(Hkv), int(T), int(d),
                                                     int(dtype), int(chunks))


def fa_bwd_workspace_size(B, Hq, T) -> int:
    return load_library().fa_bwd_workspace_size(int(B), int(Hq), int(T))


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def fa_version() -> int:
    return load_library().fa_version()


def fa_debug_sync_check(stream=None) -> int:
    return load_library().fa_debug_sync_check(_stream(stream))


def fa_last_cuda_error() -> int:
    return load_library().fa_last_cuda_error()


def fa_unit_tma(x, out, d, stream=None) -> int:
    return load_library().fa_unit_tma(_ptr(x), _ptr(out), int(d), _stream(stream))


def fa_unit_qk(q, k, s, d, stream=None) -> int:
    return load_library().fa_unit_qk(_ptr(q), _ptr(k), _ptr(s), int(d), _stream(stream))


def fa_unit_pv(p, pb, v, o, d, mode=0, lbo=0, sbo=0, stream=None) -> int:
    return load_library().fa_unit_pv(_ptr(p), _ptr(pb), _ptr(v), _ptr(o), int(d), int(mode),
                                     int(lbo), int(sbo), _stream(stream))


def fa_unit_timeout(budget_cycles, gave_up, stream=None) -> int:
    return load_library().fa_unit_timeout(int(budget_cycles), _ptr(gave_up), _stream(stream))


def fa_unit_pipe_rate(kind, iters, blocks, sink, cycles, stream=None) -> int:
    return load_library().fa_unit_pipe_rate(int(kind), int(iters), int(blocks), _ptr(sink),
                                            _ptr(cycles), _stream(stream))


# ------------------------------------------------------------------ tensor API
def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    if t.dtype == torch.float16:
        return FA_DTYPE_F16
    if t.dtype == torch.float32:
        return FA_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bfloat16, float16 or float32)")


def fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
        stream=None, kernel: str = "auto", num_splits: int | None = None, window=None,
        global_tokens=None, pack_global: bool = True):
    """Attention forward on CUDA tensors; returns (o, lse).

    q: [B, Hq, T, d]; k, v: [B, Hkv, T, d]; all contiguous CUDA tensors of one
    dtype (bfloat16, float16 or float32).  scale defaults to 1/sqrt(d).  ``out`` and
    ``lse`` may be given (shapes [B,Hq,T,d] in the input dtype and [B,Hq,T]
    float32); otherwise they are allocated with torch.  ``kernel="simt"``
    forces the fp32 CUDA-core kernel (also for 16-bit inputs); the default
    picks the kernel by dtype.  ``num_splits`` splits every row block's keys
    that many ways (16-bit inputs; None = the library's heuristic, which
    splits only shapes too small to fill the GPU); the split path's
    workspace is allocated with torch.  ``window = (wl, wr)`` restricts query
    i to the keys i - wl <= j <= i + wr (-1: unbounded side), intersected with
    the causal mask when ``causal`` is set.  ``global_tokens`` (a CUDA int32
    tensor of key indices) selects the local-global mask: ``window`` must
    then be (w, w) or None (w = 0), and query i keeps key j when |i - j| <= w
    or j is a global token (intersected with causal).  With ``pack_global``
    (default) the 16-bit path gathers the global keys into packed tiles (the
    larger workspace of fa_fwd_local_global_packed_workspace_size); False
    visits whole key tiles instead (same results).  The call is
    asynchronous on ``stream`` (default: the current torch stream).
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D tensor [B, H, T, d]")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    B, Hq, T, d = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, T, d) or tuple(v.shape) != (B, Hkv, T, d):
        raise ValueError(f"k, v must be [B, Hkv, T, d]; got {tuple(k.shape)}, {tuple(v.shape)}")
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    if kernel not in ("auto", "simt"):
        raise ValueError("kernel must be 'auto' or 'simt'")
    if num_splits is not None and int(num_splits) > 1 and (window is not None
                                                           or global_tokens is not None):
        # the band and local-global entry points have no KV split
        raise ValueError("num_splits > 1 cannot be combined with window or global_tokens")
    if global_tokens is not None:
        wl, wr = (0, 0) if window is None else (int(window[0]), int(window[1]))
        if wl != wr:
            raise ValueError("the local-global mask takes a symmetric window (w, w)")
        if (not isinstance(global_tokens, torch.Tensor) or not global_tokens.is_cuda
                or global_tokens.dtype != torch.int32 or not global_tokens.is_contiguous()):
            raise TypeError("global_tokens must be a contiguous CUDA int32 tensor")
        nbytes = (fa_fwd_local_global_packed_workspace_size(B, Hkv, T, d, code,
                                                            global_tokens.numel())
                  if pack_global else fa_fwd_local_global_workspace_size(T))
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        st = fa_fwd_local_global(q, k, v, out, lse, B, Hq, Hkv, T, d, scale, int(bool(causal)), wl,
                                 global_tokens if global_tokens.numel() else 0,
                                 global_tokens.numel(), code, ws, nbytes, stream)
        _check(st, "fa_fwd_local_global")
        return out, lse
    if window is not None:
        wl, wr = (int(x) for x in window)
        if causal:
            wr = 0 if wr < 0 else min(wr, 0)
        st = fa_fwd_window(q, k, v, out, lse, B, Hq, Hkv, T, d, scale, wl, wr, code, stream)
        _check(st, "fa_fwd_window")
        return out, lse
    if kernel == "simt":
        st = fa_fwd_simt(q, k, v, out, lse, B, Hq, Hkv, T, d, scale, int(bool(causal)), code,
                         stream)
        _check(st, "fa_fwd_simt")
        return out, lse
    splits = 1
    if code != FA_DTYPE_F32:
        splits = (fa_fwd_split_heuristic(B, Hq, Hkv, T, d, int(bool(causal)))
                  if num_splits is None else int(num_splits))
    if splits > 1:
        nbytes = fa_fwd_split_workspace_size(B, Hq, T, d, splits)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        st = fa_fwd_split(q, k, v, out, lse, B, Hq, Hkv, T, d, scale, int(bool(causal)), code,
                          splits, ws, nbytes, stream)
        _check(st, "fa_fwd_split")
    else:
        st = fa_fwd(q, k, v, out, lse, B, Hq, Hkv, T, d, scale, int(bool(causal)), code, stream)
        _check(st, "fa_fwd")
    return out, lse


def bwd(q, k, v, o, lse, d_o, causal: bool = False, scale: float | None = None, window=None,
        dq=None, dk=None, dv=None, stream=None, global_tokens=None):
    """Attention backward on CUDA tensors; returns (dq, dk, dv).

    q, k, v, o, lse are the forward's inputs and outputs (o and lse from a
    forward with the same causal flag, scale and window); d_o is the upstream
    gradient of o, like q.  dq, dk, dv may be given (shaped like q, k, v);
    otherwise they are allocated with torch, as is the small workspace.
    ``global_tokens`` selects the local-global mask as in ``fwd``.  The call
    is asynchronous on ``stream`` (default: the current torch stream).
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("d_o", d_o)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D tensor [B, H, T, d]")
        if t.dtype != q.dtype:
            raise TypeError(f"{name} must have the dtype of q")
    B, Hq, T, d = q.shape
    Hkv = k.shape[1]
    if tuple(o.shape) != tuple(q.shape) or tuple(d_o.shape) != tuple(q.shape):
        raise ValueError("o and d_o must be shaped like q")
    if tuple(k.shape) != (B, Hkv, T, d) or tuple(v.shape) != (B, Hkv, T, d):
        raise ValueError(f"k, v must be [B, Hkv, T, d]; got {tuple(k.shape)}, {tuple(v.shape)}")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, Hq, T] tensor")
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if global_tokens is not None:
        wl, wr = (0, 0) if window is None else (int(window[0]), int(window[1]))
        if wl != wr:
            raise ValueError("the local-global mask takes a symmetric window (w, w)")
        if (not isinstance(global_tokens, torch.Tensor) or not global_tokens.is_cuda
                or global_tokens.dtype != torch.int32 or not global_tokens.is_contiguous()):
            raise TypeError("global_tokens must be a contiguous CUDA int32 tensor")
        nbytes = fa_bwd_local_global_workspace_size(B, Hq, T)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        st = fa_bwd_local_global(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, T, d, scale,
                                 int(bool(causal)), wl,
                                 global_tokens if global_tokens.numel() else 0,
                                 global_tokens.numel(), code, ws, nbytes, stream)
        _check(st, "fa_bwd_local_global")
        return dq, dk, dv
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    nbytes = fa_bwd_workspace_size(B, Hq, T)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    st = fa_bwd(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, T, d, scale, int(bool(causal)), wl,
                wr, code, ws, nbytes, stream)
    _check(st, "fa_bwd")
    return dq, dk, dv


def fwd_host(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
             chunks: int = 4, workspace=None, stream=None, device=None):
    """Attention forward on host (CPU) tensors, copies overlapped with compute.

    q, k, v: contiguous CPU tensors [B, H, T, d] (pinned memory gives the
    overlap); out and lse are CPU tensors (allocated pinned when omitted).
    The batch runs in ``chunks`` pipelined chunks; the device workspace is
    allocated with torch on ``device`` (default: the current CUDA device)
    unless given.  Asynchronous on ``stream``: synchronise it before reading
    the outputs.  Returns (out, lse).
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.is_cuda:
            raise TypeError(f"{name} must be a CPU tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D tensor [B, H, T, d]")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    B, Hq, T, d = q.shape
    Hkv = k.shape[1]
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    if lse is None:
        lse = torch.empty((B, Hq, T), dtype=torch.float32).pin_memory()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    nbytes = fa_fwd_host_workspace_size(B, Hq, Hkv, T, d, code, chunks)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = fa_fwd_host(q, k, v, out, lse, B, Hq, Hkv, T, d, scale, int(bool(causal)), code, chunks,
                     workspace, nbytes, stream)
    _check(st, "fa_fwd_host")
    return out, lse


def bwd_host(q, k, v, o, lse, d_o, causal: bool = False, scale: float | None = None,
             window=None, chunks: int = 4, dq=None, dk=None, dv=None, workspace=None,
             stream=None, device=None):
    """Attention backward on host (CPU) tensors, copies overlapped with compute.

    Arguments as ``bwd`` with CPU tensors (pinned memory gives the overlap);
    dq, dk, dv are allocated pinned when omitted.  Asynchronous on ``stream``:
    synchronise it before reading the gradients.  Returns (dq, dk, dv).
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("d_o", d_o), ("lse", lse)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CPU tensor")
    B, Hq, T, d = q.shape
    Hkv = k.shape[1]
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty(q.shape, dtype=q.dtype).pin_memory() if dq is None else dq
    dk = torch.empty(k.shape, dtype=k.dtype).pin_memory() if dk is None else dk
    dv = torch.empty(v.shape, dtype=v.dtype).pin_memory() if dv is None else dv
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    nbytes = fa_bwd_host_workspace_size(B, Hq, Hkv, T, d, code, chunks)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = fa_bwd_host(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, T, d, scale, int(bool(causal)),
                     wl, wr, code, chunks, workspace, nbytes, stream)
    _check(st, "fa_bwd_host")
    return dq, dk, dv
