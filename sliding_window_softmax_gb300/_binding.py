"""ctypes binding of libnha.so (argument marshalling only: every step of the
operator runs in the library's CUDA kernels).

The names mirror the C ABI in ``include/nha.h``: :func:`nha_forward`,
:func:`nha_backward`, :func:`nha_workspace_bytes`.  Tensors are PyTorch CUDA
tensors (PyTorch supplies device memory and the stream); nothing here computes
any part of the operator, and there is no fallback: if the library is missing
or the call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnha.so")

NHA_OK = 0
STATUS = {0: "NHA_OK", 1: "NHA_ERR_INVALID_ARGUMENT", 2: "NHA_ERR_UNSUPPORTED",
          3: "NHA_ERR_WORKSPACE", 4: "NHA_ERR_CUDA", 5: "NHA_ERR_INTERNAL"}
DTYPE = {torch.float32: 0, torch.bfloat16: 1}

# Every symbol include/nha.h declares (checked by the tests).
EXPORTS = ("nha_workspace_bytes", "nha_forward", "nha_backward",
           "nha_workspace_bytes_ex", "nha_forward_ex", "nha_backward_ex",
           "nha_gate_total", "nha_state_combine", "nha_selftest_wait",
           "nha_varlen_pad", "nha_varlen_unpad",
           "nha_decode_step", "nha_decode_step_ex", "nha_decode_step_varlen",
           "nha_decode_prefill",
           "nha_forward_noalloc",
           "nha_launch_count", "nha_profile_begin", "nha_profile_end", "nha_status_string", "nha_last_error")

_lock = threading.Lock()
_lib = None


class Extras(ctypes.Structure):
    """nha_extras_t of include/nha.h (optional inputs and outputs of the _ex calls)."""
    _fields_ = [("fwd_workspace", ctypes.c_void_p), ("fwd_ws_bytes", ctypes.c_size_t),
                ("h0_k", ctypes.c_void_p), ("h0_v", ctypes.c_void_p),
                ("hT_k", ctypes.c_void_p), ("hT_v", ctypes.c_void_p),
                ("dhT_k", ctypes.c_void_p), ("dhT_v", ctypes.c_void_p),
                ("dh0_k", ctypes.c_void_p), ("dh0_v", ctypes.c_void_p),
                ("windows", ctypes.c_void_p), ("status", ctypes.c_void_p),
                ("windows_per_sequence", ctypes.c_int), ("cu_seqlens", ctypes.c_void_p)]


class ProfileRecord(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 64), ("launches", ctypes.c_int),
                ("total_ms", ctypes.c_double)]


def launch_count() -> int:
    """Kernels libnha has launched in this process."""
    return int(load_library().nha_launch_count())


def profile_begin() -> None:
    """Start bracketing every libnha kernel launch with CUDA events."""
    _raise(load_library(), load_library().nha_profile_begin())


def profile_end() -> dict:
    """End the session: {kernel name: (launches, total ms)}."""
    lib = load_library()
    recs = (ProfileRecord * 64)()
    n = lib.nha_profile_end(recs, 64)
    if n < 0:
        raise RuntimeError("nha_profile_end could not read its CUDA events")
    return {recs[i].name.decode(): (recs[i].launches, recs[i].total_ms) for i in range(min(n, 64))}


class NHAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libnha.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libnha.so not found at {p}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.nha_workspace_bytes.restype = sz
        lib.nha_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i, i]
        lib.nha_forward.restype = i
        lib.nha_forward.argtypes = [vp] * 6 + [i] * 8 + [f, vp, sz, vp]
        lib.nha_backward.restype = i
        lib.nha_backward.argtypes = [vp] * 11 + [i] * 8 + [f, vp, sz, vp]
        ep = ctypes.POINTER(Extras)
        lib.nha_workspace_bytes_ex.restype = sz
        lib.nha_workspace_bytes_ex.argtypes = [i] * 9 + [ep]
        lib.nha_forward_ex.restype = i
        lib.nha_forward_ex.argtypes = [vp] * 6 + [i] * 8 + [f, ep, vp, sz, vp]
        lib.nha_backward_ex.restype = i
        lib.nha_backward_ex.argtypes = [vp] * 11 + [i] * 8 + [f, ep, vp, sz, vp]
        lib.nha_selftest_wait.restype = i
        lib.nha_selftest_wait.argtypes = [vp, ctypes.c_longlong, vp]
        lib.nha_gate_total.restype = i
        lib.nha_gate_total.argtypes = [vp, vp] + [i] * 5 + [vp]
        lib.nha_state_combine.restype = i
        lib.nha_varlen_pad.restype = i
        lib.nha_varlen_pad.argtypes = [vp, vp, vp] + [i] * 6 + [vp]
        lib.nha_varlen_unpad.restype = i
        lib.nha_varlen_unpad.argtypes = [vp, vp, vp] + [i] * 6 + [vp]
        lib.nha_state_combine.argtypes = [vp] * 7 + [i] * 4 + [vp]
        lib.nha_decode_step.restype = i
        lib.nha_decode_step.argtypes = [vp] * 10 + [i] * 7 + [f, vp]
        lib.nha_decode_step_ex.restype = i
        lib.nha_decode_step_ex.argtypes = [vp] * 10 + [i] * 7 + [f, ctypes.c_uint, vp]
        lib.nha_decode_step_varlen.restype = i
        lib.nha_decode_step_varlen.argtypes = [vp] * 12 + [i] * 6 + [f, vp]
        lib.nha_decode_prefill.restype = i
        lib.nha_decode_prefill.argtypes = [vp] * 9 + [i] * 7 + [vp]
        lib.nha_forward_noalloc.restype = i
        lib.nha_forward_noalloc.argtypes = [vp] * 6 + [i] * 8 + [f, vp]
        lib.nha_status_string.restype = ctypes.c_char_p
        lib.nha_status_string.argtypes = [i]
        lib.nha_last_error.restype = ctypes.c_char_p
        lib.nha_last_error.argtypes = []
        lib.nha_launch_count.restype = ctypes.c_ulonglong
        lib.nha_launch_count.argtypes = []
        lib.nha_profile_begin.restype = i
        lib.nha_profile_begin.argtypes = []
        lib.nha_profile_end.restype = i
        lib.nha_profile_end.argtypes = [ctypes.POINTER(ProfileRecord), i]
        if path is None:
            _lib = lib
        return lib


def _raise(lib, rc):
    if rc != NHA_OK:
        raise NHAError(rc, lib.nha_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(name, t, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    # the library launches on the current device and takes that device's stream
    # (and, for the no-allocation forward, its scratch): tensors elsewhere would
    # be read through the wrong device's context
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{torch.cuda.current_device()}; "
                         "call under torch.cuda.device(...)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def nha_workspace_bytes(B, H, T, d, m, w, C=64, dtype=torch.bfloat16, backward=False,
                        reuse_forward=False, per_head_windows=False) -> int:
    """Workspace bytes of the forward (or backward); ``reuse_forward``: of a
    backward given the forward's workspace; ``per_head_windows``: of a call
    with a windows array or sequence lengths (nha_workspace_bytes_ex)."""
    lib = load_library()
    if reuse_forward or per_head_windows:
        ex = Extras()
        if reuse_forward:
            ex.fwd_workspace = 16  # any non-NULL value: only its presence counts here
        if per_head_windows:
            ex.windows = 16
        return int(lib.nha_workspace_bytes_ex(B, H, T, d, m, w, C, DTYPE[dtype], int(bool(backward)),
                                              ctypes.byref(ex)))
    return int(lib.nha_workspace_bytes(B, H, T, d, m, w, C, DTYPE[dtype], int(bool(backward))))


def nha_forward(q, k, v, log_alpha, w: int, C: int = 64, rope_base: float = 10000.0,
                o=None, lse=None, workspace=None, stream=None, h0=None, return_state=False, windows=None,
                status=None, cu_seqlens=None):
    """o, lse = nha_forward(q, k, v, log_alpha, w).  q, k, v [B,H,T,d]; log_alpha [B,H,T,m] fp32.

    ``h0`` = (h0k, h0v): initial slot states, fp32 [B,H,m,d] each.  With
    ``return_state`` the result is (o, lse, (hTk, hTv)), the final slot states
    (the long memory after token T - w - 1).  ``windows``: int32 [H] per-head
    or [B*H] per-sequence windows.  ``cu_seqlens``: int32 [B+1] offsets, batch
    entry b then holds a sequence of cu_seqlens[b+1] - cu_seqlens[b] tokens in
    its first rows (the rest finite padding).  Either calls nha_forward_ex."""
    lib = load_library()
    B, H, T, d = q.shape
    m = log_alpha.shape[-1]
    dt = q.dtype
    if dt not in DTYPE:
        raise TypeError(f"unsupported dtype {dt}")
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check(n, t, dt, (B, H, T, d))
    _check("log_alpha", log_alpha, torch.float32, (B, H, T, m))
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    _check("o", o, dt, (B, H, T, d))
    _check("lse", lse, torch.float32, (B, H, T))
    ex = _extras(shape=(B, H, m, d), windows=windows, cu_seqlens=cu_seqlens)
    need = int(lib.nha_workspace_bytes_ex(B, H, T, d, m, w, C, DTYPE[dt], 0, ctypes.byref(ex)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    hT = None
    if return_state:
        hT = (torch.empty((B, H, m, d), dtype=torch.float32, device=q.device),
              torch.empty((B, H, m, d), dtype=torch.float32, device=q.device))
    ex = _extras(shape=(B, H, m, d), windows=windows, status=status, cu_seqlens=cu_seqlens, h0=h0, hT=hT)
    rc = lib.nha_forward_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(o), _ptr(lse),
                            B, H, T, d, m, int(w), int(C), DTYPE[dt], float(rope_base), ctypes.byref(ex),
                            _ptr(workspace), ws_bytes, _stream_handle(stream))
    _raise(lib, rc)
    return (o, lse, hT) if return_state else (o, lse)


def nha_forward_noalloc(q, k, v, log_alpha, w: int, C: int = 64, rope_base: float = 10000.0,
                        o=None, lse=None, stream=None):
    """nha_forward using the library's built-in scratch (no workspace argument).

    For callers that cannot allocate device memory; see include/nha.h for the
    size limit and the sharing rules."""
    lib = load_library()
    B, H, T, d = q.shape
    m = log_alpha.shape[-1]
    dt = q.dtype
    if dt not in DTYPE:
        raise TypeError(f"unsupported dtype {dt}")
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check(n, t, dt, (B, H, T, d))
    _check("log_alpha", log_alpha, torch.float32, (B, H, T, m))
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device) if lse is None else lse
    _check("o", o, dt, (B, H, T, d))
    _check("lse", lse, torch.float32, (B, H, T))
    rc = lib.nha_forward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(o), _ptr(lse),
                                 B, H, T, d, m, int(w), int(C), DTYPE[dt], float(rope_base),
                                 _stream_handle(stream))
    _raise(lib, rc)
    return o, lse


STATUS_TIMEOUT = 1      # NHA_STATUS_TIMEOUT
STATUS_GATE_RANGE = 2   # NHA_STATUS_GATE_RANGE


def _extras(fwd_workspace=None, shape=None, windows=None, status=None, cu_seqlens=None, **states):
    """Extras from tensors: fwd_workspace, windows (int32 CUDA [H] per head,
    or [B*H] per sequence), cu_seqlens (int32 CUDA [B+1]), and state pairs
    given as (K, V) tuples of fp32 [B,H,m,d] CUDA tensors under the names h0,
    hT, dhT, dh0."""
    ex = Extras()
    if status is not None:
        _check("status", status, torch.int32, (1,))
        ex.status = status.data_ptr()
    if windows is not None:
        _check("windows", windows, torch.int32)
        B, H = shape[0], shape[1]
        if windows.numel() == H:
            ex.windows_per_sequence = 0
        elif windows.numel() == B * H:
            ex.windows_per_sequence = 1
        else:
            raise ValueError(f"windows has {windows.numel()} entries: expected H={H} or B*H={B * H}")
        ex.windows = windows.data_ptr()
    if cu_seqlens is not None:
        _check("cu_seqlens", cu_seqlens, torch.int32, (shape[0] + 1,))
        ex.cu_seqlens = cu_seqlens.data_ptr()
    if fwd_workspace is not None:
        _check("fwd_workspace", fwd_workspace)
        ex.fwd_workspace = fwd_workspace.data_ptr()
        ex.fwd_ws_bytes = fwd_workspace.numel() * fwd_workspace.element_size()
    for name, pair in states.items():
        if pair is None:
            continue
        kt, vt = pair
        _check(f"{name}[0]", kt, torch.float32, shape)
        _check(f"{name}[1]", vt, torch.float32, shape)
        setattr(ex, f"{name}_k", kt.data_ptr())
        setattr(ex, f"{name}_v", vt.data_ptr())
    return ex


def nha_backward(q, k, v, log_alpha, o, lse, dout, w: int, C: int = 64,
                 rope_base: float = 10000.0, dq=None, dk=None, dv=None, dlog_alpha=None,
                 workspace=None, stream=None, fwd_workspace=None, h0=None, dhT=None, windows=None,
                 status=None, cu_seqlens=None):
    """dq, dk, dv, dlog_alpha = nha_backward(q, k, v, log_alpha, o, lse, dout, w).

    ``fwd_workspace``: the workspace tensor the forward of these inputs ran
    with, untouched since; the backward then reuses the chunk states and
    rotated q, k it holds.  ``h0``: the forward's initial slot states; the
    result then ends with (dh0k, dh0v).  ``dhT``: the gradient with respect to
    the forward's final slot states.  ``windows``, ``cu_seqlens``: as for
    nha_forward (the same ones).  Calls nha_backward_ex."""
    lib = load_library()
    B, H, T, d = q.shape
    m = log_alpha.shape[-1]
    dt = q.dtype
    if dt not in DTYPE:
        raise TypeError(f"unsupported dtype {dt}")
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check(n, t, dt, (B, H, T, d))
    _check("log_alpha", log_alpha, torch.float32, (B, H, T, m))
    _check("lse", lse, torch.float32, (B, H, T))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    dlog_alpha = torch.empty_like(log_alpha) if dlog_alpha is None else dlog_alpha
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check(n, t, dt, (B, H, T, d))
    _check("dlog_alpha", dlog_alpha, torch.float32, (B, H, T, m))
    dh0 = None
    if h0 is not None:
        dh0 = (torch.empty((B, H, m, d), dtype=torch.float32, device=q.device),
               torch.empty((B, H, m, d), dtype=torch.float32, device=q.device))
    ex = _extras(fwd_workspace, shape=(B, H, m, d), windows=windows, status=status, cu_seqlens=cu_seqlens, h0=h0,
                 dhT=dhT, dh0=dh0)
    need = int(lib.nha_workspace_bytes_ex(B, H, T, d, m, w, C, DTYPE[dt], 1, ctypes.byref(ex)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.nha_backward_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(o), _ptr(lse),
                             _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dlog_alpha),
                             B, H, T, d, m, int(w), int(C), DTYPE[dt], float(rope_base), ctypes.byref(ex),
                             _ptr(workspace), ws_bytes, _stream_handle(stream))
    _raise(lib, rc)
    return (dq, dk, dv, dlog_alpha) if dh0 is None else (dq, dk, dv, dlog_alpha) + dh0


def nha_varlen_pad(packed, cu_seqlens, T: int, stream=None):
    """Packed rows [H, Ttot, *row] -> padded [B, H, T, *row] (B = len(cu_seqlens) - 1;
    rows past each sequence zero).  nha_varlen_pad of include/nha.h."""
    lib = load_library()
    _check("packed", packed)
    _check("cu_seqlens", cu_seqlens, torch.int32)
    B = cu_seqlens.numel() - 1
    H, Ttot = packed.shape[0], packed.shape[1]
    row = tuple(packed.shape[2:])
    width = 1
    for n in row:
        width *= n
    out = torch.empty((B, H, T) + row, dtype=packed.dtype, device=packed.device)
    rc = lib.nha_varlen_pad(_ptr(packed), _ptr(out), _ptr(cu_seqlens), B, H, int(T), Ttot, width,
                            packed.element_size(), _stream_handle(stream))
    _raise(lib, rc)
    return out


def nha_varlen_unpad(padded, cu_seqlens, Ttot: int, out=None, stream=None):
    """Padded rows [B, H, T, *row] -> packed [H, Ttot, *row] (each sequence's
    rows only).  nha_varlen_unpad of include/nha.h."""
    lib = load_library()
    _check("padded", padded)
    _check("cu_seqlens", cu_seqlens, torch.int32)
    B, H, T = padded.shape[0], padded.shape[1], padded.shape[2]
    row = tuple(padded.shape[3:])
    width = 1
    for n in row:
        width *= n
    if out is None:
        out = torch.zeros((H, int(Ttot)) + row, dtype=padded.dtype, device=padded.device)
    _check("out", out, padded.dtype, (H, int(Ttot)) + row)
    rc = lib.nha_varlen_unpad(_ptr(padded), _ptr(out), _ptr(cu_seqlens), B, H, T, int(Ttot), width,
                              padded.element_size(), _stream_handle(stream))
    _raise(lib, rc)
    return out


def nha_forward_varlen(q, k, v, log_alpha, cu_seqlens, max_seqlen: int, w: int, C: int = 64,
                       rope_base: float = 10000.0, stream=None, h0=None, return_state=False, windows=None,
                       status=None):
    """Forward over packed sequences: q, k, v [H, Ttot, d], log_alpha [H, Ttot, m]
    with sequence b in rows cu_seqlens[b] .. cu_seqlens[b+1] - 1 (int32 [B+1]),
    each no longer than max_seqlen.  Returns (o [H,Ttot,d], lse [H,Ttot],
    ctx) and, with return_state, the per-sequence final states [B,H,m,d]
    before ctx; ctx holds the padded tensors nha_backward_varlen needs.
    The rows move through nha_varlen_pad / nha_varlen_unpad; the sequences
    run in one nha_forward_ex call with cu_seqlens."""
    Ttot = q.shape[1]
    T = int(max_seqlen)
    qp, kp, vp = (nha_varlen_pad(x, cu_seqlens, T, stream) for x in (q, k, v))
    lp = nha_varlen_pad(log_alpha, cu_seqlens, T, stream)
    B, H = qp.shape[0], qp.shape[1]
    op = torch.zeros_like(qp)  # rows past a sequence stay finite for the backward
    lsep = torch.zeros((B, H, T), dtype=torch.float32, device=q.device)
    m, d = log_alpha.shape[-1], q.shape[-1]
    need = nha_workspace_bytes(B, H, T, d, m, w, C, q.dtype, per_head_windows=True)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    res = nha_forward(qp, kp, vp, lp, w, C, rope_base, o=op, lse=lsep, workspace=ws, stream=stream, h0=h0,
                      return_state=return_state, windows=windows, status=status, cu_seqlens=cu_seqlens)
    o = nha_varlen_unpad(op, cu_seqlens, Ttot, stream=stream)
    lse = nha_varlen_unpad(lsep.unsqueeze(-1), cu_seqlens, Ttot, stream=stream).squeeze(-1)
    ctx = dict(q=qp, k=kp, v=vp, log_alpha=lp, o=op, lse=lsep, workspace=ws, T=T, Ttot=Ttot)
    return (o, lse, res[2], ctx) if return_state else (o, lse, ctx)


def nha_backward_varlen(ctx, dout, cu_seqlens, w: int, C: int = 64, rope_base: float = 10000.0, stream=None,
                        h0=None, dhT=None, windows=None, status=None):
    """Backward of nha_forward_varlen: dout [H, Ttot, d] -> (dq, dk, dv [H,Ttot,d],
    dlog_alpha [H,Ttot,m]) and, with h0, the per-sequence (dh0k, dh0v).
    Reuses the forward's workspace held in ctx (same w, C, rope_base,
    windows and cu_seqlens)."""
    T, Ttot = ctx["T"], ctx["Ttot"]
    dop = nha_varlen_pad(dout, cu_seqlens, T, stream)
    res = nha_backward(ctx["q"], ctx["k"], ctx["v"], ctx["log_alpha"], ctx["o"], ctx["lse"], dop, w, C,
                       rope_base, stream=stream, fwd_workspace=ctx["workspace"], h0=h0, dhT=dhT,
                       windows=windows, status=status, cu_seqlens=cu_seqlens)
    grads = tuple(nha_varlen_unpad(g, cu_seqlens, Ttot, stream=stream) for g in res[:4])
    return grads + tuple(res[4:])


def nha_decode_state(B, H, d, m, w, dtype=torch.bfloat16, device="cuda"):
    """Zeroed decode state: (state_k, state_v [B,H,m,d] fp32, ring_k, ring_v [B,H,max(w,1),d] dtype,
    ring_la [B,H,max(w,1),m] fp32)."""
    n = max(int(w), 1)
    return (torch.zeros((B, H, m, d), dtype=torch.float32, device=device),
            torch.zeros((B, H, m, d), dtype=torch.float32, device=device),
            torch.zeros((B, H, n, d), dtype=dtype, device=device),
            torch.zeros((B, H, n, d), dtype=dtype, device=device),
            torch.zeros((B, H, n, m), dtype=torch.float32, device=device))


DECODE_OVERLAP = 1  # NHA_DECODE_OVERLAP


def nha_decode_step(q, k, v, log_alpha, t: int, w: int, state, rope_base: float = 10000.0, o=None,
                     stream=None, overlap=False):
    """o_t = nha_decode_step(q, k, v, log_alpha, t, w, state).

    q, k, v [B,H,d] and log_alpha [B,H,m] (fp32) are token t of every head;
    ``state`` is the tuple from :func:`nha_decode_state`, updated in place.
    ``overlap``: the kernel enqueued just before on the stream writes none of
    this state (another layer's step, say), so the step may stream its state
    in while that kernel runs (nha_decode_step_ex with NHA_DECODE_OVERLAP)."""
    lib = load_library()
    B, H, d = q.shape
    m = log_alpha.shape[-1]
    dt = q.dtype
    if dt not in DTYPE:
        raise TypeError(f"unsupported dtype {dt}")
    n = max(int(w), 1)
    sk, sv, rk, rv, rla = state
    for nm, x in (("q", q), ("k", k), ("v", v)):
        _check(nm, x, dt, (B, H, d))
    _check("log_alpha", log_alpha, torch.float32, (B, H, m))
    _check("state_k", sk, torch.float32, (B, H, m, d))
    _check("state_v", sv, torch.float32, (B, H, m, d))
    _check("ring_k", rk, dt, (B, H, n, d))
    _check("ring_v", rv, dt, (B, H, n, d))
    _check("ring_la", rla, torch.float32, (B, H, n, m))
    o = torch.empty_like(q) if o is None else o
    _check("o", o, dt, (B, H, d))
    rc = lib.nha_decode_step_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(o), _ptr(sk), _ptr(sv),
                                _ptr(rk), _ptr(rv), _ptr(rla), int(t), B, H, d, m, int(w), DTYPE[dt],
                                float(rope_base), DECODE_OVERLAP if overlap else 0, _stream_handle(stream))
    _raise(lib, rc)
    return o


def nha_decode_prefill(k, v, log_alpha, w: int, state=None, windows=None, stream=None):
    """Decode state after the prompt k, v [B,H,T,d], log_alpha [B,H,T,m]:
    returns (or fills) the tuple of :func:`nha_decode_state`, ready for
    :func:`nha_decode_step` at t = T (``windows``: per-head windows, as for
    :func:`nha_decode_step_varlen`)."""
    lib = load_library()
    B, H, T, d = k.shape
    m = log_alpha.shape[-1]
    dt = k.dtype
    if dt not in DTYPE:
        raise TypeError(f"unsupported dtype {dt}")
    _check("k", k, dt, (B, H, T, d))
    _check("v", v, dt, (B, H, T, d))
    _check("log_alpha", log_alpha, torch.float32, (B, H, T, m))
    if state is None:
        state = nha_decode_state(B, H, d, m, w, dtype=dt, device=k.device)
    n = max(int(w), 1)
    sk, sv, rk, rv, rla = state
    _check("state_k", sk, torch.float32, (B, H, m, d))
    _check("state_v", sv, torch.float32, (B, H, m, d))
    _check("ring_k", rk, dt, (B, H, n, d))
    _check("ring_v", rv, dt, (B, H, n, d))
    _check("ring_la", rla, torch.float32, (B, H, n, m))
    if windows is not None:
        _check("windows", windows, torch.int32, (H,))
    rc = lib.nha_decode_prefill(_ptr(k), _ptr(v), _ptr(log_alpha), _ptr(sk), _ptr(sv), _ptr(rk), _ptr(rv),
                                _ptr(rla), _ptr(windows), B, H, T, d, m, int(w), DTYPE[dt], _stream_handle(stream))
    _raise(lib, rc)
    return state


def nha_decode_step_varlen(q, k, v, log_alpha, positions, w: int, state, rope_base: float = 10000.0, o=None,
                           windows=None, stream=None):
    """o = nha_decode_step_varlen(q, k, v, log_alpha, positions, w, state): like
    :func:`nha_decode_step`, sequence b at position ``positions[b]`` (a CUDA
    int32 tensor [B], read on the device); ``windows`` (CUDA int32 [H], each in
    [0, w]) gives every head its own window inside the w-entry ring."""
    lib = load_library()
    B, H, d = q.shape
    m = log_alpha.shape[-1]
    dt = q.dtype
    if dt not in DTYPE:
        raise TypeError(f"unsupported dtype {dt}")
    n = max(int(w), 1)
    sk, sv, rk, rv, rla = state
    for nm, x in (("q", q), ("k", k), ("v", v)):
        _check(nm, x, dt, (B, H, d))
    _check("log_alpha", log_alpha, torch.float32, (B, H, m))
    _check("positions", positions, torch.int32, (B,))
    if windows is not None:
        _check("windows", windows, torch.int32, (H,))
    _check("state_k", sk, torch.float32, (B, H, m, d))
    _check("state_v", sv, torch.float32, (B, H, m, d))
    _check("ring_k", rk, dt, (B, H, n, d))
    _check("ring_v", rv, dt, (B, H, n, d))
    _check("ring_la", rla, torch.float32, (B, H, n, m))
    o = torch.empty_like(q) if o is None else o
    _check("o", o, dt, (B, H, d))
    rc = lib.nha_decode_step_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(o), _ptr(sk), _ptr(sv),
                                    _ptr(rk), _ptr(rv), _ptr(rla), _ptr(positions), _ptr(windows), B, H, d, m, int(w),
                                    DTYPE[dt], float(rope_base), _stream_handle(stream))
    _raise(lib, rc)
    return o


def nha_gate_total(log_alpha, w: int, stream=None):
    """decay [B,H,m] = exp(sum of log_alpha over the tokens j < T - w): the factor
    a run of these tokens applies to the state it starts from."""
    lib = load_library()
    B, H, T, m = log_alpha.shape
    _check("log_alpha", log_alpha, torch.float32, (B, H, T, m))
    decay = torch.empty((B, H, m), dtype=torch.float32, device=log_alpha.device)
    _raise(lib, lib.nha_gate_total(_ptr(log_alpha), _ptr(decay), B, H, T, m, int(w), _stream_handle(stream)))
    return decay


def nha_state_combine(decay, prev, cur, out=None, stream=None):
    """(out_k, out_v) = decay o prev + cur for state pairs (K, V) of fp32 [B,H,m,d]."""
    lib = load_library()
    B, H, m, d = cur[0].shape
    _check("decay", decay, torch.float32, (B, H, m))
    for n, t in (("prev_k", prev[0]), ("prev_v", prev[1]), ("cur_k", cur[0]), ("cur_v", cur[1])):
        _check(n, t, torch.float32, (B, H, m, d))
    if out is None:
        out = (torch.empty_like(cur[0]), torch.empty_like(cur[1]))
    rc = lib.nha_state_combine(_ptr(decay), _ptr(prev[0]), _ptr(prev[1]), _ptr(cur[0]), _ptr(cur[1]),
                               _ptr(out[0]), _ptr(out[1]), B, H, m, d, _stream_handle(stream))
    _raise(lib, rc)
    return out


def nha_selftest_wait(cycles: int, status=None, stream=None):
    """Runs one bounded wait that runs out after ``cycles`` SM clocks; returns the
    status word (int32 CUDA tensor [1]), NHA_STATUS_TIMEOUT once it has run."""
    lib = load_library()
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device="cuda")
    _check("status", status, torch.int32, (1,))
    _raise(lib, lib.nha_selftest_wait(_ptr(status), int(cycles), _stream_handle(stream)))
    return status
