"""Native Hybrid Attention (NHA) -- fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.
The product path (``sliding_window_softmax_gb300``) never imports, loads or
calls it, and the oracle imports nothing from the product.

Two independent restatements of the operator live here:

* ``nha_oracle.c`` -- token-by-token recurrent NHA in fp64 with a
  hand-derived reverse sweep for the gradients ("Native Hybrid Attention for
  Efficient Sequence Modeling", Paper-Notes page, section 关键设计/层内混合:
  the K^long_t recurrence, the single-softmax o_t equation, the token shift
  and window-only RoPE).  Wrapped below by :func:`forward` / :func:`backward`.
* ``naive.py`` -- the O(T^2) unrolled-gate closed form in PyTorch CPU fp64,
  differentiated by autograd.

Every function here takes and returns float64 numpy arrays in the layout
q, k, v, o: [B, H, T, d]; log_alpha: [B, H, T, m]; lse: [B, H, T].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nha_oracle.c")
_LIB = os.path.join(_HERE, "libnha_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libnha_oracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            L = ctypes.c_long
            lib.nha_oracle_forward.restype = ctypes.c_int
            lib.nha_oracle_forward.argtypes = [dp, dp, dp, dp, dp, dp, dp, L, L, L, L, L, L,
                                               ctypes.c_double, ctypes.c_int, dp, dp, dp, dp]
            lib.nha_oracle_backward.restype = ctypes.c_int
            lib.nha_oracle_backward.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, L, L, L, L,
                                                L, L, ctypes.c_double, ctypes.c_int, dp, dp, dp, dp,
                                                dp, dp]
            lib.nha_oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch

        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ptr_or_null(a):
    return None if a is None else _ptr(a)


def num_threads() -> int:
    """OpenMP threads the oracle uses by default (all host cores)."""
    return int(_load().nha_oracle_num_threads())


def _h0(h0, B, H, m, d):
    """(h0k, h0v) as contiguous float64 [B,H,m,d] arrays, or (None, None)."""
    if h0 is None:
        return None, None
    hk, hv = _f64(h0[0]), _f64(h0[1])
    assert hk.shape == (B, H, m, d) and hv.shape == (B, H, m, d)
    return hk, hv


def forward(q, k, v, log_alpha, w: int, rope_base: float = 10000.0, nthreads: int = 0,
            with_omega: bool = False, h0=None, return_state: bool = False):
    """fp64 NHA forward.  Returns (o, lse) or (o, lse, omega_L); with
    ``return_state`` the tuple ends with (hTk, hTv), each [B,H,m,d]: the final
    slot states, the long memory after the last token that left the window
    (token T - w - 1), h0 (or zero) when no token has.

    h0 = (h0k, h0v), each [B,H,m,d]: initial slot states (the long memory before
    token 0); with them no slot logit is masked."""
    q, k, v, la = _f64(q), _f64(k), _f64(v), _f64(log_alpha)
    B, H, T, d = q.shape
    m = la.shape[-1]
    assert k.shape == q.shape and v.shape == q.shape and la.shape[:3] == (B, H, T)
    hk, hv = _h0(h0, B, H, m, d)
    o = np.zeros_like(q)
    lse = np.zeros((B, H, T), dtype=np.float64)
    om = np.zeros((B, H, T), dtype=np.float64)
    hTk = np.zeros((B, H, m, d)) if return_state else None
    hTv = np.zeros((B, H, m, d)) if return_state else None
    rc = _load().nha_oracle_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(o), _ptr(lse),
                                    _ptr(om), B, H, T, d, m, int(w), float(rope_base),
                                    int(nthreads), _ptr_or_null(hk), _ptr_or_null(hv),
                                    _ptr_or_null(hTk), _ptr_or_null(hTv))
    if rc != 0:
        raise ValueError(f"oracle forward rejected the shape (rc={rc})")
    out = (o, lse, om) if with_omega else (o, lse)
    return out + (hTk, hTv) if return_state else out


def backward(q, k, v, log_alpha, dout, w: int, rope_base: float = 10000.0, nthreads: int = 0,
             h0=None, dhT=None):
    """fp64 NHA backward of loss = sum(o * dout) (+ <hTk, dhTk> + <hTv, dhTv> with
    dhT = (dhTk, dhTv), the gradient with respect to the final states).  Returns
    (dq, dk, dv, dlog_alpha), and with h0 = (h0k, h0v) also (dh0k, dh0v)."""
    q, k, v, la, g = _f64(q), _f64(k), _f64(v), _f64(log_alpha), _f64(dout)
    B, H, T, d = q.shape
    m = la.shape[-1]
    hk, hv = _h0(h0, B, H, m, d)
    gk, gv = _h0(dhT, B, H, m, d)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(q), np.zeros_like(q)
    dla = np.zeros_like(la)
    dhk = np.zeros((B, H, m, d)) if hk is not None else None
    dhv = np.zeros((B, H, m, d)) if hk is not None else None
    rc = _load().nha_oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(g), _ptr(dq),
                                     _ptr(dk), _ptr(dv), _ptr(dla), B, H, T, d, m, int(w),
                                     float(rope_base), int(nthreads), _ptr_or_null(hk),
                                     _ptr_or_null(hv), _ptr_or_null(dhk), _ptr_or_null(dhv),
                                     _ptr_or_null(gk), _ptr_or_null(gv))
    if rc != 0:
        raise ValueError(f"oracle backward rejected the shape (rc={rc})")
    return (dq, dk, dv, dla) if hk is None else (dq, dk, dv, dla, dhk, dhv)
