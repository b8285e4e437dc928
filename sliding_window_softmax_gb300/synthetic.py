"""Seeded synthetic inputs for the NHA operator (shared by the tests, the bench
and the oracle legs; it holds none of the operator's arithmetic).

Recipe (the pages measure this operator on no dataset; these stand in for
the layer inputs a 340M / 1.3B / 8B-hybrid NHA model would feed it):

* ``torch.Generator().manual_seed(seed)`` on the host, drawn in the order
  q, k, v, log_alpha, dout;
* q, k, v ~ N(0, 1) * d**-0.25, then cast to the dtype;
* log_alpha = logsigmoid(N(mu, 1)) in fp32, mu = 3 (mu = 4 for the
  long-context sweep);
* dout ~ N(0, 1) in the dtype.

Seeds: 1000 + workload index (1..5), plus 10 * w_index + m_index for the
window/slot grid.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    m: int
    w: int
    C: int = 64
    dtype: str = "bf16"  # "bf16" or "f32"
    mu: float = 3.0
    seed: int = 1000
    backward: bool = True

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the operator is specified on.
TINY_F32 = Workload("tiny-f32 B1 H2 T256 d64 m16 w32", 1, 2, 256, 64, 16, 32, dtype="f32", seed=1001)
LAYER_340M = Workload("340M-like B8 H16 T2048 d64 m64 w64", 8, 16, 2048, 64, 64, 64, seed=1002)
LAYER_1P3B = Workload("1.3B-like B4 H16 T2048 d128 m64 w512", 4, 16, 2048, 128, 64, 512, seed=1003)


def long_context(T: int) -> Workload:
    return Workload(f"8B-hybrid-like B1 H32 T{T} d128 m64 w512 fwd", 1, 32, T, 128, 64, 512,
                    mu=4.0, seed=1004, backward=False)


LONG_CONTEXT_T = (4096, 8192, 16384, 32768, 65536)
GRID_W = (0, 64, 256, 1024, 8192)
GRID_M = (32, 64)


def grid_point(w: int, m: int) -> Workload:
    wi, mi = GRID_W.index(w), GRID_M.index(m)
    return Workload(f"ablation B2 H16 T8192 d128 m{m} w{w}", 2, 16, 8192, 128, m, w,
                    seed=1005 + 10 * wi + mi)


def all_workloads() -> List[Workload]:
    out = [TINY_F32, LAYER_340M, LAYER_1P3B,
           LAYER_1P3B.with_(name="1.3B-like w=0 (pure slot RNN)", w=0),
           LAYER_1P3B.with_(name="1.3B-like w=T (causal attention)", w=2048)]
    out += [long_context(T) for T in LONG_CONTEXT_T]
    out += [grid_point(w, m) for w in GRID_W for m in GRID_M]
    return out


def make_inputs(wl: Workload, seed: Optional[int] = None, device="cpu", scale_qk: float = 1.0):
    """Return dict q, k, v, log_alpha, dout (host tensors unless device given).

    ``scale_qk`` multiplies q and k before the dtype cast (the "sharp" variant
    of the parity suite uses 4)."""
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    shp = (wl.B, wl.H, wl.T, wl.d)
    s = wl.d ** -0.25
    dt = wl.torch_dtype
    q = (torch.randn(shp, generator=g) * (s * scale_qk)).to(dt)
    k = (torch.randn(shp, generator=g) * (s * scale_qk)).to(dt)
    v = (torch.randn(shp, generator=g) * s).to(dt)
    la = torch.nn.functional.logsigmoid(
        torch.randn((wl.B, wl.H, wl.T, wl.m), generator=g) + wl.mu).to(torch.float32)
    dout = torch.randn(shp, generator=g).to(dt)
    out = dict(q=q, k=k, v=v, log_alpha=la, dout=dout)
    if device != "cpu":
        out = {n: t.to(device) for n, t in out.items()}
    return out


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """One decode token for B sequences through `layers` NHA layers at position t."""
    name: str
    B: int
    H: int
    d: int
    m: int
    w: int
    t: int
    layers: int
    dtype: str = "bf16"
    seed: int = 1006

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


# Serving-style decode of the 1.3B-like layer: 16 sequences, 24 layers, a full
# window and a long memory in use (t >= w).
DECODE_1P3B = DecodeWorkload("1.3B-like decode B16 H16 d128 m64 w512 t4096, 24 layers", 16, 16, 128, 64, 512,
                             4096, 24)


def make_decode_layer(dw: DecodeWorkload, layer: int, device="cuda"):
    """Token inputs (q, k, v, log_alpha [B,H,.]) and a state (state_k, state_v,
    ring_k, ring_v, ring_la) for one layer, drawn on `device` from a generator
    seeded with seed + layer: q, k, v and the ring's k, v ~ N(0,1) d**-0.25;
    log_alpha and the ring's ~ logsigmoid(N(3, 1)); the slot states
    ~ N(0,1) * 0.3 d**-0.25 (the size of a convex mix of keys)."""
    g = torch.Generator(device=device).manual_seed(dw.seed + layer)
    B, H, d, m, n = dw.B, dw.H, dw.d, dw.m, max(dw.w, 1)
    s = d ** -0.25
    dt = dw.torch_dtype

    def rn(*shape):
        return torch.randn(shape, generator=g, device=device)

    def gate(*shape):
        return torch.nn.functional.logsigmoid(rn(*shape) + 3.0)

    x = dict(q=(rn(B, H, d) * s).to(dt), k=(rn(B, H, d) * s).to(dt), v=(rn(B, H, d) * s).to(dt),
             log_alpha=gate(B, H, m))
    state = (rn(B, H, m, d) * (0.3 * s), rn(B, H, m, d) * (0.3 * s), (rn(B, H, n, d) * s).to(dt),
             (rn(B, H, n, d) * s).to(dt), gate(B, H, n, m))
    return x, state
