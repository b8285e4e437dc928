"""Naive O(T^2) unrolled-gate NHA in PyTorch CPU fp64 (autograd for gradients).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

This is a second, independent restatement of the operator ("Native Hybrid
Attention for Efficient Sequence Modeling", Paper-Notes page, section
关键设计/层内混合).  Instead of running the K^long_t recurrence token by token
it writes the state after token j in closed form, unrolling the gated update:

    K^long after token j  =  sum_{s <= j}  (prod_{r=s+1..j} alpha_r) (1 - alpha_s) (x) k_s

with the gate product taken as exp(cumsum(log_alpha)_j - cumsum(log_alpha)_s)
per slot, and V^long likewise.  The query at t reads the state after token
t - w (token shift); the window keys are s in [t-w+1, t].  RoPE is written in
its complex form: the pair (x_i, x_{i+d/2}) is the complex number
x_i + i x_{i+d/2}, multiplied by exp(i * pos * base^(-2i/d)).  One softmax
with scale 1/sqrt(d) runs over [slot logits | window logits].

With initial slot states h0 (the long memory before token 0) the state after
token j gains (prod_{r=0..j} alpha_r) h0 = exp(cumsum(log_alpha)_j) h0, queries
t < w read h0 itself, and no slot logit is masked.

Only for tiny shapes: memory is O(B H T^2 m).
"""
from __future__ import annotations

import math

import torch


def rope_complex(x: torch.Tensor, base: float) -> torch.Tensor:
    """RoPE at absolute positions 0..T-1 via complex multiplication; x [..., T, d]."""
    T, d = x.shape[-2], x.shape[-1]
    h = d // 2
    i = torch.arange(h, dtype=torch.float64)
    theta = base ** (-2.0 * i / d)
    pos = torch.arange(T, dtype=torch.float64)
    ang = pos[:, None] * theta[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)  # e^{i ang}
    z = torch.complex(x[..., :h], x[..., h:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def slot_states(x: torch.Tensor, log_alpha: torch.Tensor, h0=None) -> torch.Tensor:
    """Closed-form slot state after each token: [B,H,T(j),m,d] (h0 [B,H,m,d] or None)."""
    T = x.shape[-2]
    b = torch.cumsum(log_alpha, dim=-2)  # [B,H,T,m]
    u = -torch.expm1(log_alpha)
    jj = torch.arange(T)[:, None]
    ss = torch.arange(T)[None, :]
    causal = (ss <= jj)[None, None, :, :, None]  # [1,1,j,s,1]
    expo = b[:, :, :, None, :] - b[:, :, None, :, :]  # [B,H,j,s,m]
    expo = torch.where(causal, expo, torch.full_like(expo, -math.inf))
    decay = torch.exp(expo)
    S = torch.einsum("bhjsi,bhsi,bhsd->bhjid", decay, u, x)
    if h0 is not None:
        S = S + torch.exp(b)[..., None] * h0[:, :, None]
    return S


def nha_naive(q, k, v, log_alpha, w: int, rope_base: float = 10000.0, return_omega=False, h0k=None, h0v=None):
    """Forward of NHA for float64 tensors; returns (o, lse) [, omega_L].
    h0k, h0v [B,H,m,d]: optional initial slot states."""
    B, H, T, d = q.shape
    m = log_alpha.shape[-1]
    w = min(int(w), T)
    sigma = 1.0 / math.sqrt(d)
    SK = slot_states(k, log_alpha, h0k)  # [B,H,T,m,d]
    SV = slot_states(v, log_alpha, h0v)
    t = torch.arange(T)
    jidx = (t - w).clamp(min=0)
    SKq = SK[:, :, jidx]  # state read by query t
    SVq = SV[:, :, jidx]
    if h0k is None:
        has = t >= w
    else:  # the long memory is never empty: queries t < w read h0
        has = torch.ones(T, dtype=torch.bool)
        early = (t < w)[None, None, :, None, None]
        SKq = torch.where(early, h0k[:, :, None], SKq)
        SVq = torch.where(early, h0v[:, :, None], SVq)
    L = sigma * torch.einsum("bhtd,bhtid->bhti", q, SKq)
    L = torch.where(has[None, None, :, None], L, torch.full_like(L, -math.inf))
    qr, kr = rope_complex(q, rope_base), rope_complex(k, rope_base)
    S = sigma * torch.einsum("bhtd,bhsd->bhts", qr, kr)
    s = torch.arange(T)
    win = (s[None, :] <= t[:, None]) & (s[None, :] > t[:, None] - w)
    S = torch.where(win[None, None], S, torch.full_like(S, -math.inf))
    logits = torch.cat([L, S], dim=-1)
    lse = torch.logsumexp(logits, dim=-1)
    P = torch.exp(logits - lse[..., None])
    Pl, Pw = P[..., :m], P[..., m:]
    o = torch.einsum("bhti,bhtid->bhtd", Pl, SVq) + torch.einsum("bhts,bhsd->bhtd", Pw, v)
    if return_omega:
        return o, lse, Pl.sum(-1)
    return o, lse


def final_states(k, v, log_alpha, w: int, h0k=None, h0v=None):
    """(hTk, hTv) [B,H,m,d]: the long memory after the last token that left the
    window, token T - w - 1 (the closed-form state there; h0, or zero, when no
    token has left)."""
    B, H, T, d = k.shape
    m = log_alpha.shape[-1]
    R = T - min(int(w), T)
    if R == 0:
        z = torch.zeros(B, H, m, d, dtype=k.dtype)
        return (z if h0k is None else h0k), (z if h0v is None else h0v)
    return (slot_states(k, log_alpha, h0k)[:, :, R - 1], slot_states(v, log_alpha, h0v)[:, :, R - 1])


def nha_naive_grads(q, k, v, log_alpha, dout, w: int, rope_base: float = 10000.0, h0k=None, h0v=None,
                    dhTk=None, dhTv=None):
    """Autograd gradients of sum(o * dout) (+ <hT, dhT> when dhTk, dhTv are given):
    (dq, dk, dv, dlog_alpha[, dh0k, dh0v]), float64."""
    inputs = (q, k, v, log_alpha) + ((h0k, h0v) if h0k is not None else ())
    leaves = [x.detach().clone().to(torch.float64).requires_grad_(True) for x in inputs]
    h0 = dict(h0k=leaves[4], h0v=leaves[5]) if h0k is not None else {}
    o, _ = nha_naive(*leaves[:4], w=w, rope_base=rope_base, **h0)
    loss = (o * dout.to(torch.float64)).sum()
    if dhTk is not None:
        hk, hv = final_states(leaves[1], leaves[2], leaves[3], w, **h0)
        loss = loss + (hk * dhTk.to(torch.float64)).sum() + (hv * dhTv.to(torch.float64)).sum()
    loss.backward()
    return tuple(x.grad if x.grad is not None else torch.zeros_like(x) for x in leaves)
