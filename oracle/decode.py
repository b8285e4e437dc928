"""One recurrent NHA decode step in fp64 numpy.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): only ``tests/`` and
``bench.py``'s reference leg may import it.

The step is the token-by-token definition of the operator ("Native Hybrid
Attention for Efficient Sequence Modeling", Paper-Notes page, section
关键设计/层内混合: the K^long recurrence, the token shift that hands a token to
the long memory once it leaves the w-token window, window-only RoPE, one
softmax over the m slots and the window) taken for a single new token t:

1. if t >= w, token j = t - w leaves the window and is absorbed with its own
   gate: S^K = diag(alpha_j) S^K + u_j (x) k_j, S^V likewise (u = -expm1(log_alpha));
   the slot logits are L_i = q_t . S^K[i] / sqrt(d) (all masked while t < w);
2. the window keys are the tokens s in [max(0, t - w + 1), t], with logits
   RoPE(q_t, t) . RoPE(k_s, s) / sqrt(d) (rotate-half, theta_i = base^(-2i/d));
3. p = softmax over [L | window]; o_t = sum_i p_i S^V[i] + sum_s p_s v_s.

Between steps the caller keeps the slot states and a ring of the last w tokens
(raw k, v and log_alpha; token s in entry s mod w).  Everything is float64.

A state may start from initial slot states h0 (``DecodeState(..., init=(h0k, h0v))``):
the long memory before token 0 is then h0, and since it is never empty the
slot logits are not masked while t < w (those queries read h0 itself).
"""
from __future__ import annotations

import math

import numpy as np


def rope(x: np.ndarray, pos: int, base: float) -> np.ndarray:
    """Rotate-half RoPE of x [..., d] at absolute position pos."""
    d = x.shape[-1]
    h = d // 2
    theta = base ** (-2.0 * np.arange(h) / d)
    ang = pos * theta
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


class DecodeState:
    """Slot states S^K, S^V [B, H, m, d] and the window ring [B, H, w, .] of one layer."""

    def __init__(self, B: int, H: int, d: int, m: int, w: int, init=None):
        self.w = w
        self.S_k = np.zeros((B, H, m, d))
        self.S_v = np.zeros((B, H, m, d))
        self.has_init = init is not None
        if init is not None:
            self.S_k = np.array(init[0], dtype=np.float64).reshape(B, H, m, d)
            self.S_v = np.array(init[1], dtype=np.float64).reshape(B, H, m, d)
        n = max(w, 1)
        self.ring_k = np.zeros((B, H, n, d))
        self.ring_v = np.zeros((B, H, n, d))
        self.ring_la = np.zeros((B, H, n, m))


def decode_step(st: DecodeState, q, k, v, log_alpha, t: int, base: float = 10000.0):
    """o_t [B, H, d] for token t (q, k, v [B, H, d]; log_alpha [B, H, m]); updates st."""
    q, k, v, la = (np.asarray(a, dtype=np.float64) for a in (q, k, v, log_alpha))
    w = st.w
    d = q.shape[-1]
    scale = 1.0 / math.sqrt(d)
    # 1. the token that leaves the window enters the long memory (its own gate)
    if t - w >= 0:
        if w == 0:
            kj, vj, lj = k, v, la
        else:
            e = (t - w) % w
            kj, vj, lj = st.ring_k[:, :, e], st.ring_v[:, :, e], st.ring_la[:, :, e]
        alpha, u = np.exp(lj), -np.expm1(lj)
        st.S_k = alpha[..., None] * st.S_k + u[..., None] * kj[:, :, None, :]
        st.S_v = alpha[..., None] * st.S_v + u[..., None] * vj[:, :, None, :]
    slots = t - w >= 0 or st.has_init
    if slots:
        L = np.einsum("bhd,bhmd->bhm", q, st.S_k) * scale
    else:
        L = np.full(q.shape[:2] + (st.S_k.shape[2],), -np.inf)
    # 2. window logits over tokens max(0, t - w + 1) .. t
    qr = rope(q, t, base)
    keys, vals = [], []
    for s in range(max(0, t - w + 1), t + 1):
        if s == t:
            ks, vs = k, v
        else:
            ks, vs = st.ring_k[:, :, s % w], st.ring_v[:, :, s % w]
        keys.append(np.einsum("bhd,bhd->bh", qr, rope(ks, s, base)) * scale)
        vals.append(vs)
    logits = np.concatenate([L] + [kk[..., None] for kk in keys], axis=-1)
    # 3. one softmax over slots and window
    mx = logits.max(axis=-1, keepdims=True)
    p = np.exp(logits - mx)
    p /= p.sum(axis=-1, keepdims=True)
    m = L.shape[-1]
    o = np.einsum("bhm,bhmd->bhd", p[..., :m], st.S_v) if slots else np.zeros_like(q)
    for n, vs in enumerate(vals):
        o = o + p[..., m + n, None] * vs
    # the ring keeps the last w tokens (token t takes the entry of the token that left)
    if w > 0:
        e = t % w
        st.ring_k[:, :, e], st.ring_v[:, :, e], st.ring_la[:, :, e] = k, v, la
    return o
