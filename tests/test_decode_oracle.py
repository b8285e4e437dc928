"""Pins of the decode-step oracle (``oracle/decode.py``), CPU only.

The decode step restates the operator for one new token; run over t = 0..T-1
from empty states it must reproduce, to fp64 rounding, the full-sequence
forward of the C oracle (an independent token-by-token program with its own
RoPE and softmax code), and its slot states must equal the unrolled sum
S_J = sum_{s <= J} (prod_{r = s+1}^{J} alpha_r) u_s k_s of the recurrence.
"""
import numpy as np
import pytest

import oracle
from oracle.decode import DecodeState, decode_step


def _inputs(B, H, T, d, m, seed):
    g = np.random.default_rng(seed)
    q = g.standard_normal((B, H, T, d)) * d ** -0.25
    k = g.standard_normal((B, H, T, d)) * d ** -0.25
    v = g.standard_normal((B, H, T, d))
    la = np.log(1.0 / (1.0 + np.exp(-(g.standard_normal((B, H, T, m)) + 2.0))))  # logsigmoid(N(2, 1))
    return q, k, v, la


def _run_decode(q, k, v, la, w):
    B, H, T, d = q.shape
    st = DecodeState(B, H, d, la.shape[-1], w)
    o = np.stack([decode_step(st, q[:, :, t], k[:, :, t], v[:, :, t], la[:, :, t], t) for t in range(T)], axis=2)
    return o, st


@pytest.mark.parametrize("B,H,T,d,m,w", [
    (1, 2, 37, 8, 3, 5),    # ragged T, small window
    (2, 1, 20, 8, 2, 0),    # w = 0: slots only
    (1, 1, 15, 4, 1, 1),    # w = 1: the window is the token itself
    (1, 2, 12, 8, 4, 30),   # w > T: window attention only
    (1, 1, 64, 16, 4, 17),  # several ring wraps
])
def test_decode_steps_equal_the_full_forward(B, H, T, d, m, w):
    q, k, v, la = _inputs(B, H, T, d, m, seed=T * 7 + w)
    o_dec, _ = _run_decode(q, k, v, la, w)
    o_ref, _ = oracle.forward(q, k, v, la, w)
    assert np.max(np.abs(o_dec - o_ref)) < 1e-12


@pytest.mark.parametrize("w", [0, 3, 9])
def test_decode_states_are_the_unrolled_sum(w):
    B, H, T, d, m = 1, 2, 25, 6, 3
    q, k, v, la = _inputs(B, H, T, d, m, seed=100 + w)
    _, st = _run_decode(q, k, v, la, w)
    J = T - 1 - w  # last token absorbed by the long memory
    ref_k = np.zeros((B, H, m, d))
    ref_v = np.zeros((B, H, m, d))
    for s in range(J + 1):
        decay = np.exp(la[:, :, s + 1:J + 1].sum(axis=2))  # prod_{r = s+1}^{J} alpha_r
        u = -np.expm1(la[:, :, s])
        ref_k += (decay * u)[..., None] * k[:, :, s, None, :]
        ref_v += (decay * u)[..., None] * v[:, :, s, None, :]
    assert np.max(np.abs(st.S_k - ref_k)) < 1e-12
    assert np.max(np.abs(st.S_v - ref_v)) < 1e-12
