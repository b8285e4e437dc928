"""Pins of the oracle's optional initial slot states h0 (CPU only).

Reading: h0 = (h0k, h0v) is the long memory before token 0 (the ai.info page,
Future Directions, names learned initial slot states); the memory is then never empty, so
no slot logit is masked and queries t < w read h0 itself.  The C oracle's
forward and hand-derived backward are pinned to the unrolled closed form with
autograd, to finite differences, to the decode restatement started from h0,
and to two identities that need no formula: with w = 0 a prompt's state as h0
continues the sequence, and h0 = 0 adds m zero-logit, zero-value keys.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.decode import DecodeState, decode_step
from oracle.naive import nha_naive, nha_naive_grads


def _inputs(B, H, T, d, m, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, T, d, generator=g, dtype=torch.float64) * d ** -0.25
    k = torch.randn(B, H, T, d, generator=g, dtype=torch.float64) * d ** -0.25
    v = torch.randn(B, H, T, d, generator=g, dtype=torch.float64)
    la = torch.nn.functional.logsigmoid(torch.randn(B, H, T, m, generator=g, dtype=torch.float64) + 1.0)
    h0k = torch.randn(B, H, m, d, generator=g, dtype=torch.float64) * 0.5
    h0v = torch.randn(B, H, m, d, generator=g, dtype=torch.float64)
    dout = torch.randn(B, H, T, d, generator=g, dtype=torch.float64)
    return q, k, v, la, h0k, h0v, dout


@pytest.mark.parametrize("w", [0, 4, 17, 25])
def test_h0_forward_equals_closed_form(w):
    q, k, v, la, h0k, h0v, _ = _inputs(1, 2, 17, 8, 3, seed=40 + w)
    o, lse = oracle.forward(q, k, v, la, w, h0=(h0k, h0v))
    ro, rlse = nha_naive(q, k, v, la, w, h0k=h0k, h0v=h0v)
    assert np.abs(o - ro.numpy()).max() <= 1e-12
    assert np.abs(lse - rlse.numpy()).max() <= 1e-12


@pytest.mark.parametrize("w", [0, 3, 12, 20])
def test_h0_backward_equals_autograd(w):
    q, k, v, la, h0k, h0v, dout = _inputs(1, 2, 12, 6, 2, seed=60 + w)
    got = oracle.backward(q, k, v, la, dout, w, h0=(h0k, h0v))
    ref = nha_naive_grads(q, k, v, la, dout, w, h0k=h0k, h0v=h0v)
    assert len(got) == 6
    for name, a, b in zip(("dq", "dk", "dv", "dla", "dh0k", "dh0v"), got, ref):
        b = b.numpy()
        assert np.linalg.norm(a - b) <= 1e-10 * max(np.linalg.norm(b), 1e-30), name


def test_h0_gradient_by_finite_differences():
    q, k, v, la, h0k, h0v, dout = _inputs(1, 1, 9, 4, 2, seed=77)
    w = 3
    _, _, _, _, dh0k, dh0v = oracle.backward(q, k, v, la, dout, w, h0=(h0k, h0v))

    def loss(hk, hv):
        o, _ = oracle.forward(q, k, v, la, w, h0=(hk, hv))
        return float((o * dout.numpy()).sum())

    eps = 1e-6
    for arr, grad, which in ((h0k, dh0k, 0), (h0v, dh0v, 1)):
        for idx in [(0, 0, 0, 0), (0, 0, 1, 3), (0, 0, 0, 2)]:
            plus, minus = h0k.clone(), h0k.clone()
            plus_v, minus_v = h0v.clone(), h0v.clone()
            if which == 0:
                plus[idx] += eps
                minus[idx] -= eps
            else:
                plus_v[idx] += eps
                minus_v[idx] -= eps
            fd = (loss(plus, plus_v) - loss(minus, minus_v)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd))


def test_h0_forward_equals_the_decode_restatement():
    q, k, v, la, h0k, h0v, _ = _inputs(1, 2, 20, 8, 3, seed=90)
    w = 5
    o, _ = oracle.forward(q, k, v, la, w, h0=(h0k, h0v))
    st = DecodeState(1, 2, 8, 3, w, init=(h0k.numpy(), h0v.numpy()))
    dec = np.stack([decode_step(st, q[:, :, t].numpy(), k[:, :, t].numpy(), v[:, :, t].numpy(),
                                la[:, :, t].numpy(), t) for t in range(20)], axis=2)
    assert np.abs(o - dec).max() <= 1e-12


def test_w0_prompt_state_continues_the_sequence():
    """With w = 0 the slots read the state after token t itself; the state after a
    prompt (from the decode restatement) as h0 gives the rest of the sequence."""
    q, k, v, la, _, _, _ = _inputs(1, 2, 30, 8, 3, seed=101)
    P = 11
    o_all, lse_all = oracle.forward(q, k, v, la, 0)
    st = DecodeState(1, 2, 8, 3, 0)
    for t in range(P):
        decode_step(st, q[:, :, t].numpy(), k[:, :, t].numpy(), v[:, :, t].numpy(), la[:, :, t].numpy(), t)
    o, lse = oracle.forward(q[:, :, P:], k[:, :, P:], v[:, :, P:], la[:, :, P:], 0, h0=(st.S_k, st.S_v))
    assert np.abs(o - o_all[:, :, P:]).max() <= 1e-12
    assert np.abs(lse - lse_all[:, :, P:]).max() <= 1e-12


def test_zero_h0_adds_zero_keys_before_the_window_fills():
    q, k, v, la, h0k, h0v, _ = _inputs(1, 2, 14, 8, 3, seed=123)
    w, m = 6, 3
    o0, lse0 = oracle.forward(q, k, v, la, w)
    oz, lsez = oracle.forward(q, k, v, la, w, h0=(np.zeros_like(h0k), np.zeros_like(h0v)))
    # t >= w: the states are the same (h0 = 0 decays to 0) and no slot was masked anyway
    assert np.abs(oz[:, :, w:] - o0[:, :, w:]).max() <= 1e-12
    # t < w: m extra keys with logit 0 and value 0: Z -> Z + m, o -> o Z / (Z + m)
    Z = np.exp(lse0[:, :, :w])
    assert np.abs(lsez[:, :, :w] - np.log(Z + m)).max() <= 1e-12
    assert np.abs(oz[:, :, :w] - o0[:, :, :w] * (Z / (Z + m))[..., None]).max() <= 1e-12
