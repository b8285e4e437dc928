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


# ------------------------------------------------------------------------------------------
# Final states hT (the long memory after token T - w - 1) and their gradient dhT.
@pytest.mark.parametrize("w,with_h0", [(0, False), (4, True), (7, False), (17, True), (30, True)])
def test_final_states_equal_the_decode_restatement_and_closed_form(w, with_h0):
    from oracle.naive import final_states

    T = 17
    q, k, v, la, h0k, h0v, _ = _inputs(1, 2, T, 8, 3, seed=200 + w)
    h0 = (h0k, h0v) if with_h0 else None
    _, _, hTk, hTv = oracle.forward(q, k, v, la, w, h0=h0, return_state=True)
    # the decode restatement, run over every token, holds the same long memory
    st = DecodeState(1, 2, 8, 3, w, init=(h0k.numpy(), h0v.numpy()) if with_h0 else None)
    for t in range(T):
        decode_step(st, q[:, :, t].numpy(), k[:, :, t].numpy(), v[:, :, t].numpy(), la[:, :, t].numpy(), t)
    assert np.abs(hTk - st.S_k).max() <= 1e-12 and np.abs(hTv - st.S_v).max() <= 1e-12
    rk, rv = final_states(k, v, la, w, h0k=h0k if with_h0 else None, h0v=h0v if with_h0 else None)
    assert np.abs(hTk - rk.numpy()).max() <= 1e-12 and np.abs(hTv - rv.numpy()).max() <= 1e-12


@pytest.mark.parametrize("w,with_h0", [(0, False), (3, True), (5, False), (12, True), (20, True)])
def test_final_state_gradient_equals_autograd(w, with_h0):
    q, k, v, la, h0k, h0v, dout = _inputs(1, 2, 12, 6, 2, seed=300 + w)
    g = torch.Generator().manual_seed(301 + w)
    dhk = torch.randn(1, 2, 2, 6, generator=g, dtype=torch.float64)
    dhv = torch.randn(1, 2, 2, 6, generator=g, dtype=torch.float64)
    h0 = (h0k, h0v) if with_h0 else None
    got = oracle.backward(q, k, v, la, dout, w, h0=h0, dhT=(dhk, dhv))
    kw = dict(h0k=h0k, h0v=h0v) if with_h0 else {}
    ref = nha_naive_grads(q, k, v, la, dout, w, dhTk=dhk, dhTv=dhv, **kw)
    assert len(got) == len(ref)
    for name, a, b in zip(("dq", "dk", "dv", "dla", "dh0k", "dh0v"), got, ref):
        b = b.numpy()
        assert np.linalg.norm(a - b) <= 1e-10 * max(np.linalg.norm(b), 1e-30), name


def test_final_state_gradient_by_finite_differences():
    q, k, v, la, h0k, h0v, dout = _inputs(1, 1, 11, 4, 2, seed=401)
    w = 3
    g = torch.Generator().manual_seed(402)
    dhk = torch.randn(1, 1, 2, 4, generator=g, dtype=torch.float64).numpy()
    dhv = torch.randn(1, 1, 2, 4, generator=g, dtype=torch.float64).numpy()
    _, dk, _, dla, dh0k, _ = oracle.backward(q, k, v, la, dout, w, h0=(h0k, h0v), dhT=(dhk, dhv))

    def loss(kk, ll, hk):
        o, _, tk, tv = oracle.forward(q, kk, v, ll, w, h0=(hk, h0v), return_state=True)
        return float((o * dout.numpy()).sum() + (tk * dhk).sum() + (tv * dhv).sum())

    eps = 1e-6
    for idx in [(0, 0, 2, 1), (0, 0, 7, 0)]:  # a key that leaves the window, one still in it
        kp, km = k.clone(), k.clone()
        kp[idx] += eps
        km[idx] -= eps
        fd = (loss(kp, la, h0k) - loss(km, la, h0k)) / (2 * eps)
        assert abs(fd - dk[idx]) <= 1e-6 * max(1.0, abs(fd))
    for idx in [(0, 0, 1, 0), (0, 0, 6, 1)]:
        lp, lm = la.clone(), la.clone()
        lp[idx] += eps
        lm[idx] -= eps
        fd = (loss(k, lp, h0k) - loss(k, lm, h0k)) / (2 * eps)
        assert abs(fd - dla[idx]) <= 1e-6 * max(1.0, abs(fd))
    for idx in [(0, 0, 0, 0), (0, 0, 1, 3)]:
        hp, hm = h0k.clone(), h0k.clone()
        hp[idx] += eps
        hm[idx] -= eps
        fd = (loss(k, la, hp) - loss(k, la, hm)) / (2 * eps)
        assert abs(fd - dh0k[idx]) <= 1e-6 * max(1.0, abs(fd))


def test_segments_chained_through_final_states_reproduce_the_sequence():
    """A sequence cut into segments: each later segment runs on [the previous w
    tokens; its own tokens] from the previous segment's final state (the long
    memory after the token that left the window before the segment's halo;
    the halo's own queries read it and are dropped); the segment outputs after
    the halo are the full sequence's, and the last segment's final state is
    the full sequence's."""
    T, w = 40, 6
    q, k, v, la, _, _, _ = _inputs(1, 2, T, 8, 3, seed=501)
    o_all, lse_all, hk_all, hv_all = oracle.forward(q, k, v, la, w, return_state=True)
    # RoPE window logits depend on t - s only, so each segment may use its own positions
    cuts = [0, 13, 13 + 15, T]
    state = None  # the first segment starts the sequence: no initial state, slots masked
    for a, b in zip(cuts[:-1], cuts[1:]):
        lo = max(0, a - w)
        sl = slice(lo, b)
        o, lse, hk, hv = oracle.forward(q[:, :, sl], k[:, :, sl], v[:, :, sl], la[:, :, sl], w, h0=state,
                                        return_state=True)
        keep = a - lo
        assert np.abs(o[:, :, keep:] - o_all[:, :, a:b]).max() <= 1e-10
        assert np.abs(lse[:, :, keep:] - lse_all[:, :, a:b]).max() <= 1e-10
        state = (hk, hv)
    assert np.abs(state[0] - hk_all).max() <= 1e-12 and np.abs(state[1] - hv_all).max() <= 1e-12
