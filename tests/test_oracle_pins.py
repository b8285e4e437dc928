"""Pins for the fp64 oracle, each against something other than the oracle itself.

Source of every fact pinned here: "Native Hybrid Attention for Efficient
Sequence Modeling", Paper-Notes page -- "整体框架" (w = 0 is a pure linear
RNN, w = N is full attention; memory shapes), "关键设计/层内混合" (the
K^long_t recurrence, the single 1/sqrt(d) softmax over the concatenated
keys, omega_L, token shift, RoPE only inside the window).
"""
import math

import numpy as np
import pytest
import scipy.signal
import torch

import oracle
from oracle.naive import nha_naive, nha_naive_grads


def _rand(B, H, T, d, m, seed, mu=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, T, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, H, T, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, H, T, d, generator=g, dtype=torch.float64)
    la = torch.nn.functional.logsigmoid(torch.randn(B, H, T, m, generator=g, dtype=torch.float64) + mu)
    do = torch.randn(B, H, T, d, generator=g, dtype=torch.float64)
    return q, k, v, la, do


def _rope_polar(x, base=10000.0):
    """Textbook complex RoPE, independent of both oracles' code."""
    T, d = x.shape[-2:]
    h = d // 2
    inv = 1.0 / (base ** (torch.arange(0, d, 2, dtype=torch.float64) / d))
    ang = torch.outer(torch.arange(T, dtype=torch.float64), inv)
    z = torch.view_as_complex(torch.stack([x[..., :h], x[..., h:]], dim=-1).contiguous())
    z = z * torch.exp(1j * ang)
    r = torch.view_as_real(z)
    return torch.cat([r[..., 0], r[..., 1]], dim=-1)


# --------------------------------------------------------------------------------------
# w >= T: long memory never receives a token (all slots masked) -> causal softmax
# attention with RoPE (Paper-Notes, 关键设计/层间混合: a window as long as the
# sequence recovers full attention).  Checked against torch's SDPA.
@pytest.mark.parametrize("T,d,m,extra", [(33, 8, 3, 0), (40, 16, 4, 7), (1, 4, 2, 0)])
def test_full_window_is_causal_attention(T, d, m, extra):
    q, k, v, la, _ = _rand(2, 3, T, d, m, seed=11 + T)
    o, lse = oracle.forward(q, k, v, la, w=T + extra)
    ref = torch.nn.functional.scaled_dot_product_attention(
        _rope_polar(q), _rope_polar(k), v, is_causal=True)
    assert np.abs(o - ref.numpy()).max() <= 1e-12


# --------------------------------------------------------------------------------------
# w = 0: a pure gated-slot linear RNN read by a softmax over the m slots
# (Paper-Notes, 关键设计/层间混合: an empty window leaves a linear RNN).  With per-slot
# gates that are constant in time, each
# slot state is a first-order IIR filter of the key/value stream, which
# scipy.signal.lfilter computes: y_t = alpha y_{t-1} + (1 - alpha) x_t.
def test_zero_window_is_slot_rnn_attention():
    B, H, T, d, m = 1, 2, 29, 8, 5
    q, k, v, _, _ = _rand(B, H, T, d, m, seed=5)
    alpha = np.array([0.3, 0.9, 0.99, 0.5, 0.05])
    la = torch.tensor(np.log(alpha)).expand(B, H, T, m).contiguous()
    o, _ = oracle.forward(q, k, v, la, w=0)
    kk, vv, qq = k.numpy(), v.numpy(), q.numpy()
    ref = np.zeros_like(o)
    for b in range(B):
        for h in range(H):
            SK = np.stack([scipy.signal.lfilter([1 - a], [1, -a], kk[b, h], axis=0) for a in alpha], 1)
            SV = np.stack([scipy.signal.lfilter([1 - a], [1, -a], vv[b, h], axis=0) for a in alpha], 1)
            logits = np.einsum("td,tid->ti", qq[b, h], SK) / math.sqrt(d)
            p = torch.softmax(torch.tensor(logits), dim=-1).numpy()
            ref[b, h] = np.einsum("ti,tid->td", p, SV)
    assert np.abs(o - ref).max() <= 1e-12


# --------------------------------------------------------------------------------------
# w = 0, m = 1: the softmax over one slot is identically 1, so o_t is the
# gated moving average of v, independent of q and k; dq = dk = 0 exactly.
def test_single_slot_is_ema_and_ignores_qk():
    B, H, T, d, m = 1, 1, 37, 6, 1
    q, k, v, _, do = _rand(B, H, T, d, m, seed=9)
    a = 0.8
    la = torch.full((B, H, T, m), math.log(a), dtype=torch.float64)
    o, _ = oracle.forward(q, k, v, la, w=0)
    ema = scipy.signal.lfilter([1 - a], [1, -a], v.numpy()[0, 0], axis=0)
    assert np.abs(o[0, 0] - ema).max() <= 1e-12
    # time-varying gates: still independent of q and k
    _, _, _, la2, _ = _rand(B, H, T, d, m, seed=10)
    o1, _ = oracle.forward(q, k, v, la2, w=0)
    o2, _ = oracle.forward(q * 3 + 1, -k, v, la2, w=0)
    assert np.array_equal(o1, o2)
    dq, dk, dv, dla = oracle.backward(q, k, v, la2, do, w=0)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    assert np.abs(dv).max() > 0 and np.abs(dla).max() > 0


# --------------------------------------------------------------------------------------
# log_alpha = -40 (alpha ~ 0, 1 - alpha = 1): every slot holds exactly the
# token that left the window last (token t - w), un-rotated.  NHA is then one
# softmax over the window plus m equal copies of that token's logit, i.e. one
# extra key t - w with logit + log(m).  Pins the token-shift placement and the
# absence of position encoding on the slots.
@pytest.mark.parametrize("w", [1, 3, 7])
def test_forgetful_slots_hold_the_last_evicted_token(w):
    B, H, T, d, m = 1, 2, 23, 8, 4
    q, k, v, _, _ = _rand(B, H, T, d, m, seed=20 + w)
    la = torch.full((B, H, T, m), -40.0, dtype=torch.float64)
    o, _ = oracle.forward(q, k, v, la, w=w)
    qr, kr = _rope_polar(q), _rope_polar(k)
    t = torch.arange(T)
    S = torch.einsum("bhtd,bhsd->bhts", qr, kr) / math.sqrt(d)
    band = (t[None, :] <= t[:, None]) & (t[None, :] > t[:, None] - w)
    S = S.masked_fill(~band, -math.inf)
    j = (t - w).clamp(min=0)
    ext = torch.einsum("bhtd,bhtd->bht", q, k[:, :, j]) / math.sqrt(d) + math.log(m)
    ext = torch.where(t >= w, ext, torch.full_like(ext, -math.inf))
    P = torch.softmax(torch.cat([S, ext[..., None]], -1), -1)
    ref = P[..., :T] @ v + P[..., T:] * v[:, :, j]
    assert np.abs(o - ref.numpy()).max() <= 1e-10


# --------------------------------------------------------------------------------------
# log_alpha = -1e-12 (alpha ~ 1, 1 - alpha ~ 1e-12): the slots hold ~0 keys and
# values but are NOT masked once a token has been absorbed (t >= w).  Each slot
# adds exp(~0) = 1 to the partition and ~0 to the output:
#   o_t = o_SWA,t * Z_w / (Z_w + m)  for t >= w,   o_t = o_SWA,t  for t < w,
# with Z_w the window partition.  Pins that the mask is positional, not value
# based.  o_SWA comes from torch's SDPA with a band mask.
def test_near_unit_gates_keep_slots_unmasked():
    B, H, T, d, m, w = 1, 2, 30, 8, 6, 4
    q, k, v, _, _ = _rand(B, H, T, d, m, seed=31)
    la = torch.full((B, H, T, m), -1e-12, dtype=torch.float64)
    o, lse = oracle.forward(q, k, v, la, w=w)
    qr, kr = _rope_polar(q), _rope_polar(k)
    t = torch.arange(T)
    band = (t[None, :] <= t[:, None]) & (t[None, :] > t[:, None] - w)
    o_swa = torch.nn.functional.scaled_dot_product_attention(qr, kr, v, attn_mask=band)
    S = (torch.einsum("bhtd,bhsd->bhts", qr, kr) / math.sqrt(d)).masked_fill(~band, -math.inf)
    Zw = torch.exp(torch.logsumexp(S, -1))
    scale = torch.where(t >= w, Zw / (Zw + m), torch.ones_like(Zw))
    ref = o_swa * scale[..., None]
    assert np.abs(o - ref.numpy()).max() <= 1e-9
    ref_lse = torch.where(t >= w, torch.log(Zw + m), torch.log(Zw))
    assert np.abs(lse - ref_lse.numpy()).max() <= 1e-9


# --------------------------------------------------------------------------------------
# A worked example small enough to do by hand (d = 2, so theta_0 = 1 rad per
# position; m = 1; w = 2; T = 3; alpha = 1/2 for the absorbed token).
#   t=0: window {0}: o_0 = v_0.
#   t=1: window {0,1}: logits s_{1,0} = (R_1 q_1).(R_0 k_0)/sqrt2, s_{1,1} = q_1.k_1/sqrt2.
#   t=2: token 0 leaves the window: K^long = (1-1/2) k_0, V^long = (1-1/2) v_0;
#        slot logit q_2.K^long/sqrt2, window {1,2}.
def test_hand_worked_example():
    r2 = math.sqrt(2.0)

    def rot(x, a):
        return (x[0] * math.cos(a) - x[1] * math.sin(a), x[1] * math.cos(a) + x[0] * math.sin(a))

    def dotp(a, b):
        return a[0] * b[0] + a[1] * b[1]

    qs = [(1.0, 0.0), (0.0, 1.0), (0.5, -1.0)]
    ks = [(1.0, 0.0), (0.0, 1.0), (1.0, 1.0)]
    vs = [(2.0, 0.0), (0.0, 4.0), (-1.0, 1.0)]
    la0 = math.log(0.5)
    # t = 1
    s10 = dotp(rot(qs[1], 1.0), rot(ks[0], 0.0)) / r2  # = (R_1 q_1).k_0 / sqrt2 = -sin(1)/sqrt2
    s11 = dotp(qs[1], ks[1]) / r2
    z1 = math.exp(s10) + math.exp(s11)
    o1 = [(math.exp(s10) * vs[0][c] + math.exp(s11) * vs[1][c]) / z1 for c in range(2)]
    # t = 2
    Kl = (0.5 * ks[0][0], 0.5 * ks[0][1])
    Vl = (0.5 * vs[0][0], 0.5 * vs[0][1])
    l2 = dotp(qs[2], Kl) / r2
    s21 = dotp(rot(qs[2], 2.0), rot(ks[1], 1.0)) / r2
    s22 = dotp(qs[2], ks[2]) / r2
    e = [math.exp(l2), math.exp(s21), math.exp(s22)]
    z2 = sum(e)
    o2 = [(e[0] * Vl[c] + e[1] * vs[1][c] + e[2] * vs[2][c]) / z2 for c in range(2)]
    expect_o = np.array([vs[0], o1, o2])
    expect_lse = np.array([dotp(qs[0], ks[0]) / r2, math.log(z1), math.log(z2)])
    q = torch.tensor(qs, dtype=torch.float64)[None, None]
    k = torch.tensor(ks, dtype=torch.float64)[None, None]
    v = torch.tensor(vs, dtype=torch.float64)[None, None]
    la = torch.tensor([[la0], [-0.3], [-0.2]], dtype=torch.float64)[None, None]
    o, lse = oracle.forward(q, k, v, la, w=2)
    assert np.abs(o[0, 0] - expect_o).max() <= 1e-14
    assert np.abs(lse[0, 0] - expect_lse).max() <= 1e-14
    assert abs(s10 + math.sin(1.0) / r2) < 1e-15  # the RoPE term really is relative


# --------------------------------------------------------------------------------------
# Recurrence (C oracle) == unrolled closed form (naive.py), forward and omega_L.
@pytest.mark.parametrize("T,d,m,w", [(1, 4, 1, 0), (17, 8, 3, 3), (33, 8, 2, 5), (40, 16, 4, 40),
                                     (24, 8, 3, 0), (64, 8, 3, 13)])
def test_recurrence_equals_unrolled_formula(T, d, m, w):
    q, k, v, la, _ = _rand(2, 2, T, d, m, seed=T * 7 + w)
    o, lse, om = oracle.forward(q, k, v, la, w=w, with_omega=True)
    on, lsen, omn = nha_naive(q, k, v, la, w=w, return_omega=True)
    assert np.abs(o - on.numpy()).max() <= 1e-12
    assert np.abs(lse - lsen.numpy()).max() <= 1e-12
    assert np.abs(om - omn.numpy()).max() <= 1e-12


# --------------------------------------------------------------------------------------
# Hand-derived reverse sweep == autograd of the unrolled formula == central
# finite differences of the oracle's own forward.
GRAD_CASES = [(T, d, m, w) for T in (1, 5, 17) for d in (4, 8) for m in (1, 3)
              for w in (0, 1, 3, T)]


@pytest.mark.parametrize("T,d,m,w", GRAD_CASES)
def test_backward_matches_autograd(T, d, m, w):
    q, k, v, la, do = _rand(1, 1, T, d, m, seed=100 + T + 3 * d + 5 * m + 7 * w)
    got = oracle.backward(q, k, v, la, do, w=w)
    ref = nha_naive_grads(q, k, v, la, do, w=w)
    for a, b in zip(got, ref):
        assert np.abs(a - b.numpy()).max() <= 1e-10 * max(1.0, np.abs(b.numpy()).max())


@pytest.mark.parametrize("T,d,m,w", [(5, 4, 3, 1), (17, 8, 3, 3), (17, 4, 1, 0), (5, 8, 3, 5)])
def test_backward_matches_finite_differences(T, d, m, w):
    q, k, v, la, do = _rand(1, 1, T, d, m, seed=200 + T + w)
    grads = oracle.backward(q, k, v, la, do, w=w)
    inputs = [q.numpy().copy(), k.numpy().copy(), v.numpy().copy(), la.numpy().copy()]
    rng = np.random.default_rng(0)
    h = 1e-6

    def loss(xs):
        o, _ = oracle.forward(*xs, w=w)
        return float((o * do.numpy()).sum())

    for which in range(4):
        flat = inputs[which].reshape(-1)
        for idx in rng.choice(flat.size, size=min(8, flat.size), replace=False):
            old = flat[idx]
            flat[idx] = old + h
            lp = loss(inputs)
            flat[idx] = old - h
            lm = loss(inputs)
            flat[idx] = old
            fd = (lp - lm) / (2 * h)
            an = grads[which].reshape(-1)[idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (which, idx, fd, an)


# --------------------------------------------------------------------------------------
# Invariants of the single softmax (convexity, positional mask, causality,
# token shift, head independence).
def test_convexity_and_long_memory_share():
    q, k, v, la, _ = _rand(2, 3, 50, 8, 4, seed=3)
    for w in (0, 1, 6, 50):
        o, _, om = oracle.forward(q, k, v, la, w=w, with_omega=True)
        vmax = np.abs(v.numpy()).max(axis=2, keepdims=True)  # per (b,h,feature)
        assert np.all(np.abs(o) <= vmax + 1e-12)
        assert np.all(om >= 0) and np.all(om <= 1 + 1e-15)
        assert np.all(om[..., : min(w, 50)] == 0.0)  # slots masked while t < w
        if w == 0:
            assert np.abs(om - 1).max() <= 1e-15


def test_causality_and_token_shift():
    T, w = 40, 6
    q, k, v, la, _ = _rand(1, 1, T, 8, 3, seed=4)
    o0, _ = oracle.forward(q, k, v, la, w=w)
    s = 17
    # perturbing every input of token s leaves o_t for t < s bit-identical
    q2, k2, v2, la2 = (x.clone() for x in (q, k, v, la))
    q2[..., s, :] += 1.0; k2[..., s, :] -= 0.5; v2[..., s, :] += 2.0; la2[..., s, :] -= 0.7
    o1, _ = oracle.forward(q2, k2, v2, la2, w=w)
    assert np.array_equal(o1[..., :s, :], o0[..., :s, :])
    assert np.abs(o1[..., s, :] - o0[..., s, :]).max() > 1e-6
    # the gate of token s enters the long memory only when token s leaves the
    # window, i.e. it first affects query t = s + w
    la3 = la.clone(); la3[..., s, :] -= 0.7
    o3, _ = oracle.forward(q, k, v, la3, w=w)
    assert np.array_equal(o3[..., : s + w, :], o0[..., : s + w, :])
    assert np.abs(o3[..., s + w, :] - o0[..., s + w, :]).max() > 1e-9


def test_heads_are_independent():
    q, k, v, la, _ = _rand(2, 3, 21, 8, 3, seed=8)
    o, lse = oracle.forward(q, k, v, la, w=5)
    perm = [2, 0, 1]
    op, lsep = oracle.forward(q[:, perm], k[:, perm], v[:, perm], la[:, perm], w=5)
    assert np.array_equal(op, o[:, perm]) and np.array_equal(lsep, lse[:, perm])
