"""GPU parity: the CUDA library through the C ABI vs the fp64 oracle, on the
same seeded inputs (bf16 inputs are upcast exactly for the oracle).

Tolerances (on every element compared):
  fp32 inputs:  max |err| <= 1e-4 on o and every gradient (lse: 1e-4);
  bf16 inputs:  o: rel L2 <= 5e-3 and max |err| <= 2e-2;  lse: max |err| <= 2e-2;
                gradients (dq, dk, dv, dlog_alpha): rel L2 <= 1e-2.
Small cases compare every output; full-size workloads (in the launch
configuration the bench times) compare whole sampled heads.
"""
import numpy as np
import pytest
import torch

import oracle
from sliding_window_softmax_gb300.synthetic import (GRID_M, GRID_W, LAYER_1P3B, LAYER_340M,
                                                    LONG_CONTEXT_T, TINY_F32, Workload, grid_point,
                                                    long_context, make_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()


def _nha():
    import sliding_window_softmax_gb300 as nha

    return nha


def run_gpu(x, w, backward=True):
    nha = _nha()
    d = {n: t.cuda() for n, t in x.items()}
    o, lse = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=w)
    out = dict(o=o, lse=lse)
    if backward:
        dq, dk, dv, dla = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o, lse,
                                           d["dout"], w=w)
        out.update(dq=dq, dk=dk, dv=dv, dlog_alpha=dla)
    torch.cuda.synchronize()
    return {n: t.double().cpu().numpy() for n, t in out.items()}


def run_oracle(x, w, backward=True, heads=None):
    """Oracle outputs; ``heads`` = list of (b, h) to restrict to (returns [len(heads), T, ...])."""
    sel = dict(x)
    if heads is not None:
        sel = {n: torch.stack([t[b, h] for b, h in heads])[None] for n, t in x.items()}
    o, lse = oracle.forward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], w)
    out = dict(o=o, lse=lse)
    if backward:
        dq, dk, dv, dla = oracle.backward(sel["q"], sel["k"], sel["v"], sel["log_alpha"],
                                          sel["dout"], w)
        out.update(dq=dq, dk=dk, dv=dv, dlog_alpha=dla)
    if heads is not None:
        out = {n: a[0] for n, a in out.items()}
    return out


def pick(gpu, heads):
    return {n: np.stack([a[b, h] for b, h in heads]) for n, a in gpu.items()}


def assert_parity(gpu, ref, dtype, tag=""):
    for n in ref:
        g, r = gpu[n], ref[n]
        assert g.shape == r.shape, (n, g.shape, r.shape)
        assert np.all(np.isfinite(g)), f"{tag} {n}: non-finite values"
        err = np.abs(g - r)
        rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
        if dtype == "f32":
            assert err.max() <= 1e-4, f"{tag} {n}: max abs {err.max():.3e} > 1e-4"
        elif n == "o":
            assert rel <= 5e-3 and err.max() <= 2e-2, f"{tag} o: rel {rel:.3e} max {err.max():.3e}"
        elif n == "lse":
            # lse has no stated bound; the window logits come from bf16-rounded
            # RoPE(q), RoPE(k), whose error (~2^-8 |logit|) reaches lse directly.
            assert err.max() <= 2e-2, f"{tag} lse: max {err.max():.3e}"
        else:
            assert rel <= 1e-2, f"{tag} {n}: rel L2 {rel:.3e} > 1e-2"


# ------------------------------------------------------------------------------------------
# Small cases: several tiles and a ragged tail, every output compared.
SMALL = [
    # (B, H, T, d, m, w, dtype)
    (1, 2, 256, 64, 16, 32, "f32"),     # the tiny fp32 workload's shape
    (1, 2, 300, 64, 16, 32, "f32"),     # ragged T
    (2, 1, 333, 64, 32, 100, "f32"),    # w not a multiple of C, ragged T
    (1, 2, 200, 128, 64, 0, "f32"),     # w = 0: pure slot RNN
    (1, 1, 190, 64, 16, 190, "f32"),    # w = T: causal attention
    (1, 1, 150, 64, 16, 1000, "f32"),   # w > T
    (1, 1, 1, 64, 16, 0, "f32"),        # T = 1, slots only
    (1, 1, 1, 128, 64, 5, "f32"),       # T = 1, window only
    (1, 1, 64, 64, 16, 64, "f32"),      # exactly one tile, no slots
    (1, 2, 129, 64, 16, 1, "f32"),      # w = 1: window holds only the token itself
    (1, 2, 333, 128, 64, 70, "bf16"),
    (2, 2, 257, 64, 32, 64, "bf16"),
    (1, 2, 400, 128, 16, 0, "bf16"),
]


@pytest.mark.parametrize("B,H,T,d,m,w,dt", SMALL)
def test_small_parity(B, H, T, d, m, w, dt):
    wl = Workload(f"small {B} {H} {T} {d} {m} {w}", B, H, T, d, m, w, dtype=dt,
                  seed=4000 + T + d + m + w)
    x = make_inputs(wl)
    assert_parity(run_gpu(x, w), run_oracle(x, w), dt, tag=wl.name)


def test_sharp_softmax_variant():
    """q, k scaled by 4: a peaked softmax (the workloads' own is near uniform)."""
    wl = Workload("sharp", 1, 2, 320, 128, 64, 96, dtype="f32", seed=77)
    x = make_inputs(wl, scale_qk=4.0)
    assert_parity(run_gpu(x, 96), run_oracle(x, 96), "f32", tag="sharp f32")
    wl = wl.with_(dtype="bf16")
    x = make_inputs(wl, scale_qk=4.0)
    assert_parity(run_gpu(x, 96), run_oracle(x, 96), "bf16", tag="sharp bf16")


def test_chunking_invariance_of_head_layout():
    """Heads are independent: the same head gives the same result in any batch slot."""
    wl = Workload("perm", 2, 3, 200, 64, 16, 40, dtype="f32", seed=5)
    x = make_inputs(wl)
    a = run_gpu(x, 40)
    perm = [2, 0, 1]
    xp = {n: t[:, perm].contiguous() for n, t in x.items()}
    b = run_gpu(xp, 40)
    for n in a:
        assert np.array_equal(a[n][:, perm], b[n])


def test_repeated_calls_are_deterministic():
    wl = Workload("det", 1, 2, 300, 128, 64, 70, dtype="bf16", seed=6)
    x = make_inputs(wl)
    a, b = run_gpu(x, 70), run_gpu(x, 70)
    for n in a:
        assert np.array_equal(a[n], b[n]), n


def test_two_streams_match_serial_calls():
    """Forward and backward of two problems enqueued on two user streams with no
    synchronisation between them (the library's side stream and events are
    shared by both) give bit-identical results to serial calls."""
    nha = _nha()
    wls = [Workload("s1", 1, 2, 300, 128, 64, 70, dtype="bf16", seed=11),
           Workload("s2", 2, 1, 257, 64, 32, 33, dtype="bf16", seed=12)]
    xs = [make_inputs(wl) for wl in wls]
    serial = [run_gpu(x, wl.w) for x, wl in zip(xs, wls)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    ds = [{n: t.cuda() for n, t in x.items()} for x in xs]
    torch.cuda.synchronize()
    for d, wl, st in zip(ds, wls, streams):
        with torch.cuda.stream(st):
            o, lse = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=wl.w, stream=st)
            g = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o, lse, d["dout"], w=wl.w,
                                 stream=st)
            outs.append(dict(o=o, lse=lse, dq=g[0], dk=g[1], dv=g[2], dlog_alpha=g[3]))
    torch.cuda.synchronize()
    for got, ref in zip(outs, serial):
        for n, t in got.items():
            assert np.array_equal(t.double().cpu().numpy(), ref[n]), n


# ------------------------------------------------------------------------------------------
# The specified workloads at full size; sampled heads compared with the oracle.
def test_tiny_f32_workload():
    x = make_inputs(TINY_F32)
    assert_parity(run_gpu(x, TINY_F32.w), run_oracle(x, TINY_F32.w), "f32", tag=TINY_F32.name)


@pytest.mark.parametrize("wl", [LAYER_340M, LAYER_1P3B,
                                LAYER_1P3B.with_(name="1.3B w=0", w=0),
                                LAYER_1P3B.with_(name="1.3B w=T", w=2048)],
                         ids=lambda w: w.name)
def test_layer_workloads(wl):
    x = make_inputs(wl)
    gpu = run_gpu(x, wl.w)
    heads = [(0, 0), (wl.B - 1, wl.H - 1)]
    assert_parity(pick(gpu, heads), run_oracle(x, wl.w, heads=heads), wl.dtype, tag=wl.name)


@pytest.mark.parametrize("T", LONG_CONTEXT_T)
def test_long_context_forward(T):
    wl = long_context(T)
    x = make_inputs(wl)
    gpu = run_gpu(x, wl.w, backward=False)
    heads = [(0, 31)]
    assert_parity(pick(gpu, heads), run_oracle(x, wl.w, backward=False, heads=heads), "bf16",
                  tag=wl.name)


@pytest.mark.parametrize("w", GRID_W)
@pytest.mark.parametrize("m", GRID_M)
def test_window_slot_grid(w, m):
    """Forward and backward at every grid point; one whole head (at w = 8192 the
    oracle's backward of one head is a full causal attention over 8192 tokens)."""
    wl = grid_point(w, m)
    x = make_inputs(wl)
    gpu = run_gpu(x, wl.w)
    heads = [(1, 15)]
    ref = run_oracle(x, wl.w, heads=heads)
    assert_parity(pick(gpu, heads), ref, "bf16", tag=wl.name)


def test_layer_1p3b_every_head():
    """The 1.3B-like layer (B4 H16 T2048 d128 m64 w512, bf16): all 64 heads,
    forward and backward, element by element."""
    wl = LAYER_1P3B
    x = make_inputs(wl)
    assert_parity(run_gpu(x, wl.w), run_oracle(x, wl.w), "bf16", tag=wl.name + " all heads")
