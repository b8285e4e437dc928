"""GPU parity of the recurrent decode step (nha_decode_step through the C ABI)
against the fp64 oracle, on seeded inputs (bf16 inputs upcast exactly).

* Step-by-step runs from zero states over ragged lengths: every o_t against
  the oracle's full-sequence forward, and the final slot states against the
  oracle's own decode recurrence; the ring holds raw copies (bit-exact).
* Serving-sized batches at a late position t: one step from a random state
  and ring, against the oracle's decode step on the same state.
* The prefill entry point, per-sequence positions (continuous batching, CUDA
  graph replay with positions advanced on the device) and per-head windows:
  every output against the oracle's forward over that sequence and head.

Tolerances: fp32: max |err| <= 1e-4 on o, <= 1e-5 on the states;
bf16: o rel L2 <= 5e-3 and max |err| <= 2e-2 (o is rounded to bf16),
states max |err| <= 1e-4 (fp32 arithmetic on exact inputs).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.decode import DecodeState, decode_step
from sliding_window_softmax_gb300.synthetic import Workload, make_inputs

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


def _np(t):
    return t.double().cpu().numpy()


def _check_o(g, r, dtype, tag):
    assert np.all(np.isfinite(g)), tag
    err = np.abs(g - r).max()
    if dtype == "f32":
        assert err <= 1e-4, f"{tag}: max abs {err:.3e}"
    else:
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        assert rel <= 5e-3 and err <= 2e-2, f"{tag}: rel {rel:.3e} max abs {err:.3e}"


STEP_CASES = [
    # B, H, T, d, m, w, dtype
    (1, 2, 150, 64, 16, 37, "f32"),    # ring wraps several times, ragged T
    (1, 2, 150, 64, 16, 37, "bf16"),
    (2, 1, 70, 128, 64, 0, "bf16"),    # w = 0: slots only
    (1, 1, 40, 128, 32, 1, "f32"),     # w = 1: the window is the token itself
    (1, 3, 50, 64, 64, 80, "bf16"),    # w > T: window attention only
    (2, 2, 300, 128, 64, 128, "bf16"),
]


@pytest.mark.parametrize("B,H,T,d,m,w,dtype", STEP_CASES)
def test_decode_steps_match_the_forward_oracle(B, H, T, d, m, w, dtype):
    nha = _nha()
    wl = Workload("decode steps", B, H, T, d, m, w, dtype=dtype, seed=2000 + T + w + m)
    x = make_inputs(wl)
    dev = {n: t.cuda() for n, t in x.items()}
    state = nha.nha_decode_state(B, H, d, m, w, dtype=wl.torch_dtype)
    outs = []
    for t in range(T):
        o = nha.nha_decode_step(dev["q"][:, :, t].contiguous(), dev["k"][:, :, t].contiguous(),
                                dev["v"][:, :, t].contiguous(), dev["log_alpha"][:, :, t].contiguous(),
                                t, w, state)
        outs.append(o)
    torch.cuda.synchronize()
    o_gpu = _np(torch.stack(outs, dim=2))
    o_ref, _ = oracle.forward(x["q"], x["k"], x["v"], x["log_alpha"], w)
    _check_o(o_gpu, o_ref, dtype, f"decode B{B} H{H} T{T} d{d} m{m} w{w} {dtype}")
    # final states against the oracle's decode recurrence; the ring is raw copies
    st = DecodeState(B, H, d, m, w)
    for t in range(T):
        decode_step(st, _np(x["q"][:, :, t]), _np(x["k"][:, :, t]), _np(x["v"][:, :, t]),
                    _np(x["log_alpha"][:, :, t]), t)
    tol = 1e-5 if dtype == "f32" else 1e-4
    assert np.abs(_np(state[0]) - st.S_k).max() <= tol
    assert np.abs(_np(state[1]) - st.S_v).max() <= tol
    if w > 0:
        assert np.array_equal(_np(state[2]), st.ring_k)
        assert np.array_equal(_np(state[3]), st.ring_v)
        assert np.array_equal(_np(state[4]), st.ring_la)


BATCH_CASES = [
    # B, H, d, m, w, t, dtype: decode batches of a 1.3B-like layer (d128 m64 w512)
    (16, 16, 128, 64, 512, 4096, "bf16"),   # 256 heads: one CTA per head
    (1, 2, 128, 64, 512, 4096, "bf16"),     # 2 heads: 8-CTA clusters
    (4, 16, 128, 64, 512, 700, "f32"),
    (8, 16, 64, 64, 64, 2047, "bf16"),      # 340M-like layer
    (2, 16, 128, 32, 8192, 5000, "bf16"),   # window not yet full: slots masked
    (1, 32, 128, 64, 512, 65535, "bf16"),   # long context, last position supported by the forward sizes
]


@pytest.mark.parametrize("B,H,d,m,w,t,dtype", BATCH_CASES)
def test_decode_batch_matches_the_decode_oracle(B, H, d, m, w, t, dtype):
    nha = _nha()
    g = torch.Generator().manual_seed(3000 + B * H + w + t)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    n = max(w, 1)
    s = d ** -0.25
    q, k, v = ((torch.randn((B, H, d), generator=g) * s).to(tdt) for _ in range(3))
    la = torch.nn.functional.logsigmoid(torch.randn((B, H, m), generator=g) + 3.0)
    # a state of the magnitude the recurrence reaches (a convex mix of keys) and a full ring
    sk0 = torch.randn((B, H, m, d), generator=g) * (0.3 * s)
    sv0 = torch.randn((B, H, m, d), generator=g) * (0.3 * s)
    rk0 = (torch.randn((B, H, n, d), generator=g) * s).to(tdt)
    rv0 = (torch.randn((B, H, n, d), generator=g) * s).to(tdt)
    rla0 = torch.nn.functional.logsigmoid(torch.randn((B, H, n, m), generator=g) + 3.0)
    state = tuple(a.cuda() for a in (sk0, sv0, rk0, rv0, rla0))
    o = nha.nha_decode_step(q.cuda(), k.cuda(), v.cuda(), la.cuda(), t, w, state)
    torch.cuda.synchronize()
    st = DecodeState(B, H, d, m, w)
    st.S_k, st.S_v, st.ring_k, st.ring_v, st.ring_la = (_np(a) for a in (sk0, sv0, rk0, rv0, rla0))
    o_ref = decode_step(st, _np(q), _np(k), _np(v), _np(la), t)
    _check_o(_np(o), o_ref, dtype, f"decode batch B{B} H{H} d{d} m{m} w{w} t{t} {dtype}")
    tol = 1e-5 if dtype == "f32" else 1e-4
    assert np.abs(_np(state[0]) - st.S_k).max() <= tol
    assert np.abs(_np(state[1]) - st.S_v).max() <= tol
    assert np.array_equal(_np(state[2]), st.ring_k)
    assert np.array_equal(_np(state[3]), st.ring_v)
    assert np.array_equal(_np(state[4]), st.ring_la)


def test_decode_matches_the_library_forward():
    """Decoding a whole bf16 sequence token by token gives the o of the
    library's chunkwise forward on the same inputs (two independent GPU paths)."""
    nha = _nha()
    wl = Workload("decode after prefill", 1, 4, 200, 128, 64, 48, seed=4000)
    x = make_inputs(wl, device="cuda")
    o_fwd, _ = nha.nha_forward(x["q"], x["k"], x["v"], x["log_alpha"], w=wl.w)
    state = nha.nha_decode_state(1, 4, 128, 64, 48, dtype=torch.bfloat16)
    outs = [nha.nha_decode_step(x["q"][:, :, t].contiguous(), x["k"][:, :, t].contiguous(),
                                x["v"][:, :, t].contiguous(), x["log_alpha"][:, :, t].contiguous(),
                                t, wl.w, state) for t in range(wl.T)]
    o_dec = torch.stack(outs, dim=2)
    torch.cuda.synchronize()
    a, b = _np(o_dec), _np(o_fwd)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) <= 5e-3


def test_decode_bench_workload_layer_matches_the_oracle():
    """The decode workload the benchmark times (same inputs, same launch)."""
    nha = _nha()
    from sliding_window_softmax_gb300.synthetic import DECODE_1P3B, make_decode_layer

    dw = DECODE_1P3B
    x, state = make_decode_layer(dw, 0, device="cuda")
    st = DecodeState(dw.B, dw.H, dw.d, dw.m, dw.w)
    st.S_k, st.S_v, st.ring_k, st.ring_v, st.ring_la = (_np(a) for a in state)
    o = nha.nha_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], dw.t, dw.w, state)
    torch.cuda.synchronize()
    o_ref = decode_step(st, _np(x["q"]), _np(x["k"]), _np(x["v"]), _np(x["log_alpha"]), dw.t)
    _check_o(_np(o), o_ref, dw.dtype, dw.name)
    assert np.abs(_np(state[0]) - st.S_k).max() <= 1e-4
    assert np.abs(_np(state[1]) - st.S_v).max() <= 1e-4


@pytest.mark.parametrize("ks", ["1", "2", "4", "8"])
def test_decode_every_cluster_size(ks, monkeypatch):
    """The result does not depend on how many CTAs share a head (tuning override)."""
    monkeypatch.setenv("NHA_DECODE_CLUSTER", ks)
    test_decode_batch_matches_the_decode_oracle(2, 4, 128, 64, 512, 1000, "bf16")
    test_decode_batch_matches_the_decode_oracle(1, 3, 64, 16, 100, 60, "f32")


PREFILL_CASES = [
    # B, H, T (prompt), K (decoded after it), d, m, w, dtype
    (1, 2, 200, 30, 128, 64, 48, "bf16"),
    (2, 1, 100, 20, 64, 16, 0, "f32"),     # w = 0: no ring
    (1, 2, 20, 40, 64, 32, 64, "bf16"),    # prompt shorter than the window: no slot state yet
    (1, 1, 0, 12, 128, 16, 5, "f32"),      # empty prompt
    (2, 4, 700, 6, 128, 64, 512, "bf16"),  # 1.3B-like head shape, ring wrapped
    (1, 2, 333, 25, 64, 64, 37, "f32"),
]


@pytest.mark.parametrize("B,H,T,K,d,m,w,dtype", PREFILL_CASES)
def test_prefill_then_decode_matches_the_forward_oracle(B, H, T, K, d, m, w, dtype):
    """nha_decode_prefill on a prompt of T tokens, then nha_decode_step for
    t = T .. T+K-1: the o of those tokens against the oracle's forward over all
    T+K tokens; the prefilled state against the decode oracle after T steps."""
    nha = _nha()
    wl = Workload("prefill", B, H, T + K, d, m, w, dtype=dtype, seed=5000 + T + K + w)
    x = make_inputs(wl)
    dev = {n: t.cuda() for n, t in x.items()}
    state = nha.nha_decode_prefill(dev["k"][:, :, :T].contiguous(), dev["v"][:, :, :T].contiguous(),
                                   dev["log_alpha"][:, :, :T].contiguous(), w)
    torch.cuda.synchronize()
    st = DecodeState(B, H, d, m, w)
    for t in range(T):
        decode_step(st, _np(x["q"][:, :, t]), _np(x["k"][:, :, t]), _np(x["v"][:, :, t]),
                    _np(x["log_alpha"][:, :, t]), t)
    tol = 1e-5 if dtype == "f32" else 1e-4
    assert np.abs(_np(state[0]) - st.S_k).max() <= tol
    assert np.abs(_np(state[1]) - st.S_v).max() <= tol
    if w > 0:
        assert np.array_equal(_np(state[2]), st.ring_k)
        assert np.array_equal(_np(state[3]), st.ring_v)
        assert np.array_equal(_np(state[4]), st.ring_la)
    outs = [nha.nha_decode_step(dev["q"][:, :, t].contiguous(), dev["k"][:, :, t].contiguous(),
                                dev["v"][:, :, t].contiguous(), dev["log_alpha"][:, :, t].contiguous(),
                                t, w, state) for t in range(T, T + K)]
    torch.cuda.synchronize()
    o_ref, _ = oracle.forward(x["q"], x["k"], x["v"], x["log_alpha"], w)
    _check_o(_np(torch.stack(outs, dim=2)), o_ref[:, :, T:], dtype, f"prefill T{T} + decode {K} w{w} {dtype}")


def test_varlen_decode_continuous_batch():
    """Sequences with prompts of different lengths, each prefilled on its own,
    then decoded together with nha_decode_step_varlen: every sequence against
    the oracle's forward over its own tokens.  The last steps replay a CUDA
    graph that decodes and then advances the positions on the device."""
    nha = _nha()
    B, H, d, m, w, K = 4, 2, 128, 64, 64, 8
    prompts = [0, 30, 300, 1000]
    wl = Workload("varlen", B, H, max(prompts) + K, d, m, w, seed=6000)
    x = make_inputs(wl)
    dev = {n: t.cuda() for n, t in x.items()}
    state = nha.nha_decode_state(B, H, d, m, w, dtype=torch.bfloat16)
    for b, T in enumerate(prompts):
        sub = tuple(a[b:b + 1] for a in state)
        nha.nha_decode_prefill(dev["k"][b:b + 1, :, :T].contiguous(), dev["v"][b:b + 1, :, :T].contiguous(),
                               dev["log_alpha"][b:b + 1, :, :T].contiguous(), w, state=sub)
    pos = torch.tensor(prompts, dtype=torch.int32, device="cuda")
    idx = (pos.long()[:, None, None].expand(B, H, 1))

    def token(n, step):  # token prompts[b] + step of every sequence, [B, H, .]
        src = dev[n]
        i = (idx + step)[..., None].expand(B, H, 1, src.shape[-1])
        return torch.gather(src, 2, i)[:, :, 0].contiguous()

    outs = []
    for step in range(K // 2):  # eager calls
        outs.append(nha.nha_decode_step_varlen(token("q", step), token("k", step), token("v", step),
                                               token("log_alpha", step), pos, w, state))
        pos += 1
    # graph: fixed input buffers, decode, then advance the positions on the device
    bufs = {n: token(n, K // 2) for n in ("q", "k", "v", "log_alpha")}
    o_buf = torch.empty_like(bufs["q"])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nha.nha_decode_step_varlen(bufs["q"], bufs["k"], bufs["v"], bufs["log_alpha"], pos, w, state, o=o_buf)
        pos.add_(1)
    for step in range(K // 2, K):
        for n in bufs:
            bufs[n].copy_(token(n, step))
        g.replay()
        outs.append(o_buf.clone())
    torch.cuda.synchronize()
    assert pos.cpu().tolist() == [T + K for T in prompts]
    got = _np(torch.stack(outs, dim=2))
    for b, T in enumerate(prompts):
        sel = {n: t[b:b + 1, :, :T + K] for n, t in x.items()}
        o_ref, _ = oracle.forward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], w)
        _check_o(got[b:b + 1], o_ref[:, :, T:], "bf16", f"varlen sequence {b} (prompt {T})")


def test_varlen_position_out_of_range_is_nan_and_leaves_the_state():
    nha = _nha()
    B, H, d, m, w = 2, 2, 64, 16, 8
    g = torch.Generator().manual_seed(6100)
    q, k, v = ((torch.randn((B, H, d), generator=g) * d ** -0.25).float() for _ in range(3))
    la = torch.nn.functional.logsigmoid(torch.randn((B, H, m), generator=g) + 3.0)
    sk0 = torch.randn((B, H, m, d), generator=g) * 0.1
    sv0 = torch.randn((B, H, m, d), generator=g) * 0.1
    rk0, rv0 = (torch.randn((B, H, w, d), generator=g) * 0.3 for _ in range(2))
    rla0 = torch.nn.functional.logsigmoid(torch.randn((B, H, w, m), generator=g) + 3.0)
    state = tuple(a.cuda() for a in (sk0, sv0, rk0, rv0, rla0))
    pos = torch.tensor([-1, 20], dtype=torch.int32, device="cuda")
    o = nha.nha_decode_step_varlen(q.cuda(), k.cuda(), v.cuda(), la.cuda(), pos, w, state)
    torch.cuda.synchronize()
    o = _np(o)
    assert np.all(np.isnan(o[0]))
    for a, a0 in zip(state, (sk0, sv0, rk0, rv0, rla0)):
        assert np.array_equal(_np(a[0]), _np(a0[0]))
    st = DecodeState(1, H, d, m, w)
    st.S_k, st.S_v, st.ring_k, st.ring_v, st.ring_la = (_np(a[1:2]) for a in (sk0, sv0, rk0, rv0, rla0))
    o_ref = decode_step(st, _np(q[1:2]), _np(k[1:2]), _np(v[1:2]), _np(la[1:2]), 20)
    _check_o(o[1:2], o_ref, "f32", "varlen sequence 1")
    assert np.abs(_np(state[0][1:2]) - st.S_k).max() <= 1e-5


@pytest.mark.parametrize("d,m,dtype", [(64, 16, "f32"), (128, 64, "bf16")])
def test_per_head_windows_prefill_and_varlen_decode(d, m, dtype):
    """Heads with windows 0, 5, 37 and 64 inside one 64-entry ring: prefill on
    prompts of 50 and 200 tokens, then varlen decode; each (sequence, head)
    against the oracle's forward with that head's own window."""
    nha = _nha()
    B, H, w, K = 2, 4, 64, 6
    wins, prompts = [0, 5, 37, 64], [50, 200]
    wl = Workload("per-head windows", B, H, max(prompts) + K + 1, d, m, w, dtype=dtype, seed=7000 + d)
    x = make_inputs(wl)
    dev = {n: t.cuda() for n, t in x.items()}
    windows = torch.tensor(wins, dtype=torch.int32, device="cuda")
    state = nha.nha_decode_state(B, H, d, m, w, dtype=wl.torch_dtype)
    for b, T in enumerate(prompts):
        sub = tuple(a[b:b + 1] for a in state)
        nha.nha_decode_prefill(dev["k"][b:b + 1, :, :T].contiguous(), dev["v"][b:b + 1, :, :T].contiguous(),
                               dev["log_alpha"][b:b + 1, :, :T].contiguous(), w, state=sub, windows=windows)
    pos = torch.tensor(prompts, dtype=torch.int32, device="cuda")
    outs = []
    for step in range(K):
        tok = {n: torch.stack([dev[n][b, :, prompts[b] + step] for b in range(B)]).contiguous() for n in dev}
        outs.append(nha.nha_decode_step_varlen(tok["q"], tok["k"], tok["v"], tok["log_alpha"], pos, w, state,
                                               windows=windows))
        pos += 1
    torch.cuda.synchronize()
    got = _np(torch.stack(outs, dim=2))
    for b, T in enumerate(prompts):
        for h, wh in enumerate(wins):
            sel = {n: t[b:b + 1, h:h + 1, :T + K] for n, t in x.items()}
            o_ref, _ = oracle.forward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], wh)
            _check_o(got[b:b + 1, h:h + 1], o_ref[:, :, T:], dtype, f"sequence {b} head {h} window {wh}")
    # a window beyond the ring: NaN for that head, its state untouched
    before = [a.clone() for a in state]
    bad = torch.tensor([w + 1] + wins[1:], dtype=torch.int32, device="cuda")
    tok = {n: torch.stack([dev[n][b, :, prompts[b] + K] for b in range(B)]).contiguous() for n in dev}
    o = nha.nha_decode_step_varlen(tok["q"], tok["k"], tok["v"], tok["log_alpha"], pos, w, state, windows=bad)
    torch.cuda.synchronize()
    assert torch.isnan(o[:, 0]).all() and not torch.isnan(o[:, 1:]).any()
    for a, a0 in zip(state, before):
        assert torch.equal(a[:, 0], a0[:, 0])


@pytest.mark.parametrize("graph", [False, True])
def test_overlapped_launches_of_interleaved_layers(graph):
    """Layers decoding in turn with NHA_DECODE_OVERLAP (each launch streams its
    state in while the previous layer's kernel runs) give the plain launches'
    outputs and states bit for bit, eagerly and replayed from a CUDA graph;
    the first layer's outputs also match the decode oracle."""
    from sliding_window_softmax_gb300.synthetic import DecodeWorkload, make_decode_layer

    nha = _nha()
    dw = DecodeWorkload("overlap", B=3, H=4, d=128, m=64, w=96, t=500, layers=3, dtype="bf16", seed=2101)
    base = [make_decode_layer(dw, i) for i in range(dw.layers)]

    def clone(st):
        return tuple(x.clone() for x in st)

    plain = [clone(st) for _, st in base]
    over = [clone(st) for _, st in base]
    ref = DecodeState(dw.B, dw.H, dw.d, dw.m, dw.w)
    ref.S_k, ref.S_v, ref.ring_k, ref.ring_v, ref.ring_la = (_np(x) for x in base[0][1])
    g = torch.Generator(device="cuda").manual_seed(2102)
    steps = 4
    xs = [[dict(q=(torch.randn(3, 4, 128, generator=g, device="cuda") * 128 ** -0.25).bfloat16(),
                k=(torch.randn(3, 4, 128, generator=g, device="cuda") * 128 ** -0.25).bfloat16(),
                v=(torch.randn(3, 4, 128, generator=g, device="cuda") * 128 ** -0.25).bfloat16(),
                log_alpha=torch.nn.functional.logsigmoid(torch.randn(3, 4, 64, generator=g, device="cuda") + 3))
           for _ in range(dw.layers)] for _ in range(steps)]
    o_plain = [[torch.empty(3, 4, 128, dtype=torch.bfloat16, device="cuda") for _ in range(dw.layers)]
               for _ in range(steps)]
    o_over = [[torch.empty_like(o) for o in row] for row in o_plain]
    for s in range(steps):
        for i in range(dw.layers):
            x = xs[s][i]
            nha.nha_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], dw.t + s, dw.w, plain[i], o=o_plain[s][i])

    def run_overlapped():
        for s in range(steps):
            for i in range(dw.layers):
                x = xs[s][i]
                nha.nha_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], dw.t + s, dw.w, over[i],
                                    o=o_over[s][i], overlap=True)

    if graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=side):
            run_overlapped()
        torch.cuda.current_stream().wait_stream(side)
        cg.replay()
    else:
        run_overlapped()
    torch.cuda.synchronize()
    for s in range(steps):
        for i in range(dw.layers):
            assert torch.equal(o_plain[s][i], o_over[s][i]), f"step {s} layer {i}"
    for i in range(dw.layers):
        for a, b in zip(plain[i], over[i]):
            assert torch.equal(a, b), f"layer {i} state"
    for s in range(steps):
        x = xs[s][0]
        ro = decode_step(ref, _np(x["q"]), _np(x["k"]), _np(x["v"]), _np(x["log_alpha"]), dw.t + s)
        _check_o(_np(o_plain[s][0]), ro, "bf16", f"layer 0 step {s}")

