"""Initial and final slot states of the chunkwise operator on the GPU, through
the C ABI (nha_forward_ex / nha_backward_ex), against the fp64 oracle on the
same inputs.

Reading (the ai.info page, Future Directions: learned initial slot states;
the Paper-Notes page, Chunkwise 并行计算: a state carried from chunk to chunk):
h0 is the long memory before token 0, so no slot logit is masked and queries
t < w read h0 itself; hT is the long memory after token T - w - 1; dhT is the
gradient with respect to hT and dh0 the gradient with respect to h0.

Tolerances are the operator's: fp32 max |err| <= 1e-4 on every output; bf16
o rel L2 <= 5e-3 and max |err| <= 2e-2, gradients (dh0 included) rel L2 <=
1e-2, lse max |err| <= 2e-2, and the final states (fp32 sums of bf16 products)
rel L2 <= 5e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from sliding_window_softmax_gb300.synthetic import LAYER_1P3B, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()


def _states(B, H, m, d, seed):
    """h0 ~ N(0,1) 0.3 d^-0.25 for keys (the size of a convex mix of keys), N(0,1)
    for values; dhT ~ N(0,1) 0.1."""
    g = torch.Generator().manual_seed(seed)
    h0k = torch.randn(B, H, m, d, generator=g) * 0.3 * d ** -0.25
    h0v = torch.randn(B, H, m, d, generator=g)
    dhk = torch.randn(B, H, m, d, generator=g) * 0.1
    dhv = torch.randn(B, H, m, d, generator=g) * 0.1
    return h0k, h0v, dhk, dhv


def _cmp(name, g, r, dtype, kind):
    g = g.double().cpu().numpy() if hasattr(g, "cpu") else g
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite"
    err = np.abs(g - r)
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    if dtype == "f32":
        assert err.max() <= 1e-4, f"{name}: max abs {err.max():.3e}"
    elif kind == "o":
        assert rel <= 5e-3 and err.max() <= 2e-2, f"{name}: rel {rel:.3e} max {err.max():.3e}"
    elif kind == "lse":
        assert err.max() <= 2e-2, f"{name}: max {err.max():.3e}"
    elif kind == "state":
        assert rel <= 5e-3, f"{name}: rel {rel:.3e}"
    else:
        assert rel <= 1e-2, f"{name}: rel L2 {rel:.3e}"


CASES = [
    Workload("states f32", 1, 2, 300, 64, 16, 32, dtype="f32", seed=1101),
    Workload("states f32 w=0", 1, 2, 200, 128, 32, 0, dtype="f32", seed=1102),
    Workload("states f32 w>T", 1, 1, 150, 64, 16, 400, dtype="f32", seed=1103),
    Workload("states bf16", 2, 2, 333, 128, 64, 70, dtype="bf16", seed=1104),
    Workload("states bf16 w=0", 1, 2, 257, 64, 32, 0, dtype="bf16", seed=1105),
    Workload("states bf16 w>T", 1, 2, 200, 128, 16, 300, dtype="bf16", seed=1106),
    Workload("states bf16 w=1", 1, 2, 129, 64, 16, 1, dtype="bf16", seed=1107),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("reuse", [False, True])
def test_initial_and_final_states_match_the_oracle(wl, reuse):
    import sliding_window_softmax_gb300 as nha

    x = make_inputs(wl)
    h0k, h0v, dhk, dhv = _states(wl.B, wl.H, wl.m, wl.d, wl.seed + 7)
    d = {n: t.cuda() for n, t in x.items()}
    h0 = (h0k.cuda(), h0v.cuda())
    dhT = (dhk.cuda(), dhv.cuda())
    B, H, T, D = d["q"].shape
    wsf = torch.empty(max(1, nha.nha_workspace_bytes(B, H, T, D, wl.m, wl.w, dtype=d["q"].dtype)),
                      dtype=torch.uint8, device="cuda")
    o, lse, (hk, hv) = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=wl.w, h0=h0,
                                       return_state=True, workspace=wsf)
    g = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o, lse, d["dout"], w=wl.w, h0=h0, dhT=dhT,
                         fwd_workspace=wsf if reuse else None)
    torch.cuda.synchronize()
    ro, rlse, rhk, rhv = oracle.forward(x["q"], x["k"], x["v"], x["log_alpha"], wl.w, h0=(h0k, h0v),
                                        return_state=True)
    rg = oracle.backward(x["q"], x["k"], x["v"], x["log_alpha"], x["dout"], wl.w, h0=(h0k, h0v),
                         dhT=(dhk, dhv))
    tag = f"{wl.name} reuse={reuse}"
    _cmp(f"{tag} o", o, ro, wl.dtype, "o")
    _cmp(f"{tag} lse", lse, rlse, wl.dtype, "lse")
    _cmp(f"{tag} hTk", hk, rhk, wl.dtype, "state")
    _cmp(f"{tag} hTv", hv, rhv, wl.dtype, "state")
    for name, a, r in zip(("dq", "dk", "dv", "dlog_alpha", "dh0k", "dh0v"), g, rg):
        _cmp(f"{tag} {name}", a, r, wl.dtype, "grad")


def test_final_states_without_initial_states():
    """hT alone (no h0): the slots of queries t < w stay masked; hT is the state
    after token T - w - 1; dhT flows into dk, dv and dlog_alpha."""
    import sliding_window_softmax_gb300 as nha

    wl = Workload("hT only", 1, 2, 300, 128, 64, 40, dtype="bf16", seed=1201)
    x = make_inputs(wl)
    _, _, dhk, dhv = _states(1, 2, 64, 128, 1202)
    d = {n: t.cuda() for n, t in x.items()}
    o, lse, (hk, hv) = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=wl.w, return_state=True)
    g = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o, lse, d["dout"], w=wl.w,
                         dhT=(dhk.cuda(), dhv.cuda()))
    torch.cuda.synchronize()
    ro, _, rhk, rhv = oracle.forward(x["q"], x["k"], x["v"], x["log_alpha"], wl.w, return_state=True)
    rg = oracle.backward(x["q"], x["k"], x["v"], x["log_alpha"], x["dout"], wl.w, dhT=(dhk, dhv))
    _cmp("o", o, ro, "bf16", "o")
    _cmp("hTk", hk, rhk, "bf16", "state")
    _cmp("hTv", hv, rhv, "bf16", "state")
    assert len(g) == 4
    for name, a, r in zip(("dq", "dk", "dv", "dlog_alpha"), g, rg):
        _cmp(name, a, r, "bf16", "grad")


def test_full_size_layer_with_states():
    """The 1.3B-like layer (B4 H16 T2048 d128 m64 w512, bf16) with initial states
    and a final-state gradient; two whole heads compared."""
    import sliding_window_softmax_gb300 as nha

    wl = LAYER_1P3B
    x = make_inputs(wl)
    h0k, h0v, dhk, dhv = _states(wl.B, wl.H, wl.m, wl.d, 1301)
    d = {n: t.cuda() for n, t in x.items()}
    o, lse, (hk, hv) = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=wl.w,
                                       h0=(h0k.cuda(), h0v.cuda()), return_state=True)
    g = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o, lse, d["dout"], w=wl.w,
                         h0=(h0k.cuda(), h0v.cuda()), dhT=(dhk.cuda(), dhv.cuda()))
    torch.cuda.synchronize()
    heads = [(0, 3), (3, 12)]
    sel = {n: torch.stack([t[b, h] for b, h in heads])[None] for n, t in x.items()}
    st = {n: torch.stack([t[b, h] for b, h in heads])[None] for n, t in
          dict(h0k=h0k, h0v=h0v, dhk=dhk, dhv=dhv).items()}
    ro, rlse, rhk, rhv = oracle.forward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], wl.w,
                                        h0=(st["h0k"], st["h0v"]), return_state=True)
    rg = oracle.backward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], sel["dout"], wl.w,
                         h0=(st["h0k"], st["h0v"]), dhT=(st["dhk"], st["dhv"]))

    def pick(t):
        return np.stack([t[b, h].double().cpu().numpy() for b, h in heads])[None]

    _cmp("o", pick(o), ro, "bf16", "o")
    _cmp("lse", pick(lse), rlse, "bf16", "lse")
    _cmp("hTk", pick(hk), rhk, "bf16", "state")
    _cmp("hTv", pick(hv), rhv, "bf16", "state")
    for name, a, r in zip(("dq", "dk", "dv", "dlog_alpha", "dh0k", "dh0v"), g, rg):
        _cmp(name, pick(a), r, "bf16", "grad")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_segments_chained_through_final_states(dtype):
    """A 1000-token sequence in three segments on the GPU: each later segment
    runs on [the previous w tokens; its tokens] from the previous segment's hT;
    its outputs after those w queries equal the oracle's full-sequence outputs,
    and the last hT equals the full sequence's."""
    import sliding_window_softmax_gb300 as nha

    wl = Workload("segments", 1, 2, 1000, 128, 32, 96, dtype=dtype, seed=1401)
    x = make_inputs(wl)
    ro, rlse, rhk, rhv = oracle.forward(x["q"], x["k"], x["v"], x["log_alpha"], wl.w, return_state=True)
    d = {n: t.cuda() for n, t in x.items()}
    cuts = [0, 333, 700, 1000]
    state = None
    for a, b in zip(cuts[:-1], cuts[1:]):
        lo = max(0, a - wl.w)
        seg = {n: t[:, :, lo:b].contiguous() for n, t in d.items()}
        o, lse, state = nha.nha_forward(seg["q"], seg["k"], seg["v"], seg["log_alpha"], w=wl.w, h0=state,
                                        return_state=True)
        keep = a - lo
        _cmp(f"segment {a}:{b} o", o[:, :, keep:], ro[:, :, a:b], dtype, "o")
        _cmp(f"segment {a}:{b} lse", lse[:, :, keep:], rlse[:, :, a:b], dtype, "lse")
    torch.cuda.synchronize()
    _cmp("final hTk", state[0], rhk, dtype, "state")
    _cmp("final hTv", state[1], rhv, dtype, "state")


@pytest.mark.parametrize("windows", [None, [100, 0]])
def test_long_chunk_scan_with_slot_states(windows):
    """Few heads over many chunks (127 and 128 chunks of 64 tokens), h0 in
    and hT out, compared with the oracle, forward and backward, with per-head
    windows (so the heads have different chunk counts)."""
    import sliding_window_softmax_gb300 as nha

    wl = Workload("long scan", 1, 2, 8192, 64, 16, 100, dtype="bf16", seed=2201)
    x = make_inputs(wl)
    g = torch.Generator().manual_seed(2202)
    h0 = (torch.randn(1, 2, 16, 64, generator=g) * 0.3 * 64 ** -0.25, torch.randn(1, 2, 16, 64, generator=g))
    dhT = (torch.randn(1, 2, 16, 64, generator=g) * 0.1, torch.randn(1, 2, 16, 64, generator=g) * 0.1)
    d = {n: t.cuda() for n, t in x.items()}
    hd = tuple(t.cuda() for t in h0)
    gd = tuple(t.cuda() for t in dhT)
    wv = None if windows is None else torch.tensor(windows, dtype=torch.int32, device="cuda")
    o, lse, hT = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=wl.w, h0=hd, return_state=True,
                                 windows=wv)
    gr = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o, lse, d["dout"], w=wl.w, h0=hd, dhT=gd,
                          windows=wv)
    torch.cuda.synchronize()
    got = dict(o=o, lse=lse, hTk=hT[0], hTv=hT[1], dq=gr[0], dk=gr[1], dv=gr[2], dlog_alpha=gr[3], dh0k=gr[4],
               dh0v=gr[5])
    got = {n: t.double().cpu().numpy() for n, t in got.items()}
    for h in range(2):
        wh = wl.w if windows is None else windows[h]
        sel = {n: t[:, h:h + 1] for n, t in x.items()}
        hs = (h0[0][:, h:h + 1], h0[1][:, h:h + 1])
        gs = (dhT[0][:, h:h + 1], dhT[1][:, h:h + 1])
        fo = oracle.forward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], wh, h0=hs, return_state=True)
        rg = oracle.backward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], sel["dout"], wh, h0=hs, dhT=gs)
        ref = dict(o=fo[0], lse=fo[1], hTk=fo[2], hTv=fo[3], dq=rg[0], dk=rg[1], dv=rg[2], dlog_alpha=rg[3],
                   dh0k=rg[4], dh0v=rg[5])
        for n, r in ref.items():
            gv = got[n][:, h:h + 1]
            err = np.abs(gv - r)
            rel = np.linalg.norm(gv - r) / max(np.linalg.norm(r), 1e-30)
            assert np.all(np.isfinite(gv)), f"head {h} {n}: non-finite"
            if n == "lse":
                assert err.max() <= 2e-2, f"head {h} {n}: max {err.max():.3e}"
            elif n in ("o", "hTk", "hTv"):
                assert rel <= 5e-3 and err.max() <= 2e-2, f"head {h} {n}: rel {rel:.3e} max {err.max():.3e}"
            else:
                assert rel <= 1e-2, f"head {h} {n}: rel {rel:.3e}"
