"""Sequences of different lengths in one call (nha_extras_t cu_seqlens), on
the GPU through the C ABI: packed sequences are moved into the padded layout
(nha_varlen_pad), run in one forward and one backward with per-sequence
lengths, moved back (nha_varlen_unpad), and every sequence is compared with
the fp64 oracle run on that sequence alone, forward and backward, with and
without initial / final slot states, and with per-sequence windows (windows
holding B * H entries).

Tolerances are the operator's: fp32 max |err| <= 1e-4; bf16 o rel L2 <= 5e-3
and max |err| <= 2e-2, lse max |err| <= 2e-2, gradients rel L2 <= 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from sliding_window_softmax_gb300.synthetic import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()


def _cmp(name, g, r, dtype, kind):
    err = np.abs(g - r)
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    assert np.all(np.isfinite(g)), f"{name}: non-finite"
    if dtype == "f32":
        assert err.max() <= 1e-4, f"{name}: max abs {err.max():.3e}"
    elif kind == "o":
        assert rel <= 5e-3 and err.max() <= 2e-2, f"{name}: rel {rel:.3e} max {err.max():.3e}"
    elif kind == "lse":
        assert err.max() <= 2e-2, f"{name}: max {err.max():.3e}"
    else:
        assert rel <= 1e-2, f"{name}: rel L2 {rel:.3e}"


def _packed(lens, H, d, m, w, dtype, seed):
    """Packed inputs [H, Ttot, ...] drawn as one B = 1 workload of Ttot tokens."""
    Ttot = int(sum(lens))
    wl = Workload("varlen", 1, H, Ttot, d, m, w, dtype=dtype, seed=seed)
    x = make_inputs(wl)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return x, cu


def _run(x, cu, lens, w, windows=None, h0=None, dhT=None):
    import sliding_window_softmax_gb300 as nha

    d = {n: t[0].cuda() for n, t in x.items()}  # [H, Ttot, ...]
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    wv = None if windows is None else torch.tensor(windows, dtype=torch.int32, device="cuda").flatten()
    hd = None if h0 is None else (h0[0].cuda(), h0[1].cuda())
    gd = None if dhT is None else (dhT[0].cuda(), dhT[1].cuda())
    Tmax = max(1, int(max(lens)))
    res = nha.nha_forward_varlen(d["q"], d["k"], d["v"], d["log_alpha"], cu_d, Tmax, w, h0=hd,
                                 return_state=h0 is not None, windows=wv)
    o, lse, ctx = res[0], res[1], res[-1]
    g = nha.nha_backward_varlen(ctx, d["dout"], cu_d, w, h0=hd, dhT=gd, windows=wv)
    torch.cuda.synchronize()
    got = dict(o=o, lse=lse, dq=g[0], dk=g[1], dv=g[2], dlog_alpha=g[3])
    if h0 is not None:
        got.update(hTk=res[2][0], hTv=res[2][1], dh0k=g[4], dh0v=g[5])
    return {n: t.double().cpu().numpy() for n, t in got.items()}


def _check(x, cu, lens, w, got, dtype, windows=None, h0=None, dhT=None):
    H = x["q"].shape[1]
    for b, Tb in enumerate(lens):
        a, e = int(cu[b]), int(cu[b + 1])
        for h in range(H):
            wh = w if windows is None else min(max(int(np.asarray(windows)[b][h]), 0), w)
            hs = None if h0 is None else (h0[0][b:b + 1, h:h + 1], h0[1][b:b + 1, h:h + 1])
            gs = None if dhT is None else (dhT[0][b:b + 1, h:h + 1], dhT[1][b:b + 1, h:h + 1])
            tag = f"seq {b} (T={Tb}) head {h} (w={wh})"
            if Tb == 0:  # no tokens: the final state is h0, its gradient flows to dh0 unchanged
                if h0 is not None:
                    for n, ref in (("hTk", hs[0]), ("hTv", hs[1]), ("dh0k", gs[0]), ("dh0v", gs[1])):
                        assert np.array_equal(got[n][b:b + 1, h:h + 1], ref.double().numpy()), f"{tag} {n}"
                continue
            sel = {n: t[:, h:h + 1, a:e] for n, t in x.items()}
            fo = oracle.forward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], wh, h0=hs,
                                return_state=h0 is not None)
            rg = oracle.backward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], sel["dout"], wh, h0=hs, dhT=gs)
            ref = dict(o=fo[0], lse=fo[1], dq=rg[0], dk=rg[1], dv=rg[2], dlog_alpha=rg[3])
            if h0 is not None:
                ref.update(hTk=fo[2], hTv=fo[3], dh0k=rg[4], dh0v=rg[5])
            for n, r in ref.items():
                if n in ("hTk", "hTv", "dh0k", "dh0v"):
                    gv = got[n][b:b + 1, h:h + 1]
                elif n == "lse":
                    gv = got[n][h:h + 1, a:e][None]
                else:
                    gv = got[n][h:h + 1, a:e][None]
                kind = "o" if n in ("o", "hTk", "hTv") else ("lse" if n == "lse" else "grad")
                _cmp(f"{tag} {n}", gv, r, dtype, kind)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_varlen_sequences_match_each_sequence_alone(dtype):
    # lengths around the 64-token chunks and 128-row tiles, one shorter than
    # the window, one of a single token, one empty
    lens = [700, 129, 0, 64, 1, 333] if dtype == "bf16" else [300, 65, 0, 1, 130]
    d, m, w = (128, 64, 200) if dtype == "bf16" else (64, 16, 90)
    x, cu = _packed(lens, 2, d, m, w, dtype, seed=1901)
    got = _run(x, cu, lens, w)
    _check(x, cu, lens, w, got, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_varlen_with_slot_states(dtype):
    lens = [333, 0, 90, 201]
    B, H, d, m, w = len(lens), 2, 64, 32, 100
    x, cu = _packed(lens, H, d, m, w, dtype, seed=1902)
    g = torch.Generator().manual_seed(1903)
    h0 = (torch.randn(B, H, m, d, generator=g) * 0.3 * d ** -0.25, torch.randn(B, H, m, d, generator=g))
    dhT = (torch.randn(B, H, m, d, generator=g) * 0.1, torch.randn(B, H, m, d, generator=g) * 0.1)
    got = _run(x, cu, lens, w, h0=h0, dhT=dhT)
    _check(x, cu, lens, w, got, dtype, h0=h0, dhT=dhT)


def test_varlen_with_per_sequence_windows():
    lens = [400, 150, 77]
    B, H, d, m, w = len(lens), 3, 128, 64, 256
    x, cu = _packed(lens, H, d, m, w, "bf16", seed=1904)
    windows = [[0, 37, 256], [256, 64, 5], [100, 1000, -3]]  # per (sequence, head); clamped to [0, w]
    got = _run(x, cu, lens, w, windows=windows)
    _check(x, cu, lens, w, got, "bf16", windows=windows)


def test_full_length_sequences_equal_the_batched_call():
    """cu_seqlens with every sequence T tokens long gives the batched results bit for bit."""
    import sliding_window_softmax_gb300 as nha

    wl = Workload("varlen uniform", 2, 2, 300, 128, 64, 70, dtype="bf16", seed=1905)
    x = make_inputs(wl)
    dd = {n: t.cuda() for n, t in x.items()}
    cu = torch.tensor([0, 300, 600], dtype=torch.int32, device="cuda")
    o1, l1 = nha.nha_forward(dd["q"], dd["k"], dd["v"], dd["log_alpha"], w=70)
    o2, l2 = nha.nha_forward(dd["q"], dd["k"], dd["v"], dd["log_alpha"], w=70, cu_seqlens=cu)
    g1 = nha.nha_backward(dd["q"], dd["k"], dd["v"], dd["log_alpha"], o1, l1, dd["dout"], w=70)
    g2 = nha.nha_backward(dd["q"], dd["k"], dd["v"], dd["log_alpha"], o2, l2, dd["dout"], w=70, cu_seqlens=cu)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("dtype,width", [(torch.bfloat16, 128), (torch.float32, 16), (torch.float32, 1),
                                         (torch.bfloat16, 6)])
def test_pad_unpad_move_rows_exactly(dtype, width):
    import sliding_window_softmax_gb300 as nha

    lens = [5, 0, 17, 1, 9]
    T = 12  # shorter than the 17-token sequence: its rows past T are dropped
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    H, Ttot = 3, int(cu[-1])
    g = torch.Generator().manual_seed(1906)
    packed = torch.randn(H, Ttot, width, generator=g).to(dtype)
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    padded = nha.nha_varlen_pad(packed.cuda(), cu_d, T)
    back = nha.nha_varlen_unpad(padded, cu_d, Ttot)
    torch.cuda.synchronize()
    ref = torch.zeros(len(lens), H, T, width, dtype=dtype)
    ref_back = torch.zeros(H, Ttot, width, dtype=dtype)
    for b, n in enumerate(lens):
        n = min(n, T)
        ref[b, :, :n] = packed[:, cu[b]:cu[b] + n]
        ref_back[:, cu[b]:cu[b] + n] = packed[:, cu[b]:cu[b] + n]
    assert torch.equal(padded.cpu(), ref)
    assert torch.equal(back.cpu(), ref_back)
