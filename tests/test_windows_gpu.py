"""Per-head windows in the chunkwise forward and backward (nha_extras_t
windows, a device array read by the kernels), on the GPU through the C ABI:
every head of one call is compared with the fp64 oracle run at that head's
own window (the ai.info page: randomised window sizes in training and
per-layer / per-head window schedules).

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


def _run(wl, windows, h0=None, reuse=False):
    import sliding_window_softmax_gb300 as nha

    x = make_inputs(wl)
    d = {n: t.cuda() for n, t in x.items()}
    wv = torch.tensor(windows, dtype=torch.int32, device="cuda")
    B, H, T, D = d["q"].shape
    wsf = torch.empty(max(1, nha.nha_workspace_bytes(B, H, T, D, wl.m, wl.w, dtype=d["q"].dtype,
                                                     per_head_windows=True)), dtype=torch.uint8, device="cuda")
    hd = None if h0 is None else (h0[0].cuda(), h0[1].cuda())
    out = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=wl.w, windows=wv, workspace=wsf, h0=hd,
                          return_state=h0 is not None)
    o, lse = out[0], out[1]
    g = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o, lse, d["dout"], w=wl.w, windows=wv, h0=hd,
                         fwd_workspace=wsf if reuse else None)
    torch.cuda.synchronize()
    got = dict(o=o, lse=lse, dq=g[0], dk=g[1], dv=g[2], dlog_alpha=g[3])
    if h0 is not None:
        got.update(hTk=out[2][0], hTv=out[2][1], dh0k=g[4], dh0v=g[5])
    return x, {n: t.double().cpu().numpy() for n, t in got.items()}


def _check_heads(wl, windows, x, got, h0=None):
    for h, wh in enumerate(windows):
        wh = min(max(wh, 0), wl.w)
        sel = {n: t[:, h:h + 1] for n, t in x.items()}
        hs = None if h0 is None else (h0[0][:, h:h + 1], h0[1][:, h:h + 1])
        fo = oracle.forward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], wh, h0=hs,
                            return_state=h0 is not None)
        rg = oracle.backward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], sel["dout"], wh, h0=hs)
        ref = dict(o=fo[0], lse=fo[1], dq=rg[0], dk=rg[1], dv=rg[2], dlog_alpha=rg[3])
        if h0 is not None:
            ref.update(hTk=fo[2], hTv=fo[3], dh0k=rg[4], dh0v=rg[5])
        for n, r in ref.items():
            kind = "o" if n in ("o", "hTk", "hTv") else ("lse" if n == "lse" else "grad")
            _cmp(f"{wl.name} head {h} (w={wh}) {n}", got[n][:, h:h + 1], r, wl.dtype, kind)


@pytest.mark.parametrize("reuse", [False, True])
def test_per_head_windows_bf16(reuse):
    wl = Workload("windows bf16", 2, 4, 700, 128, 64, 512, dtype="bf16", seed=1501)
    windows = [0, 37, 64, 512]
    x, got = _run(wl, windows, reuse=reuse)
    _check_heads(wl, windows, x, got)


def test_per_head_windows_fp32():
    wl = Workload("windows f32", 1, 4, 300, 64, 16, 100, dtype="f32", seed=1502)
    windows = [0, 37, 64, 100]
    x, got = _run(wl, windows)
    _check_heads(wl, windows, x, got)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_per_head_windows_with_slot_states(dtype):
    wl = Workload("windows states", 1, 4, 333, 64, 32, 200, dtype=dtype, seed=1503)
    windows = [5, 0, 200, 130]
    g = torch.Generator().manual_seed(1504)
    h0 = (torch.randn(1, 4, 32, 64, generator=g) * 0.3 * 64 ** -0.25, torch.randn(1, 4, 32, 64, generator=g))
    x, got = _run(wl, windows, h0=h0, reuse=dtype == "bf16")
    _check_heads(wl, windows, x, got, h0=h0)


def test_out_of_range_windows_are_clamped():
    wl = Workload("windows clamp", 1, 3, 260, 64, 16, 90, dtype="bf16", seed=1505)
    windows = [-7, 40, 100000]
    x, got = _run(wl, windows)
    _check_heads(wl, windows, x, got)


def test_uniform_windows_array_equals_the_scalar_window():
    """A windows array holding w for every head gives the scalar-w results bit for bit."""
    import sliding_window_softmax_gb300 as nha

    wl = Workload("windows uniform", 1, 3, 333, 128, 64, 70, dtype="bf16", seed=1506)
    x = make_inputs(wl)
    d = {n: t.cuda() for n, t in x.items()}
    wv = torch.full((3,), 70, dtype=torch.int32, device="cuda")
    o1, l1 = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=70)
    o2, l2 = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=70, windows=wv)
    g1 = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o1, l1, d["dout"], w=70)
    g2 = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o2, l2, d["dout"], w=70, windows=wv)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
