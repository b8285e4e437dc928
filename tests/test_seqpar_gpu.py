"""Sequence parallelism on the GPU: one sequence cut into segments, each run by
the library's kernels on [its w-token halo; its tokens] from the initial state
an associative scan of per-segment summaries gives (nha_gate_total for the
decay, the zero-start final state, nha_state_combine for the scan), backward
with the reverse scan of the state gradients.  Compared with the fp64 oracle
on the whole sequence; the operator's tolerances (fp32 max |err| <= 1e-4;
bf16 o rel L2 <= 5e-3 and max |err| <= 2e-2, lse max |err| <= 2e-2,
gradients rel L2 <= 1e-2).  Multi-GPU exchange: tests/test_seqpar.py (gloo);
every box here has one GPU, so the multi-rank path is unmeasured on hardware.
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
    g = g.double().cpu().numpy()
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


def test_gate_total_and_state_combine():
    import sliding_window_softmax_gb300 as nha

    g = torch.Generator().manual_seed(1601)
    la = torch.nn.functional.logsigmoid(torch.randn(2, 3, 150, 32, generator=g) + 3.0)
    dec = nha.nha_gate_total(la.cuda(), 40)
    ref = torch.exp(la[:, :, :110].double().sum(2))
    assert torch.allclose(dec.double().cpu(), ref, rtol=1e-5, atol=0)
    assert torch.equal(nha.nha_gate_total(la.cuda(), 150).cpu(), torch.ones(2, 3, 32))
    prev = (torch.randn(2, 3, 32, 64, generator=g), torch.randn(2, 3, 32, 64, generator=g))
    cur = (torch.randn(2, 3, 32, 64, generator=g), torch.randn(2, 3, 32, 64, generator=g))
    out = nha.nha_state_combine(dec, tuple(t.cuda() for t in prev), tuple(t.cuda() for t in cur))
    for o, p, c in zip(out, prev, cur):
        want = dec.cpu()[..., None] * p + c
        assert torch.allclose(o.cpu(), want, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("dtype,n,w", [("f32", 3, 96), ("bf16", 3, 96), ("bf16", 4, 300), ("bf16", 2, 0)])
def test_segments_on_one_gpu_equal_the_whole_sequence(dtype, n, w):
    from sliding_window_softmax_gb300.seqpar import backward_segments, forward_segments

    wl = Workload("seqpar", 1, 2, 1100, 128, 32, w, dtype=dtype, seed=1700 + n + w)
    x = make_inputs(wl)
    d = {k: t.cuda() for k, t in x.items()}
    o, lse, ctx = forward_segments(d["q"], d["k"], d["v"], d["log_alpha"], w, n)
    grads = backward_segments(ctx, d["dout"])
    torch.cuda.synchronize()
    ro, rlse = oracle.forward(x["q"], x["k"], x["v"], x["log_alpha"], w)
    rg = oracle.backward(x["q"], x["k"], x["v"], x["log_alpha"], x["dout"], w)
    _cmp("o", o, ro, dtype, "o")
    _cmp("lse", lse, rlse, dtype, "lse")
    for name, a, r in zip(("dq", "dk", "dv", "dlog_alpha"), grads, rg):
        _cmp(name, a, r, dtype, "grad")
