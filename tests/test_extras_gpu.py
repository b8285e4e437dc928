"""The extended calls (nha_forward_ex / nha_backward_ex) on the GPU, through the
C ABI: the backward that reuses the forward's workspace (chunk states, gate
totals, RoPE table, rotated q and k) gives bit-identical gradients to the
backward that forms them again."""
import numpy as np
import pytest
import torch

from sliding_window_softmax_gb300.synthetic import LAYER_1P3B, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()


CASES = [
    Workload("reuse f32", 1, 2, 300, 64, 16, 32, dtype="f32", seed=901),
    Workload("reuse bf16", 2, 2, 333, 128, 64, 70, dtype="bf16", seed=902),
    Workload("reuse bf16 w=0", 1, 2, 257, 64, 32, 0, dtype="bf16", seed=903),
    Workload("reuse bf16 w>T", 1, 1, 200, 128, 16, 500, dtype="bf16", seed=904),
    LAYER_1P3B,
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_backward_reusing_the_forward_workspace_is_identical(wl):
    import sliding_window_softmax_gb300 as nha

    d = {n: t.cuda() for n, t in make_inputs(wl).items()}
    B, H, T, D = d["q"].shape
    wsf = torch.empty(nha.nha_workspace_bytes(B, H, T, D, wl.m, wl.w, dtype=d["q"].dtype),
                      dtype=torch.uint8, device="cuda")
    own = nha.nha_workspace_bytes(B, H, T, D, wl.m, wl.w, dtype=d["q"].dtype, backward=True,
                                  reuse_forward=True)
    full = nha.nha_workspace_bytes(B, H, T, D, wl.m, wl.w, dtype=d["q"].dtype, backward=True)
    assert own < full
    o, lse = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=wl.w, workspace=wsf)
    plain = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o, lse, d["dout"], w=wl.w)
    wsb = torch.full((own,), 0xFF, dtype=torch.uint8, device="cuda")  # stale contents must not matter
    reused = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o, lse, d["dout"], w=wl.w,
                              workspace=wsb, fwd_workspace=wsf)
    torch.cuda.synchronize()
    for name, a, b in zip(("dq", "dk", "dv", "dlog_alpha"), plain, reused):
        assert torch.equal(a, b), name
        assert bool(torch.isfinite(a.float()).all()), name
