"""The device-side status word of a call (nha_extras_t.status), on the GPU: set
to zero by every forward and backward, bit NHA_STATUS_GATE_RANGE when a chunk's
per-slot log_alpha sum leaves the range where the intra-chunk factorisation is
exact, and bit NHA_STATUS_TIMEOUT when a bounded wait gives up, shown by the
self-test wait on a barrier that nothing arrives at.  Nothing here faults or
waits without a bound."""
import pytest
import torch

from sliding_window_softmax_gb300.synthetic import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()


def test_selftest_wait_reports_a_wait_that_ran_out():
    import sliding_window_softmax_gb300 as nha

    st = nha.nha_selftest_wait(100_000)
    torch.cuda.synchronize()
    assert int(st.item()) == nha._binding.STATUS_TIMEOUT
    # the context is still usable: a forward afterwards runs and reports nothing
    wl = Workload("after", 1, 2, 200, 64, 16, 32, dtype="bf16", seed=1801)
    d = {n: t.cuda() for n, t in make_inputs(wl).items()}
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    o, lse = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=32, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and bool(torch.isfinite(o.float()).all())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gate_range_is_reported(dtype):
    import sliding_window_softmax_gb300 as nha

    wl = Workload("gates", 1, 2, 300, 64, 16, 40, dtype=dtype, seed=1802)
    d = {n: t.cuda() for n, t in make_inputs(wl).items()}
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    o, lse = nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=40, status=status)
    g = nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o, lse, d["dout"], w=40)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # one head whose gates close hard: log_alpha = -40 sums to -2560 over a chunk
    la = d["log_alpha"].clone()
    la[0, 1] = -40.0
    o, lse = nha.nha_forward(d["q"], d["k"], d["v"], la, w=40, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & nha._binding.STATUS_GATE_RANGE
    bst = torch.zeros((1,), dtype=torch.int32, device="cuda")
    nha.nha_backward(d["q"], d["k"], d["v"], la, o, lse, d["dout"], w=40, status=bst)
    torch.cuda.synchronize()
    assert int(bst.item()) & nha._binding.STATUS_GATE_RANGE
    # the next ordinary call clears it
    nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], w=40, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
