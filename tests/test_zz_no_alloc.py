"""The forward entry point that allocates nothing (nha_forward_noalloc).

It serves callers that cannot allocate device memory -- plugins that are
handed only their input and output buffers, processes whose device memory
belongs to another allocator.  It
takes its workspace from a fixed scratch array compiled into the library.
This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()
    import sliding_window_softmax_gb300 as nha

    return nha.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_forward_matches_forward_twice(lib, dtype):
    import sliding_window_softmax_gb300 as nha
    from sliding_window_softmax_gb300.synthetic import Workload, make_inputs

    wl = Workload("noalloc", 1, 4, 1000, 128, 64, 100, dtype=dtype, seed=321)
    x = {n: t.cuda() for n, t in make_inputs(wl).items()}
    B, H, T, d = x["q"].shape
    assert lib.nha_workspace_bytes(B, H, T, d, wl.m, wl.w, 64, 1 if dtype == "bf16" else 0, 0) <= (32 << 20)
    ref_o, ref_lse = nha.nha_forward(x["q"], x["k"], x["v"], x["log_alpha"], w=wl.w)
    torch.cuda.synchronize()
    dt = 1 if dtype == "bf16" else 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):  # the second call reuses the scratch left by the first
        o = torch.full_like(x["q"], float("nan"))
        lse = torch.full((B, H, T), float("nan"), device="cuda")
        rc = lib.nha_forward_noalloc(_p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["log_alpha"]), _p(o),
                                     _p(lse), B, H, T, d, wl.m, wl.w, 64, dt, 10000.0, stream)
        assert rc == 0, lib.nha_last_error()
        torch.cuda.synchronize()
        g, r = o.double().cpu().numpy(), ref_o.double().cpu().numpy()
        assert np.all(np.isfinite(g))
        err = np.abs(g - r)
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        if dtype == "f32":
            assert err.max() <= 1e-4
        else:
            assert rel <= 5e-3 and err.max() <= 2e-2
        assert np.abs(lse.double().cpu().numpy() - ref_lse.double().cpu().numpy()).max() <= 2e-2
