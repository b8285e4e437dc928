"""Host logic of bench.py (no GPU): the algorithmic byte and flop models the
roofline fractions divide by, the per-kernel source hash that keeps a stored
ncu traffic figure tied to the kernel it was measured on, and its parser."""
import dataclasses
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sliding_window_softmax_gb300.synthetic import DECODE_1P3B, LAYER_1P3B, Workload  # noqa: E402


def test_decode_bytes_hand_count():
    dw = dataclasses.replace(DECODE_1P3B, B=1, H=1, d=64, m=16, w=4, t=10)
    # states 16 m d (read + write, K and V, fp32); window tokens t-3 .. t-1 from the
    # ring (2 d e each); the leaving token and its gate; token t into the ring;
    # q, k, v, o (4 d e) and log_alpha (4 m)
    states, window, leaving, ring_write, io = 16 * 16 * 64, 3 * 2 * 64 * 2, 2 * 64 * 2 + 64, 2 * 64 * 2 + 64, \
        4 * 64 * 2 + 64
    assert bench.decode_bytes(dw) == states + window + leaving + ring_write + io
    # no token leaves while t < w; w = 0 has no ring
    assert bench.decode_bytes(dataclasses.replace(dw, t=2)) == states + window + ring_write + io
    assert bench.decode_bytes(dataclasses.replace(dw, w=0)) == states + io
    # linear in the heads
    assert bench.decode_bytes(dataclasses.replace(dw, B=3, H=5)) == 15 * bench.decode_bytes(dw)


def test_work_model_conventions():
    wl = Workload("tiny", 1, 1, 10, 64, 16, 4)
    mdl = bench.work_model(wl)
    n_sum = sum(min(t + 1, 4) for t in range(10))
    assert mdl["n_sum"] == n_sum and mdl["R"] == 6
    assert mdl["fwd_flops"] == 4 * 64 * n_sum + 8 * 16 * 64 * 6
    assert mdl["step_flops"] == 3.5 * mdl["fwd_flops"]
    assert mdl["fwd_bytes"] == 10 * (4 * 64 * 2 + 4 * 16 + 4)
    assert mdl["step_bytes"] == mdl["fwd_bytes"] + 10 * (8 * 64 * 2 + 8 * 16 + 4)
    # every kernel the bench can name as dominant has a model
    big = bench.work_model(LAYER_1P3B)["kernels"]
    for k in ("fwd_tc", "bwd_sk_tc", "bwd_sq_tc", "bwd_wkv_tc", "bwd_wdq_tc", "state_scan", "adj_scan", "rope_qk"):
        assert big[k][1] > 0


def _reader_with(changes):
    def reader(name):
        if name in changes:
            return changes[name]
        with open(os.path.join(bench.CSRC, name), "rb") as fh:
            return fh.read()
    return reader


def test_kernel_source_hash_follows_the_kernels_own_sources():
    h_dec, h_fwd = bench.kernel_source_hash("decode_step"), bench.kernel_source_hash("fwd_tc")
    assert h_dec != h_fwd and bench.kernel_source_hash("no_such_kernel") == "none"
    # a change in the decode file moves only the decode hash ...
    src = open(os.path.join(bench.CSRC, "nha_decode.cu"), "rb").read()
    r = _reader_with({"nha_decode.cu": src + b"\n// edited\n"})
    assert bench.kernel_source_hash("decode_step", r) != h_dec
    assert bench.kernel_source_hash("fwd_tc", r) == h_fwd
    # ... a change in a header both include moves both
    com = open(os.path.join(bench.CSRC, "nha_common.cuh"), "rb").read()
    r = _reader_with({"nha_common.cuh": com + b"\n// edited\n"})
    assert bench.kernel_source_hash("decode_step", r) != h_dec
    assert bench.kernel_source_hash("fwd_tc", r) != h_fwd


def test_traffic_lines_parse_and_match_only_their_sources():
    path = os.path.join(ROOT, "profiles", "traffic.md")
    lines = [ln.split() for ln in open(path) if ln.strip().startswith("traffic ")]
    assert lines, "no traffic lines"
    for _, kernel, workload, digest, nbytes in lines:
        got = bench.ncu_traffic(kernel, workload)
        if digest == bench.kernel_source_hash(kernel):
            assert got == pytest.approx(float(nbytes))
        else:
            assert got is None
        assert bench.ncu_traffic(kernel, workload + "-other") is None


def test_step_roofline_frac_is_the_step_figure():
    mdl = bench.work_model(LAYER_1P3B)
    peaks = {"hbm_gbs": 6781.4, "bf16_tflops": 1926.9}
    t_roof, roof = bench.step_roofline(mdl, peaks, 0.5)
    # the 1.3B-like layer is HBM-bound: 504 MB of algorithmic bytes per step
    assert roof["bound"] == "hbm" and roof["algorithmic_bytes"] == mdl["step_bytes"]
    assert abs(mdl["step_bytes"] / 1e6 - 503.3) < 1.5
    assert roof["frac"] == pytest.approx(t_roof / 0.5e-3)
    assert t_roof == pytest.approx(mdl["step_bytes"] / 6781.4e9)
    # the w = T endpoint is tensor-bound
    wt = bench.work_model(LAYER_1P3B.with_(w=2048))
    t2, r2 = bench.step_roofline(wt, peaks, 1.0)
    assert r2["bound"] == "tensor" and r2["frac"] == pytest.approx(t2 / 1e-3)
    _, rf = bench.step_roofline(mdl, peaks, 0.2, backward=False)
    assert rf["algorithmic_bytes"] == mdl["fwd_bytes"]


def test_step_traffic_needs_every_kernel():
    assert bench.step_traffic({"no_such_kernel": 1.0}, "1.3B") is None
    assert bench.step_traffic({}, "1.3B") == 0.0
