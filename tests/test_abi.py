"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol include/nha.h declares, and validates arguments before it
enqueues anything."""
import ctypes
import os
import re

import pytest

import sliding_window_softmax_gb300 as nha
from sliding_window_softmax_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build_library()
    return nha.load_library()


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "nha.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(nha_[a-z_]+)\s*\(", src))


def test_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert declared == set(_binding.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_workspace_bytes(lib):
    f = lib.nha_workspace_bytes
    assert f(1, 2, 256, 64, 16, 32, 64, 0, 0) > 0
    assert f(1, 2, 256, 64, 16, 32, 64, 0, 1) > f(1, 2, 256, 64, 16, 32, 64, 0, 0)
    assert 0 < f(1, 2, 256, 64, 16, 256, 64, 0, 0) < f(1, 2, 256, 64, 16, 32, 64, 0, 0)  # w >= T: no slot states
    assert f(1, 2, 256, 96, 16, 32, 64, 0, 0) == 0  # unsupported d
    assert f(1, 2, 256, 64, 16, 32, 32, 0, 0) == 0  # unsupported C
    assert f(-1, 2, 256, 64, 16, 32, 64, 0, 0) == 0
    # grows linearly in T (chunked states, no T^2 term)
    a = f(1, 1, 4096, 128, 64, 512, 64, 1, 1)
    b = f(1, 1, 8192, 128, 64, 512, 64, 1, 1)
    assert 1.9 < b / a < 2.2


def _fwd(lib, q=1, **kw):
    args = dict(B=1, H=1, T=16, d=64, m=16, w=4, C=64, dt=1, base=10000.0, ws=None, ws_bytes=0)
    args.update(kw)
    p = ctypes.c_void_p(q * 4096) if q else None  # never dereferenced: validation fails first
    return lib.nha_forward(p, p, p, p, p, p, args["B"], args["H"], args["T"], args["d"], args["m"],
                           args["w"], args["C"], args["dt"], args["base"], args["ws"],
                           args["ws_bytes"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), 2), (dict(m=8), 2), (dict(C=128), 2), (dict(T=(1 << 18) + 1), 2),
    (dict(w=-1), 1), (dict(B=-2), 1), (dict(dt=7), 1), (dict(base=0.0), 1),
    (dict(base=float("nan")), 1), (dict(m=0), 1),
])
def test_forward_rejects_bad_arguments(lib, kw, status):
    assert _fwd(lib, **kw) == status
    assert lib.nha_last_error()


def test_forward_null_and_misaligned_and_workspace(lib):
    assert _fwd(lib, q=0) == 1 and b"NULL" in lib.nha_last_error()
    p = ctypes.c_void_p(4096 + 4)
    rc = lib.nha_forward(p, p, p, p, p, p, 1, 1, 16, 64, 16, 4, 64, 1, 10000.0, None, 0, None)
    assert rc == 1 and b"aligned" in lib.nha_last_error()
    # valid pointers but no workspace where one is needed (w < T)
    assert _fwd(lib) == 3 and b"workspace" in lib.nha_last_error()
    # the library only checks the size: too small by one byte is rejected too
    need = lib.nha_workspace_bytes(1, 1, 16, 64, 16, 4, 64, 1, 0)
    assert _fwd(lib, ws=ctypes.c_void_p(1 << 20), ws_bytes=need - 1) == 3


def test_empty_inputs_are_a_no_op(lib):
    # B*H*T == 0: nothing to do, NULL pointers allowed, no CUDA call made
    assert _fwd(lib, q=0, T=0) == 0
    assert _fwd(lib, q=0, B=0) == 0
    assert lib.nha_backward(*([None] * 11), 1, 1, 0, 64, 16, 4, 64, 1, 10000.0, None, 0, None) == 0


def test_backward_validation(lib):
    p = ctypes.c_void_p(4096)
    ptrs = [p] * 11
    assert lib.nha_backward(*ptrs, 1, 1, 16, 64, 16, 4, 64, 1, 10000.0, None, 0, None) == 3
    ptrs[6] = None
    assert lib.nha_backward(*ptrs, 1, 1, 16, 64, 16, 4, 64, 1, 10000.0, None, 0, None) == 1
    assert b"dout" in lib.nha_last_error()


def test_status_strings(lib):
    for code, name in _binding.STATUS.items():
        assert lib.nha_status_string(code).decode() == name


def test_fault_injection_on_host(lib, monkeypatch):
    monkeypatch.setenv("NHA_FAULT_INJECT", "validate")
    assert _fwd(lib) == 5 and b"injected" in lib.nha_last_error()
    monkeypatch.setenv("NHA_FAULT_INJECT", "forward_launch")
    need = lib.nha_workspace_bytes(1, 1, 16, 64, 16, 4, 64, 1, 0)
    # validation passes, the injected failure stops the call before any launch
    assert _fwd(lib, ws=ctypes.c_void_p(1 << 20), ws_bytes=need) == 5
    monkeypatch.delenv("NHA_FAULT_INJECT")


def test_python_binding_rejects_cpu_tensors(lib):
    import torch

    x = torch.zeros(1, 1, 8, 64)
    with pytest.raises(TypeError):
        nha.nha_forward(x, x, x, torch.zeros(1, 1, 8, 16), w=2)


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sliding_window_softmax_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if not f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                continue
            src = open(os.path.join(dirpath, f), errors="ignore").read()
            assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
            assert "nha_oracle" not in src, f


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    # 2 x 16 heads of 2048 tokens at d = 128, m = 64 need more than the 32 MiB
    # built-in scratch: rejected during validation, before any CUDA call.
    p = ctypes.c_void_p(4096)
    rc = lib.nha_forward_noalloc(p, p, p, p, p, p, 2, 16, 2048, 128, 64, 512, 64, 1, 10000.0, None)
    assert rc == 3 and b"built-in scratch" in lib.nha_last_error()
    # an invalid shape reports its own reason
    assert lib.nha_forward_noalloc(p, p, p, p, p, p, 1, 1, 16, 96, 16, 4, 64, 1, 10000.0, None) == 2


def _dec(lib, q=1, **kw):
    args = dict(t=5, B=1, H=1, d=64, m=16, w=4, dt=1, base=10000.0, ring=True)
    args.update(kw)
    p = ctypes.c_void_p(q * 4096) if q else None  # never dereferenced: validation fails first
    r = p if args["ring"] else None
    return lib.nha_decode_step(p, p, p, p, p, p, p, r, r, r, args["t"], args["B"], args["H"], args["d"],
                               args["m"], args["w"], args["dt"], args["base"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), 2), (dict(m=8), 2), (dict(t=1 << 18), 2), (dict(w=(1 << 18) + 1), 2),
    (dict(t=-1), 1), (dict(w=-1), 1), (dict(B=-1), 1), (dict(dt=3), 1), (dict(base=1.0), 1),
    (dict(base=float("inf")), 1), (dict(m=0), 1),
])
def test_decode_rejects_bad_arguments(lib, kw, status):
    assert _dec(lib, **kw) == status
    assert lib.nha_last_error()


def test_decode_pointer_checks(lib):
    assert _dec(lib, q=0) == 1 and b"NULL" in lib.nha_last_error()
    # the ring is required when w > 0 ...
    assert _dec(lib, ring=False) == 1 and b"ring_k" in lib.nha_last_error()
    p, bad = ctypes.c_void_p(4096), ctypes.c_void_p(4096 + 8)
    assert lib.nha_decode_step(p, p, p, p, p, bad, p, p, p, p, 0, 1, 1, 64, 16, 4, 1, 1e4, None) == 1
    assert b"state_k" in lib.nha_last_error() and b"aligned" in lib.nha_last_error()
    # no heads: a no-op that touches nothing
    assert _dec(lib, q=0, B=0) == 0


def test_decode_fault_injection_on_host(lib, monkeypatch):
    # ... and unused when w = 0: validation passes, the injected failure stops the call
    monkeypatch.setenv("NHA_FAULT_INJECT", "decode_launch")
    assert _dec(lib, ring=False, w=0) == 5 and b"decode_launch" in lib.nha_last_error()
    monkeypatch.delenv("NHA_FAULT_INJECT")


def _pre(lib, q=1, **kw):
    args = dict(B=1, H=1, T=16, d=64, m=16, w=4, dt=1, ring=True)
    args.update(kw)
    p = ctypes.c_void_p(q * 4096) if q else None  # never dereferenced: validation fails first
    r = p if args["ring"] else None
    return lib.nha_decode_prefill(p, p, p, p, p, r, r, r, args.get("win"), args["B"], args["H"], args["T"],
                                  args["d"], args["m"], args["w"], args["dt"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), 2), (dict(m=8), 2), (dict(T=(1 << 18) + 1), 2), (dict(w=(1 << 18) + 1), 2),
    (dict(T=-1), 1), (dict(w=-1), 1), (dict(H=-1), 1), (dict(dt=9), 1), (dict(m=0), 1),
])
def test_prefill_rejects_bad_arguments(lib, kw, status):
    assert _pre(lib, **kw) == status
    assert lib.nha_last_error()


def test_prefill_pointer_checks(lib, monkeypatch):
    assert _pre(lib, q=0) == 1 and b"NULL" in lib.nha_last_error()
    assert _pre(lib, ring=False) == 1 and b"ring_k" in lib.nha_last_error()
    p = ctypes.c_void_p(4096)
    assert lib.nha_decode_prefill(p, None, p, p, p, p, p, p, None, 1, 1, 16, 64, 16, 4, 1, None) == 1
    assert b"v is NULL" in lib.nha_last_error()
    assert _pre(lib, q=0, B=0) == 0  # no heads: nothing to do
    assert _pre(lib, win=ctypes.c_void_p(4097)) == 1 and b"windows" in lib.nha_last_error()
    # T = 0 reads no prompt and w = 0 uses no ring: validation passes, the injected failure stops the call
    monkeypatch.setenv("NHA_FAULT_INJECT", "prefill_launch")
    assert lib.nha_decode_prefill(None, None, None, p, p, None, None, None, None, 1, 1, 0, 64, 16, 0, 1, None) == 5
    monkeypatch.delenv("NHA_FAULT_INJECT")


def test_decode_varlen_validation(lib, monkeypatch):
    p = ctypes.c_void_p(4096)
    args = [p] * 10
    # positions are required (unless there are no heads) and must be 4-byte aligned
    assert lib.nha_decode_step_varlen(*args, None, None, 2, 1, 64, 16, 4, 1, 1e4, None) == 1
    assert b"positions" in lib.nha_last_error()
    assert lib.nha_decode_step_varlen(*args, ctypes.c_void_p(4098), None, 2, 1, 64, 16, 4, 1, 1e4, None) == 1
    assert b"aligned" in lib.nha_last_error()
    assert lib.nha_decode_step_varlen(*args, p, ctypes.c_void_p(4097), 2, 1, 64, 16, 4, 1, 1e4, None) == 1
    assert b"windows" in lib.nha_last_error()
    assert lib.nha_decode_step_varlen(*([None] * 10), None, None, 0, 1, 64, 16, 4, 1, 1e4, None) == 0
    assert lib.nha_decode_step_varlen(*args, p, None, 2, 1, 96, 16, 4, 1, 1e4, None) == 2
    monkeypatch.setenv("NHA_FAULT_INJECT", "decode_launch")
    assert lib.nha_decode_step_varlen(*args, p, p, 2, 1, 64, 16, 4, 1, 1e4, None) == 5
    monkeypatch.delenv("NHA_FAULT_INJECT")


def test_public_header_is_plain_c_and_links_against_the_library(lib, tmp_path):
    """include/nha.h compiles as C99 (no C++ in the ABI), and a C program that
    takes the address of every declared entry point links against libnha.so."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = sorted(_declared_symbols())
    src = tmp_path / "abi.c"
    src.write_text('#include "nha.h"\ntypedef void (*fn_t)(void);\n'
                   + "static fn_t volatile table[] = {\n"
                   + "".join(f"    (fn_t){n},\n" for n in names)
                   + "};\nint main(void) { return table[0] == 0; }\n")
    exe = tmp_path / "abi"
    libdir = os.path.dirname(_binding.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", f"-I{os.path.join(ROOT, 'include')}",
                        str(src), "-o", str(exe), f"-L{libdir}", "-l:libnha.so"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_extended_calls_validate_their_extras(lib):
    ex = _binding.Extras()
    f = lib.nha_workspace_bytes_ex
    full = lib.nha_workspace_bytes(1, 2, 256, 64, 16, 32, 64, 1, 1)
    # without extras the _ex sizes are the plain ones
    assert f(1, 2, 256, 64, 16, 32, 64, 1, 1, None) == full
    assert f(1, 2, 256, 64, 16, 32, 64, 1, 1, ctypes.byref(ex)) == full
    ex.fwd_workspace = 4096
    own = f(1, 2, 256, 64, 16, 32, 64, 1, 1, ctypes.byref(ex))
    assert 0 < own < full
    p = ctypes.c_void_p(4096)
    fwd_need = lib.nha_workspace_bytes(1, 2, 256, 64, 16, 32, 64, 1, 0)
    # the forward takes no forward workspace
    rc = lib.nha_forward_ex(p, p, p, p, p, p, 1, 2, 256, 64, 16, 32, 64, 1, 10000.0, ctypes.byref(ex), p,
                            1 << 30, None)
    assert rc == 1 and b"backward only" in lib.nha_last_error()
    # a forward workspace smaller than the forward's plan is refused
    ex.fwd_ws_bytes = fwd_need - 256
    rc = lib.nha_backward_ex(p, p, p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 16, 32, 64, 1, 10000.0,
                             ctypes.byref(ex), p, own, None)
    assert rc == 3 and b"forward workspace" in lib.nha_last_error()
    # the backward's own workspace may be the smaller size
    rc = lib.nha_backward_ex(p, p, p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 16, 32, 64, 1, 10000.0,
                             ctypes.byref(ex), p, own - 256, None)
    assert rc == 3


def test_extended_calls_validate_state_pointers(lib):
    p = ctypes.c_void_p(4096)
    args = (p, p, p, p, p, p, 1, 2, 256, 64, 16, 32, 64, 1, 10000.0)
    ex = _binding.Extras()
    ex.h0_k = 4096  # without h0_v
    assert lib.nha_forward_ex(*args, ctypes.byref(ex), p, 1 << 30, None) == 1
    assert b"together" in lib.nha_last_error()
    ex = _binding.Extras()
    ex.dhT_k = ex.dhT_v = 4096  # a backward input given to the forward
    assert lib.nha_forward_ex(*args, ctypes.byref(ex), p, 1 << 30, None) == 1
    ex = _binding.Extras()
    ex.h0_k, ex.h0_v = 4096, 4100  # misaligned
    assert lib.nha_forward_ex(*args, ctypes.byref(ex), p, 1 << 30, None) == 1
    ex = _binding.Extras()
    ex.dh0_k = ex.dh0_v = 4096  # dh0 without h0
    bargs = (p, p, p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 16, 32, 64, 1, 10000.0)
    assert lib.nha_backward_ex(*bargs, ctypes.byref(ex), p, 1 << 30, None) == 1
    assert b"needs h0" in lib.nha_last_error()
    ex = _binding.Extras()
    ex.hT_k = ex.hT_v = 4096  # a forward output given to the backward
    assert lib.nha_backward_ex(*bargs, ctypes.byref(ex), p, 1 << 30, None) == 1


def test_selftest_wait_validates(lib):
    p = ctypes.c_void_p(4096)
    assert lib.nha_selftest_wait(None, 1000, None) == 1
    assert lib.nha_selftest_wait(ctypes.c_void_p(4098), 1000, None) == 1
    assert lib.nha_selftest_wait(p, 0, None) == 1
    assert lib.nha_selftest_wait(p, (1 << 32) + 1, None) == 1


def test_varlen_extras_and_copies_validate(lib):
    p = ctypes.c_void_p(4096)
    args = (p, p, p, p, p, p, 1, 2, 256, 64, 16, 32, 64, 1, 10000.0)
    ex = _binding.Extras()
    ex.windows_per_sequence = 1  # without a windows array
    assert lib.nha_forward_ex(*args, ctypes.byref(ex), p, 1 << 30, None) == 1
    assert b"without a windows array" in lib.nha_last_error()
    ex = _binding.Extras()
    ex.windows, ex.windows_per_sequence = 4096, 2
    assert lib.nha_forward_ex(*args, ctypes.byref(ex), p, 1 << 30, None) == 1
    ex = _binding.Extras()
    ex.cu_seqlens = 4098  # misaligned
    assert lib.nha_forward_ex(*args, ctypes.byref(ex), p, 1 << 30, None) == 1
    assert b"cu_seqlens" in lib.nha_last_error()
    # sequence lengths lay the workspace out like per-head windows
    ex = _binding.Extras()
    ex.cu_seqlens = 4096
    win = _binding.Extras()
    win.windows = 4096
    f = lib.nha_workspace_bytes_ex
    assert f(2, 2, 300, 64, 16, 100, 64, 1, 1, ctypes.byref(ex)) == f(2, 2, 300, 64, 16, 100, 64, 1, 1,
                                                                       ctypes.byref(win))
    assert f(2, 2, 300, 64, 16, 100, 64, 1, 1, ctypes.byref(ex)) > lib.nha_workspace_bytes(2, 2, 300, 64, 16, 100,
                                                                                          64, 1, 1)
    # pad / unpad: sizes, element size, row bytes, pointers
    for fn in (lib.nha_varlen_pad, lib.nha_varlen_unpad):
        assert fn(p, p, p, 2, 2, 10, 20, 8, 3, None) == 1           # elem_bytes neither 2 nor 4
        assert fn(p, p, p, 2, 2, 10, 20, 3, 2, None) == 1           # 6-byte rows
        assert fn(p, p, p, -1, 2, 10, 20, 8, 4, None) == 1
        assert fn(p, p, p, 2, 2, 10, 20, 0, 4, None) == 1
        assert fn(None, p, p, 2, 2, 10, 20, 8, 4, None) == 1
        assert fn(p, p, ctypes.c_void_p(4098), 2, 2, 10, 20, 8, 4, None) == 1
        assert fn(p, p, p, 0, 2, 10, 20, 8, 4, None) == 0           # nothing to move


def test_decode_ex_rejects_unknown_flags(lib):
    p = ctypes.c_void_p(4096)
    args = (p,) * 10 + (0, 1, 1, 64, 16, 4, 1, 10000.0)
    assert lib.nha_decode_step_ex(*args, 2, None) == 1 and b"flags" in lib.nha_last_error()
    assert lib.nha_decode_step_ex(*args, 0x80000000, None) == 1
