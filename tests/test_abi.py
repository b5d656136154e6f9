"""The C-ABI library builds, loads without a GPU, and exports every entry
point ``include/maxsim.h`` declares (no compute calls here).  Also the
argument checks that return before anything touches a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "maxsim.h")


@pytest.fixture(scope="module")
def lib():
    from late_interaction_retrieval_maxsim_gb300 import _build
    _build.build()
    import late_interaction_retrieval_maxsim_gb300 as m
    return m.load_library()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(maxsim_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ["maxsim_forward", "maxsim_backward", "maxsim_build_csr", "maxsim_device_status",
              "maxsim_forward_workspace_size", "maxsim_backward_workspace_size",
              "maxsim_status_string", "maxsim_abi_version"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} missing from libmaxsim.so"


def test_abi_version_and_status_strings(lib):
    assert lib.maxsim_abi_version() == 1
    for code in range(6):
        assert lib.maxsim_status_string(code)


def test_workspace_sizes(lib):
    # short queries need no forward workspace; long ones keep per-chunk partials
    assert lib.maxsim_forward_workspace_size(16, 32, 50000, 128, 0) == 0
    big = lib.maxsim_forward_workspace_size(1, 1024, 10000, 128, 0)
    assert big >= 32 * 10000 * 4
    assert lib.maxsim_forward_workspace_size(1, 1024, 10000, 128, 2) >= 32 * 10000 * 8
    assert lib.maxsim_backward_workspace_size(256, 32, 256, 46080) >= (46081 + 256 * 256 * 32) * 4


def test_argument_errors_return_before_touching_the_device(lib):
    vp = ctypes.c_void_p
    # bounded-wait self-test: limit out of range -> invalid argument
    lib.maxsim_selftest_bounded_wait.argtypes = [ctypes.c_uint32, vp]
    assert lib.maxsim_selftest_bounded_wait(0, None) == 1
    assert lib.maxsim_selftest_bounded_wait(1_000_001, None) == 1
    # dim != 128 -> unsupported; bad dtype -> unsupported
    f = lib.maxsim_forward
    assert f(vp(16), vp(16), 1, 32, vp(16), vp(16), 1, 10, 64, 0, 1.0, 1.0,
             vp(16), None, None, None, 0, None) == 2
    assert f(vp(16), vp(16), 1, 32, vp(16), vp(16), 1, 10, 128, 7, 1.0, 1.0,
             vp(16), None, None, None, 0, None) == 2
    # negative sizes / null scores -> invalid argument
    assert f(vp(16), vp(16), -1, 32, vp(16), vp(16), 1, 10, 128, 0, 1.0, 1.0,
             vp(16), None, None, None, 0, None) == 1
    assert f(vp(16), vp(16), 1, 32, vp(16), vp(16), 1, 10, 128, 0, 1.0, 1.0,
             None, None, None, None, 0, None) == 1
    # misaligned Q -> invalid argument
    assert f(vp(18), vp(16), 1, 32, vp(16), vp(16), 1, 10, 128, 0, 1.0, 1.0,
             vp(16), None, None, None, 0, None) == 1
    # INT8 without scales -> invalid argument
    assert f(vp(16), vp(16), 1, 32, vp(16), vp(16), 1, 10, 128, 2, 0.0, 1.0,
             vp(16), None, None, None, 0, None) == 1
    # long queries without the workspace -> workspace error
    assert f(vp(16), vp(16), 1, 1024, vp(16), vp(16), 1, 10, 128, 0, 1.0, 1.0,
             vp(16), None, None, None, 0, None) == 3
    # empty problem: nothing to do
    assert f(None, None, 0, 32, None, None, 0, 0, 128, 0, 1.0, 1.0,
             None, None, None, None, 0, None) == 0
    b = lib.maxsim_backward
    assert b(vp(16), vp(16), vp(16), vp(16), 1, 32, vp(16), vp(16), 1, 10, 128, 2,
             vp(16), vp(16), vp(16), 1 << 20, None) == 2          # INT8 backward
    assert b(vp(16), vp(16), vp(16), vp(16), 1, 32, vp(16), vp(16), 1, 10, 128, 0,
             vp(16), vp(16), None, 0, None) == 3                  # no workspace
    c = lib.maxsim_build_csr
    assert c(vp(16), vp(16), 1, 32, vp(16), 1, 10, None, vp(16), vp(16), 1 << 20, None) == 1


def test_host_corpus_argument_errors_return_before_touching_the_device(lib):
    """maxsim_forward_host plans its blocks on the host; plan errors and a
    short workspace return before any CUDA call."""
    vp = ctypes.c_void_p
    lib.maxsim_forward_host.argtypes = [vp, vp, ctypes.c_int32, ctypes.c_int32, vp, vp, ctypes.c_int32,
                                        ctypes.c_int64, ctypes.c_int32, ctypes.c_int, ctypes.c_float,
                                        ctypes.c_float, vp, vp, vp, ctypes.c_int32, ctypes.c_int64, vp,
                                        ctypes.c_size_t, vp, vp]
    lib.maxsim_forward_host_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                       ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                                       ctypes.c_int]
    lib.maxsim_forward_host_workspace_size.restype = ctypes.c_size_t
    cu = (ctypes.c_int32 * 4)(0, 5, 40, 41)
    cu_bad = (ctypes.c_int32 * 4)(1, 5, 40, 41)
    host = vp(ctypes.addressof(cu))

    def call(cu_arr, block_docs, block_tokens, ws_bytes, total=41, dim=128):
        return lib.maxsim_forward_host(vp(16), vp(16), 1, 32, host, vp(ctypes.addressof(cu_arr)), 3, total, dim,
                                       0, 1.0, 1.0, vp(16), None, None, block_docs, block_tokens, vp(256),
                                       ws_bytes, None, None)

    need = lib.maxsim_forward_host_workspace_size(1, 32, 3, 2, 64, 128, 0)
    # two staging blocks of 64 rows x 256 B plus the corpus's and a block's offsets
    assert need >= 2 * 64 * 256 + 4 * 4 + 3 * 4
    assert call(cu, 2, 64, need, dim=64) == 2          # dim != 128
    assert call(cu, 0, 64, need) == 1                  # no documents per block
    assert call(cu, 2, 0, need) == 1                   # no tokens per block
    assert call(cu, 2, 34, need) == 1                  # document 1 has 35 tokens
    assert call(cu_bad, 2, 64, need) == 1              # cu[0] != 0
    assert call(cu, 2, 64, need, total=40) == 1        # cu[n_docs] != total
    assert call(cu, 2, 64, need - 1) == 3              # workspace too small
    assert lib.maxsim_forward_host_workspace_size(1, 32, 3, 0, 64, 128, 0) == 0


def test_bench_case_mode_parses_without_a_gpu():
    """bench.py's single-case mode (the command the profiles run) imports and
    parses its arguments on a machine without a GPU (it touches the device
    only when a case runs)."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "bench.py", "--help"], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "chamfer" in r.stdout and "--case" in r.stdout


def test_backward_rejects_misaligned_rows(lib):
    """Rows are moved with vector loads and stores: a pointer off a 16-byte
    boundary is an argument error, reported before any device work."""
    vp = ctypes.c_void_p
    b = lib.maxsim_backward
    ws = 1 << 20
    ok = [vp(256), vp(256), vp(256), vp(256), 1, 32, vp(256), vp(256), 1, 10, 128, 0,
          vp(256), vp(256), vp(256), ws, None]
    for pos in (2, 6, 12, 13):          # Q, D, dQ, dD
        args = list(ok)
        args[pos] = vp(256 + 8)
        assert b(*args) == 1


def test_noalloc_binding_checks_outputs_before_any_call(lib):
    """maxsim_forward_noalloc writes into caller-provided outputs without
    bounds checks, so the binding rejects a wrong shape, dtype or rank before
    anything reaches the library (host tensors: the checks come before the
    device check)."""
    import torch

    import late_interaction_retrieval_maxsim_gb300 as m
    Q = torch.zeros((2, 40, 128), dtype=torch.float16)
    D = torch.zeros((100, 128), dtype=torch.float16)
    ql = torch.tensor([40, 3], dtype=torch.int32)
    cu = torch.tensor([0, 60, 100], dtype=torch.int32)
    ok_s = torch.zeros((2, 2))
    cases = [
        (dict(scores=torch.zeros((2, 1))), ValueError, "scores must have shape"),
        (dict(scores=torch.zeros((2, 2), dtype=torch.float64)), TypeError, "scores must be"),
        (dict(scores=ok_s, argmax=torch.zeros((2, 2, 39), dtype=torch.int32)), ValueError, "argmax must have shape"),
        (dict(scores=ok_s, argmax=torch.zeros((2, 2, 40), dtype=torch.int64)), TypeError, "argmax must be"),
        (dict(scores=ok_s, raw_scores=torch.zeros((1, 2), dtype=torch.int64)), ValueError, "raw_scores must have"),
        (dict(scores=ok_s, raw_scores=torch.zeros((2, 2), dtype=torch.int32)), TypeError, "raw_scores must be"),
        (dict(scores=torch.zeros((4, 2))[::2]), ValueError, "contiguous"),
    ]
    for kw, exc, msg in cases:
        with pytest.raises(exc, match=msg):
            m.maxsim_forward_noalloc(Q, ql, D, cu, **kw)
    with pytest.raises(ValueError, match="Q must be"):
        m.maxsim_forward_noalloc(Q[0], ql, D, cu, ok_s)
    with pytest.raises(ValueError, match="Q must be"):
        m.maxsim_forward_noalloc(Q, ql, D[:, :64], cu, ok_s)
    # well-formed outputs get as far as the device check
    with pytest.raises(ValueError, match="CUDA device"):
        m.maxsim_forward_noalloc(Q, ql, D, cu, ok_s, argmax=torch.zeros((2, 2, 40), dtype=torch.int32))
    # the allocating forward checks caller-provided outputs the same way
    with pytest.raises(ValueError, match="scores must have shape"):
        m.maxsim_forward(Q, ql, D, cu, scores=torch.zeros((3, 2)))


def test_l2_probe_rejects_bad_arguments(lib):
    """Argument errors return before any device work."""
    vp = ctypes.c_void_p
    p = lib.maxsim_probe_l2_read
    assert p(None, 1 << 20, 1, vp(256), None) == 1        # no buffer
    assert p(vp(256), 1 << 20, 1, None, None) == 1        # no sink
    assert p(vp(264), 1 << 20, 1, vp(256), None) == 1     # buffer off a 16-byte boundary
    assert p(vp(256), 1000, 1, vp(256), None) == 1        # not a multiple of 16 bytes
    assert p(vp(256), 1 << 20, 0, vp(256), None) == 1     # no pass
