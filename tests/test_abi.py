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
