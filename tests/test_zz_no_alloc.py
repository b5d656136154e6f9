"""maxsim_forward_noalloc -- the forward for callers that cannot allocate
device memory (a plugin inside a host framework that owns every device
allocation, or a serving loop that must never call cudaMalloc / cudaFree
because they can synchronise the device).  Its scratch is one fixed array
owned by the library, so these tests call it through the C ABI and compare
it with maxsim_forward (which gets a caller-allocated workspace) on the same
inputs, twice in a row: the second call runs on whatever the first one left
in the shared array.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from maxsim_testlib import SCORE_TOL_PER_TOKEN, random_case

pytestmark = pytest.mark.gpu

ERR_WORKSPACE = 3


def _noalloc(lib, Q, ql, D, cu, scores, argmax=None, raw=None, qs=1.0, ds=1.0):
    vp = ctypes.c_void_p
    code = {torch.float16: 0, torch.bfloat16: 1, torch.int8: 2}[Q.dtype]
    return lib.maxsim_forward_noalloc(
        vp(Q.data_ptr()), vp(ql.data_ptr()), Q.shape[0], Q.shape[1], vp(D.data_ptr()), vp(cu.data_ptr()),
        cu.numel() - 1, D.shape[0], Q.shape[2], code, float(qs), float(ds), vp(scores.data_ptr()),
        None if raw is None else vp(raw.data_ptr()), None if argmax is None else vp(argmax.data_ptr()),
        vp(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_forward_two_calls(ops):
    """Queries longer than 32 tokens keep per-chunk partial sums in the
    scratch; two different problems in a row reuse it."""
    lib = ops.load_library()
    cases = [
        random_case(3, 100, [1, 130, 0, 257, 64, 500] * 4, "fp16", [100, 64, 33], seed=41),
        random_case(2, 1024, [1024, 700, 3, 1300], "bf16", [1024, 999], seed=42),
    ]
    for Q, ql, D, cu in cases:
        ref_s, ref_a, _ = ops.maxsim_forward(Q, ql, D, cu)
        tol = SCORE_TOL_PER_TOKEN * ql.float().clamp(min=1)[:, None]
        for _ in range(2):
            s = torch.full_like(ref_s, float("nan"))
            a = torch.full_like(ref_a, -7)
            assert _noalloc(lib, Q, ql, D, cu, s, a) == 0
            torch.cuda.synchronize()
            assert ops.maxsim_device_status() == 0
            finite = torch.isfinite(ref_s)
            assert torch.equal(torch.isfinite(s), finite)
            assert torch.all((s[finite] - ref_s[finite]).abs() <= tol.expand_as(s)[finite])
            assert torch.equal(a, ref_a)


def test_noalloc_int8_two_calls(ops):
    """INT8 keeps an FP16 copy of Q and int64 partial sums in the scratch."""
    lib = ops.load_library()
    rng = np.random.default_rng(43)
    lengths = [40, 1, 300, 0, 129]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device="cuda")
    Q = torch.from_numpy(rng.integers(-127, 128, (2, 70, 128)).astype(np.int8)).cuda()
    D = torch.from_numpy(rng.integers(-127, 128, (sum(lengths), 128)).astype(np.int8)).cuda()
    ql = torch.tensor([70, 35], dtype=torch.int32, device="cuda")
    ref_s, ref_a, ref_r = ops.maxsim_forward(Q, ql, D, cu, q_scale=0.01, d_scale=0.02, want_raw=True)
    for _ in range(2):
        s = torch.empty_like(ref_s)
        a = torch.empty_like(ref_a)
        r = torch.empty_like(ref_r)
        assert _noalloc(lib, Q, ql, D, cu, s, a, r, 0.01, 0.02) == 0
        torch.cuda.synchronize()
        assert ops.maxsim_device_status() == 0
        assert torch.equal(r, ref_r) and torch.equal(a, ref_a) and torch.equal(s, ref_s)


def test_noalloc_rejects_sizes_beyond_the_array(ops):
    """1 query x 1024 tokens x 40,000 documents needs 5.1 MB of partial sums,
    more than the 4 MiB array: refused before anything is enqueued."""
    lib = ops.load_library()
    vp = ctypes.c_void_p
    st = lib.maxsim_forward_noalloc(vp(256), vp(256), 1, 1024, vp(256), vp(256), 40_000, 40_000, 128, 0,
                                    1.0, 1.0, vp(256), None, None, None)
    assert st == ERR_WORKSPACE
