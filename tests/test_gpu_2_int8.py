"""GPU INT8 x INT8 forward: bit-exact against the oracle's int64 arithmetic
(Flash-MaxSim §4.3.1, one symmetric scale per tensor)."""
import numpy as np
import pytest
import torch

import oracle
from late_interaction_retrieval_maxsim_gb300 import synthetic as syn
from maxsim_testlib import THREADS

pytestmark = pytest.mark.gpu


def _run_and_check(ops, Q, ql, D, cu, qs, ds, docs=None):
    scores, argmax, raw = ops.maxsim_forward(Q, ql, D, cu, q_scale=qs, d_scale=ds, want_raw=True)
    assert ops.maxsim_device_status() == 0
    n_docs = cu.numel() - 1
    docs = list(range(n_docs)) if docs is None else docs
    cu_h = cu.cpu().numpy()
    Dh = torch.cat([D[int(cu_h[b]):int(cu_h[b + 1])] for b in docs]).cpu().numpy() if docs else \
        np.zeros((0, 128), np.int8)
    lens = [int(cu_h[b + 1] - cu_h[b]) for b in docs]
    cu_sub = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ref = oracle.forward_i8(Q.cpu().numpy(), ql.cpu().numpy(), Dh, cu_sub, qs, ds, threads=THREADS)
    P = Q.shape[0] * len(docs)
    assert np.array_equal(raw[:, docs].cpu().numpy().reshape(P), ref["raw"])
    assert np.array_equal(scores[:, docs].cpu().numpy().reshape(P), ref["score"])
    assert np.array_equal(argmax[:, docs].cpu().numpy().reshape(P, Q.shape[1]), ref["argmax"])
    return scores, argmax, raw


def _rand_i8(shape, rng):
    return torch.from_numpy(rng.integers(-127, 128, shape).astype(np.int8)).cuda()


@pytest.mark.parametrize("lq_max,q_lens", [(32, [32, 17, 0, 1]), (8, [8, 3]), (100, [100, 64, 1])])
def test_random_ragged_bit_exact(ops, lq_max, q_lens):
    rng = np.random.default_rng(lq_max)
    lengths = [1, 15, 16, 17, 0, 127, 128, 129, 255, 256, 257, 3, 400]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32).cuda()
    Q = _rand_i8((len(q_lens), lq_max, 128), rng)
    D = _rand_i8((sum(lengths), 128), rng)
    ql = torch.tensor(q_lens, dtype=torch.int32).cuda()
    _run_and_check(ops, Q, ql, D, cu, np.float32(0.0037), np.float32(0.0041))


def test_extreme_magnitudes(ops):
    """All entries +-127: |dot| reaches 128 * 127^2 = 2,064,512."""
    Q = torch.full((2, 32, 128), 127, dtype=torch.int8)
    Q[1] = -127
    Q[0, 5:9] = -127
    D = torch.full((300, 128), 127, dtype=torch.int8)
    D[7] = -127
    D[150:, ::2] = -127
    cu = torch.tensor([0, 100, 300], dtype=torch.int32)
    ql = torch.tensor([32, 30], dtype=torch.int32)
    _, _, raw = _run_and_check(ops, Q.cuda(), ql.cuda(), D.cuda(), cu.cuda(), np.float32(1.0), np.float32(1.0))
    assert raw[0, 0].item() == 32 * 2064512


def test_ties_lowest_index(ops):
    rng = np.random.default_rng(5)
    Q = _rand_i8((1, 32, 128), rng)
    row = _rand_i8((1, 128), rng)
    D = row.repeat(260, 1)
    cu = torch.tensor([0, 130, 260], dtype=torch.int32).cuda()
    ql = torch.tensor([32], dtype=torch.int32).cuda()
    _, argmax, _ = _run_and_check(ops, Q, ql, D, cu, np.float32(0.5), np.float32(0.25))
    assert torch.all(argmax == 0)


def test_int8_varlen_full_size_sampled(ops):
    """32 queries Lq=32 vs 100,000 docs Ld~U[32,512], per-tensor scales;
    48 sampled documents bit-exact."""
    x = syn.make_inputs(syn.WORKLOADS["int8_varlen"], device="cuda")
    rng = np.random.default_rng(1)
    docs = sorted(set(rng.integers(0, 100_000, 44).tolist()) | {0, 1, 99_998, 99_999})
    _run_and_check(ops, x["Q"], x["q_lens"], x["D"], x["cu_seqlens"], x["q_scale"], x["d_scale"], docs=docs)
