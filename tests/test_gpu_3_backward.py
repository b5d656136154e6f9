"""GPU backward: inverse-grid CSR bit-exact against the oracle, dQ / dD
within 1e-4 of max|grad| (Flash-MaxSim §4.2, Eqs. (2)-(3), Alg. 3)."""
import numpy as np
import pytest
import torch

import oracle
from late_interaction_retrieval_maxsim_gb300 import synthetic as syn
from maxsim_testlib import GRAD_TOL, random_case

pytestmark = pytest.mark.gpu


def _contrastive_grad(scores):
    """grad = softmax(scores / 0.05) - onehot(diagonal), row-wise (the
    in-batch-negatives workload's synthetic upstream gradient)."""
    n = scores.shape[0]
    g = torch.softmax(scores / 0.05, dim=1)
    g[torch.arange(n), torch.arange(n) % scores.shape[1]] -= 1.0
    return g.contiguous()


def _check_csr(ops, argmax, ql, cu, total):
    row_ptr, col_idx = ops.maxsim_build_csr(argmax, ql, cu, total)
    assert ops.maxsim_device_status() == 0
    rp, ci = oracle.build_csr(argmax.cpu().numpy(), ql.cpu().numpy(), cu.cpu().numpy())
    assert np.array_equal(row_ptr.cpu().numpy().astype(np.int64), rp)
    assert np.array_equal(col_idx.cpu().numpy().astype(np.int64), ci)


def _check_backward(ops, g, argmax, Q, ql, D, cu, dtype):
    dQ, dD = ops.maxsim_backward(g, argmax, Q, ql, D, cu)
    assert ops.maxsim_device_status() == 0
    qd = oracle.decode(dtype, syn.bits_u16(Q))
    dd = oracle.decode(dtype, syn.bits_u16(D))
    rq, rd = oracle.backward_f64(g.double().cpu().numpy(), argmax.cpu().numpy(), qd,
                                 ql.cpu().numpy(), dd, cu.cpu().numpy())
    for got, want in ((dQ, rq), (dD, rd)):
        scale = float(np.abs(want).max())
        err = float(np.abs(got.double().cpu().numpy() - want).max())
        assert err <= GRAD_TOL * scale, f"gradient error {err:.3e} (max |grad| {scale:.3e})"
    return dQ, dD


def test_training_workload_csr_and_gradients(ops):
    """256 queries Lq=32 x 256 docs Ld=180, BF16: forward, contrastive grad,
    CSR (bit-exact) and dQ / dD."""
    x = syn.make_inputs(syn.WORKLOADS["train"], device="cuda")
    Q, ql, D, cu = x["Q"], x["q_lens"], x["D"], x["cu_seqlens"]
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    g = _contrastive_grad(scores)
    _check_csr(ops, argmax, ql, cu, D.shape[0])
    dQ, dD = _check_backward(ops, g, argmax, Q, ql, D, cu, "bf16")
    # deterministic: a second run gives the same bits
    dQ2, dD2 = ops.maxsim_backward(g, argmax, Q, ql, D, cu)
    assert torch.equal(dQ, dQ2) and torch.equal(dD, dD2)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_ragged_with_empty_docs_and_padding(ops, dtype):
    lengths = [5, 0, 130, 1, 257, 0, 33]
    Q, ql, D, cu = random_case(4, 40, lengths, dtype, [40, 0, 17, 33], seed=21)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    scores = torch.where(torch.isfinite(scores), scores, torch.zeros_like(scores))
    g = torch.randn(scores.shape, device="cuda", generator=torch.Generator("cuda").manual_seed(3))
    _check_csr(ops, argmax, ql, cu, D.shape[0])
    dQ, dD = _check_backward(ops, g, argmax, Q, ql, D, cu, dtype)
    assert torch.all(dQ[1] == 0) and torch.all(dQ[2, 17:] == 0)


def test_long_queries_colpali_like(ops):
    """Queries of hundreds of tokens against page-length documents (the
    ColPali training shape of Flash-MaxSim §5 "Training Step", scaled down):
    CSR bit-exact, dQ / dD within tolerance."""
    lengths = [700, 1024, 3, 512, 1000, 257]
    Q, ql, D, cu = random_case(6, 300, lengths, "bf16", [300, 1, 129, 257, 32, 300], seed=41)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    g = _contrastive_grad(scores)
    _check_csr(ops, argmax, ql, cu, D.shape[0])
    _check_backward(ops, g, argmax, Q, ql, D, cu, "bf16")


def test_csr_documents_split_into_chunks(ops):
    """16 queries x 1024 tokens: each document's 16,384 candidate sources are
    split into several chunks placed by separate CTAs; the CSR must still be
    the unique stable argsort (hot tokens make many sources share a row
    across chunk borders)."""
    lengths = [1024] * 10 + [3, 700, 1]
    Q, ql, D, cu = random_case(16, 1024, lengths, "bf16", [1024] * 8 + [1000, 1, 0, 512] + [700] * 4, seed=43)
    D[cu[0]:cu[0] + 4] = Q[0, :4]            # a few document tokens that many query tokens pick
    _, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    _check_csr(ops, argmax, ql, cu, D.shape[0])
    g = torch.randn((16, len(lengths)), device="cuda", generator=torch.Generator("cuda").manual_seed(4))
    _check_backward(ops, g, argmax, Q, ql, D, cu, "bf16")


def test_many_candidates_several_sort_chunks(ops):
    """20,480 candidates per document (40 queries x 512 tokens): the
    backward sorts each document's sources in five chunks whose runs dD reads
    as one list; CSR bit-exact, gradients within tolerance, identical bits
    on a second run."""
    lengths = [300, 1024, 1, 0, 700, 129, 2000]
    q_lens = [512, 500, 1, 0, 256, 512, 33, 400] * 5
    Q, ql, D, cu = random_case(40, 512, lengths, "bf16", q_lens, seed=61)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    g = _contrastive_grad(torch.where(torch.isfinite(scores), scores, torch.zeros_like(scores)))
    _check_csr(ops, argmax, ql, cu, D.shape[0])
    dQ, dD = _check_backward(ops, g, argmax, Q, ql, D, cu, "bf16")
    dQ2, dD2 = ops.maxsim_backward(g, argmax, Q, ql, D, cu)
    assert torch.equal(dQ, dQ2) and torch.equal(dD, dD2)


def test_sort_long_documents_windows(ops):
    """The backward's per-document sort on documents longer than its
    256-token window, one of them longer than 4,096 tokens, with a few hot
    tokens: gradients within tolerance, bits identical run to run."""
    lengths = [5000, 257, 256, 255, 1, 0, 3000]
    Q, ql, D, cu = random_case(12, 64, lengths, "fp16", [64, 1, 0, 63] * 3, seed=62)
    D[cu[0] + 4000:cu[0] + 4004] = Q[0, :4]
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    g = torch.randn(scores.shape, device="cuda", generator=torch.Generator("cuda").manual_seed(6))
    dQ, dD = _check_backward(ops, g, argmax, Q, ql, D, cu, "fp16")
    dQ2, dD2 = ops.maxsim_backward(g, argmax, Q, ql, D, cu)
    assert torch.equal(dQ, dQ2) and torch.equal(dD, dD2)


def test_hot_tokens_skewed_argmax(ops):
    """A skewed winner map (half the rows pick token 0 of their document):
    the CSR keeps ascending source order inside each hot row."""
    rng = np.random.default_rng(8)
    lengths = [180] * 64
    Q, ql, D, cu = random_case(128, 32, lengths, "bf16", seed=31)
    am = np.where(rng.random((128, 64, 32)) < 0.5, 0, rng.integers(0, 180, (128, 64, 32)))
    argmax = torch.tensor(am, dtype=torch.int32, device="cuda")
    _check_csr(ops, argmax, ql, cu, D.shape[0])
    g = torch.randn((128, 64), device="cuda", generator=torch.Generator("cuda").manual_seed(4))
    _check_backward(ops, g, argmax, Q, ql, D, cu, "bf16")


def test_out_of_range_argmax_is_reported(ops):
    """An argmax entry outside its document is skipped by the bounds check
    and reported through the device status word."""
    Q, ql, D, cu = random_case(2, 4, [10, 6], "fp16", [4, 4], seed=2)
    argmax = torch.zeros((2, 2, 4), dtype=torch.int32, device="cuda")
    argmax[1, 1, 2] = 6          # document 1 has tokens 0..5
    ops.maxsim_build_csr(argmax, ql, cu, D.shape[0])
    assert ops.maxsim_device_status(clear=True) == 0x201
    assert ops.maxsim_device_status() == 0


def _counted_matches_plain(ops, Q, ql, D, cu):
    s0, a0, _ = ops.maxsim_forward(Q, ql, D, cu)
    s1, a1, bws = ops.maxsim_forward_with_counts(Q, ql, D, cu)
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    assert torch.equal(s0, s1) and torch.equal(a0, a1)
    g = torch.where(torch.isfinite(s0), s0, torch.zeros_like(s0))
    g = torch.softmax(g / 0.05, dim=1).contiguous()
    dq0, dd0 = ops.maxsim_backward(g, a0, Q, ql, D, cu)
    dq1, dd1 = ops.maxsim_backward_with_counts(g, a1, Q, ql, D, cu, bws)
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    assert torch.equal(dq0, dq1) and torch.equal(dd0, dd1)


@pytest.mark.parametrize("case", ["train", "ragged", "long"])
def test_training_pair_names_equal_the_plain_pair(ops, case):
    """maxsim_forward_with_counts / maxsim_backward_with_counts (the
    training pair under its earlier names; the backward now sorts each
    document's sources itself) give the same bits as maxsim_forward /
    maxsim_backward."""
    if case == "train":
        x = syn.make_inputs(syn.WORKLOADS["train"], device="cuda")
        Q, ql, D, cu = x["Q"], x["q_lens"], x["D"], x["cu_seqlens"]
    elif case == "ragged":
        Q, ql, D, cu = random_case(4, 40, [5, 0, 130, 1, 257, 0, 33], "fp16", [40, 0, 17, 33], seed=51)
    else:
        Q, ql, D, cu = random_case(3, 300, [700, 64, 3, 1024], "bf16", [300, 129, 1], seed=52)
    _counted_matches_plain(ops, Q, ql, D, cu)


def test_out_of_range_argmax_in_backward_contributes_nothing(ops):
    """maxsim_backward with an argmax entry outside its document: the status
    word reports it and both gradients equal the oracle's for the same
    argmax with that entry dropped (-1)."""
    Q, ql, D, cu = random_case(3, 8, [10, 6, 40], "bf16", [8, 5, 8], seed=71)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    g = torch.randn(scores.shape, device="cuda", generator=torch.Generator("cuda").manual_seed(9))
    bad = argmax.clone()
    bad[2, 1, 3] = 6           # document 1 has tokens 0..5
    bad[0, 2, 7] = -5
    ops.maxsim_device_status(clear=True)
    dQ, dD = ops.maxsim_backward(g, bad, Q, ql, D, cu)
    torch.cuda.synchronize()
    assert ops.maxsim_device_status(clear=True) == 0x201
    dropped = bad.clone()
    dropped[2, 1, 3] = -1
    dropped[0, 2, 7] = -1
    rq, rd = oracle.backward_f64(g.double().cpu().numpy(), dropped.cpu().numpy(),
                                 oracle.decode("bf16", syn.bits_u16(Q)), ql.cpu().numpy(),
                                 oracle.decode("bf16", syn.bits_u16(D)), cu.cpu().numpy())
    for got, want in ((dQ, rq), (dD, rd)):
        assert np.abs(got.double().cpu().numpy() - want).max() <= GRAD_TOL * np.abs(want).max()
    assert ops.maxsim_device_status() == 0


def test_colpali_training_shape_full_size(ops):
    """64 queries x 1024 tokens vs 64 documents x 1024 tokens, BF16 (the
    ColPali training step bench.py times): forward on sampled pairs, then
    every dQ / dD element against the oracle, and identical bits on a
    second backward."""
    from maxsim_testlib import check_forward
    x = syn.make_inputs(syn.WORKLOADS["train_colpali"], device="cuda")
    Q, ql, D, cu = x["Q"], x["q_lens"], x["D"], x["cu_seqlens"]
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert ops.maxsim_device_status() == 0
    check_forward("bf16", Q, ql, D, cu, scores, argmax, pairs=[(0, 0), (5, 63), (63, 7), (31, 32)])
    g = _contrastive_grad(scores)
    dQ, dD = _check_backward(ops, g, argmax, Q, ql, D, cu, "bf16")
    dQ2, dD2 = ops.maxsim_backward(g, argmax, Q, ql, D, cu)
    assert torch.equal(dQ, dQ2) and torch.equal(dD, dD2)


@pytest.mark.parametrize("case", ["odd_lq", "unaligned_argmax"])
def test_sort_scalar_argmax_loads(ops, case):
    """The sort loads four argmax entries at once only when lq_max is a
    multiple of 4 and the argmax is 16-byte aligned: an odd lq_max, and an
    argmax view that starts 4 bytes into its buffer, take the one-entry path
    and give the same gradients as the oracle."""
    lq = 7 if case == "odd_lq" else 8
    Q, ql, D, cu = random_case(5, lq, [40, 3, 0, 130, 17], "fp16", [lq, 1, lq - 2, 0, lq], seed=77)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    if case == "unaligned_argmax":
        buf = torch.empty(argmax.numel() + 1, dtype=torch.int32, device="cuda")
        view = buf[1:].view(argmax.shape)
        view.copy_(argmax)
        assert view.data_ptr() % 16 != 0
        argmax = view
    g = torch.randn(scores.shape, device="cuda", generator=torch.Generator("cuda").manual_seed(12))
    _check_csr(ops, argmax.contiguous(), ql, cu, D.shape[0])
    _check_backward(ops, g, argmax, Q, ql, D, cu, "fp16")
