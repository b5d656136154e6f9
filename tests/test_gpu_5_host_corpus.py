"""Out-of-core scoring (Flash-MaxSim §5 "Out-of-Core Corpus Scaling"): the
corpus stays in host memory and is streamed to the device in blocks of
documents.  A document's score does not depend on which other documents
share a launch, so the streamed forward must give the same bits as the
in-HBM forward over the whole corpus, and both agree with the oracle."""
import numpy as np
import pytest
import torch

from maxsim_testlib import check_forward, random_case

pytestmark = pytest.mark.gpu


def _host(ops, Q, ql, D, cu, pinned=True, **kw):
    D_h = D.cpu()
    if pinned:
        D_h = D_h.pin_memory()
    cu_h = cu.cpu()
    out = ops.maxsim_forward_host(Q, ql, D_h, cu_h, **kw)
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    return out


LENGTHS = [1, 130, 0, 257, 64, 500, 3, 33, 0, 128, 129, 7] * 3


@pytest.mark.parametrize("block_docs,block_tokens,overlap", [
    (1, 512, True), (3, 600, True), (5, 1000, False), (36, 512, True), (1000, 100000, True)])
def test_streamed_equals_resident_fp16(ops, block_docs, block_tokens, overlap):
    Q, ql, D, cu = random_case(4, 32, LENGTHS, "fp16", [32, 17, 1, 0], seed=91)
    ref_s, ref_a, _ = ops.maxsim_forward(Q, ql, D, cu)
    s, a, _ = _host(ops, Q, ql, D, cu, block_docs=block_docs, block_tokens=block_tokens,
                    with_argmax=True, overlap=overlap)
    assert torch.equal(s, ref_s) and torch.equal(a, ref_a)


def test_streamed_long_queries_bf16_matches_oracle(ops):
    """Queries of more than 32 tokens go through per-chunk partial sums,
    whose scratch is shared by all blocks."""
    Q, ql, D, cu = random_case(2, 100, LENGTHS, "bf16", [100, 45], seed=92)
    ref_s, ref_a, _ = ops.maxsim_forward(Q, ql, D, cu)
    s, a, _ = _host(ops, Q, ql, D, cu, block_docs=4, block_tokens=700, with_argmax=True)
    assert torch.equal(s, ref_s) and torch.equal(a, ref_a)
    check_forward("bf16", Q, ql, D, cu, s, a)


def test_streamed_pageable_host_memory(ops):
    Q, ql, D, cu = random_case(3, 32, LENGTHS, "fp16", seed=93)
    ref_s, _, _ = ops.maxsim_forward(Q, ql, D, cu, with_argmax=False)
    s, a, _ = _host(ops, Q, ql, D, cu, pinned=False, block_docs=7, block_tokens=800)
    assert a is None and torch.equal(s, ref_s)


def test_streamed_int8_bit_exact(ops):
    rng = np.random.default_rng(94)
    lengths = [40, 1, 300, 0, 129, 77, 512, 2]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device="cuda")
    Q = torch.from_numpy(rng.integers(-127, 128, (3, 70, 128)).astype(np.int8)).cuda()
    D = torch.from_numpy(rng.integers(-127, 128, (sum(lengths), 128)).astype(np.int8)).cuda()
    ql = torch.tensor([70, 35, 1], dtype=torch.int32, device="cuda")
    ref = ops.maxsim_forward(Q, ql, D, cu, q_scale=0.01, d_scale=0.02, want_raw=True)
    out = _host(ops, Q, ql, D, cu, block_docs=3, block_tokens=600, with_argmax=True, q_scale=0.01,
                d_scale=0.02, want_raw=True)
    for x, y in zip(out, ref):
        assert torch.equal(x, y)


def test_streamed_block_of_empty_documents(ops):
    """Blocks {0, 1}, {2, 3}, {4}: the middle one has no token and takes the
    no-token path."""
    lengths = [5, 9, 0, 0, 9]
    Q, ql, D, cu = random_case(2, 8, lengths, "fp16", [8, 0], seed=95)
    ref_s, ref_a, _ = ops.maxsim_forward(Q, ql, D, cu)
    s, a, _ = _host(ops, Q, ql, D, cu, block_docs=2, block_tokens=14, with_argmax=True)
    assert torch.equal(s, ref_s) and torch.equal(a, ref_a)
    assert torch.isinf(s[0, 2:4]).all() and (s[1] == 0).all()


def test_streamed_rejects_a_document_longer_than_a_block(ops):
    Q, ql, D, cu = random_case(1, 8, [10, 300], "fp16", seed=96)
    with pytest.raises(ops.MaxSimError):
        ops.maxsim_forward_host(Q, ql, D.cpu(), cu.cpu(), block_docs=4, block_tokens=256)
