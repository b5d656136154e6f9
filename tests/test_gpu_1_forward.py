"""GPU parity of the fused forward (FP16/BF16) against the CPU oracle,
through the C ABI.  Flash-MaxSim §4.1 (Alg. 2), §4.1.1, §4.3.2."""
import numpy as np
import pytest
import torch

import oracle
from late_interaction_retrieval_maxsim_gb300 import synthetic as syn
from maxsim_testlib import check_forward, random_case

pytestmark = pytest.mark.gpu


def test_tiny_workload_every_pair(ops):
    """1 query Lq=32 vs 256 docs Ld=128, FP16, seed 0: all 256 scores and the
    [256, 32] argmax."""
    x = syn.make_inputs(syn.WORKLOADS["tiny"], device="cuda")
    scores, argmax, _ = ops.maxsim_forward(x["Q"], x["q_lens"], x["D"], x["cu_seqlens"])
    assert ops.maxsim_device_status() == 0
    check_forward("fp16", x["Q"], x["q_lens"], x["D"], x["cu_seqlens"], scores, argmax)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("lq_max,q_lens", [
    (1, [1, 0, 1]),
    (7, [7, 3, 1, 0]),
    (31, [31, 16]),
    (32, [32, 1, 31, 32, 5]),
    (33, [33, 32, 1]),
    (64, [64, 40]),
    (100, [100, 99, 33, 0]),
])
def test_edge_shapes_ragged(ops, dtype, lq_max, q_lens):
    """Ragged documents straddling tile and chunk edges, empty documents,
    padded and empty queries."""
    lengths = [1, 15, 16, 17, 0, 31, 32, 33, 127, 128, 129, 0, 255, 256, 257, 3, 511, 2]
    Q, ql, D, cu = random_case(len(q_lens), lq_max, lengths, dtype, q_lens, seed=lq_max)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert ops.maxsim_device_status() == 0
    check_forward(dtype, Q, ql, D, cu, scores, argmax)


def test_long_query_split_across_groups(ops):
    """Lq = 1024 and 1000: a query spans two CTAs' row groups; partial sums
    per 32-token chunk are combined in order."""
    lengths = [1024, 700, 1, 1300, 0, 129]
    Q, ql, D, cu = random_case(2, 1024, lengths, "fp16", [1024, 1000], seed=5)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert ops.maxsim_device_status() == 0
    check_forward("fp16", Q, ql, D, cu, scores, argmax)


def test_many_queries_several_groups(ops):
    """40 queries x 32 tokens = 1280 padded rows: three row groups."""
    rng = np.random.default_rng(3)
    lengths = rng.integers(1, 300, 60).tolist()
    q_lens = rng.integers(0, 33, 40).tolist()
    Q, ql, D, cu = random_case(40, 32, lengths, "bf16", q_lens, seed=9)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert ops.maxsim_device_status() == 0
    check_forward("bf16", Q, ql, D, cu, scores, argmax)


@pytest.mark.parametrize("n_q", [9, 12, 16, 20])
def test_row_group_shapes(ops, n_q):
    """Row counts that pick each M-tile layout: 288 and 384 padded rows run
    one four-M-tile CTA per SM with one or more empty M-tiles; 512 and 640
    rows run two CTAs of two M-tiles per SM, 640 with a half-empty last
    group.  Ragged documents and queries, with and without the argmax."""
    rng = np.random.default_rng(40 + n_q)
    lengths = rng.integers(0, 400, 300).tolist()
    q_lens = rng.integers(1, 33, n_q).tolist()
    q_lens[-1] = 32
    Q, ql, D, cu = random_case(n_q, 32, lengths, "fp16", q_lens, seed=n_q)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert ops.maxsim_device_status() == 0
    check_forward("fp16", Q, ql, D, cu, scores, argmax)
    s2, _, _ = ops.maxsim_forward(Q, ql, D, cu, with_argmax=False)
    assert torch.equal(scores, s2)


def test_without_argmax_same_scores(ops):
    Q, ql, D, cu = random_case(3, 32, [100, 7, 300, 129, 0, 64], "fp16", [32, 20, 1], seed=2)
    s1, a1, _ = ops.maxsim_forward(Q, ql, D, cu)
    s2, a2, _ = ops.maxsim_forward(Q, ql, D, cu, with_argmax=False)
    assert a2 is None
    assert torch.equal(s1, s2)


def test_run_to_run_bitwise(ops):
    Q, ql, D, cu = random_case(5, 48, [200, 33, 512, 1, 90] * 20, "bf16", [48, 47, 1, 32, 0], seed=4)
    s1, a1, _ = ops.maxsim_forward(Q, ql, D, cu)
    s2, a2, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert torch.equal(s1, s2) and torch.equal(a1, a2)


def test_closed_form_exact_copies(ops):
    """D holds exact copies of the unit-norm query rows (four +-0.5 entries):
    the score is exactly Lq and each argmax is the copy's position."""
    rng = np.random.default_rng(11)
    lq, ld = 32, 300
    rows = []
    seen = set()
    while len(rows) < lq + ld:
        idx = tuple(sorted(rng.choice(128, 4, replace=False).tolist()))
        sg = tuple(rng.choice([-1, 1], 4).tolist())
        if (idx, sg) in seen:
            continue
        seen.add((idx, sg))
        v = np.zeros(128)
        v[list(idx)] = 0.5 * np.array(sg)
        rows.append(v)
    rows = np.array(rows)
    Qh = rows[:lq]
    Dh = rows[lq:].copy()
    pos = rng.choice(ld, lq, replace=False)
    Dh[pos] = Qh
    Q = torch.tensor(Qh, dtype=torch.float16, device="cuda").view(1, lq, 128)
    D = torch.tensor(np.concatenate([Dh, Dh]), dtype=torch.float16, device="cuda")
    cu = torch.tensor([0, ld, 2 * ld], dtype=torch.int32, device="cuda")
    ql = torch.tensor([lq], dtype=torch.int32, device="cuda")
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert scores.cpu().tolist() == [[float(lq), float(lq)]]
    assert np.array_equal(argmax[0, 0].cpu().numpy(), pos)
    assert np.array_equal(argmax[0, 1].cpu().numpy(), pos)


def test_one_hot_ties_lowest_index(ops):
    """One-hot rows: values are 0/1, so ties are everywhere; every argmax must
    be the first matching token, or 0 when nothing matches."""
    rng = np.random.default_rng(12)
    lq, ld = 32, 200
    a = rng.integers(0, 128, lq)
    c = rng.integers(0, 128, ld)
    Qh = np.zeros((lq, 128)); Qh[np.arange(lq), a] = 1
    Dh = np.zeros((ld, 128)); Dh[np.arange(ld), c] = 1
    Q = torch.tensor(Qh, dtype=torch.bfloat16, device="cuda").view(1, lq, 128)
    D = torch.tensor(Dh, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, ld], dtype=torch.int32, device="cuda")
    ql = torch.tensor([lq], dtype=torch.int32, device="cuda")
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    expect = sum(1 for ai in a if ai in set(c.tolist()))
    assert scores.item() == float(expect)
    for i, ai in enumerate(a):
        hits = np.nonzero(c == ai)[0]
        assert argmax[0, 0, i].item() == (hits[0] if hits.size else 0)


def test_all_documents_empty(ops):
    Q, ql, D, cu = random_case(2, 8, [0, 0, 0], "fp16", [8, 0])
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    s = scores.cpu().numpy()
    assert np.all(np.isneginf(s[0])) and np.all(s[1] == 0)
    assert torch.all(argmax == -1)


def test_colbert_varlen_full_size_sampled(ops):
    """16 queries Lq=32 vs 50,000 packed docs Ld~U[32,300], FP16 (the
    launch the benchmark times); 48 sampled documents against every query."""
    x = syn.make_inputs(syn.WORKLOADS["colbert_varlen"], device="cuda")
    scores, argmax, _ = ops.maxsim_forward(x["Q"], x["q_lens"], x["D"], x["cu_seqlens"])
    assert ops.maxsim_device_status() == 0
    rng = np.random.default_rng(0)
    docs = sorted(set(rng.integers(0, 50_000, 44).tolist()) | {0, 1, 49_998, 49_999})
    check_forward("fp16", x["Q"], x["q_lens"], x["D"], x["cu_seqlens"], scores, argmax, docs=docs)
    # invariants over every pair: unit vectors bound each score by Lq
    assert torch.all(scores <= 32.0 + 1e-3) and torch.all(scores > 0)


def test_colpali_full_size_sampled(ops):
    """1 query Lq=1024 vs 10,000 docs Ld=1024, FP16; 12 sampled documents."""
    x = syn.make_inputs(syn.WORKLOADS["colpali"], device="cuda")
    scores, argmax, _ = ops.maxsim_forward(x["Q"], x["q_lens"], x["D"], x["cu_seqlens"])
    assert ops.maxsim_device_status() == 0
    docs = [0, 1, 37, 2500, 5003, 7777, 9998, 9999, 75, 76, 151, 152]
    check_forward("fp16", x["Q"], x["q_lens"], x["D"], x["cu_seqlens"], scores, argmax, docs=docs)
    assert torch.all(scores <= 1024.0 + 1e-2)


def test_training_forward_every_pair(ops):
    """256 queries Lq=32 x 256 docs Ld=180, BF16: all 65,536 pairs."""
    x = syn.make_inputs(syn.WORKLOADS["train"], device="cuda")
    scores, argmax, _ = ops.maxsim_forward(x["Q"], x["q_lens"], x["D"], x["cu_seqlens"])
    assert ops.maxsim_device_status() == 0
    check_forward("bf16", x["Q"], x["q_lens"], x["D"], x["cu_seqlens"], scores, argmax)


def _pow2_bf16_case(seed):
    """BF16 inputs built from powers of two whose dot products are exact in
    FP32: every query row is (2^-40, 2^-40, 2^-40, 0, ...).  "Peak" documents
    hold the largest value 2^-77 = <q, (2^-37, 0, ...)> at column m and, at a
    lower column p, its float predecessor 2^-77 - 2^-101 =
    <q, (255 * 2^-45, 255 * 2^-53, 255 * 2^-61, 0, ...)> (three products of
    255 * 2^-85, 2^-93, 2^-101: 24 bits in all); their other tokens are zero.
    "Filler" documents between them hold 2^-70 everywhere, so a document
    boundary inside a 32-column chunk meets a right-hand maximum in the
    range of the fast indicator.  Exact ties and values make the argmax
    unique: it must be m, bit for bit."""
    rng = np.random.default_rng(seed)
    q = np.zeros(128)
    q[:3] = 2.0 ** -40
    top = np.zeros(128)
    top[0] = 2.0 ** -37
    pred = np.zeros(128)
    pred[:3] = [255 * 2.0 ** -45, 255 * 2.0 ** -53, 255 * 2.0 ** -61]
    fill = np.zeros(128)
    fill[0] = 2.0 ** -30
    rows, lengths, expect = [], [], []
    for k in range(120):
        if k % 2 == 0:
            ld = int(rng.integers(2, 90))
            p = int(rng.integers(0, ld - 1))
            m = p + 1 if rng.random() < 0.7 else int(rng.integers(p + 1, ld))
            doc = np.zeros((ld, 128))
            doc[p] = pred
            doc[m] = top
            expect.append(m)
        else:
            ld = int(rng.integers(1, 40))
            doc = np.tile(fill, (ld, 1))
            expect.append(0)
        rows.append(doc)
        lengths.append(ld)
    D = torch.tensor(np.concatenate(rows), dtype=torch.bfloat16, device="cuda")
    Q = torch.tensor(np.tile(q, (32, 1)), dtype=torch.bfloat16, device="cuda").view(1, 32, 128)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device="cuda")
    ql = torch.tensor([32], dtype=torch.int32, device="cuda")
    # the stored values are the intended powers of two
    assert float(D[cu[0] + int(np.argmax(rows[0][:, 0] == 2.0 ** -37)), 0]) == 2.0 ** -37
    return Q, ql, D, cu, np.array(expect)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_argmax_exact_at_tiny_power_of_two_maxima(ops, seed):
    """A row maximum of exactly 2^-77 next to its float predecessor: the
    exact argmax search must tell them apart (a fast-path bound one binade
    too low reports the predecessor or a zero column).  Argmax bit-exact
    against the oracle; scores exact (sums of powers of two)."""
    Q, ql, D, cu, expect = _pow2_bf16_case(seed)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert ops.maxsim_device_status() == 0
    ref = oracle.forward_bits("bf16", syn.bits_u16(Q), ql.cpu().numpy(), syn.bits_u16(D), cu.cpu().numpy())
    assert np.array_equal(ref["argmax"][:, 0], expect)           # the construction is what it claims
    assert np.array_equal(argmax[0].cpu().numpy(), ref["argmax"])
    assert np.array_equal(scores[0].double().cpu().numpy(), ref["score"])


@pytest.mark.parametrize("n_q,lq_max", [(1, 32), (4, 8), (3, 32)])
def test_split_column_epilogue_many_tiny_documents(ops, n_q, lq_max):
    """Up to 128 query rows run two epilogue warps per TMEM lane quarter,
    each folding half of every tile's columns, merged per document: 600
    documents of 0-5 tokens (many document ends per chunk, so the merge
    buffer fills in the middle of a chunk) plus a few long ones, every pair
    checked; bits identical run to run."""
    rng = np.random.default_rng(70 + n_q)
    lengths = rng.integers(0, 6, 600).tolist()
    lengths[100] = 300
    lengths[400] = 129
    q_lens = [lq_max] + rng.integers(0, lq_max + 1, n_q - 1).tolist()
    Q, ql, D, cu = random_case(n_q, lq_max, lengths, "bf16", q_lens, seed=80 + n_q)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert ops.maxsim_device_status() == 0
    check_forward("bf16", Q, ql, D, cu, scores, argmax)
    s2, a2, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert torch.equal(scores, s2) and torch.equal(argmax, a2)


def test_split_column_epilogue_ties_across_halves(ops):
    """Equal maxima in both column halves of a tile (the same document token
    repeated at columns t and t + 64): the merge keeps the lower column."""
    rng = np.random.default_rng(13)
    lq, ld = 32, 256
    Qh = rng.standard_normal((lq, 128))
    Qh /= np.linalg.norm(Qh, axis=1, keepdims=True)
    Dh = rng.standard_normal((ld, 128))
    Dh /= np.linalg.norm(Dh, axis=1, keepdims=True)
    hot = rng.choice(64, lq, replace=False)
    Dh[hot] = Qh                   # each query token's best match in the first half ...
    Dh[hot + 64] = Qh              # ... repeated 64 columns later (second half)
    Dh[hot + 192] = Qh             # and in the next tile's second half
    Q = torch.tensor(Qh, dtype=torch.float16, device="cuda").view(1, lq, 128)
    D = torch.tensor(Dh, dtype=torch.float16, device="cuda")
    cu = torch.tensor([0, ld], dtype=torch.int32, device="cuda")
    ql = torch.tensor([lq], dtype=torch.int32, device="cuda")
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert ops.maxsim_device_status() == 0
    assert np.array_equal(argmax[0, 0].cpu().numpy(), hot)
    check_forward("fp16", Q, ql, D, cu, scores, argmax)


def test_single_query_full_size_sampled(ops):
    """1 query Lq=32 vs the 50,000 ColBERT documents (the single-query launch
    the benchmark times: one M-tile, split-column epilogue); 48 sampled
    documents."""
    x = syn.make_inputs(syn.WORKLOADS["colbert_1q"], device="cuda")
    scores, argmax, _ = ops.maxsim_forward(x["Q"], x["q_lens"], x["D"], x["cu_seqlens"])
    assert ops.maxsim_device_status() == 0
    rng = np.random.default_rng(1)
    docs = sorted(set(rng.integers(0, 50_000, 44).tolist()) | {0, 1, 49_998, 49_999})
    check_forward("fp16", x["Q"], x["q_lens"], x["D"], x["cu_seqlens"], scores, argmax, docs=docs)
