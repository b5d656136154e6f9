"""The INT8 variants of Flash-MaxSim §4.3.1 / §4.1 on the GPU against the
oracle:

  * INT8 with one scale per token against the binary64 oracle: argmax equal
    wherever the exact top-2 gap exceeds 2^-22 |max| (the kernel ranks the
    products rounded once to binary32, a monotone rounding), a near-maximum
    elsewhere; scores within 1e-4 per query token;
  * row-wise top-K: ids and values bit-exact;
  * the two-stage INT8 -> FP16 top-K scan: the stage-2 candidates exactly
    (the per-tensor INT8 stage is exact), the final ranking within the FP16
    score tolerance; the FP16 corpus in device memory or in pinned host
    memory gives the same bits."""
import numpy as np
import pytest
import torch

import oracle
from late_interaction_retrieval_maxsim_gb300 import synthetic as syn
from maxsim_testlib import SCORE_TOL_PER_TOKEN, THREADS, check_int8_token

pytestmark = pytest.mark.gpu


def _token_case(n_q, lq, lengths, q_lens=None, seed=0):
    cu = syn.cu_seqlens_from_lengths(torch.as_tensor(lengths, dtype=torch.int32))
    total = int(cu[-1])
    Q8, qs = syn.unit_tokens_int8_per_token(n_q * lq, 128, seed + 1, "cuda")
    D8, ds = syn.unit_tokens_int8_per_token(total, 128, seed + 2, "cuda")
    q_lens = torch.tensor(q_lens if q_lens is not None else [lq] * n_q, dtype=torch.int32, device="cuda")
    return Q8.view(n_q, lq, 128), qs.view(n_q, lq), q_lens, D8, ds, cu.cuda()


def _check_token(ops, Q8, qs, ql, D8, ds, cu):
    s, a = ops.maxsim_forward_int8_per_token(Q8, qs, ql, D8, ds, cu)
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    check_int8_token(Q8.cpu().numpy(), qs.cpu().numpy(), ql.cpu().numpy(), D8.cpu().numpy(), ds.cpu().numpy(),
                     cu.cpu().numpy(), s.cpu().numpy(), a.cpu().numpy())
    # the value-only instantiation gives the same scores
    s2, _ = ops.maxsim_forward_int8_per_token(Q8, qs, ql, D8, ds, cu, with_argmax=False)
    assert torch.equal(s2, s)


LENGTHS = [1, 130, 0, 257, 64, 500, 3, 33, 0, 128, 129, 7, 31, 32, 95]


@pytest.mark.parametrize("n_q,lq,q_lens", [
    (1, 32, None),              # one M-tile
    (3, 8, [8, 5, 0]),          # several queries per 32-row slice
    (6, 32, [32, 1, 17, 32, 0, 30]),   # two M-tiles
    (9, 32, None),              # four M-tiles
    (2, 70, [70, 41]),          # per-chunk partial sums
])
def test_int8_per_token_matches_oracle(ops, n_q, lq, q_lens):
    _check_token(ops, *_token_case(n_q, lq, LENGTHS * 2, q_lens, seed=n_q * 100 + lq))


def test_int8_per_token_zero_scales(ops):
    """All-zero document tokens (scale 0) rank as 0."""
    Q8, qs, ql, D8, ds, cu = _token_case(2, 32, [40, 3, 200], seed=5)
    D8[10:20] = 0
    ds[10:20] = 0
    ds[41] = 0
    _check_token(ops, Q8, qs, ql, D8, ds, cu)


@pytest.mark.parametrize("n_rows,n_cols,k", [(1, 1, 1), (3, 100, 10), (5, 5000, 1000), (2, 100_000, 4096),
                                             (4, 37, 64), (2, 4096, 4096)])
def test_topk_bit_exact(ops, n_rows, n_cols, k):
    g = torch.Generator("cuda").manual_seed(n_cols + k)
    vals = torch.randint(-50, 50, (n_rows, n_cols), generator=g, device="cuda").float() / 7.0
    vals[:, ::11] = float("-inf")
    ids, v = ops.maxsim_topk(vals, k)
    torch.cuda.synchronize()
    rid, rv = oracle.topk(vals.cpu().numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.array_equal(v.cpu().numpy(), rv.astype(np.float32))


def test_topk_strided_rows(ops):
    g = torch.Generator("cuda").manual_seed(3)
    big = torch.randn((4, 3000), generator=g, device="cuda")
    vals = big[:, 100:2100]
    ids, v = ops.maxsim_topk(vals, 300)
    rid, rv = oracle.topk(vals.cpu().numpy(), 300)
    assert np.array_equal(ids.cpu().numpy(), rid) and np.array_equal(v.cpu().numpy(), rv)


def _rerank_case(n_q, lq, n_docs, lo, hi, seed):
    lengths = syn.doc_lengths(n_docs, lo, hi, seed)
    cu = syn.cu_seqlens_from_lengths(lengths)
    total = int(cu[-1])
    Q16 = syn.unit_tokens(n_q * lq, 128, seed + 1, "fp16", "cuda").view(n_q, lq, 128)
    D16 = syn.unit_tokens(total, 128, seed + 2, "fp16", "cuda")
    Q8, qs = syn.unit_tokens_int8(n_q * lq, 128, seed + 1, "cuda")
    D8, ds = syn.unit_tokens_int8(total, 128, seed + 2, "cuda")
    ql = torch.full((n_q,), lq, dtype=torch.int32, device="cuda")
    return Q8.view(n_q, lq, 128), qs, D8, ds, Q16, D16, ql, cu.cuda()


def _check_final(ids, scores, ref, s2_ref_of, tol):
    """ids sorted by the kernel's own scores; each score within tol of the
    oracle's stage-2 score of that document; the kept set equals the
    oracle's except where the oracle's scores are within 2 tol of the cut."""
    ids, scores = ids.cpu().numpy(), scores.double().cpu().numpy()
    for q in range(ids.shape[0]):
        assert np.all(np.diff(scores[q]) <= 0)
        for j, d in enumerate(ids[q]):
            assert abs(scores[q, j] - s2_ref_of(q, d)) <= tol
        cut = ref["scores"][q, -1]
        sure = set(int(d) for d, s in zip(ref["ids"][q], ref["scores"][q]) if s > cut + 2 * tol)
        assert sure <= set(int(d) for d in ids[q])


def test_two_stage_rerank_matches_oracle(ops):
    Q8, qs, D8, ds, Q16, D16, ql, cu = _rerank_case(3, 32, 600, 32, 200, seed=17)
    kc, k = 64, 10
    ids, scores, cand = ops.maxsim_rerank_two_stage(Q8, D8, Q16, D16, ql, cu, k_candidates=kc, k=k,
                                                    q_scale=qs, d_scale=ds, return_candidates=True)
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    ref = oracle.rerank_two_stage(Q8.cpu().numpy(), D8.cpu().numpy(), qs, ds, "fp16", syn.bits_u16(Q16),
                                  syn.bits_u16(D16), ql.cpu().numpy(), cu.cpu().numpy(), kc, k, threads=THREADS)
    assert np.array_equal(cand.cpu().numpy(), ref["cand_ids"])
    qb, db = syn.bits_u16(Q16), syn.bits_u16(D16)
    cu_h = cu.cpu().numpy()

    def s2_of(q, d):
        return oracle.forward_bits("fp16", qb, ql.cpu().numpy(), db, cu_h, pairs=[[q, d]])["score"][0]
    _check_final(ids, scores, ref, s2_of, SCORE_TOL_PER_TOKEN * 32)

    # the FP16 corpus read from pinned host memory gives the same bits
    ids_h, scores_h, _ = ops.maxsim_rerank_two_stage(Q8, D8, Q16, D16.cpu().pin_memory(), ql, cu,
                                                     k_candidates=kc, k=k, q_scale=qs, d_scale=ds)
    torch.cuda.synchronize()
    assert torch.equal(ids_h, ids) and torch.equal(scores_h, scores)


def test_two_stage_rerank_long_queries_bf16_per_token(ops):
    """Queries longer than 32 tokens (per-chunk partials in both stages),
    BF16 stage 2, per-token INT8 stage 1 (its candidates are compared by
    the oracle's stage-1 scores, which differ from the kernel's by rounding)."""
    n_q, lq, seed = 2, 64, 23
    lengths = syn.doc_lengths(300, 16, 150, seed)
    cu = syn.cu_seqlens_from_lengths(lengths)
    total = int(cu[-1])
    Q8, qs = syn.unit_tokens_int8_per_token(n_q * lq, 128, seed + 1, "cuda")
    D8, ds = syn.unit_tokens_int8_per_token(total, 128, seed + 2, "cuda")
    Q16 = syn.unit_tokens(n_q * lq, 128, seed + 1, "bf16", "cuda").view(n_q, lq, 128)
    D16 = syn.unit_tokens(total, 128, seed + 2, "bf16", "cuda")
    ql = torch.tensor([64, 40], dtype=torch.int32, device="cuda")
    cu_d = cu.cuda()
    kc, k = 40, 8
    ids, scores, cand = ops.maxsim_rerank_two_stage(Q8.view(n_q, lq, 128), D8, Q16, D16, ql, cu_d,
                                                    k_candidates=kc, k=k, q_tok_scales=qs.view(n_q, lq),
                                                    d_tok_scales=ds, return_candidates=True)
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    ref = oracle.rerank_two_stage(Q8.view(n_q, lq, 128).cpu().numpy(), D8.cpu().numpy(), 1.0, 1.0, "bf16",
                                  syn.bits_u16(Q16), syn.bits_u16(D16), ql.cpu().numpy(), cu.numpy(), kc, k,
                                  q_tok_scales=qs.view(n_q, lq).cpu().numpy(), d_tok_scales=ds.cpu().numpy(),
                                  threads=THREADS)
    tol1 = SCORE_TOL_PER_TOKEN * lq
    for q in range(n_q):
        got = ref["stage1"][q, cand[q].cpu().numpy()]
        assert got.min() >= ref["stage1"][q][ref["cand_ids"][q]].min() - 2 * tol1
    qb, db = syn.bits_u16(Q16), syn.bits_u16(D16)

    def s2_of(q, d):
        return oracle.forward_bits("bf16", qb, ql.cpu().numpy(), db, cu.numpy(), pairs=[[q, d]])["score"][0]
    for q in range(n_q):
        for j, d in enumerate(ids[q].cpu().numpy()):
            assert int(d) in set(cand[q].cpu().numpy().tolist())
            assert abs(float(scores[q, j]) - s2_of(q, d)) <= tol1
        assert np.all(np.diff(scores[q].cpu().numpy()) <= 0)


def test_two_stage_rerank_fewer_documents_than_candidates(ops):
    Q8, qs, D8, ds, Q16, D16, ql, cu = _rerank_case(2, 16, 5, 3, 40, seed=29)
    ids, scores, cand = ops.maxsim_rerank_two_stage(Q8, D8, Q16, D16, ql, cu, k_candidates=8, k=7,
                                                    q_scale=qs, d_scale=ds, return_candidates=True)
    torch.cuda.synchronize()
    ids = ids.cpu().numpy()
    assert np.all(ids[:, 5:] == -1) and np.all(np.isneginf(scores[:, 5:].cpu().numpy()))
    assert all(sorted(ids[q, :5].tolist()) == [0, 1, 2, 3, 4] for q in range(2))
    assert np.all(cand[:, 5:].cpu().numpy() == -1)


def test_int8_per_token_full_size_sampled(ops):
    """The INT8 varlen workload at full size (32 x 32 queries vs 100,000
    documents, Ld ~ U[32, 512]) with per-token scales: argmax and scores
    against the binary64 oracle on 40 sampled documents."""
    w = syn.WORKLOADS["int8_varlen"]
    cu = syn.cu_seqlens_from_lengths(syn.doc_lengths(w.n_docs, w.ld_lo, w.ld_hi, w.seed))
    total = int(cu[-1])
    Q8, qs = syn.unit_tokens_int8_per_token(w.n_q * w.lq, 128, w.seed + 1, "cuda")
    D8, ds = syn.unit_tokens_int8_per_token(total, 128, w.seed + 2, "cuda")
    Q8, qs = Q8.view(w.n_q, w.lq, 128), qs.view(w.n_q, w.lq)
    ql = torch.full((w.n_q,), w.lq, dtype=torch.int32, device="cuda")
    s, a = ops.maxsim_forward_int8_per_token(Q8, qs, ql, D8, ds, cu.cuda())
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    rng = np.random.default_rng(3)
    docs = sorted(set(rng.integers(0, w.n_docs, 36).tolist()) | {0, 1, w.n_docs - 2, w.n_docs - 1})
    cu_h = cu.numpy()
    D_sub = torch.cat([D8[int(cu_h[b]):int(cu_h[b + 1])] for b in docs])
    ds_sub = torch.cat([ds[int(cu_h[b]):int(cu_h[b + 1])] for b in docs])
    cu_sub = np.concatenate([[0], np.cumsum([int(cu_h[b + 1] - cu_h[b]) for b in docs])]).astype(np.int32)
    idx = torch.as_tensor(docs, device="cuda")
    check_int8_token(Q8.cpu().numpy(), qs.cpu().numpy(), ql.cpu().numpy(), D_sub.cpu().numpy(),
                     ds_sub.cpu().numpy(), cu_sub, s[:, idx].cpu().numpy(), a[:, idx].cpu().numpy())


def test_two_stage_rerank_full_size_sampled(ops):
    """The scan at the benchmark's size (32 x 32 queries vs 100,000 documents,
    1,000 candidates, 100 kept): the candidates are exactly the row-wise
    top-1000 of the INT8 scores (a property at any size), and sampled final
    scores match the oracle's FP16 rescoring."""
    w = syn.WORKLOADS["int8_varlen"]
    cu = syn.cu_seqlens_from_lengths(syn.doc_lengths(w.n_docs, w.ld_lo, w.ld_hi, w.seed))
    total = int(cu[-1])
    Q8, qs = syn.unit_tokens_int8(w.n_q * w.lq, 128, w.seed + 1, "cuda")
    D8, ds = syn.unit_tokens_int8(total, 128, w.seed + 2, "cuda")
    Q8 = Q8.view(w.n_q, w.lq, 128)
    Q16 = syn.unit_tokens(w.n_q * w.lq, 128, w.seed + 1, "fp16", "cuda").view(w.n_q, w.lq, 128)
    D16 = syn.unit_tokens(total, 128, w.seed + 2, "fp16", "cuda")
    ql = torch.full((w.n_q,), w.lq, dtype=torch.int32, device="cuda")
    cu_d = cu.cuda()
    ids, scores, cand = ops.maxsim_rerank_two_stage(Q8, D8, Q16, D16, ql, cu_d, k_candidates=1000, k=100,
                                                    q_scale=qs, d_scale=ds, max_doc_len=w.ld_hi,
                                                    return_candidates=True)
    s1, _, _ = ops.maxsim_forward(Q8, ql, D8, cu_d, with_argmax=False, q_scale=qs, d_scale=ds)
    top_ids, _ = ops.maxsim_topk(s1, 1000)
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    assert torch.equal(cand, top_ids)
    assert all(set(ids[q].tolist()) <= set(cand[q].tolist()) for q in range(w.n_q))
    assert torch.all(scores[:, :-1] >= scores[:, 1:])
    qb, db = syn.bits_u16(Q16), syn.bits_u16(D16)
    rng = np.random.default_rng(4)
    pairs = [(int(q), int(ids[q, j])) for q in rng.integers(0, w.n_q, 6) for j in rng.integers(0, 100, 4)]
    ref = oracle.forward_bits("fp16", qb, ql.cpu().numpy(), db, cu.numpy(), pairs=pairs, threads=THREADS)["score"]
    got = np.array([float(scores[q, (ids[q] == d).nonzero()[0, 0]]) for q, d in pairs])
    assert np.abs(got - ref).max() <= SCORE_TOL_PER_TOKEN * w.lq
