"""Pins for the oracle's top-K selection and two-stage rerank (Flash-MaxSim
§4.1 "Kernel Family": the two-stage INT8 -> FP16 top-K scan).  CPU only.

  * top-K against a pure-Python sort on (value descending, column
    ascending), with heavy ties, -inf and k beyond the row length;
  * the two-stage rerank with k_candidates = n_docs keeps every document, so
    it must equal the FP16 oracle's full ranking cut at k, whatever the INT8
    stage says;
  * one-hot inputs whose INT8 and FP16 scores are the same integers rank the
    same in both stages, and the closed form fixes the answer."""
import numpy as np

import oracle
from late_interaction_retrieval_maxsim_gb300 import synthetic as syn

RNG = np.random.default_rng(7)


def _py_topk(row, k):
    order = sorted(range(len(row)), key=lambda c: (-row[c], c))[:k]
    ids = order + [-1] * (k - len(order))
    vals = [row[c] for c in order] + [-np.inf] * (k - len(order))
    return ids, vals


def test_topk_against_python_sort_with_ties():
    vals = RNG.integers(-3, 4, (5, 40)).astype(np.float64)
    vals[1, ::3] = -np.inf
    for k in (1, 5, 17, 40, 55):
        ids, v = oracle.topk(vals, k)
        for r in range(vals.shape[0]):
            pi, pv = _py_topk(list(vals[r]), k)
            assert list(ids[r]) == pi
            assert list(v[r]) == pv


def test_topk_id_map():
    vals = np.array([[0.5, 2.0, 2.0, 1.0]])
    ids, v = oracle.topk(vals, 3, ids=np.array([[10, 11, 12, 13]]))
    assert list(ids[0]) == [11, 12, 13] and list(v[0]) == [2.0, 2.0, 1.0]


def _bits_case(n_q=2, lq=6, lengths=(4, 9, 1, 7, 3, 12, 5, 8), seed=5):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    Q16 = syn.unit_tokens(n_q * lq, 128, seed, "fp16").view(n_q, lq, 128)
    D16 = syn.unit_tokens(int(cu[-1]), 128, seed + 1, "fp16")
    Q8, _ = syn.unit_tokens_int8_per_token(n_q * lq, 128, seed)
    D8, _ = syn.unit_tokens_int8_per_token(int(cu[-1]), 128, seed + 1)
    return (Q8.view(n_q, lq, 128).numpy(), D8.numpy(), syn.bits_u16(Q16), syn.bits_u16(D16),
            np.full(n_q, lq, np.int32), cu)


def test_rerank_keeping_every_document_equals_the_fp16_ranking():
    Q8, D8, Qb, Db, q_lens, cu = _bits_case()
    n_docs = len(cu) - 1
    out = oracle.rerank_two_stage(Q8, D8, 0.01, 0.01, "fp16", Qb, Db, q_lens, cu, n_docs, 5)
    full = oracle.forward_bits("fp16", Qb, q_lens, Db, cu)["score"].reshape(len(q_lens), n_docs)
    ids, vals = oracle.topk(full, 5)
    assert np.array_equal(out["ids"], ids)
    assert np.array_equal(out["scores"], vals)


def test_rerank_one_hot_closed_form():
    """Q token i = e_{a_i}, D token t = e_{c_t} (exact in INT8 with scale 1
    and in FP16): score(q, b) = #{i : a_i occurs in document b}."""
    lq, dim = 4, 128
    a = np.array([[3, 7, 9, 11], [5, 5, 6, 60]])
    docs = [[3, 7], [9], [1, 2, 3, 7, 9, 11], [5, 6], [60, 5, 5], [100]]
    lengths = [len(d) for d in docs]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    Q8 = np.zeros((2, lq, dim), np.int8)
    for q in range(2):
        Q8[q, np.arange(lq), a[q]] = 1
    D8 = np.zeros((int(cu[-1]), dim), np.int8)
    D8[np.arange(int(cu[-1])), np.concatenate(docs)] = 1
    Qb = np.where(Q8 == 1, np.uint16(0x3C00), np.uint16(0)).astype(np.uint16)   # FP16 1.0
    Db = np.where(D8 == 1, np.uint16(0x3C00), np.uint16(0)).astype(np.uint16)
    out = oracle.rerank_two_stage(Q8, D8, 1.0, 1.0, "fp16", Qb, Db, [4, 4], cu, 3, 2)
    expect = np.array([[sum(x in d for x in a[q]) for d in docs] for q in range(2)], np.float64)
    for q in range(2):
        order = sorted(range(len(docs)), key=lambda b: (-expect[q, b], b))
        assert list(out["cand_ids"][q]) == order[:3]
        assert list(out["ids"][q]) == order[:2]
        assert list(out["scores"][q]) == [expect[q, b] for b in order[:2]]
