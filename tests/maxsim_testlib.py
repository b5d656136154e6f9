"""Helpers shared by the GPU parity tests: run the CUDA path through the C
ABI, run the oracle on the same stored bits, and compare with the acceptance
rules:

  scores   |score_gpu - score_oracle| <= 1e-4 * Lq   (Lq = q_lens[q], >= 1);
           -inf exactly where the oracle has -inf.
  argmax   equal to the oracle wherever the oracle's top-2 gap exceeds
               thr = min(1e-3, 1e-3 * |max| + 2^-15 * s),
           s = |q_i| * max_t |d_t| (the Cauchy-Schwarz bound on every value of
           the row); elsewhere the kernel's choice must be a near-maximum: its
           exact value >= oracle max - thr.  The 2^-15 * s term is twice the
           worst-case error of a 128-term FP32 dot product (128 * 2^-23 * s),
           so a correct kernel can never differ where the rule demands
           equality; the relative term catches a wrong choice among values
           that are all tiny.  Padding rows are -1.
  INT8     bit-exact (raw int64, fp32 score, argmax).
  per-token INT8   argmax equal where the exact top-2 gap > 2^-22 * |max|
           (four half-ulps of binary32), a near-maximum within that bound
           elsewhere; scores within 1e-4 * Lq.
  Chamfer  distance within 2^-18 of the oracle's binary64 minimum; index
           equal where the binary64 top-2 gap > 2^-19 of the second
           distance, a near-minimum (within 2^-19) elsewhere.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from late_interaction_retrieval_maxsim_gb300 import synthetic as syn

SCORE_TOL_PER_TOKEN = 1e-4
ARGMAX_GAP = 1e-3
ARGMAX_REL_GAP = 1e-3
ARGMAX_ROUND = 2.0 ** -15
TOKEN_REL_GAP = 2.0 ** -22
CHAMFER_DIST_REL = 2.0 ** -18
CHAMFER_GAP_REL = 2.0 ** -19
GRAD_TOL = 1e-4
THREADS = max(1, min(16, os.cpu_count() or 1))

DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def random_case(n_q, lq_max, lengths, dtype="fp16", q_lens=None, seed=0, device="cuda"):
    """Unit-norm N(0,1) tokens (the workload recipe) for arbitrary lengths."""
    lengths = torch.as_tensor(lengths, dtype=torch.int32)
    cu = syn.cu_seqlens_from_lengths(lengths)
    total = int(cu[-1])
    Q = syn.unit_tokens(n_q * lq_max, 128, seed + 1, dtype, device).view(n_q, lq_max, 128)
    D = syn.unit_tokens(total, 128, seed + 2, dtype, device)
    if q_lens is None:
        q_lens = [lq_max] * n_q
    ql = torch.as_tensor(q_lens, dtype=torch.int32, device=device)
    return Q, ql, D, cu.to(device)


def sub_batch(D, cu, docs):
    """Host copy of the rows of the chosen documents, with its own cu."""
    cu_h = cu.cpu().numpy().astype(np.int64)
    pieces, lens = [], []
    for b in docs:
        pieces.append(D[int(cu_h[b]):int(cu_h[b + 1])])
        lens.append(int(cu_h[b + 1] - cu_h[b]))
    Dsub = torch.cat(pieces) if pieces else D[:0]
    cu_sub = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return Dsub, cu_sub


def _row_scale(dtype, qb, db, cu, pq, pb):
    """s[p, i] = |Q[pq[p], i]| * max over document pb[p] of |D_t| (0 for an
    empty document)."""
    qn = np.sqrt((oracle.decode(dtype, qb) ** 2).sum(-1))            # [n_q, lq_max]
    dn = np.sqrt((oracle.decode(dtype, db) ** 2).sum(-1))            # [total]
    n_docs = len(cu) - 1
    dmax = np.zeros(n_docs)
    for b in range(n_docs):
        if cu[b + 1] > cu[b]:
            dmax[b] = dn[cu[b]:cu[b + 1]].max()
    return qn[pq] * dmax[pb][:, None]


def argmax_threshold(rowmax, scale):
    """The gap above which the kernel must reproduce the oracle's argmax, and
    the slack of a near-maximum elsewhere."""
    with np.errstate(invalid="ignore"):
        rel = ARGMAX_REL_GAP * np.abs(np.nan_to_num(rowmax, nan=0.0, neginf=0.0)) + ARGMAX_ROUND * scale
    return np.minimum(ARGMAX_GAP, rel)


def check_forward(dtype, Q, ql, D, cu, scores, argmax, docs=None, queries=None, pairs=None):
    """Compare GPU outputs with the oracle on all pairs, on the pairs
    (queries x docs) when given, or on an explicit list of (q, b) pairs.
    Returns the max |score error| / Lq."""
    n_q, lq_max, _ = Q.shape
    n_docs = cu.numel() - 1
    if pairs is not None:
        pairs = np.asarray(pairs, np.int64).reshape(-1, 2)
        qb, db = syn.bits_u16(Q), syn.bits_u16(D)
        cu_ref = cu.cpu().numpy().astype(np.int32)
        ql_all = ql.cpu().numpy()
        pq, pb = pairs[:, 0], pairs[:, 1]
        ref = oracle.forward_bits(dtype, qb, ql_all, db, cu_ref, pairs=pairs, want_rowmax=True, threads=THREADS)
        qi, bi = torch.as_tensor(pq), torch.as_tensor(pb)
        s_gpu = scores.cpu()[qi, bi].double().numpy()
        a_gpu = None if argmax is None else argmax.cpu()[qi, bi].numpy()
        lq_of_pair = np.maximum(ql_all[pq], 1)
        q_of, b_of = pq, pb
    else:
        docs = list(range(n_docs)) if docs is None else list(docs)
        queries = list(range(n_q)) if queries is None else list(queries)
        Dsub, cu_ref = sub_batch(D, cu, docs)
        qb, db = syn.bits_u16(Q[queries]), syn.bits_u16(Dsub)
        ql_sub = ql[queries].cpu().numpy()
        ref = oracle.forward_bits(dtype, qb, ql_sub, db, cu_ref, want_rowmax=True, threads=THREADS)
        P = len(queries) * len(docs)
        s_gpu = scores[queries][:, docs].double().cpu().numpy().reshape(P)
        a_gpu = None if argmax is None else argmax[queries][:, docs].cpu().numpy().reshape(P, lq_max)
        lq_of_pair = np.repeat(np.maximum(ql_sub, 1), len(docs))
        q_of = np.repeat(np.arange(len(queries)), len(docs))
        b_of = np.tile(np.arange(len(docs)), len(queries))
    s_ref = ref["score"]
    neg = np.isneginf(s_ref)
    assert np.array_equal(np.isneginf(s_gpu), neg), "-inf pattern differs"
    err = np.abs(s_gpu[~neg] - s_ref[~neg]) / lq_of_pair[~neg]
    worst = float(err.max()) if err.size else 0.0
    assert worst <= SCORE_TOL_PER_TOKEN, f"score error {worst:.3e} per token"
    if a_gpu is not None:
        a_ref = ref["argmax"]
        pad = a_ref == -1
        assert np.array_equal(a_gpu[pad], a_ref[pad]), "padding / empty-doc rows must be -1"
        thr = argmax_threshold(ref["rowmax"], _row_scale(dtype, qb, db, cu_ref, q_of, b_of))
        sure = (ref["gap"] > thr) & ~pad
        assert np.array_equal(a_gpu[sure], a_ref[sure]), \
            f"argmax differs on {(a_gpu[sure] != a_ref[sure]).sum()} unambiguous rows"
        near = ~sure & ~pad
        if near.any():
            pi, ii = np.nonzero(near)
            tt = a_gpu[pi, ii]
            assert np.all(tt >= 0)
            v = oracle.dot_bits(dtype, qb, db, cu_ref, q_of[pi], b_of[pi], ii, tt)
            assert np.all(v >= ref["rowmax"][pi, ii] - thr[pi, ii]), "argmax is not a near-maximum"
    return worst


def check_int8_token(Q8, qs, ql, D8, ds, cu, scores, argmax):
    """Per-token INT8 outputs against the binary64 oracle (rules above), on
    every pair.  Host numpy inputs."""
    n_q, lq = Q8.shape[:2]
    cu = np.asarray(cu, np.int32)
    n_docs = len(cu) - 1
    ref = oracle.forward_i8_token(Q8, qs, ql, D8, ds, cu, want_rowmax=True, threads=THREADS)
    a_ref = ref["argmax"].reshape(n_q, n_docs, lq)
    a_gpu = np.asarray(argmax).reshape(n_q, n_docs, lq)
    pad = a_ref == -1
    assert np.array_equal(a_gpu[pad], a_ref[pad]), "padding / empty-doc rows must be -1"
    best = ref["rowmax"].reshape(n_q, n_docs, lq)
    gap = ref["gap"].reshape(n_q, n_docs, lq)
    with np.errstate(invalid="ignore"):
        bound = TOKEN_REL_GAP * np.abs(np.where(pad, 0.0, best))
    sure = (gap > bound) & ~pad
    assert np.array_equal(a_gpu[sure], a_ref[sure]), \
        f"argmax differs on {(a_gpu[sure] != a_ref[sure]).sum()} unambiguous rows"
    near = ~sure & ~pad
    if near.any():
        qq, bb, ii = np.nonzero(near)
        v = oracle.dot_i8_token(Q8, D8, ds, cu, qq, bb, ii, a_gpu[qq, bb, ii])
        assert np.all(v >= best[qq, bb, ii] - bound[qq, bb, ii]), "argmax is not a near-maximum"
    s_ref = ref["score"].reshape(n_q, n_docs)
    s_gpu = np.asarray(scores, np.float64)
    neg = np.isneginf(s_ref)
    assert np.array_equal(np.isneginf(s_gpu), neg)
    lqs = np.maximum(np.asarray(ql), 1)[:, None].repeat(n_docs, 1)
    assert np.all(np.abs(s_gpu[~neg] - s_ref[~neg]) <= SCORE_TOL_PER_TOKEN * lqs[~neg])
    return int(sure.sum()), int(near.sum())


def check_chamfer_nn(S, cu_s, T, cu_t, dist, arg, rows=None):
    """Kernel nearest neighbours (dist float32, arg local index) of the
    sources S against the binary64 oracle (rules above).  Host numpy inputs;
    ``rows`` restricts the check to those global source indices (of a single
    item)."""
    if rows is not None:
        S = S[rows]
        cu_s = np.array([0, len(rows)], np.int32)
        dist, arg = dist[rows], arg[rows]
    d_ref, a_ref, gap = oracle.chamfer_nn(S, cu_s, T, cu_t, want_gap=True)
    dist = np.asarray(dist, np.float64)
    empty = a_ref == -1
    assert np.array_equal(arg[empty], a_ref[empty]) and np.all(np.isposinf(dist[empty]))
    ok = ~empty
    assert np.all(np.abs(dist[ok] - d_ref[ok]) <= CHAMFER_DIST_REL * d_ref[ok]), "distance off"
    sure = ok & (gap > CHAMFER_GAP_REL * (d_ref + gap))
    assert np.array_equal(arg[sure], a_ref[sure]), \
        f"nearest index differs on {(arg[sure] != a_ref[sure]).sum()} unambiguous points"
    near = ok & ~sure
    if near.any():
        item = np.searchsorted(np.asarray(cu_s), np.nonzero(near)[0], side="right") - 1
        t_glob = np.asarray(cu_t)[item] + arg[near]
        v = oracle.chamfer_pair_dist(S, T, np.nonzero(near)[0], t_glob)
        assert np.all(v <= d_ref[near] * (1 + CHAMFER_GAP_REL)), "not a near-minimum"
    return int(sure.sum()), int(near.sum())
