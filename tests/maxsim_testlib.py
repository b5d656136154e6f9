"""Helpers shared by the GPU parity tests: run the CUDA path through the C
ABI, run the oracle on the same stored bits, and compare with the acceptance
rules:

  scores   |score_gpu - score_oracle| <= 1e-4 * Lq   (Lq = q_lens[q], >= 1);
           -inf exactly where the oracle has -inf.
  argmax   equal to the oracle wherever the oracle's top-2 gap > 1e-3;
           elsewhere the kernel's choice must be a near-maximum: its exact
           value >= oracle max - 1e-3.  Padding rows are -1.
  INT8     bit-exact (raw int64, fp32 score, argmax).
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from late_interaction_retrieval_maxsim_gb300 import synthetic as syn

SCORE_TOL_PER_TOKEN = 1e-4
ARGMAX_GAP = 1e-3
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


def check_forward(dtype, Q, ql, D, cu, scores, argmax, docs=None, queries=None):
    """Compare GPU outputs with the oracle on all pairs, or on the pairs
    (queries x docs) when given.  Returns the max |score error| / Lq."""
    n_q, lq_max, _ = Q.shape
    n_docs = cu.numel() - 1
    docs = list(range(n_docs)) if docs is None else list(docs)
    queries = list(range(n_q)) if queries is None else list(queries)
    Dsub, cu_sub = sub_batch(D, cu, docs)
    Qsub = Q[queries]
    ql_sub = ql[queries].cpu().numpy()
    qb, db = syn.bits_u16(Qsub), syn.bits_u16(Dsub)
    ref = oracle.forward_bits(dtype, qb, ql_sub, db, cu_sub, want_rowmax=True, threads=THREADS)
    P = len(queries) * len(docs)
    s_gpu = scores[queries][:, docs].double().cpu().numpy().reshape(P)
    s_ref = ref["score"]
    lq_of_pair = np.repeat(np.maximum(ql_sub, 1), len(docs))
    neg = np.isneginf(s_ref)
    assert np.array_equal(np.isneginf(s_gpu), neg), "-inf pattern differs"
    err = np.abs(s_gpu[~neg] - s_ref[~neg]) / lq_of_pair[~neg]
    worst = float(err.max()) if err.size else 0.0
    assert worst <= SCORE_TOL_PER_TOKEN, f"score error {worst:.3e} per token"
    if argmax is not None:
        a_gpu = argmax[queries][:, docs].cpu().numpy().reshape(P, lq_max)
        a_ref = ref["argmax"]
        gap = ref["gap"]
        sure = gap > ARGMAX_GAP
        assert np.array_equal(a_gpu[sure], a_ref[sure]), \
            f"argmax differs on {(a_gpu[sure] != a_ref[sure]).sum()} unambiguous rows"
        pad = a_ref == -1
        assert np.array_equal(a_gpu[pad], a_ref[pad]), "padding / empty-doc rows must be -1"
        near = ~sure & ~pad
        if near.any():
            pi, ii = np.nonzero(near)
            qq = pi // len(docs)
            bb = pi % len(docs)
            tt = a_gpu[pi, ii]
            assert np.all(tt >= 0)
            v = oracle.dot_bits(dtype, qb, db, cu_sub, qq, bb, ii, tt)
            assert np.all(v >= ref["rowmax"][pi, ii] - ARGMAX_GAP), "argmax is not a near-maximum"
    return worst
