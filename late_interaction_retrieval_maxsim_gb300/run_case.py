"""Run one case of a library entry point a few times on ``cuda:0``.

A driver for profilers (``ncu -k ... python -m
late_interaction_retrieval_maxsim_gb300.run_case forward ...``) and for
quick checks: it builds seeded synthetic inputs with ``synthetic``, calls the
entry point ``--reps`` times, synchronises and checks the device status word.

    python -m late_interaction_retrieval_maxsim_gb300.run_case forward \\
        --workload colbert_varlen --n-docs 5000 --reps 2 [--value-only]
    python -m late_interaction_retrieval_maxsim_gb300.run_case int8-token --n-docs 5000
    python -m late_interaction_retrieval_maxsim_gb300.run_case backward --workload train
    python -m late_interaction_retrieval_maxsim_gb300.run_case chamfer --points 20000
    python -m late_interaction_retrieval_maxsim_gb300.run_case rerank --n-docs 20000
    python -m late_interaction_retrieval_maxsim_gb300.run_case host --n-docs 20000
"""
from __future__ import annotations

import argparse
import sys

import torch

from . import (maxsim_backward, maxsim_chamfer_backward, maxsim_chamfer_forward, maxsim_device_status,
               maxsim_forward, maxsim_forward_host, maxsim_forward_int8_per_token, maxsim_rerank_two_stage)
from . import synthetic as syn


def _forward(a):
    w = syn.WORKLOADS[a.workload]
    x = syn.make_inputs(w, device="cuda", n_docs=a.n_docs)
    kw = dict(q_scale=x["q_scale"], d_scale=x["d_scale"])
    s, am, _ = maxsim_forward(x["Q"], x["q_lens"], x["D"], x["cu_seqlens"], with_argmax=not a.value_only, **kw)
    for _ in range(a.reps - 1):
        maxsim_forward(x["Q"], x["q_lens"], x["D"], x["cu_seqlens"], with_argmax=not a.value_only, scores=s,
                       argmax=am, **kw)


def _int8_token(a):
    w = syn.WORKLOADS["int8_varlen"]
    n_docs = a.n_docs or w.n_docs
    cu = syn.cu_seqlens_from_lengths(syn.doc_lengths(w.n_docs, w.ld_lo, w.ld_hi, w.seed)[:n_docs]).cuda()
    Q8, qs = syn.unit_tokens_int8_per_token(w.n_q * w.lq, w.dim, w.seed + 1, "cuda")
    D8, ds = syn.unit_tokens_int8_per_token(int(cu[-1]), w.dim, w.seed + 2, "cuda")
    ql = torch.full((w.n_q,), w.lq, dtype=torch.int32, device="cuda")
    for _ in range(a.reps):
        maxsim_forward_int8_per_token(Q8.view(w.n_q, w.lq, w.dim), qs.view(w.n_q, w.lq), ql, D8, ds, cu,
                                      with_argmax=not a.value_only)


def _backward(a):
    w = syn.WORKLOADS[a.workload]
    x = syn.make_inputs(w, device="cuda", n_docs=a.n_docs)
    Q, ql, D, cu = x["Q"], x["q_lens"], x["D"], x["cu_seqlens"]
    s, am, _ = maxsim_forward(Q, ql, D, cu)
    g = torch.softmax(s / 0.05, dim=1).contiguous()
    for _ in range(a.reps):
        maxsim_backward(g, am, Q, ql, D, cu)


def _chamfer(a):
    g = torch.Generator("cuda").manual_seed(0)
    P = torch.rand((a.points, 3), generator=g, device="cuda")
    Q = torch.rand((a.points, 3), generator=g, device="cuda")
    cu = torch.tensor([0, a.points], dtype=torch.int32, device="cuda")
    for _ in range(a.reps):
        _, _, apq, _, aqp = maxsim_chamfer_forward(P, cu, Q, cu)
        maxsim_chamfer_backward(torch.ones(1, device="cuda"), P, cu, Q, cu, apq, aqp)


def _rerank(a):
    """Two-stage scan on the INT8 varlen workload: 1,000 candidates, 100 kept."""
    w = syn.WORKLOADS["int8_varlen"]
    n_docs = a.n_docs or w.n_docs
    cu = syn.cu_seqlens_from_lengths(syn.doc_lengths(w.n_docs, w.ld_lo, w.ld_hi, w.seed)[:n_docs]).cuda()
    total = int(cu[-1])
    Q8, qs = syn.unit_tokens_int8(w.n_q * w.lq, w.dim, w.seed + 1, "cuda")
    D8, ds = syn.unit_tokens_int8(total, w.dim, w.seed + 2, "cuda")
    Q16 = syn.unit_tokens(w.n_q * w.lq, w.dim, w.seed + 1, "fp16", "cuda").view(w.n_q, w.lq, w.dim)
    D16 = syn.unit_tokens(total, w.dim, w.seed + 2, "fp16", "cuda")
    ql = torch.full((w.n_q,), w.lq, dtype=torch.int32, device="cuda")
    for _ in range(a.reps):
        maxsim_rerank_two_stage(Q8.view(w.n_q, w.lq, w.dim), D8, Q16, D16, ql, cu, k_candidates=1000, k=100,
                                q_scale=qs, d_scale=ds, max_doc_len=w.ld_hi)


def _host(a):
    """Out-of-core forward: the ColBERT workload's corpus in pinned host
    memory, streamed in blocks of 5,000 documents."""
    w = syn.WORKLOADS["colbert_varlen"]
    x = syn.make_inputs(w, device="cuda", n_docs=a.n_docs)
    D_h = x["D"].cpu().pin_memory()
    cu_h = x["cu_seqlens"].cpu().pin_memory()
    for _ in range(a.reps):
        maxsim_forward_host(x["Q"], x["q_lens"], D_h, cu_h, block_docs=5000, block_tokens=5000 * w.ld_hi,
                            with_argmax=True)
    torch.cuda.synchronize()


CASES = {"forward": _forward, "int8-token": _int8_token, "backward": _backward, "chamfer": _chamfer,
         "rerank": _rerank, "host": _host}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--workload", default="colbert_varlen", choices=sorted(syn.WORKLOADS))
    ap.add_argument("--n-docs", type=int, default=None, help="first n documents of the workload")
    ap.add_argument("--points", type=int, default=20_000, help="points per cloud (chamfer)")
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--value-only", action="store_true", help="forward without the argmax output")
    a = ap.parse_args(argv)
    torch.cuda.set_device(0)
    CASES[a.case](a)
    torch.cuda.synchronize()
    status = maxsim_device_status()
    if status != 0:
        print(f"device status word {status:#x}", file=sys.stderr)
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
