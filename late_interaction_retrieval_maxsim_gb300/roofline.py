"""Algorithmic work model of the fused MaxSim path (bytes and FLOPs).

These counts are what the roofline fractions divide by a measured kernel
time.  They restate the IO model of "FLASH-MAXSIM: IO-Aware Fused Kernels for
Late-Interaction Retrieval" §4.1.2 (Theorem 1: the fused forward reads each
operand once and writes Theta(N_q B) scalars; the naive path additionally
writes and reads the [B, Lq, Ld] similarity tensor), and are pinned to the
figures the pages print (Table 2 and the 21 GB figure of §1).
"""
from __future__ import annotations


def naive_hbm_bytes(n_docs: int, lq: int, ld: int, dim: int = 128,
                    in_bytes: int = 2, s_bytes: int = 4) -> int:
    """Materialised path (§3.1, Alg. 1): one write and one read of the FP32
    similarity tensor plus the document embeddings read once."""
    return 2 * n_docs * lq * ld * s_bytes + n_docs * ld * dim * in_bytes


def fused_input_bytes(n_docs: int, ld: int, dim: int = 128, in_bytes: int = 2) -> int:
    """Fused path (Theorem 1): the document embeddings read once."""
    return n_docs * ld * dim * in_bytes


def materialised_tensor_bytes(n_docs: int, lq: int, ld: int, s_bytes: int = 2) -> int:
    """Size of the [B, Lq, Ld] similarity tensor (§1)."""
    return n_docs * lq * ld * s_bytes


def forward_flops(sum_q_tokens: int, total_d_tokens: int, dim: int = 128) -> int:
    """2 d FLOPs per (query token, document token) pair; every query is scored
    against every document, so the pairs are sum_q Lq(q) x sum_b Ld(b)."""
    return 2 * dim * sum_q_tokens * total_d_tokens


def forward_hbm_bytes(n_q: int, lq_max: int, n_docs: int, total_d_tokens: int,
                      dim: int = 128, in_bytes: int = 2, argmax: bool = True) -> int:
    """Algorithmic HBM bytes of one fused forward launch: Q and D read once,
    cu_seqlens and q_lens read once, scores (FP32) and the optional INT32
    argmax written once."""
    b = (n_q * lq_max * dim + total_d_tokens * dim) * in_bytes
    b += (n_docs + 1) * 4 + n_q * 4
    b += n_q * n_docs * 4
    if argmax:
        b += n_q * n_docs * lq_max * 4
    return b


def backward_hbm_bytes(n_q: int, lq_max: int, n_docs: int, total_d_tokens: int,
                       n_sources: int, dim: int = 128, in_bytes: int = 2) -> dict:
    """Algorithmic HBM bytes of the backward (Alg. 3): argmax and grad read,
    CSR written and read back, Q and D read once, dQ and dD (FP32) written."""
    parts = {
        "argmax": n_q * n_docs * lq_max * 4,
        "grad": n_q * n_docs * 4,
        "csr": 2 * (n_sources * 4 + (total_d_tokens + 1) * 4),
        "Q": n_q * lq_max * dim * in_bytes,
        "D": total_d_tokens * dim * in_bytes,
        "dQ": n_q * lq_max * dim * 4,
        "dD": total_d_tokens * dim * 4,
    }
    parts["total"] = sum(parts.values())
    return parts
