"""Seeded synthetic inputs shaped like the late-interaction workloads.

This module only *draws* inputs: document lengths, token embeddings
(N(0,1) in fp32, L2-normalised per token, then rounded to the storage type),
and symmetric INT8 quantisation with one scale per tensor or per token.  It holds none of the MaxSim
arithmetic, so both the CUDA path and the CPU oracle can consume its output.

Recipe (the same for every workload; see ``WORKLOADS``):
  1. document lengths from a CPU ``torch.Generator`` seeded with ``seed``,
     uniform integers in [ld_lo, ld_hi];
  2. Q, then D, drawn from a generator on the target device seeded with
     ``seed + 1`` (Q) and ``seed + 2`` (D), in row chunks;
  3. each token row divided by its fp32 L2 norm, then cast (round to nearest
     even) to FP16/BF16, or quantised to INT8 with s = max|x| / 127 over the
     whole tensor and q = clamp(round_half_even(x / s), -127, 127).

The shapes follow the ColBERT / ColPali settings of "FLASH-MAXSIM: IO-Aware
Fused Kernels for Late-Interaction Retrieval" (§3.1 and Table 1); no dataset
is read -- seeded synthetic embeddings stand in for the BEIR / ViDoRe-style
corpora the pages evaluate on.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

DIM = 128
_CHUNK_ROWS = 1 << 20


@dataclass(frozen=True)
class Workload:
    """Shape of one synthetic workload."""
    name: str
    n_q: int
    lq: int
    n_docs: int
    ld_lo: int
    ld_hi: int
    dtype: str            # "fp16" | "bf16" | "int8"
    seed: int = 0
    dim: int = DIM
    note: str = field(default="", compare=False)

    @property
    def uniform(self) -> bool:
        return self.ld_lo == self.ld_hi


WORKLOADS = {
    "tiny": Workload("tiny", 1, 32, 256, 128, 128, "fp16",
                     note="1 query Lq=32 vs 256 docs Ld=128, FP16"),
    "colbert_varlen": Workload("colbert_varlen", 16, 32, 50_000, 32, 300, "fp16",
                               note="16 queries Lq=32 vs 50,000 docs Ld~U[32,300], packed"),
    "colbert_1q": Workload("colbert_1q", 1, 32, 50_000, 32, 300, "fp16",
                           note="1 query Lq=32 vs the 50,000 ColBERT documents (single-query rerank, HBM-bound)"),
    "colpali": Workload("colpali", 1, 1024, 10_000, 1024, 1024, "fp16",
                        note="1 query Lq=1024 vs 10,000 docs Ld=1024"),
    "train": Workload("train", 256, 32, 256, 180, 180, "bf16",
                      note="256 queries Lq=32 x 256 docs Ld=180, BF16, fwd+bwd"),
    "train_colpali": Workload("train_colpali", 64, 1024, 64, 1024, 1024, "bf16",
                              note="64 queries Lq=1024 x 64 docs Ld=1024, BF16, fwd+bwd"),
    "int8_varlen": Workload("int8_varlen", 32, 32, 100_000, 32, 512, "int8",
                            note="32 queries Lq=32 vs 100,000 docs Ld~U[32,512], INT8"),
}

TORCH_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16, "int8": torch.int8}


def doc_lengths(n_docs: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Uniform integer document lengths in [lo, hi] (CPU int32)."""
    if lo == hi:
        return torch.full((n_docs,), lo, dtype=torch.int32)
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randint(lo, hi + 1, (n_docs,), generator=g, dtype=torch.int64).to(torch.int32)


def cu_seqlens_from_lengths(lengths: torch.Tensor) -> torch.Tensor:
    """[0, l0, l0+l1, ...] as int32 (CPU)."""
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lengths.to(torch.int64), 0)
    if int(cu[-1]) >= 2**31:
        raise ValueError("total token count exceeds int32")
    return cu.to(torch.int32)


def _unit_rows(n_rows: int, dim: int, gen: torch.Generator, device) -> torch.Tensor:
    x = torch.randn((n_rows, dim), generator=gen, device=device, dtype=torch.float32)
    return x / x.norm(dim=1, keepdim=True)


def unit_tokens(n_rows: int, dim: int, seed: int, dtype: str, device="cpu") -> torch.Tensor:
    """[n_rows, dim] unit-norm token rows stored as FP16/BF16 (see recipe)."""
    out = torch.empty((n_rows, dim), dtype=TORCH_DTYPES[dtype], device=device)
    gen = torch.Generator(device=device).manual_seed(seed)
    for s in range(0, n_rows, _CHUNK_ROWS):
        e = min(n_rows, s + _CHUNK_ROWS)
        out[s:e] = _unit_rows(e - s, dim, gen, device).to(out.dtype)
    return out


def unit_tokens_int8(n_rows: int, dim: int, seed: int, device="cpu"):
    """[n_rows, dim] unit-norm rows quantised to INT8 with one symmetric scale.

    Two passes over the same seeded stream: the first finds max|x|, the second
    quantises.  Returns (int8 tensor, scale as a Python float32 value)."""
    gen = torch.Generator(device=device).manual_seed(seed)
    amax = torch.zeros((), dtype=torch.float32, device=device)
    for s in range(0, n_rows, _CHUNK_ROWS):
        e = min(n_rows, s + _CHUNK_ROWS)
        amax = torch.maximum(amax, _unit_rows(e - s, dim, gen, device).abs().max())
    scale = (amax / 127.0).to(torch.float32)
    out = torch.empty((n_rows, dim), dtype=torch.int8, device=device)
    gen = torch.Generator(device=device).manual_seed(seed)
    for s in range(0, n_rows, _CHUNK_ROWS):
        e = min(n_rows, s + _CHUNK_ROWS)
        x = _unit_rows(e - s, dim, gen, device)
        out[s:e] = torch.clamp(torch.round(x / scale), -127, 127).to(torch.int8)
    return out, float(scale.item())


def unit_tokens_int8_per_token(n_rows: int, dim: int, seed: int, device="cpu", with_fp16: bool = False):
    """[n_rows, dim] unit-norm rows (the same seeded stream as unit_tokens)
    quantised to INT8 with one symmetric scale per row: s = max|x| / 127 in
    FP32, code = clamp(round-half-even(x / s), -127, 127).  Returns (int8
    codes, float32 scales [n_rows]) and, with ``with_fp16``, the FP16 rows
    the codes came from."""
    gen = torch.Generator(device=device).manual_seed(seed)
    codes = torch.empty((n_rows, dim), dtype=torch.int8, device=device)
    scales = torch.empty((n_rows,), dtype=torch.float32, device=device)
    f16 = torch.empty((n_rows, dim), dtype=torch.float16, device=device) if with_fp16 else None
    for s in range(0, n_rows, _CHUNK_ROWS):
        e = min(n_rows, s + _CHUNK_ROWS)
        x = _unit_rows(e - s, dim, gen, device)
        sc = (x.abs().amax(dim=1) / 127.0).to(torch.float32)
        safe = torch.where(sc > 0, sc, torch.ones_like(sc))
        codes[s:e] = torch.clamp(torch.round(x / safe[:, None]), -127, 127).to(torch.int8)
        scales[s:e] = sc
        if with_fp16:
            f16[s:e] = x.to(torch.float16)
    return (codes, scales, f16) if with_fp16 else (codes, scales)


def make_inputs(w: Workload, device="cpu", n_docs: int | None = None, n_q: int | None = None):
    """Materialise a workload.  ``n_docs`` / ``n_q`` override the counts (the
    lengths of the first n_docs documents and the first n_q queries of the
    full draw are kept, so a reduced case is a prefix of the full one).

    Returns a dict with Q [n_q, lq, dim], q_lens [n_q] (int32, device),
    D [total, dim], cu_seqlens [n_docs+1] (int32, device), lengths (CPU),
    and q_scale / d_scale for INT8."""
    nd = w.n_docs if n_docs is None else n_docs
    nq = w.n_q if n_q is None else n_q
    lengths = doc_lengths(w.n_docs, w.ld_lo, w.ld_hi, w.seed)[:nd].clone()
    cu = cu_seqlens_from_lengths(lengths)
    total = int(cu[-1])
    out = {"workload": w, "lengths": lengths, "cu_seqlens": cu.to(device),
           "q_lens": torch.full((nq,), w.lq, dtype=torch.int32, device=device)}
    if w.dtype == "int8":
        Qf, qs = unit_tokens_int8(nq * w.lq, w.dim, w.seed + 1, device)
        Df, ds = unit_tokens_int8(total, w.dim, w.seed + 2, device)
        out.update(Q=Qf.view(nq, w.lq, w.dim), D=Df, q_scale=qs, d_scale=ds)
    else:
        out.update(Q=unit_tokens(nq * w.lq, w.dim, w.seed + 1, w.dtype, device).view(nq, w.lq, w.dim),
                   D=unit_tokens(total, w.dim, w.seed + 2, w.dtype, device),
                   q_scale=1.0, d_scale=1.0)
    return out


def bits_u16(t: torch.Tensor):
    """Stored 16-bit patterns of an FP16/BF16 tensor as a numpy uint16 array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
