"""CPU oracle for the fused MaxSim operator -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library's product path never does:
it shares no code with this oracle, and the oracle never imports the library.

The arithmetic lives in ``oracle.c`` (plain C, binary64 / int64); this module
only marshals numpy arrays through ctypes.  Each entry point names the passage
of "FLASH-MAXSIM: IO-Aware Fused Kernels for Late-Interaction Retrieval"
(arXiv 2605.29517) it follows.

Every function is pinned by CPU tests (``tests/test_oracle_*.py``) against
closed forms, invariants, brute force and finite differences.
"""
from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from ._build import build_oracle, library_path

__all__ = [
    "decode", "forward_bits", "forward_f64", "forward_i8", "forward_i8_token", "dot_bits",
    "backward_f64", "build_csr", "topk", "rerank_two_stage", "chamfer_nn", "chamfer_forward",
    "chamfer_backward", "chamfer_csr", "chamfer_pair_dist", "dot_i8_token", "DTYPE_CODES",
]

DTYPE_CODES = {"fp16": 0, "bf16": 1}

_lib = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i8p = np.ctypeslib.ndpointer(dtype=np.int8, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_vp = ctypes.c_void_p


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        build_oracle()
    lib = ctypes.CDLL(path)
    I32, I64, F32, INT = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    lib.oracle_decode.argtypes = [INT, _u16p, _f64p, I64]
    lib.oracle_decode.restype = INT
    lib.oracle_forward_f64.argtypes = [_f64p, _i32p, I32, I32, _f64p, _i32p, I32, I32,
                                       I64, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.oracle_forward_f64.restype = INT
    lib.oracle_forward_bits.argtypes = [INT, _u16p, _i32p, I32, I32, _u16p, _i32p, I32, I32,
                                        I64, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.oracle_forward_bits.restype = INT
    lib.oracle_dot_bits.argtypes = [INT, _u16p, I32, _u16p, _i32p, I32, I64,
                                    _i32p, _i32p, _i32p, _i32p, _f64p]
    lib.oracle_dot_bits.restype = INT
    lib.oracle_forward_i8.argtypes = [_i8p, _i32p, I32, I32, _i8p, _i32p, I32, I32, F32, F32,
                                      I64, _vp, _vp, _vp, _vp, _vp]
    lib.oracle_forward_i8.restype = INT
    lib.oracle_forward_i8_token.argtypes = [_i8p, _f32p, _i32p, I32, I32, _i8p, _f32p, _i32p, I32, I32,
                                            I64, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.oracle_forward_i8_token.restype = INT
    lib.oracle_dot_i8_token.argtypes = [_i8p, I32, _i8p, _f32p, _i32p, I32, I64, _i32p, _i32p, _i32p, _i32p,
                                        _f64p]
    lib.oracle_dot_i8_token.restype = INT
    lib.oracle_chamfer_pair_dist.argtypes = [_f32p, _f32p, I64, _i32p, _i32p, _f64p]
    lib.oracle_chamfer_pair_dist.restype = INT
    lib.oracle_chamfer_nn.argtypes = [_f32p, _i32p, _f32p, _i32p, I32, _f64p, _i32p, _vp]
    lib.oracle_chamfer_nn.restype = INT
    lib.oracle_chamfer_reduce.argtypes = [_f64p, _i32p, _f64p, _i32p, I32, _f64p]
    lib.oracle_chamfer_reduce.restype = INT
    lib.oracle_chamfer_backward.argtypes = [_f32p, _i32p, _f32p, _i32p, I32, _i32p, _i32p, _f64p, _f64p, _f64p]
    lib.oracle_chamfer_backward.restype = INT
    lib.oracle_backward_f64.argtypes = [_f64p, _i32p, _f64p, _i32p, I32, I32, _f64p, _i32p,
                                        I32, I32, _f64p, _f64p]
    lib.oracle_backward_f64.restype = INT
    lib.oracle_build_csr.argtypes = [_i32p, _i32p, I32, I32, _i32p, I32, _i64p, _i64p]
    lib.oracle_build_csr.restype = I64
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _pairs(pairs, n_q, n_docs):
    if pairs is None:
        qq, bb = np.divmod(np.arange(n_q * n_docs, dtype=np.int64), max(n_docs, 1))
        return qq.astype(np.int32), bb.astype(np.int32)
    pairs = np.asarray(pairs, dtype=np.int32).reshape(-1, 2)
    return np.ascontiguousarray(pairs[:, 0]), np.ascontiguousarray(pairs[:, 1])


def decode(dtype: str, bits: np.ndarray) -> np.ndarray:
    """Exact binary64 value of stored FP16 / BF16 patterns (uint16 array)."""
    lib = _load()
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    rc = lib.oracle_decode(DTYPE_CODES[dtype], bits.reshape(-1), out.reshape(-1), bits.size)
    if rc != 0:
        raise ValueError("oracle_decode failed")
    return out


def _run_chunks(n_pairs, threads, fn):
    """Split [0, n_pairs) into contiguous chunks evaluated on a thread pool.

    The C calls release the GIL, so chunks run on separate cores."""
    threads = max(1, int(threads))
    if threads == 1 or n_pairs < 2 * threads:
        fn(0, n_pairs)
        return
    step = (n_pairs + threads - 1) // threads
    with ThreadPoolExecutor(max_workers=threads) as ex:
        futs = [ex.submit(fn, s, min(n_pairs, s + step)) for s in range(0, n_pairs, step)]
        for f in futs:
            f.result()


def forward_bits(dtype: str, Q_bits, q_lens, D_bits, cu_seqlens, pairs=None,
                 want_rowmax=False, threads=1):
    """Flash-MaxSim §1 Eq. (1) on stored FP16/BF16 patterns, in binary64.

    Q_bits: uint16 [n_q, lq_max, dim]; D_bits: uint16 [total_tokens, dim];
    cu_seqlens: int32 [n_docs + 1].  ``pairs``: optional int array [P, 2] of
    (q, b); default = every pair in (q, b) row-major order.
    Returns dict(score [P] f64, argmax [P, lq_max] i32, and when want_rowmax,
    rowmax [P, lq_max] f64 and gap [P, lq_max] f64 = top-1 minus top-2).
    """
    lib = _load()
    Q_bits = _c(Q_bits, np.uint16)
    D_bits = _c(D_bits, np.uint16)
    q_lens = _c(q_lens, np.int32)
    cu = _c(cu_seqlens, np.int32)
    n_q, lq_max, dim = Q_bits.shape
    n_docs = cu.shape[0] - 1
    pq, pb = _pairs(pairs, n_q, n_docs)
    P = pq.shape[0]
    score = np.empty(P, np.float64)
    argmax = np.empty((P, lq_max), np.int32)
    rowmax = np.empty((P, lq_max), np.float64) if want_rowmax else None
    gap = np.empty((P, lq_max), np.float64) if want_rowmax else None
    code = DTYPE_CODES[dtype]

    def run(s, e):
        if e <= s:
            return
        rc = lib.oracle_forward_bits(
            code, Q_bits.reshape(-1), q_lens, n_q, lq_max, D_bits.reshape(-1), cu, n_docs, dim,
            e - s, _ptr(pq[s:e]), _ptr(pb[s:e]), _ptr(score[s:e]), _ptr(argmax[s:e]),
            _ptr(None if rowmax is None else rowmax[s:e]), _ptr(None if gap is None else gap[s:e]))
        if rc != 0:
            raise ValueError(f"oracle_forward_bits failed ({rc})")

    _run_chunks(P, threads, run)
    out = {"score": score, "argmax": argmax}
    if want_rowmax:
        out["rowmax"] = rowmax
        out["gap"] = gap
    return out


def forward_f64(Q, q_lens, D, cu_seqlens, pairs=None, want_rowmax=False):
    """Flash-MaxSim §1 Eq. (1) on binary64 inputs (used by the finite-difference
    and closed-form pins).  Shapes as in forward_bits."""
    lib = _load()
    Q = _c(Q, np.float64)
    D = _c(D, np.float64)
    q_lens = _c(q_lens, np.int32)
    cu = _c(cu_seqlens, np.int32)
    n_q, lq_max, dim = Q.shape
    n_docs = cu.shape[0] - 1
    pq, pb = _pairs(pairs, n_q, n_docs)
    P = pq.shape[0]
    score = np.empty(P, np.float64)
    argmax = np.empty((P, lq_max), np.int32)
    rowmax = np.empty((P, lq_max), np.float64)
    gap = np.empty((P, lq_max), np.float64)
    Dflat = D.reshape(-1) if D.size else np.zeros(1, np.float64)
    rc = lib.oracle_forward_f64(Q.reshape(-1), q_lens, n_q, lq_max, Dflat, cu, n_docs, dim,
                                P, _ptr(pq), _ptr(pb), _ptr(score), _ptr(argmax),
                                _ptr(rowmax), _ptr(gap))
    if rc != 0:
        raise ValueError(f"oracle_forward_f64 failed ({rc})")
    out = {"score": score, "argmax": argmax}
    if want_rowmax:
        out["rowmax"] = rowmax
        out["gap"] = gap
    return out


def dot_bits(dtype, Q_bits, D_bits, cu_seqlens, q, b, i, t):
    """Exact <Q[q,i], D[cu[b]+t]> for arrays of (q, b, i, t)."""
    lib = _load()
    Q_bits = _c(Q_bits, np.uint16)
    D_bits = _c(D_bits, np.uint16)
    cu = _c(cu_seqlens, np.int32)
    n_q, lq_max, dim = Q_bits.shape
    q, b, i, t = (_c(x, np.int32).reshape(-1) for x in (q, b, i, t))
    out = np.empty(q.shape[0], np.float64)
    rc = lib.oracle_dot_bits(DTYPE_CODES[dtype], Q_bits.reshape(-1), lq_max, D_bits.reshape(-1),
                             cu, dim, q.shape[0], q, b, i, t, out)
    if rc != 0:
        raise ValueError("oracle_dot_bits failed")
    return out


def forward_i8(Q, q_lens, D, cu_seqlens, q_scale, d_scale, pairs=None, threads=1):
    """Flash-MaxSim §4.3.1 INT8 x INT8 MaxSim with one scale per tensor:
    exact int dots, int maxima (lowest t on ties), int64 sum, one scale.
    Returns dict(raw [P] int64, score [P] f32, argmax [P, lq_max] i32)."""
    lib = _load()
    Q = _c(Q, np.int8)
    D = _c(D, np.int8)
    q_lens = _c(q_lens, np.int32)
    cu = _c(cu_seqlens, np.int32)
    n_q, lq_max, dim = Q.shape
    n_docs = cu.shape[0] - 1
    pq, pb = _pairs(pairs, n_q, n_docs)
    P = pq.shape[0]
    raw = np.empty(P, np.int64)
    score = np.empty(P, np.float32)
    argmax = np.empty((P, lq_max), np.int32)
    Dflat = D.reshape(-1) if D.size else np.zeros(1, np.int8)

    def run(s, e):
        if e <= s:
            return
        rc = lib.oracle_forward_i8(Q.reshape(-1), q_lens, n_q, lq_max, Dflat, cu, n_docs, dim,
                                   float(q_scale), float(d_scale), e - s, _ptr(pq[s:e]),
                                   _ptr(pb[s:e]), _ptr(raw[s:e]), _ptr(score[s:e]),
                                   _ptr(argmax[s:e]))
        if rc != 0:
            raise ValueError(f"oracle_forward_i8 failed ({rc})")

    _run_chunks(P, threads, run)
    return {"raw": raw, "score": score, "argmax": argmax}


def forward_i8_token(Q, q_scales, q_lens, D, d_scales, cu_seqlens, pairs=None, want_rowmax=False,
                     threads=1):
    """Flash-MaxSim §4.3.1 INT8 x INT8 MaxSim with one scale per token (the
    reading in oracle.c, R6): the value ranked is the exact product
    dot * d_scale[t] in binary64, the row maximum (lowest t on ties) is
    multiplied by the query token's scale and summed in binary64.  Q int8
    [n_q, lq_max, dim], q_scales f32 [n_q, lq_max], D int8 [total, dim],
    d_scales f32 [total].  Returns dict(score [P] f64, argmax [P, lq_max]
    i32, and when want_rowmax, rowmax [P, lq_max] f64 and gap [P, lq_max] f64
    = top-1 minus top-2)."""
    lib = _load()
    Q = _c(Q, np.int8)
    D = _c(D, np.int8)
    qs = _c(q_scales, np.float32)
    ds = _c(d_scales, np.float32)
    q_lens = _c(q_lens, np.int32)
    cu = _c(cu_seqlens, np.int32)
    n_q, lq_max, dim = Q.shape
    n_docs = cu.shape[0] - 1
    pq, pb = _pairs(pairs, n_q, n_docs)
    P = pq.shape[0]
    score = np.empty(P, np.float64)
    argmax = np.empty((P, lq_max), np.int32)
    rowmax = np.empty((P, lq_max), np.float64) if want_rowmax else None
    gap = np.empty((P, lq_max), np.float64) if want_rowmax else None
    Dflat = D.reshape(-1) if D.size else np.zeros(1, np.int8)
    dsflat = ds.reshape(-1) if ds.size else np.zeros(1, np.float32)

    def run(s, e):
        if e <= s:
            return
        rc = lib.oracle_forward_i8_token(Q.reshape(-1), qs.reshape(-1), q_lens, n_q, lq_max, Dflat, dsflat,
                                         cu, n_docs, dim, e - s, _ptr(pq[s:e]), _ptr(pb[s:e]),
                                         _ptr(score[s:e]), _ptr(argmax[s:e]),
                                         _ptr(None if rowmax is None else rowmax[s:e]),
                                         _ptr(None if gap is None else gap[s:e]))
        if rc != 0:
            raise ValueError(f"oracle_forward_i8_token failed ({rc})")

    _run_chunks(P, threads, run)
    out = {"score": score, "argmax": argmax}
    if want_rowmax:
        out["rowmax"] = rowmax
        out["gap"] = gap
    return out


def dot_i8_token(Q, D, d_scales, cu_seqlens, q, b, i, t):
    """Exact ranked value dot(Q[q,i], D[cu[b]+t]) * d_scales[cu[b]+t] (R6)
    for arrays of (q, b, i, t)."""
    lib = _load()
    Q = _c(Q, np.int8)
    D = _c(D, np.int8)
    ds = _c(d_scales, np.float32)
    cu = _c(cu_seqlens, np.int32)
    n_q, lq_max, dim = Q.shape
    q, b, i, t = (_c(x, np.int32).reshape(-1) for x in (q, b, i, t))
    out = np.empty(q.shape[0], np.float64)
    lib.oracle_dot_i8_token(Q.reshape(-1), lq_max, D.reshape(-1), ds.reshape(-1), cu, dim, q.shape[0],
                            q, b, i, t, out)
    return out


def topk(values, k, ids=None):
    """Per row of ``values`` [n_rows, n], the k largest entries in descending
    order, ties to the lower column (a stable sort on the negated values).
    Rows with fewer than k columns are padded with id -1 and value -inf.
    ``ids`` [n_rows, n] maps a column to the id reported (default: the
    column).  Returns (ids [n_rows, k] int32, values [n_rows, k])."""
    values = np.asarray(values)
    n_rows, n = values.shape
    out_ids = np.full((n_rows, k), -1, np.int32)
    out_val = np.full((n_rows, k), -np.inf, values.dtype)
    m = min(k, n)
    for r in range(n_rows):
        order = np.argsort(-values[r], kind="stable")[:m]
        out_ids[r, :m] = order if ids is None else np.asarray(ids)[r, order]
        out_val[r, :m] = values[r, order]
    return out_ids, out_val


def rerank_two_stage(Q8, D8, q_scale, d_scale, dtype16, Q16_bits, D16_bits, q_lens, cu_seqlens, k_candidates,
                     k, q_tok_scales=None, d_tok_scales=None, threads=1):
    """The two-stage INT8 -> FP16 top-K scan of Flash-MaxSim §4.1 ("Kernel
    Family"), read plainly: score every document with the INT8 MaxSim (one
    scale per tensor, or per token when both token-scale arrays are given),
    keep each query's k_candidates best documents (ties to the lower
    document index), rescore those with the FP16/BF16 MaxSim and return each
    query's k best of them.  Returns dict(cand_ids [n_q, k_candidates],
    stage1 [n_q, n_docs], ids [n_q, k], scores [n_q, k] (binary64))."""
    q_lens = _c(q_lens, np.int32)
    cu = _c(cu_seqlens, np.int32)
    n_q = q_lens.shape[0]
    n_docs = cu.shape[0] - 1
    if q_tok_scales is not None:
        s1 = forward_i8_token(Q8, q_tok_scales, q_lens, D8, d_tok_scales, cu, threads=threads)["score"]
    else:
        s1 = forward_i8(Q8, q_lens, D8, cu, q_scale, d_scale, threads=threads)["score"]
    s1 = s1.reshape(n_q, n_docs)
    cand, _ = topk(s1, k_candidates)
    pairs = np.array([(q, b) for q in range(n_q) for b in cand[q] if b >= 0], np.int32).reshape(-1, 2)
    s2 = np.full((n_q, k_candidates), -np.inf)
    if len(pairs):
        sc = forward_bits(dtype16, Q16_bits, q_lens, D16_bits, cu, pairs=pairs, threads=threads)["score"]
        pos = 0
        for q in range(n_q):
            m = int((cand[q] >= 0).sum())
            s2[q, :m] = sc[pos:pos + m]
            pos += m
    ids, scores = topk(s2, k, ids=cand)
    return {"cand_ids": cand, "stage1": s1, "ids": ids, "scores": scores}


def _pts(a):
    a = _c(a, np.float32).reshape(-1, 3)
    return a if a.size else np.zeros((1, 3), np.float32)


def chamfer_nn(S, cu_s, T, cu_t, want_gap=False):
    """Nearest target of every source point (reading R7 in oracle.c): binary64
    squared distances [total_s] and target indices local to the item
    [total_s]; with want_gap also the second-smallest distance minus the
    smallest [total_s]."""
    lib = _load()
    cu_s, cu_t = _c(cu_s, np.int32), _c(cu_t, np.int32)
    n = int(cu_s[-1])
    dist = np.empty(max(n, 1), np.float64)
    arg = np.empty(max(n, 1), np.int32)
    gap = np.empty(max(n, 1), np.float64) if want_gap else None
    rc = lib.oracle_chamfer_nn(_pts(S).reshape(-1), cu_s, _pts(T).reshape(-1), cu_t, cu_s.shape[0] - 1, dist, arg,
                               _ptr(gap))
    if rc != 0:
        raise ValueError("oracle_chamfer_nn failed")
    if want_gap:
        return dist[:n], arg[:n], gap[:n]
    return dist[:n], arg[:n]


def chamfer_pair_dist(S, T, s_idx, t_idx):
    """Squared distances (R7) of (source, target) index pairs (global indices
    into the packed point arrays), binary64."""
    lib = _load()
    s_idx, t_idx = _c(s_idx, np.int32).reshape(-1), _c(t_idx, np.int32).reshape(-1)
    out = np.empty(s_idx.shape[0], np.float64)
    lib.oracle_chamfer_pair_dist(_pts(S).reshape(-1), _pts(T).reshape(-1), s_idx.shape[0], s_idx, t_idx, out)
    return out


def chamfer_forward(P, cu_p, Q, cu_q):
    """Chamfer distance of every item (Flash-MaxSim §4.2, "Generalization to
    Chamfer Distance"), binary64: dict(cd [B], dist_pq, arg_pq, gap_pq,
    dist_qp, arg_qp, gap_qp)."""
    lib = _load()
    cu_p, cu_q = _c(cu_p, np.int32), _c(cu_q, np.int32)
    d_pq, a_pq, g_pq = chamfer_nn(P, cu_p, Q, cu_q, want_gap=True)
    d_qp, a_qp, g_qp = chamfer_nn(Q, cu_q, P, cu_p, want_gap=True)
    B = cu_p.shape[0] - 1
    cd = np.empty(max(B, 1), np.float64)
    lib.oracle_chamfer_reduce(np.ascontiguousarray(d_pq) if d_pq.size else np.zeros(1, np.float64), cu_p,
                              np.ascontiguousarray(d_qp) if d_qp.size else np.zeros(1, np.float64), cu_q, B, cd)
    return {"cd": cd[:B], "dist_pq": d_pq, "arg_pq": a_pq, "gap_pq": g_pq, "dist_qp": d_qp, "arg_qp": a_qp,
            "gap_qp": g_qp}


def chamfer_backward(P, cu_p, Q, cu_q, arg_pq, arg_qp, grad):
    """Gradient of sum_b grad[b] * cd[b] for given nearest-neighbour indices,
    in binary64 scatter form.  Returns (dP [N, 3], dQ [M, 3]) float64."""
    lib = _load()
    cu_p, cu_q = _c(cu_p, np.int32), _c(cu_q, np.int32)
    N, M = int(cu_p[-1]), int(cu_q[-1])
    dP = np.zeros(max(3 * N, 1), np.float64)
    dQ = np.zeros(max(3 * M, 1), np.float64)
    a_pq = _c(arg_pq, np.int32) if N else np.zeros(1, np.int32)
    a_qp = _c(arg_qp, np.int32) if M else np.zeros(1, np.int32)
    rc = lib.oracle_chamfer_backward(_pts(P).reshape(-1), cu_p, _pts(Q).reshape(-1), cu_q, cu_p.shape[0] - 1,
                                     a_pq, a_qp, _c(grad, np.float64), dP, dQ)
    if rc != 0:
        raise ValueError("oracle_chamfer_backward failed")
    return dP[:3 * N].reshape(N, 3), dQ[:3 * M].reshape(M, 3)


def chamfer_csr(arg, cu_src, cu_dst):
    """Inverse of a nearest-neighbour map (Flash-MaxSim §4.2.2 applied to
    Chamfer): source i of item b points at destination cu_dst[b] + arg[i];
    row_ptr [total_dst + 1] = exclusive cumulative count per destination,
    col_idx = sources ordered by destination, ascending source within one
    (a stable argsort of the destinations).  Sources with arg -1 are left
    out."""
    arg = np.asarray(arg, np.int64)
    cu_src, cu_dst = np.asarray(cu_src, np.int64), np.asarray(cu_dst, np.int64)
    item = np.repeat(np.arange(len(cu_src) - 1), np.diff(cu_src))
    keep = arg >= 0
    dst = cu_dst[item[keep]] + arg[keep]
    src = np.nonzero(keep)[0]
    order = np.argsort(dst, kind="stable")
    row_ptr = np.zeros(int(cu_dst[-1]) + 1, np.int64)
    np.add.at(row_ptr, dst + 1, 1)
    return np.cumsum(row_ptr).astype(np.int32), src[order].astype(np.int32)


def backward_f64(grad, argmax, Q, q_lens, D, cu_seqlens):
    """Flash-MaxSim §4.2.1 Eqs. (2)-(3) in scatter form, binary64.
    grad [n_q, n_docs]; argmax [n_q, n_docs, lq_max]; Q [n_q, lq_max, dim]
    (float64 values); D [total, dim].  Returns (dQ, dD) in float64."""
    lib = _load()
    grad = _c(grad, np.float64)
    argmax = _c(argmax, np.int32)
    Q = _c(Q, np.float64)
    D = _c(D, np.float64)
    q_lens = _c(q_lens, np.int32)
    cu = _c(cu_seqlens, np.int32)
    n_q, lq_max, dim = Q.shape
    n_docs = cu.shape[0] - 1
    total = int(cu[-1]) if n_docs > 0 else 0
    dQ = np.empty((n_q, lq_max, dim), np.float64)
    dD = np.empty((max(total, 1), dim), np.float64)
    Dflat = D.reshape(-1) if D.size else np.zeros(1, np.float64)
    rc = lib.oracle_backward_f64(grad.reshape(-1), argmax.reshape(-1), Q.reshape(-1), q_lens,
                                 n_q, lq_max, Dflat, cu, n_docs, dim,
                                 dQ.reshape(-1), dD.reshape(-1))
    if rc != 0:
        raise ValueError(f"oracle_backward_f64 failed ({rc})")
    return dQ, dD[:total]


def build_csr(argmax, q_lens, cu_seqlens):
    """Flash-MaxSim §4.2.2 / Alg. 3 step 1: inverse-grid CSR of the argmax map.
    Returns (row_ptr [total+1] int64, col_idx [nnz] int64)."""
    lib = _load()
    argmax = _c(argmax, np.int32)
    q_lens = _c(q_lens, np.int32)
    cu = _c(cu_seqlens, np.int32)
    n_q, n_docs, lq_max = argmax.shape
    total = int(cu[-1]) if n_docs > 0 else 0
    row_ptr = np.empty(total + 1, np.int64)
    col_idx = np.empty(max(1, n_q * n_docs * lq_max), np.int64)
    nnz = lib.oracle_build_csr(argmax.reshape(-1), q_lens, n_q, lq_max, cu, n_docs,
                               row_ptr, col_idx)
    if nnz < 0:
        raise ValueError(f"oracle_build_csr failed ({nnz})")
    return row_ptr, col_idx[:nnz]
