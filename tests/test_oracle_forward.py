"""Pins for the oracle's forward (Flash-MaxSim §1 Eq. (1), §4.1, §4.3.2).

Each test checks the oracle against something other than itself: closed
forms, invariants the pages state, brute force through numpy, or the
definition of the storage formats.  CPU only.
"""
import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


def _f16_bits(x):
    return np.ascontiguousarray(np.asarray(x, np.float16)).view(np.uint16)


def _cu(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


# --------------------------------------------------------------------------
# storage decoding: every one of the 65,536 patterns, against numpy / torch
# --------------------------------------------------------------------------

def test_decode_fp16_every_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode("fp16", bits)
    ref = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_decode_bf16_every_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode("bf16", bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def test_one_hot_integer_scores_and_lowest_index():
    """Q_i = e_{a_i}, D_t = e_{c_t}: <Q_i, D_t> = [a_i == c_t], so the score is
    #{i : a_i in {c_t}}, the argmax is the first t with c_t = a_i, and when
    no token matches every value is 0 and the lowest index (0) wins."""
    dim = 128
    lq, ld = 24, 40
    a = RNG.integers(0, dim, lq)
    c = RNG.integers(0, dim, ld)
    a[0] = dim - 1                   # last coordinate: catches a dropped term
    c[ld - 1] = dim - 1
    a[1] = c[5]
    c[17] = c[5]                     # a duplicate: the lower index must win
    Q = np.zeros((1, lq, dim))
    Q[0, np.arange(lq), a] = 1.0
    D = np.zeros((ld, dim))
    D[np.arange(ld), c] = 1.0
    out = oracle.forward_f64(Q, [lq], D, [0, ld])
    expect = sum(1 for ai in a if ai in set(c.tolist()))
    assert out["score"][0] == float(expect)
    for i, ai in enumerate(a):
        hits = np.nonzero(c == ai)[0]
        assert out["argmax"][0, i] == (hits[0] if hits.size else 0)


def _signed_quads(n, dim, rng):
    """Rows with four entries of +-0.5 and zeros elsewhere: exactly unit norm
    in FP16, and two distinct rows have inner product <= 0.75."""
    rows = set()
    out = []
    while len(out) < n:
        idx = tuple(sorted(rng.choice(dim, 4, replace=False).tolist()))
        sg = tuple(rng.choice([-1, 1], 4).tolist())
        if (idx, sg) in rows:
            continue
        rows.add((idx, sg))
        v = np.zeros(dim)
        v[list(idx)] = 0.5 * np.array(sg)
        out.append(v)
    return np.array(out)


def test_exact_copies_score_equals_lq():
    """A document holding exact copies of the unit-norm query rows scores
    exactly Lq, with each argmax at the (first) copy."""
    dim, lq, ld = 128, 32, 96
    rows = _signed_quads(lq + ld, dim, RNG)
    Q = rows[:lq][None]
    D = rows[lq:].copy()
    pos = RNG.choice(ld, lq, replace=False)
    D[pos] = Q[0]
    dup = pos[3]
    other = [t for t in range(dup) if t not in set(pos.tolist())]
    if other:                          # a second, earlier copy of row 3
        D[other[0]] = Q[0, 3]
    Qb, Db = _f16_bits(Q), _f16_bits(D)
    out = oracle.forward_bits("fp16", Qb, [lq], Db, [0, ld])
    assert out["score"][0] == float(lq)
    exp = pos.copy()
    if other:
        exp[3] = other[0]
    assert np.array_equal(out["argmax"][0], exp)


def test_negative_scores_still_pick_the_maximum():
    """All inner products negative: the maximum (closest to zero) is taken,
    never a padding zero (masking with -inf, §4.1.1)."""
    dim = 128
    q = np.zeros(dim)
    q[7] = 1.0
    D = np.zeros((5, dim))
    D[:, 7] = [-0.5, -0.25, -0.75, -0.125, -1.0]
    out = oracle.forward_f64(q[None, None], [1], D, [0, 5])
    assert out["score"][0] == -0.125
    assert out["argmax"][0, 0] == 3


# --------------------------------------------------------------------------
# brute force through numpy (the materialised path of §3.1, Alg. 1)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_brute_force_materialised(dtype):
    n_q, lq_max, dim = 3, 9, 128
    lengths = np.array([1, 7, 16, 33, 2])
    cu = _cu(lengths)
    q_lens = np.array([9, 4, 1], np.int32)
    Qf = torch.randn(n_q, lq_max, dim, generator=torch.Generator().manual_seed(5))
    Df = torch.randn(int(cu[-1]), dim, generator=torch.Generator().manual_seed(6))
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    Qb = Qf.to(tdt).view(torch.int16).numpy().view(np.uint16)
    Db = Df.to(tdt).view(torch.int16).numpy().view(np.uint16)
    out = oracle.forward_bits(dtype, Qb, q_lens, Db, cu, want_rowmax=True)
    Qv = Qf.to(tdt).double().numpy()
    Dv = Df.to(tdt).double().numpy()
    p = 0
    for q in range(n_q):
        for b in range(len(lengths)):
            S = np.einsum("id,td->it", Qv[q, :q_lens[q]], Dv[cu[b]:cu[b + 1]])
            m = S.max(axis=1)
            assert out["score"][p] == pytest.approx(m.sum(), rel=1e-12, abs=1e-12)
            am = S.argmax(axis=1)       # numpy returns the first maximum
            gap = out["gap"][p, :q_lens[q]]
            sure = gap > 1e-9
            assert np.array_equal(out["argmax"][p, :q_lens[q]][sure], am[sure])
            assert np.all(out["argmax"][p, q_lens[q]:] == -1)
            p += 1


def test_pairs_subset_matches_full():
    n_q, lq, dim = 2, 5, 128
    lengths = np.array([3, 8, 1, 12])
    cu = _cu(lengths)
    Q = RNG.standard_normal((n_q, lq, dim))
    D = RNG.standard_normal((int(cu[-1]), dim))
    full = oracle.forward_f64(Q, [5, 3], D, cu)
    pairs = np.array([[1, 3], [0, 0], [1, 1]])
    sub = oracle.forward_f64(Q, [5, 3], D, cu, pairs=pairs)
    for k, (q, b) in enumerate(pairs):
        assert sub["score"][k] == full["score"][q * 4 + b]
        assert np.array_equal(sub["argmax"][k], full["argmax"][q * 4 + b])


def test_bits_path_matches_f64_path():
    n_q, lq, dim = 2, 6, 128
    lengths = np.array([4, 9, 2])
    cu = _cu(lengths)
    Q = RNG.standard_normal((n_q, lq, dim)).astype(np.float16)
    D = RNG.standard_normal((int(cu[-1]), dim)).astype(np.float16)
    a = oracle.forward_bits("fp16", Q.view(np.uint16), [6, 2], D.view(np.uint16), cu)
    b = oracle.forward_f64(Q.astype(np.float64), [6, 2], D.astype(np.float64), cu)
    assert np.array_equal(a["score"], b["score"])
    assert np.array_equal(a["argmax"], b["argmax"])


# --------------------------------------------------------------------------
# invariants and special cases
# --------------------------------------------------------------------------

def test_score_bounded_by_lq_for_unit_vectors():
    dim, lq = 128, 32
    Q = RNG.standard_normal((1, lq, dim))
    Q /= np.linalg.norm(Q, axis=-1, keepdims=True)
    D = RNG.standard_normal((200, dim))
    D /= np.linalg.norm(D, axis=-1, keepdims=True)
    out = oracle.forward_f64(Q, [lq], D, [0, 100, 200])
    assert np.all(out["score"] <= lq + 1e-12)
    assert np.all(out["score"] > 0)


def test_doc_token_permutation_invariance():
    dim, lq, ld = 128, 16, 50
    Q = RNG.standard_normal((1, lq, dim))
    D = RNG.standard_normal((ld, dim))
    perm = RNG.permutation(ld)
    a = oracle.forward_f64(Q, [lq], D, [0, ld], want_rowmax=True)
    b = oracle.forward_f64(Q, [lq], D[perm], [0, ld])
    assert a["score"][0] == b["score"][0]
    # D[perm][k] = D[perm[k]]  =>  the winner t of D appears at k = inv[t]
    inv = np.argsort(perm)
    assert np.array_equal(b["argmax"][0], inv[a["argmax"][0]])


def test_query_chunk_additivity():
    """§4.1: the sum of maxima decomposes over query chunks."""
    dim, lq = 128, 40
    Q = RNG.standard_normal((1, lq, dim))
    D = RNG.standard_normal((70, dim))
    cu = [0, 30, 70]
    whole = oracle.forward_f64(Q, [lq], D, cu)["score"]
    first = oracle.forward_f64(Q[:, :17], [17], D, cu)["score"]
    rest = oracle.forward_f64(Q[:, 17:], [lq - 17], D, cu)["score"]
    np.testing.assert_allclose(whole, first + rest, rtol=1e-13, atol=1e-12)


def test_varlen_equals_per_document_dense():
    """§4.3.2 / §5.5: the packed cu_seqlens result equals scoring each
    document on its own, exactly."""
    dim, lq = 128, 8
    lengths = np.array([5, 1, 0, 13, 7])
    cu = _cu(lengths)
    Q = RNG.standard_normal((2, lq, dim))
    D = RNG.standard_normal((int(cu[-1]), dim))
    packed = oracle.forward_f64(Q, [8, 5], D, cu)
    for b in range(len(lengths)):
        alone = oracle.forward_f64(Q, [8, 5], D[cu[b]:cu[b + 1]], [0, lengths[b]])
        for q in range(2):
            assert packed["score"][q * 5 + b] == alone["score"][q] or (
                np.isneginf(packed["score"][q * 5 + b]) and np.isneginf(alone["score"][q]))
            assert np.array_equal(packed["argmax"][q * 5 + b], alone["argmax"][q])


def test_positive_homogeneity():
    dim, lq = 128, 12
    Q = RNG.standard_normal((1, lq, dim))
    D = RNG.standard_normal((20, dim))
    a = oracle.forward_f64(Q, [lq], D, [0, 20])
    b = oracle.forward_f64(Q, [lq], 4.0 * D, [0, 20])
    assert b["score"][0] == 4.0 * a["score"][0]
    assert np.array_equal(a["argmax"], b["argmax"])


def test_single_doc_token_is_inner_product_of_query_sum():
    dim, lq = 128, 10
    Q = RNG.standard_normal((1, lq, dim))
    d = RNG.standard_normal((1, dim))
    out = oracle.forward_f64(Q, [lq], d, [0, 1])
    assert out["score"][0] == pytest.approx(float(Q[0].sum(0) @ d[0]), rel=1e-12)
    assert np.all(out["argmax"][0] == 0)


def test_single_query_token_is_max_of_matvec():
    dim = 128
    q = RNG.standard_normal((1, 1, dim))
    D = RNG.standard_normal((64, dim))
    out = oracle.forward_f64(q, [1], D, [0, 64])
    v = D @ q[0, 0]
    assert out["score"][0] == pytest.approx(v.max(), rel=1e-12)
    assert out["argmax"][0, 0] == int(np.argmax(v))


def test_empty_document_and_empty_query():
    """Readings: an empty document scores -inf with argmax -1; a query with
    no valid tokens scores 0 with argmax -1 everywhere."""
    dim = 128
    Q = RNG.standard_normal((2, 4, dim))
    D = RNG.standard_normal((3, dim))
    cu = [0, 0, 3]
    out = oracle.forward_f64(Q, [4, 0], D, cu)
    assert np.isneginf(out["score"][0])
    assert np.all(out["argmax"][0] == -1)
    assert out["score"][2] == 0.0 and out["score"][3] == 0.0
    assert np.all(out["argmax"][2:] == -1)
    assert np.isfinite(out["score"][1])


def test_padded_query_rows_are_ignored():
    dim = 128
    Q = RNG.standard_normal((1, 6, dim))
    D = RNG.standard_normal((9, dim))
    a = oracle.forward_f64(Q, [4], D, [0, 9])
    Q2 = Q.copy()
    Q2[0, 4:] = 1e3                    # garbage in the padding
    b = oracle.forward_f64(Q2, [4], D, [0, 9])
    assert a["score"][0] == b["score"][0]
    assert np.all(b["argmax"][0, 4:] == -1)


def test_skeptic_recipe_lengths():
    """The pages' suggested check (random pairs at lengths 128/256/512): the
    oracle agrees with the materialised numpy path on those shapes."""
    dim = 128
    for lq, ld in [(128, 256), (256, 512), (512, 128)]:
        Q = RNG.standard_normal((1, lq, dim)).astype(np.float16)
        D = RNG.standard_normal((ld, dim)).astype(np.float16)
        out = oracle.forward_bits("fp16", Q.view(np.uint16), [lq], D.view(np.uint16), [0, ld])
        S = Q[0].astype(np.float64) @ D.astype(np.float64).T
        assert out["score"][0] == pytest.approx(S.max(1).sum(), rel=1e-12)


def test_dot_bits_matches_decoded_product():
    dim = 128
    Q = RNG.standard_normal((2, 3, dim)).astype(np.float16)
    D = RNG.standard_normal((10, dim)).astype(np.float16)
    cu = np.array([0, 4, 10], np.int32)
    v = oracle.dot_bits("fp16", Q.view(np.uint16), D.view(np.uint16), cu,
                        [1, 0], [1, 0], [2, 0], [5, 3])
    assert v[0] == pytest.approx(float(Q[1, 2].astype(np.float64) @ D[9].astype(np.float64)), rel=1e-14)
    assert v[1] == pytest.approx(float(Q[0, 0].astype(np.float64) @ D[3].astype(np.float64)), rel=1e-14)
