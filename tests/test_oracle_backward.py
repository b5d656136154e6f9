"""Pins for the oracle's backward (Flash-MaxSim §4.2.1 Eqs. (2)-(3)) and its
inverse-grid CSR (§4.2.2, Alg. 3 step 1).  CPU only.

Finite differences of L = sum_{q,b} g[q,b] * score(q,b) in binary64 on
tie-free inputs (the score is piecewise linear, so central differences are
exact up to rounding while no argmax flips), Euler's identity for the
degree-1 homogeneous score, and the CSR against numpy's own bincount /
cumsum / stable argsort.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(7)


def _cu(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def _tie_free(n_q, lq, lengths, dim=128, min_gap=1e-2, seed=0):
    rng = np.random.default_rng(seed)
    cu = _cu(lengths)
    while True:
        Q = rng.standard_normal((n_q, lq, dim))
        D = rng.standard_normal((int(cu[-1]), dim))
        out = oracle.forward_f64(Q, [lq] * n_q, D, cu, want_rowmax=True)
        if np.all(out["gap"][np.isfinite(out["gap"])] > min_gap):
            return Q, D, cu, out


def _loss(Q, q_lens, D, cu, g):
    s = oracle.forward_f64(Q, q_lens, D, cu)["score"]
    return float((s * g.reshape(-1)).sum())


def test_finite_differences():
    n_q, lq = 2, 3
    lengths = np.array([4, 1, 6])
    Q, D, cu, fwd = _tie_free(n_q, lq, lengths, dim=128, seed=3)
    q_lens = np.array([lq, lq], np.int32)
    g = RNG.standard_normal((n_q, len(lengths)))
    argmax = fwd["argmax"].reshape(n_q, len(lengths), lq)
    dQ, dD = oracle.backward_f64(g, argmax, Q, q_lens, D, cu)
    h = 1e-4
    for _ in range(40):
        q, i, k = RNG.integers(0, n_q), RNG.integers(0, lq), RNG.integers(0, 128)
        Qp, Qm = Q.copy(), Q.copy()
        Qp[q, i, k] += h
        Qm[q, i, k] -= h
        fd = (_loss(Qp, q_lens, D, cu, g) - _loss(Qm, q_lens, D, cu, g)) / (2 * h)
        assert fd == pytest.approx(dQ[q, i, k], rel=1e-6, abs=1e-8)
    for _ in range(40):
        r, k = RNG.integers(0, D.shape[0]), RNG.integers(0, 128)
        Dp, Dm = D.copy(), D.copy()
        Dp[r, k] += h
        Dm[r, k] -= h
        fd = (_loss(Q, q_lens, Dp, cu, g) - _loss(Q, q_lens, Dm, cu, g)) / (2 * h)
        assert fd == pytest.approx(dD[r, k], rel=1e-6, abs=1e-8)


def test_euler_identity_and_unselected_rows():
    """score is positively homogeneous of degree 1 in Q and in D, so
    sum <dQ, Q> = sum <dD, D> = sum g * score; rows nobody selected get 0."""
    n_q, lq = 3, 5
    lengths = np.array([7, 2, 9, 4])
    Q, D, cu, fwd = _tie_free(n_q, lq, lengths, seed=11)
    q_lens = np.array([5, 2, 4], np.int32)
    fwd = oracle.forward_f64(Q, q_lens, D, cu)
    g = RNG.standard_normal((n_q, len(lengths)))
    argmax = fwd["argmax"].reshape(n_q, len(lengths), lq)
    dQ, dD = oracle.backward_f64(g, argmax, Q, q_lens, D, cu)
    total = float((g.reshape(-1) * fwd["score"]).sum())
    assert float((dQ * Q).sum()) == pytest.approx(total, rel=1e-12)
    assert float((dD * D).sum()) == pytest.approx(total, rel=1e-12)
    for q in range(n_q):
        assert np.all(dQ[q, q_lens[q]:] == 0)
    selected = np.zeros(D.shape[0], bool)
    for q in range(n_q):
        for b in range(len(lengths)):
            for i in range(q_lens[q]):
                selected[cu[b] + argmax[q, b, i]] = True
    assert np.all(dD[~selected] == 0)
    assert np.all(np.abs(dD[selected]).sum(1) > 0)


def test_backward_rejects_out_of_range_argmax():
    Q = RNG.standard_normal((1, 2, 128))
    D = RNG.standard_normal((3, 128))
    with pytest.raises(ValueError):
        oracle.backward_f64(np.ones((1, 1)), np.array([[[0, 3]]], np.int32), Q, [2], D, [0, 3])


def _numpy_csr(argmax, q_lens, cu):
    """Alg. 3 step 1 with numpy's primitives: dst -> bincount -> cumsum, and
    a stable argsort of dst."""
    n_q, n_docs, lq_max = argmax.shape
    q = np.arange(n_q)[:, None, None]
    b = np.arange(n_docs)[None, :, None]
    i = np.arange(lq_max)[None, None, :]
    valid = (i < np.asarray(q_lens)[:, None, None]) & (argmax >= 0)
    src = ((q * n_docs + b) * lq_max + i)
    dst = (np.asarray(cu)[:-1][None, :, None] + argmax)
    src, dst = src[valid], dst[valid]
    order = np.argsort(dst, kind="stable")
    row_ptr = np.concatenate([[0], np.cumsum(np.bincount(dst, minlength=int(cu[-1])))])
    return row_ptr, src[order]


def test_csr_matches_numpy_primitives():
    n_q, lq = 4, 6
    lengths = np.array([5, 0, 3, 11, 1])
    cu = _cu(lengths)
    q_lens = np.array([6, 2, 0, 5], np.int32)
    argmax = -np.ones((n_q, len(lengths), lq), np.int32)
    for q in range(n_q):
        for b in range(len(lengths)):
            if lengths[b]:
                # skewed: many rows hit token 0 (a hot token)
                argmax[q, b, :q_lens[q]] = np.where(RNG.random(q_lens[q]) < 0.5, 0,
                                                    RNG.integers(0, lengths[b], q_lens[q]))
    row_ptr, col_idx = oracle.build_csr(argmax, q_lens, cu)
    rp, ci = _numpy_csr(argmax, q_lens, cu)
    assert np.array_equal(row_ptr, rp)
    assert np.array_equal(col_idx, ci)
    nonempty = int((lengths > 0).sum())
    assert row_ptr[-1] == int(q_lens.sum()) * nonempty
    for r in range(int(cu[-1])):
        seg = col_idx[row_ptr[r]:row_ptr[r + 1]]
        assert np.all(np.diff(seg) > 0)          # ascending sources in a row


def test_dd_through_csr_equals_scatter():
    """The destination-owned reduction over the CSR (Alg. 3 step 2) gives the
    scatter-form dD of Eq. (3)."""
    n_q, lq = 3, 4
    lengths = np.array([6, 3, 8])
    cu = _cu(lengths)
    Q = RNG.standard_normal((n_q, lq, 128))
    D = RNG.standard_normal((int(cu[-1]), 128))
    q_lens = np.array([4, 4, 3], np.int32)
    fwd = oracle.forward_f64(Q, q_lens, D, cu)
    argmax = fwd["argmax"].reshape(n_q, 3, lq)
    g = RNG.standard_normal((n_q, 3))
    _, dD = oracle.backward_f64(g, argmax, Q, q_lens, D, cu)
    row_ptr, col_idx = oracle.build_csr(argmax, q_lens, cu)
    dD2 = np.zeros_like(dD)
    for r in range(int(cu[-1])):
        for s in col_idx[row_ptr[r]:row_ptr[r + 1]]:
            q, rem = divmod(int(s), 3 * lq)
            b, i = divmod(rem, lq)
            dD2[r] += g[q, b] * Q[q, i]
    np.testing.assert_allclose(dD2, dD, rtol=1e-13, atol=1e-13)
