"""Pins for the oracle's INT8 x INT8 forward (Flash-MaxSim §4.3.1, read with
one symmetric scale per tensor).  Exact integer arithmetic: checked against an
int64 numpy brute force and adversarial extremes.  CPU only."""
import numpy as np

import oracle

RNG = np.random.default_rng(99)


def _cu(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def _brute(Q, q_lens, D, cu, qs, ds):
    n_q = Q.shape[0]
    n_docs = len(cu) - 1
    raw = np.zeros((n_q, n_docs), np.int64)
    arg = -np.ones((n_q, n_docs, Q.shape[1]), np.int32)
    for q in range(n_q):
        for b in range(n_docs):
            S = Q[q, :q_lens[q]].astype(np.int64) @ D[cu[b]:cu[b + 1]].astype(np.int64).T
            if S.shape[1] == 0:
                raw[q, b] = np.iinfo(np.int64).min if q_lens[q] else 0
                continue
            raw[q, b] = S.max(1).sum()
            arg[q, b, :q_lens[q]] = S.argmax(1)
    score = np.where(raw == np.iinfo(np.int64).min, -np.inf,
                     (raw.astype(np.float64) * (np.float64(qs) * np.float64(ds)))).astype(np.float32)
    return raw, score, arg


def test_random_against_int64_brute_force():
    lengths = np.array([3, 40, 1, 17, 0, 64])
    cu = _cu(lengths)
    Q = RNG.integers(-127, 128, (3, 20, 128)).astype(np.int8)
    D = RNG.integers(-127, 128, (int(cu[-1]), 128)).astype(np.int8)
    q_lens = np.array([20, 7, 0], np.int32)
    qs, ds = np.float32(0.0037), np.float32(0.0041)
    out = oracle.forward_i8(Q, q_lens, D, cu, qs, ds)
    raw, score, arg = _brute(Q, q_lens, D, cu, qs, ds)
    assert np.array_equal(out["raw"], raw.reshape(-1))
    assert np.array_equal(out["score"], score.reshape(-1))
    assert np.array_equal(out["argmax"], arg.reshape(-1, 20))


def test_extreme_magnitudes_fit_int32():
    """All entries +-127: |dot| reaches 128 * 127^2 = 2,064,512."""
    Q = np.full((1, 2, 128), 127, np.int8)
    Q[0, 1] = -127
    D = np.full((3, 128), 127, np.int8)
    D[1] = -127
    out = oracle.forward_i8(Q, [2], D, [0, 3], 1.0, 1.0)
    assert out["raw"][0] == 2 * 128 * 127 * 127
    assert np.array_equal(out["argmax"][0], [0, 1])
    assert out["score"][0] == np.float32(2 * 2064512)


def test_ties_go_to_lowest_index():
    Q = RNG.integers(-127, 128, (1, 4, 128)).astype(np.int8)
    D = np.repeat(RNG.integers(-127, 128, (1, 128)).astype(np.int8), 6, axis=0)
    out = oracle.forward_i8(Q, [4], D, [0, 6], 1.0, 1.0)
    assert np.all(out["argmax"][0] == 0)


def test_alternating_signs_cancel():
    q = np.tile(np.array([127, -127], np.int8), 64)[None, None]
    D = np.stack([np.full(128, 127, np.int8), np.tile(np.array([1, -1], np.int8), 64)])
    out = oracle.forward_i8(q, [1], D, [0, 2], 1.0, 1.0)
    assert out["raw"][0] == 128 * 127
    assert out["argmax"][0, 0] == 1


def test_scale_applied_once_in_binary64():
    Q = RNG.integers(-127, 128, (1, 32, 128)).astype(np.int8)
    D = RNG.integers(-127, 128, (50, 128)).astype(np.int8)
    qs, ds = np.float32(1 / 300), np.float32(1 / 257)
    out = oracle.forward_i8(Q, [32], D, [0, 50], qs, ds)
    S = Q[0].astype(np.int64) @ D.astype(np.int64).T
    raw = int(S.max(1).sum())
    assert out["raw"][0] == raw
    assert out["score"][0] == np.float32(float(raw) * (float(qs) * float(ds)))
