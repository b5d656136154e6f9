"""Pins for the oracle's INT8 forward with one scale per token (Flash-MaxSim
§4.3.1, per-token symmetric quantisation; the reading: rank the exact real
products dot * s_D[t] -- exact in binary64 -- take the lowest index of the
maximum, multiply it by s_Q[i], sum in binary64).  CPU only.

  * unit scales reduce it to the per-tensor INT8 forward with scale 1, whose
    raw integer sums are exact;
  * for arbitrary scales an independent float64 numpy brute force (integer
    matrix product, one exact product with the scale, first-occurrence
    argmax, a sequential sum) agrees bit for bit, top-2 gaps included;
  * two products that round to the same binary32 value are still told
    apart (the ranking is exact, not rounded);
  * a planted mistake (the query scale dropped) fails the brute force."""
import numpy as np

import oracle

RNG = np.random.default_rng(2024)


def _cu(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def _case(n_q=3, lq=12, lengths=(5, 33, 1, 0, 17, 64), seed=0):
    rng = np.random.default_rng(seed)
    cu = _cu(np.array(lengths))
    Q = rng.integers(-127, 128, (n_q, lq, 128)).astype(np.int8)
    D = rng.integers(-127, 128, (int(cu[-1]), 128)).astype(np.int8)
    q_lens = np.array([lq] + [max(0, lq - 5 * k) for k in range(1, n_q)], np.int32)
    return Q, q_lens, D, cu


def _brute_exact(Q, q_lens, D, cu, qs, ds):
    """float64 brute force: the integer dots (below 2^24) times the binary32
    scales are exact in float64; the score sums query tokens in order."""
    n_q, lq = Q.shape[:2]
    n_docs = len(cu) - 1
    score = np.zeros((n_q, n_docs))
    arg = -np.ones((n_q, n_docs, lq), np.int32)
    for q in range(n_q):
        for b in range(n_docs):
            S = Q[q, :q_lens[q]].astype(np.float64) @ D[cu[b]:cu[b + 1]].astype(np.float64).T
            S = S * ds[cu[b]:cu[b + 1]].astype(np.float64)[None, :]
            if S.shape[1] == 0:
                score[q, b] = -np.inf if q_lens[q] else 0.0
                continue
            arg[q, b, :q_lens[q]] = S.argmax(1)
            acc = 0.0
            for i, v in enumerate(S.max(1)):
                acc += float(qs[q, i]) * float(v)
            score[q, b] = acc
    return score, arg


def test_unit_scales_equal_the_per_tensor_forward():
    Q, q_lens, D, cu = _case()
    qs = np.ones(Q.shape[:2], np.float32)
    ds = np.ones(D.shape[0], np.float32)
    tok = oracle.forward_i8_token(Q, qs, q_lens, D, ds, cu)
    ten = oracle.forward_i8(Q, q_lens, D, cu, 1.0, 1.0)
    finite = ten["raw"] != np.iinfo(np.int64).min
    assert np.array_equal(tok["score"][finite], ten["raw"][finite].astype(np.float64))
    assert np.all(np.isneginf(tok["score"][~finite]))
    assert np.array_equal(tok["argmax"], ten["argmax"])


def test_power_of_two_scales_match_float64_brute_force_exactly():
    Q, q_lens, D, cu = _case(seed=1)
    qs = np.exp2(RNG.integers(-12, -4, Q.shape[:2])).astype(np.float32)
    ds = np.exp2(RNG.integers(-12, -4, D.shape[0])).astype(np.float32)
    out = oracle.forward_i8_token(Q, qs, q_lens, D, ds, cu)
    score, arg = _brute_exact(Q, q_lens, D, cu, qs, ds)
    assert np.array_equal(out["score"], score.reshape(-1))
    assert np.array_equal(out["argmax"], arg.reshape(-1, Q.shape[1]))


def test_dropping_the_query_scale_is_caught():
    """The brute force above is sensitive to the query-token scale."""
    Q, q_lens, D, cu = _case(seed=2)
    qs = np.exp2(RNG.integers(-12, -4, Q.shape[:2])).astype(np.float32)
    ds = np.exp2(RNG.integers(-12, -4, D.shape[0])).astype(np.float32)
    out = oracle.forward_i8_token(Q, qs, q_lens, D, ds, cu)
    wrong, _ = _brute_exact(Q, q_lens, D, cu, np.ones_like(qs), ds)
    finite = np.isfinite(wrong.reshape(-1)) & (wrong.reshape(-1) != 0)
    assert not np.array_equal(out["score"][finite], wrong.reshape(-1)[finite])


def test_general_scales_match_float64_brute_force_exactly():
    Q, q_lens, D, cu = _case(seed=3)
    qs = RNG.uniform(1e-3, 1e-2, Q.shape[:2]).astype(np.float32)
    ds = RNG.uniform(1e-3, 1e-2, D.shape[0]).astype(np.float32)
    out = oracle.forward_i8_token(Q, qs, q_lens, D, ds, cu, want_rowmax=True)
    score, arg = _brute_exact(Q, q_lens, D, cu, qs, ds)
    assert np.array_equal(out["score"], score.reshape(-1))
    assert np.array_equal(out["argmax"], arg.reshape(-1, Q.shape[1]))
    n_q, lq = Q.shape[:2]
    n_docs = len(cu) - 1
    for q in range(n_q):
        for b in range(n_docs):
            p = q * n_docs + b
            S = Q[q, :q_lens[q]].astype(np.float64) @ D[cu[b]:cu[b + 1]].astype(np.float64).T
            S = S * ds[cu[b]:cu[b + 1]].astype(np.float64)[None, :]
            if S.shape[1] == 0 or q_lens[q] == 0:
                continue
            srt = np.sort(S, 1)
            assert np.array_equal(out["rowmax"][p, :q_lens[q]], srt[:, -1])
            if S.shape[1] >= 2:
                assert np.array_equal(out["gap"][p, :q_lens[q]], srt[:, -1] - srt[:, -2])


def test_ranking_is_exact_not_rounded_to_binary32():
    """Token 0 has value 1 x 2^20, token 1 has 3 x (349525 + 11/32) =
    2^20 + 1/32.  Rounded to binary32 (spacing 1/8 at 2^20) both are 2^20 and
    the lower index would win; exactly, token 1 is the maximum by 1/32."""
    Q = np.zeros((1, 1, 128), np.int8)
    Q[0, 0, 0] = 1
    D = np.zeros((2, 128), np.int8)
    D[0, 0] = 1
    D[1, 0] = 3
    ds = np.array([2.0 ** 20, 349525.0 + 11.0 / 32.0], np.float32)
    assert float(ds[1]) == 349525.0 + 11.0 / 32.0                       # exact in binary32
    assert np.float32(3) * ds[1] == np.float32(2.0 ** 20)               # the binary32 products tie
    out = oracle.forward_i8_token(Q, np.ones((1, 1), np.float32), [1], D, ds, np.array([0, 2], np.int32),
                                  want_rowmax=True)
    assert out["argmax"][0, 0] == 1
    assert out["rowmax"][0, 0] == 2.0 ** 20 + 1.0 / 32.0
    assert out["gap"][0, 0] == 1.0 / 32.0


def test_empty_documents_and_empty_queries():
    Q, q_lens, D, cu = _case(n_q=2, lq=4, lengths=(0, 3, 0), seed=4)
    q_lens = np.array([4, 0], np.int32)
    qs = np.full(Q.shape[:2], 0.5, np.float32)
    ds = np.full(D.shape[0], 0.25, np.float32)
    out = oracle.forward_i8_token(Q, qs, q_lens, D, ds, cu)
    sc = out["score"].reshape(2, 3)
    assert np.isneginf(sc[0, 0]) and np.isneginf(sc[0, 2]) and np.isfinite(sc[0, 1])
    assert np.array_equal(sc[1], [0.0, 0.0, 0.0])
    assert np.all(out["argmax"].reshape(2, 3, 4)[0, 0] == -1)
    assert np.all(out["argmax"].reshape(2, 3, 4)[1] == -1)


def test_zero_scale_token_ranks_as_zero():
    """A document token quantised from an all-zero vector has scale 0: its
    value is 0 for every query token."""
    Q = np.full((1, 1, 128), 1, np.int8)
    D = np.stack([np.full(128, -1, np.int8), np.full(128, 5, np.int8)])
    cu = _cu(np.array([2]))
    out = oracle.forward_i8_token(Q, np.ones((1, 1), np.float32), [1], D, np.array([1.0, 0.0], np.float32), cu)
    # token 0: -128 * 1 = -128; token 1: 640 * 0 = 0 -> token 1 wins
    assert out["argmax"][0, 0] == 1 and out["score"][0] == 0.0


def test_value_of_a_chosen_token_matches_brute_force():
    """oracle.dot_i8_token (used to judge the kernel's near-tie choices)
    returns the exact ranked value of any (q, b, i, t)."""
    Q, q_lens, D, cu = _case(seed=6)
    ds = RNG.uniform(1e-3, 1e-2, D.shape[0]).astype(np.float32)
    rng = np.random.default_rng(7)
    n_docs = len(cu) - 1
    docs = [b for b in range(n_docs) if cu[b + 1] > cu[b]]
    bb = rng.choice(docs, 50)
    qq = rng.integers(0, Q.shape[0], 50)
    ii = rng.integers(0, Q.shape[1], 50)
    tt = np.array([rng.integers(0, cu[b + 1] - cu[b]) for b in bb])
    got = oracle.dot_i8_token(Q, D, ds, cu, qq, bb, ii, tt)
    want = [float(Q[q, i].astype(np.int64) @ D[cu[b] + t].astype(np.int64)) * float(ds[cu[b] + t])
            for q, b, i, t in zip(qq, bb, ii, tt)]
    assert np.array_equal(got, np.array(want))
