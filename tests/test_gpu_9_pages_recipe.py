"""The concrete test the pith.science review page proposes for this method
("concrete_test"): forward scores and backward gradients compared element
by element with a reference MaxSim on 128 random (query length, document
length) pairs drawn from {128, 256, 512}, in FP16 and in INT8; scores within
1e-5 and gradients within 1e-4.

Here the reference is the oracle (binary64 / int64).  The 128 pairs are
batched as 128 queries x 128 documents and pair k is (query k, document k);
the upstream gradient is nonzero on those pairs only.  Scores must meet the
page's 1e-5 relative bound and the 1e-4 * Lq bound, gradients 1e-4 of
max|grad|, the argmax the rule of maxsim_testlib; the INT8 forward (one scale
per tensor) is bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from late_interaction_retrieval_maxsim_gb300 import synthetic as syn
from maxsim_testlib import GRAD_TOL, THREADS, check_forward

pytestmark = pytest.mark.gpu

N_PAIRS = 128
LENGTHS = (128, 256, 512)


def _recipe(seed=0):
    rng = np.random.default_rng(seed)
    q_lens = rng.choice(LENGTHS, N_PAIRS).astype(np.int32)
    d_lens = rng.choice(LENGTHS, N_PAIRS).astype(np.int32)
    cu = syn.cu_seqlens_from_lengths(torch.as_tensor(d_lens))
    return q_lens, d_lens, cu


def test_pages_recipe_fp16_scores_and_gradients(ops):
    q_lens, _, cu = _recipe()
    lq_max = int(max(LENGTHS))
    total = int(cu[-1])
    Q = syn.unit_tokens(N_PAIRS * lq_max, 128, 101, "fp16", "cuda").view(N_PAIRS, lq_max, 128)
    D = syn.unit_tokens(total, 128, 102, "fp16", "cuda")
    ql = torch.as_tensor(q_lens, device="cuda")
    cu_d = cu.cuda()
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu_d)
    assert ops.maxsim_device_status() == 0
    diag = [(k, k) for k in range(N_PAIRS)]
    check_forward("fp16", Q, ql, D, cu_d, scores, argmax, pairs=diag)
    qb, db = syn.bits_u16(Q), syn.bits_u16(D)
    ref = oracle.forward_bits("fp16", qb, q_lens, db, cu.numpy(), pairs=diag, threads=THREADS)["score"]
    got = scores.diagonal().double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 1e-5 * np.abs(ref)), "the page's 1e-5 relative score bound"

    g = torch.zeros((N_PAIRS, N_PAIRS), device="cuda")
    g.diagonal().copy_(torch.randn(N_PAIRS, device="cuda", generator=torch.Generator("cuda").manual_seed(7)))
    dQ, dD = ops.maxsim_backward(g, argmax, Q, ql, D, cu_d)
    assert ops.maxsim_device_status() == 0
    rq, rd = oracle.backward_f64(g.double().cpu().numpy(), argmax.cpu().numpy(), oracle.decode("fp16", qb),
                                 q_lens, oracle.decode("fp16", db), cu.numpy())
    for got_g, want in ((dQ, rq), (dD, rd)):
        err = float(np.abs(got_g.double().cpu().numpy() - want).max())
        assert err <= GRAD_TOL * float(np.abs(want).max()), f"gradient error {err:.3e}"


def test_pages_recipe_int8_bit_exact(ops):
    q_lens, _, cu = _recipe(seed=1)
    lq_max = int(max(LENGTHS))
    total = int(cu[-1])
    Q8, qs = syn.unit_tokens_int8(N_PAIRS * lq_max, 128, 201, "cuda")
    D8, ds = syn.unit_tokens_int8(total, 128, 202, "cuda")
    Q8 = Q8.view(N_PAIRS, lq_max, 128)
    ql = torch.as_tensor(q_lens, device="cuda")
    scores, argmax, raw = ops.maxsim_forward(Q8, ql, D8, cu.cuda(), q_scale=qs, d_scale=ds, want_raw=True)
    assert ops.maxsim_device_status() == 0
    diag = [(k, k) for k in range(N_PAIRS)]
    ref = oracle.forward_i8(Q8.cpu().numpy(), q_lens, D8.cpu().numpy(), cu.numpy(), qs, ds, pairs=diag,
                            threads=THREADS)
    k = torch.arange(N_PAIRS)
    assert np.array_equal(raw.cpu()[k, k].numpy(), ref["raw"])
    assert np.array_equal(scores.cpu()[k, k].numpy(), ref["score"])
    assert np.array_equal(argmax.cpu()[k, k].numpy(), ref["argmax"])
