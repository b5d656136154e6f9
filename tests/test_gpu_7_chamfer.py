"""Chamfer distance on the GPU (Flash-MaxSim §4.2 "Generalization to Chamfer
Distance") against the oracle:

  * nearest-neighbour distances and indices against the binary64 oracle:
    distance within 2^-18 of the exact minimum (the kernel evaluates it in
    binary32), index equal wherever the exact top-2 gap exceeds 2^-19 of the
    second distance and a near-minimum elsewhere -- on ragged batches with
    empty sets and duplicated points, and on a large pair split into target
    slices (sampled points); on integer coordinates both sides are exact and
    every index and distance must match bit for bit (lowest index on ties);
  * the per-item distance within 2^-17 relative;
  * the inverse CSR bit-exact; gradients within 1e-4 of the largest
    gradient; every output identical on a second run."""
import numpy as np
import pytest
import torch

import oracle
from maxsim_testlib import check_chamfer_nn

pytestmark = pytest.mark.gpu

CD_REL = 2.0 ** -17


def _cloud(sizes, seed, dup_every=0):
    g = torch.Generator("cuda").manual_seed(seed)
    total = int(sum(sizes))
    X = torch.rand((total, 3), generator=g, device="cuda") * 2 - 1
    if dup_every and total > dup_every:
        X[dup_every::dup_every] = X[0:total - dup_every:dup_every][: X[dup_every::dup_every].shape[0]]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(sizes)]), dtype=torch.int32, device="cuda")
    return X.contiguous(), cu


def _check_forward(ops, P, cu_p, Q, cu_q, exact=False):
    cd, d_pq, a_pq, d_qp, a_qp = ops.maxsim_chamfer_forward(P, cu_p, Q, cu_q)
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    Ph, Qh, cph, cqh = P.cpu().numpy(), Q.cpu().numpy(), cu_p.cpu().numpy(), cu_q.cpu().numpy()
    ref = oracle.chamfer_forward(Ph, cph, Qh, cqh)
    if exact:
        assert np.array_equal(d_pq.double().cpu().numpy(), ref["dist_pq"])
        assert np.array_equal(a_pq.cpu().numpy(), ref["arg_pq"])
        assert np.array_equal(d_qp.double().cpu().numpy(), ref["dist_qp"])
        assert np.array_equal(a_qp.cpu().numpy(), ref["arg_qp"])
    else:
        check_chamfer_nn(Ph, cph, Qh, cqh, d_pq.cpu().numpy(), a_pq.cpu().numpy())
        check_chamfer_nn(Qh, cqh, Ph, cph, d_qp.cpu().numpy(), a_qp.cpu().numpy())
    got, want = cd.double().cpu().numpy(), ref["cd"]
    assert np.array_equal(np.isinf(got), np.isinf(want))
    fin = np.isfinite(want)
    assert np.all(np.abs(got[fin] - want[fin]) <= CD_REL * np.abs(want[fin]))
    return cd, d_pq, a_pq, d_qp, a_qp


def test_forward_ragged_batch_with_empty_sets(ops):
    P, cu_p = _cloud([0, 1, 100, 1500, 5000, 37], seed=1, dup_every=7)
    Q, cu_q = _cloud([3, 0, 2000, 1500, 700, 1], seed=2, dup_every=5)
    _check_forward(ops, P, cu_p, Q, cu_q)


def test_forward_integer_coordinates_bit_exact(ops):
    """Integer coordinates: every distance is exact in binary32 and binary64,
    ties are everywhere, and the lowest index must win them."""
    g = torch.Generator("cuda").manual_seed(14)
    P = torch.randint(-12, 13, (2600, 3), generator=g, device="cuda").float()
    Q = torch.randint(-12, 13, (3100, 3), generator=g, device="cuda").float()
    cu_p = torch.tensor([0, 100, 100, 2600], dtype=torch.int32, device="cuda")
    cu_q = torch.tensor([0, 1, 1100, 3100], dtype=torch.int32, device="cuda")
    _check_forward(ops, P, cu_p, Q, cu_q, exact=True)


def test_forward_identical_sets(ops):
    P, cu = _cloud([3000], seed=3)
    cd, d_pq, a_pq, _, _ = _check_forward(ops, P, cu, P.clone(), cu)
    assert float(cd[0]) == 0.0
    assert torch.equal(a_pq.cpu(), torch.arange(3000, dtype=torch.int32))


def test_forward_large_pair_sliced(ops):
    """60,000 x 50,000 points: the target set is split into slices merged in
    order; sampled points are checked against the oracle one by one."""
    P, cu_p = _cloud([60_000], seed=4, dup_every=1000)
    Q, cu_q = _cloud([50_000], seed=5, dup_every=999)
    cd, d_pq, a_pq, d_qp, a_qp = ops.maxsim_chamfer_forward(P, cu_p, Q, cu_q)
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    rng = np.random.default_rng(6)
    for S, T, d, a in ((P, Q, d_pq, a_pq), (Q, P, d_qp, a_qp)):
        idx = np.sort(rng.choice(S.shape[0], 400, replace=False))
        check_chamfer_nn(S.cpu().numpy(), np.array([0, S.shape[0]], np.int32), T.cpu().numpy(),
                         np.array([0, T.shape[0]], np.int32), d.cpu().numpy(), a.cpu().numpy(), rows=idx)
    ref_cd = float(d_pq.double().mean() + d_qp.double().mean())
    assert abs(float(cd[0]) - ref_cd) <= 1e-6 * ref_cd


def test_csr_bit_exact(ops):
    P, cu_p = _cloud([400, 0, 2500, 9], seed=7)
    Q, cu_q = _cloud([50, 30, 100, 0], seed=8)
    _, _, a_pq, _, _ = ops.maxsim_chamfer_forward(P, cu_p, Q, cu_q)
    row_ptr, col = ops.maxsim_chamfer_build_csr(a_pq, cu_p, cu_q, Q.shape[0])
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    r_row, r_col = oracle.chamfer_csr(a_pq.cpu().numpy(), cu_p.cpu().numpy(), cu_q.cpu().numpy())
    assert np.array_equal(row_ptr.cpu().numpy(), r_row)
    n = int(r_row[-1])
    assert np.array_equal(col.cpu().numpy()[:n], r_col)


def test_csr_many_passes(ops):
    """More than 2^16 destinations: three 8-bit radix passes, hot rows."""
    n_src, n_dst = 300_000, 70_000
    g = torch.Generator("cuda").manual_seed(9)
    arg = torch.randint(0, n_dst, (n_src,), generator=g, device="cuda", dtype=torch.int32)
    arg[::3] = 12345
    arg[1::17] = -1
    cu_src = torch.tensor([0, n_src], dtype=torch.int32, device="cuda")
    cu_dst = torch.tensor([0, n_dst], dtype=torch.int32, device="cuda")
    row_ptr, col = ops.maxsim_chamfer_build_csr(arg, cu_src, cu_dst, n_dst)
    torch.cuda.synchronize()
    r_row, r_col = oracle.chamfer_csr(arg.cpu().numpy(), [0, n_src], [0, n_dst])
    assert np.array_equal(row_ptr.cpu().numpy(), r_row)
    assert np.array_equal(col.cpu().numpy()[:int(r_row[-1])], r_col)


def test_backward_matches_oracle_and_is_deterministic(ops):
    P, cu_p = _cloud([300, 1200, 0, 64], seed=10)
    Q, cu_q = _cloud([200, 900, 5, 0], seed=11)
    g = torch.tensor([1.0, -0.5, 2.0, 0.25], device="cuda")
    cd, _, a_pq, _, a_qp = ops.maxsim_chamfer_forward(P, cu_p, Q, cu_q)
    dP, dQ = ops.maxsim_chamfer_backward(g, P, cu_p, Q, cu_q, a_pq, a_qp)
    torch.cuda.synchronize()
    assert ops.maxsim_device_status() == 0
    rP, rQ = oracle.chamfer_backward(P.cpu().numpy(), cu_p.cpu().numpy(), Q.cpu().numpy(), cu_q.cpu().numpy(),
                                     a_pq.cpu().numpy(), a_qp.cpu().numpy(), g.double().cpu().numpy())
    scale = max(np.abs(rP).max(), np.abs(rQ).max())
    assert np.abs(dP.double().cpu().numpy() - rP).max() <= 1e-4 * scale
    assert np.abs(dQ.double().cpu().numpy() - rQ).max() <= 1e-4 * scale
    dP2, dQ2 = ops.maxsim_chamfer_backward(g, P, cu_p, Q, cu_q, a_pq, a_qp)
    torch.cuda.synchronize()
    assert torch.equal(dP, dP2) and torch.equal(dQ, dQ2)


def test_backward_matches_torch_autograd(ops):
    """The materialised fp32 form of the same loss, differentiated by torch."""
    P, cu_p = _cloud([500], seed=12)
    Q, cu_q = _cloud([400], seed=13)
    cd, _, a_pq, _, a_qp = ops.maxsim_chamfer_forward(P, cu_p, Q, cu_q)
    Pr, Qr = P.clone().requires_grad_(True), Q.clone().requires_grad_(True)
    D = ((Pr[:, None, :] - Qr[None, :, :]) ** 2).sum(-1)
    loss = D.min(1).values.mean() + D.min(0).values.mean()
    loss.backward()
    dP, dQ = ops.maxsim_chamfer_backward(torch.ones(1, device="cuda"), P, cu_p, Q, cu_q, a_pq, a_qp)
    assert abs(float(loss.detach()) - float(cd[0])) <= 1e-5 * float(loss.detach())
    assert torch.allclose(dP, Pr.grad, atol=1e-5 * float(Pr.grad.abs().max()), rtol=1e-3)
    assert torch.allclose(dQ, Qr.grad, atol=1e-5 * float(Qr.grad.abs().max()), rtol=1e-3)
