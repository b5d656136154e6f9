"""The autograd entry point against a plain PyTorch fp32 reference: the
materialised einsum -> max -> sum of Flash-MaxSim §3.1 differentiated by
torch.autograd, on tie-free inputs (so the max is differentiable there)."""
import pytest
import torch

from maxsim_testlib import random_case

pytestmark = pytest.mark.gpu


def _torch_reference(Q, D, q_lens, cu):
    """fp32 materialised MaxSim per (query, document) pair, differentiable."""
    n_q = Q.shape[0]
    cu_h = cu.tolist()
    rows = []
    for q in range(n_q):
        qi = Q[q, : int(q_lens[q])]
        row = []
        for b in range(len(cu_h) - 1):
            S = qi @ D[cu_h[b]:cu_h[b + 1]].T
            row.append(S.max(dim=1).values.sum())
        rows.append(torch.stack(row))
    return torch.stack(rows)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_autograd_matches_torch_reference(ops, dtype):
    from late_interaction_retrieval_maxsim_gb300.autograd import maxsim
    name = "fp16" if dtype == torch.float16 else "bf16"
    lengths = [7, 130, 1, 64, 200]
    Q, ql, D, cu = random_case(3, 40, lengths, name, [40, 33, 12], seed=77)
    g = torch.randn((3, len(lengths)), device="cuda", generator=torch.Generator("cuda").manual_seed(5))

    Qa = Q.clone().requires_grad_(True)
    Da = D.clone().requires_grad_(True)
    s = maxsim(Qa, Da, ql, cu)
    (s * g).sum().backward()

    Qr = Q.float().clone().requires_grad_(True)
    Dr = D.float().clone().requires_grad_(True)
    sr = _torch_reference(Qr, Dr, ql.cpu(), cu.cpu())
    (sr * g).sum().backward()

    assert torch.allclose(s, sr.detach(), atol=1e-4 * 40, rtol=0)
    # gradients are computed in FP32 by the kernels, then rounded to the input dtype
    tol = 1e-2 * max(1.0, float(Qr.grad.abs().max()))
    assert torch.allclose(Qa.grad.float(), Qr.grad, atol=tol, rtol=0)
    tol = 1e-2 * max(1.0, float(Dr.grad.abs().max()))
    assert torch.allclose(Da.grad.float(), Dr.grad, atol=tol, rtol=0)


@pytest.mark.parametrize("lq", [32, 100])
def test_autograd_grads_equal_the_c_abi_backward(ops, lq):
    """Bit-equal to the C ABI's forward + backward (32- and 100-token
    queries)."""
    from late_interaction_retrieval_maxsim_gb300.autograd import maxsim
    Q, ql, D, cu = random_case(4, lq, [180] * 16, "bf16", seed=78)
    Qa = Q.clone().requires_grad_(True)
    Da = D.clone().requires_grad_(True)
    s = maxsim(Qa, Da, ql, cu)
    g = torch.softmax(s.detach() / 0.05, dim=1)
    s.backward(g)
    _, am, _ = ops.maxsim_forward(Q, ql, D, cu)
    dQ, dD = ops.maxsim_backward(g.contiguous(), am, Q, ql, D, cu)
    assert torch.equal(Qa.grad, dQ.to(torch.bfloat16))
    assert torch.equal(Da.grad, dD.to(torch.bfloat16))


def test_autograd_second_backward_through_the_same_graph(ops):
    """A second backward through the retained graph gives the same
    gradients as the first."""
    from late_interaction_retrieval_maxsim_gb300.autograd import maxsim
    Q, ql, D, cu = random_case(4, 32, [180] * 8, "bf16", seed=79)
    Qa = Q.clone().requires_grad_(True)
    Da = D.clone().requires_grad_(True)
    s = maxsim(Qa, Da, ql, cu)
    g = torch.softmax(s.detach() / 0.05, dim=1)
    s.backward(g, retain_graph=True)
    gq, gd = Qa.grad.clone(), Da.grad.clone()
    Qa.grad = None
    Da.grad = None
    s.backward(g)
    assert torch.equal(Qa.grad, gq) and torch.equal(Da.grad, gd)
