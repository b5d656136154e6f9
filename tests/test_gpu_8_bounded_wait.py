"""The kernels' failure path on the GPU, without a fault: a CTA holding tensor
memory waits on a barrier that nothing completes; its bounded wait must give
up, record its code in the device status word, release the tensor memory and
leave the context usable."""
import time

import pytest
import torch

from maxsim_testlib import check_forward, random_case

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_reports(ops):
    assert ops.maxsim_device_status() == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ops.maxsim_selftest_bounded_wait(20_000)            # 20 ms
    code = ops.maxsim_device_status(clear=True)
    elapsed = time.perf_counter() - t0
    assert code == 0x105
    assert elapsed >= 0.019
    assert ops.maxsim_device_status() == 0               # cleared


def test_context_usable_after_expired_waits(ops):
    """Two expired self-tests in a row (each allocates and must have freed
    tensor memory), then a forward that allocates it again."""
    for _ in range(2):
        ops.maxsim_selftest_bounded_wait(2_000)
    assert ops.maxsim_device_status(clear=True) == 0x105
    Q, ql, D, cu = random_case(2, 32, [40, 129, 7], "fp16", [32, 5], seed=3)
    scores, argmax, _ = ops.maxsim_forward(Q, ql, D, cu)
    assert ops.maxsim_device_status() == 0
    check_forward("fp16", Q, ql, D, cu, scores, argmax)


def test_limit_out_of_range_is_rejected(ops):
    with pytest.raises(Exception):
        ops.maxsim_selftest_bounded_wait(0)
    with pytest.raises(Exception):
        ops.maxsim_selftest_bounded_wait(2_000_000)
    assert ops.maxsim_device_status() == 0
