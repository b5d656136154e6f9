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


def test_l2_read_probe_reads_every_word(ops):
    """The L2 read probe (the measuring stick of the backward's roofline)
    folds every 16-byte word it reads into its sink: with one pass the XOR of
    all sink words equals the XOR of all 32-bit words of the buffer."""
    import numpy as np
    g = torch.Generator("cuda").manual_seed(5)
    buf = torch.randint(-2**31, 2**31 - 1, (3 << 20,), generator=g, dtype=torch.int64, device="cuda")
    buf = buf.to(torch.int32)                       # 12 MiB of random words
    sink = ops.maxsim_probe_l2_read(buf, 1)
    torch.cuda.synchronize()
    words = buf.cpu().numpy().view(np.uint32)
    want = int(np.bitwise_xor.reduce(words))
    got = int(np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint64)))
    assert got == want
    # an even number of passes cancels out
    sink2 = ops.maxsim_probe_l2_read(buf, 2)
    torch.cuda.synchronize()
    assert int(np.bitwise_xor.reduce(sink2.cpu().numpy().view(np.uint64))) == 0
