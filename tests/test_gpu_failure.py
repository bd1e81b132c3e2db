"""The kernels' failure path on the GPU, reached without a fault or a hang.

kvq_selftest_wait runs one CTA that starts a real bulk copy into shared
memory and then waits, with the bounded wait of the split attention kernels
(which = 0) or of the weight ring (which = 1), on an mbarrier that nothing
ever arrives at.  The wait must give up after its bound (~1 s), raise
KVQ_ERRBIT_TIMEOUT, let the copy it started land before the CTA exits, and
leave the context usable: library calls after it still match the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import oracle_pins as pins
from gpu_harness import dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", [0, 1], ids=["split_attention_wait", "weight_ring_wait"])
def test_bounded_wait_gives_up_and_drains(kvq, which):
    src = torch.arange(16, dtype=torch.int32, device="cuda") + 0x5A5A0000
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    landed = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    kvq.kvq_selftest_wait(which, src, err, landed)
    torch.cuda.synchronize()
    took = time.monotonic() - t0
    assert int(err.item()) == kvq.ERRBIT_TIMEOUT
    assert int(landed.item()) == 0x5A5A0000, "the drained copy did not land"
    assert 0.05 < took < 30.0, took

    # the context is still usable: a weight-only product (ring kernel) after it
    rng = np.random.default_rng(17 + which)
    w, s, x = pins.random_wq_case(rng, oracle.W_INT4, 1, 200, 1536)
    y = torch.full((1, 200), float("nan"), dtype=torch.float32, device="cuda")
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_wq_gemm(oracle.W_INT4, dev(w), dev(s.view(np.int16)),
                    dev(x.view(np.int16)).view(torch.bfloat16), y, err_word=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    ref = oracle.wq_gemm(oracle.W_INT4, w, s, x)
    got = y.cpu().numpy().astype(np.float64)
    scale = np.abs(pins._bf16_to_f64(x)) @ np.abs(pins.numpy_int4_weights(w, s, 128)).T
    assert np.all(np.abs(got - ref) <= 1e-5 * scale + 1e-30)


def test_selftest_arguments(kvq):
    L = kvq.load()
    buf = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    assert L.kvq_selftest_wait(2, p, p, p, None) == 1     # which
    assert L.kvq_selftest_wait(0, None, p, p, None) == 1  # src
    assert L.kvq_selftest_wait(0, p + 4, p, p, None) == 1  # alignment
