"""Failure detection without a GPU fault: a bounded in-kernel wait that runs
out (an mbarrier phase that nothing completes) reports GQ_ERR_TIMEOUT
through the device status word, the kernel returns normally, the status is
cleared by reading it, and the context keeps working."""

import time

import numpy as np
import pytest

import block_quantized_matvec_gq_gb300 as gq
import oracle
import synth
from gpu_util import assert_within, dev, packed, torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_reports_and_leaves_the_context_usable():
    t = torch()
    assert gq.gq_device_status() == gq.GQ_OK  # clean start (reads and clears)
    t0 = time.time()
    gq.gq_selftest_bounded_wait()
    assert gq.gq_device_status(reset=False) == gq.GQ_ERR_TIMEOUT
    elapsed = time.time() - t0
    assert 1.0 < elapsed < 30.0, elapsed  # the wait's limit (about 2 s), not a hang
    assert gq.gq_device_status() == gq.GQ_ERR_TIMEOUT  # read and clear
    assert gq.gq_device_status() == gq.GQ_OK
    # the context still runs kernels correctly
    rows, K = 64, 256
    W = synth.q4_0_weights(rows, K, synth.stream(77, 0))
    x = synth.normal(K, synth.stream(77, 1))
    y = t.empty(rows, dtype=t.float32, device="cuda")
    gq.gq_q4_0_matvec(packed(oracle.FORMAT_Q4_0, W, rows, K), dev(x), y, rows, K)
    t.cuda.synchronize()
    y_ref, a_ref = oracle.matvec(oracle.FORMAT_Q4_0, W, x, rows, K)
    assert_within(y.cpu().numpy(), y_ref, a_ref, what="after the timeout")
