"""The allocation-free top-k entry point (gq_logits_topk_noalloc).

Some callers cannot allocate device memory at all -- for instance a serving
loop that must not call cudaMalloc once it runs (the allocation would
synchronize the device or stall the loop), or a host runtime that only hands
the library its input and output buffers.  For them the tied-logit top-k
keeps its per-CTA key lists in a fixed array inside libgq instead of a
caller-provided workspace.  This test calls that entry point through the C
ABI twice in a row (the array keeps the previous call's contents) and checks
each result against the workspace entry point on the same inputs.

The file is named so that pytest collects it last.
"""

import numpy as np
import pytest

import block_quantized_matvec_gq_gb300 as gq
import oracle
import synth
from gpu_util import dev, packed, torch

pytestmark = pytest.mark.gpu


def _with_workspace(Wp, x, rows, K, k, cap):
    t = torch()
    wsb = gq.gq_logits_topk_workspace_bytes(rows, K, k)
    ws = t.zeros(wsb, dtype=t.uint8, device="cuda")
    idx = t.empty(k, dtype=t.int32, device="cuda")
    val = t.empty(k, dtype=t.float32, device="cuda")
    logits = t.empty(rows, dtype=t.float32, device="cuda")
    gq.gq_logits_topk(Wp, x, cap, k, idx, val, logits, ws, wsb, rows, K)
    t.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy(), logits.cpu().numpy()


def _no_alloc(Wp, x, rows, K, k, cap):
    t = torch()
    idx = t.full((k,), -1, dtype=t.int32, device="cuda")
    val = t.full((k,), float("nan"), dtype=t.float32, device="cuda")
    logits = t.empty(rows, dtype=t.float32, device="cuda")
    gq.gq_logits_topk_noalloc(Wp, x, cap, k, idx, val, logits, rows, K)
    t.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy(), logits.cpu().numpy()


def test_no_alloc_top_k_matches_workspace_entry_point_on_two_calls():
    t = torch()
    # two different problems back to back: the second call must not see the
    # first one's key lists (they are left in the shared array)
    cases = [(50000, 5376, 10, 30.0, 70), (7001, 1024, 64, 0.0, 71)]
    for rows, K, k, cap, seed in cases:
        W = synth.q8_0_weights(rows, K, synth.stream(seed, 0))
        Wp = packed(oracle.FORMAT_Q8_0, W, rows, K)
        x = dev(synth.normal(K, synth.stream(seed, 1)))
        ref_idx, ref_val, ref_logits = _with_workspace(Wp, x, rows, K, k, cap)
        got_idx, got_val, got_logits = _no_alloc(Wp, x, rows, K, k, cap)
        # same kernels, same geometry: the results agree exactly (the tests'
        # tolerance for this path is exact agreement of indices)
        assert np.array_equal(got_idx, ref_idx)
        assert np.array_equal(got_val, ref_val)
        assert np.array_equal(got_logits, ref_logits)
    assert gq.gq_device_status() == gq.GQ_OK


def test_no_alloc_top_k_rejects_what_the_workspace_form_rejects():
    t = torch()
    W = t.zeros(gq.gq_packed_bytes(1, 64, 64), dtype=t.uint8, device="cuda")
    x = t.zeros(64, dtype=t.float32, device="cuda")
    idx = t.empty(8, dtype=t.int32, device="cuda")
    val = t.empty(8, dtype=t.float32, device="cuda")
    with pytest.raises(gq.GQError) as e:
        gq.gq_logits_topk_noalloc(W, x, 30.0, 65, idx, val, None, 64, 64)
    assert e.value.status == gq.GQ_ERR_SHAPE
    with pytest.raises(gq.GQError) as e:
        gq.gq_logits_topk_noalloc(W, x, 30.0, 8, idx, val, None, 64, 48)
    assert e.value.status == gq.GQ_ERR_SHAPE
