"""GPU parity of the Q8_0 tied-logit projection with soft-cap and top-k.

Values: every returned (and materialized) capped logit lies within
  bound_i = 1e-5 * sum_j |w_ij x_j| + 2^-20 * (|l_i| + |l'_i|)
of the oracle's capped value (the first term is the matvec bound, which the
soft-cap can only shrink since its slope is <= 1; the second covers the f32
division, tanhf and the final product).  Indices: equal to the oracle's full
sort wherever the neighbouring capped values are further apart than their
summed bounds; inside a run of near-ties, equal as sets; across the k-th
boundary, members of the run.  Exact ties (duplicate rows) and NaN rows
follow the ranking rule exactly.
"""

import math

import numpy as np
import pytest

import block_quantized_matvec_gq_gb300 as gq
import oracle
import synth
from gpu_util import dev, guarded, packed, torch

pytestmark = pytest.mark.gpu


def gpu_logits_topk(Wp, x, rows, K, k, softcap, with_logits=True):
    t = torch()
    wsb = gq.gq_logits_topk_workspace_bytes(rows, K, k)
    ws = t.zeros(wsb, dtype=t.uint8, device="cuda")  # zero-filled once before first use
    idx = t.full((k,), -1, dtype=t.int32, device="cuda")
    val = t.full((k,), float("nan"), dtype=t.float32, device="cuda")
    full, logits, check = guarded(rows, t.float32) if with_logits else (None, None, lambda: None)
    gq.gq_logits_topk(Wp, dev(x) if isinstance(x, np.ndarray) else x, softcap, k, idx, val, logits, ws,
                      wsb, rows, K)
    t.cuda.synchronize()
    check()
    return idx.cpu().numpy(), val.cpu().numpy(), (logits.cpu().numpy() if with_logits else None)


def capped(v, cap):
    return np.array([oracle.softcap(float(a), cap) for a in v]) if cap > 0 else v.copy()


def check_topk(idx, val, l_ref, a_ref, cap, k):
    c_ref = capped(l_ref, cap)
    bound = 1e-5 * a_ref + 2.0 ** -20 * (np.abs(l_ref) + np.abs(c_ref))
    ridx, rval = oracle.topk(c_ref, min(len(c_ref), k + 64))
    n = len(ridx)
    # values of what the GPU returned
    for p in range(k):
        i = idx[p]
        assert 0 <= i < len(l_ref)
        if math.isnan(c_ref[i]):
            assert math.isnan(val[p])
        else:
            assert abs(val[p] - c_ref[i]) <= bound[i], (p, i, val[p], c_ref[i], bound[i])
    # near-tie runs in the oracle order
    close = [False] * (n - 1)
    for p in range(n - 1):
        a, b = ridx[p], ridx[p + 1]
        va, vb = c_ref[a], c_ref[b]
        if math.isnan(va) or math.isnan(vb):
            close[p] = False      # NaN order is exact: after every number, by row
        else:
            close[p] = abs(va - vb) <= bound[a] + bound[b]
    p = 0
    while p < k:
        q = p
        while q < n - 1 and close[q]:
            q += 1
        # run = positions p..q in the oracle order
        if q == p:
            assert idx[p] == ridx[p], (p, idx[p], ridx[p])
        else:
            run = set(int(v) for v in ridx[p:q + 1])
            hi = min(q, k - 1)
            got = set(int(v) for v in idx[p:hi + 1])
            assert got <= run, (p, q, got, run)
            if q <= k - 1:
                assert got == run
        p = q + 1


@pytest.mark.parametrize("rows,K,k,cap", [(1, 32, 1, 30.0), (64, 64, 10, 30.0), (1000, 256, 10, 30.0),
                                          (5000, 512, 64, 0.0), (4097, 5376, 10, 30.0),
                                          (70001, 1024, 33, 30.0), (513, 2304, 40, 5.0)])
def test_logits_topk_matches_oracle(rows, K, k, cap):
    seed = 20 + rows + K
    W = synth.q8_0_weights(rows, K, synth.stream(seed, 0))
    x = synth.normal(K, synth.stream(seed, 1))
    Wp = packed(oracle.FORMAT_Q8_0, W, rows, K)
    idx, val, logits = gpu_logits_topk(Wp, x, rows, K, k, cap)
    l_ref, a_ref = oracle.matvec(oracle.FORMAT_Q8_0, W, x, rows, K)
    c_ref = capped(l_ref, cap)
    bound = 1e-5 * a_ref + 2.0 ** -20 * (np.abs(l_ref) + np.abs(c_ref))
    assert np.all(np.abs(logits - c_ref) <= bound)
    check_topk(idx, val, l_ref, a_ref, cap, k)


def test_logits_topk_full_262144x5376_workload():
    rows, K, k, cap = 262144, 5376, 10, 30.0
    W, x = synth.q8_0_logits_inputs()
    Wp = packed(oracle.FORMAT_Q8_0, W, rows, K)
    idx, val, logits = gpu_logits_topk(Wp, x, rows, K, k, cap)
    l_ref, a_ref = oracle.matvec(oracle.FORMAT_Q8_0, W, x, rows, K)
    c_ref = capped(l_ref, cap)
    bound = 1e-5 * a_ref + 2.0 ** -20 * (np.abs(l_ref) + np.abs(c_ref))
    assert np.all(np.abs(logits - c_ref) <= bound)
    check_topk(idx, val, l_ref, a_ref, cap, k)
    # the top-k alone (no logits output) gives the same answer
    idx2, val2, _ = gpu_logits_topk(Wp, x, rows, K, k, cap, with_logits=False)
    assert np.array_equal(idx, idx2) and np.array_equal(val, val2)


def _gpu_order(logits):
    return sorted(range(len(logits)),
                  key=lambda i: (np.isnan(logits[i]), -logits[i] if not np.isnan(logits[i]) else 0.0, i))


def test_exact_ties_rank_by_lower_row_and_nan_rows_rank_last():
    rows, K, k = 300, 64, 40
    W = synth.q8_0_weights(rows, K, synth.stream(44, 0))
    x = synth.normal(K, synth.stream(44, 1))
    l_ref, _ = oracle.matvec(oracle.FORMAT_Q8_0, W, x, rows, K)
    top = int(np.argmax(l_ref))
    W = W.reshape(rows, K // 32, 34)
    # rows 10, 150, 299 duplicate the largest row: bitwise-equal logits, a tie at the top
    for r in (10, 150, 299):
        W[r] = W[top]
    # rows with a NaN scale give NaN logits
    nan_half = np.array([np.nan], np.float16).view(np.uint8)
    for r in (0, 5, 120):
        W[r, 0, 0:2] = nan_half
    Wp = packed(oracle.FORMAT_Q8_0, W.reshape(rows, -1), rows, K)
    for cap in (0.0, 30.0):
        idx, val, logits = gpu_logits_topk(Wp, x, rows, K, k, cap)
        for r in (10, 150, 299):
            assert logits[r] == logits[top]
        assert all(np.isnan(logits[r]) for r in (0, 5, 120))
        assert list(idx) == _gpu_order(logits)[:k]
        group = sorted({10, 150, 299, top})
        assert list(idx[:len(group)]) == group
    # every row requested: the NaN rows come last, in row order
    small = 40
    Ws = W[:small].reshape(small, -1)
    Wps = packed(oracle.FORMAT_Q8_0, Ws, small, K)
    idx, val, logits = gpu_logits_topk(Wps, x, small, K, small, 30.0)
    assert list(idx) == _gpu_order(logits)
    assert list(idx[-2:]) == [0, 5] and np.all(np.isnan(val[-2:]))


def test_all_nan_rows_return_lowest_indices():
    rows, K, k = 50, 32, 7
    W = synth.q8_0_weights(rows, K, synth.stream(45, 0)).reshape(rows, 1, 34)
    W[:, 0, 0:2] = np.array([np.nan], np.float16).view(np.uint8)
    Wp = packed(oracle.FORMAT_Q8_0, W.reshape(rows, -1), rows, K)
    idx, val, _ = gpu_logits_topk(Wp, synth.normal(K, synth.stream(45, 1)), rows, K, k, 30.0)
    assert list(idx) == list(range(k))
    assert np.all(np.isnan(val))


def test_repeat_runs_identical_and_workspace_errors():
    t = torch()
    rows, K, k = 20000, 768, 16
    W = synth.q8_0_weights(rows, K, synth.stream(46, 0))
    Wp = packed(oracle.FORMAT_Q8_0, W, rows, K)
    x = synth.normal(K, synth.stream(46, 1))
    a = gpu_logits_topk(Wp, x, rows, K, k, 30.0)
    b = gpu_logits_topk(Wp, x, rows, K, k, 30.0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    wsb = gq.gq_logits_topk_workspace_bytes(rows, K, k)
    ws = t.zeros(wsb, dtype=t.uint8, device="cuda")  # zero-filled once before first use
    idx = t.empty(k, dtype=t.int32, device="cuda")
    val = t.empty(k, dtype=t.float32, device="cuda")
    with pytest.raises(gq.GQError) as e:
        gq.gq_logits_topk(Wp, dev(x), 30.0, k, idx, val, None, ws, wsb - 8, rows, K)
    assert e.value.status == gq.GQ_ERR_WORKSPACE
    with pytest.raises(gq.GQError) as e:
        gq.gq_logits_topk(Wp, dev(x), 30.0, 65, idx, val, None, ws, wsb, rows, K)
    assert e.value.status == gq.GQ_ERR_SHAPE
    with pytest.raises(gq.GQError) as e:
        gq.gq_logits_topk(Wp, dev(x), 30.0, k, idx, val, None, None, wsb, rows, K)
    assert e.value.status == gq.GQ_ERR_WORKSPACE


def test_workspace_reused_across_calls_and_grid_sizes():
    """The finished-CTA counter at the start of the workspace is back at zero
    after every call: one workspace serves calls of different row counts
    (different grids) in any order with the same results as fresh ones."""
    t = torch()
    K, k = 2048, 12
    shapes = [(60000, 1), (3000, 2), (60000, 3), (700, 4), (3000, 5)]
    big = max(gq.gq_logits_topk_workspace_bytes(r, K, k) for r, _ in shapes)
    shared = t.zeros(big, dtype=t.uint8, device="cuda")
    for rows, seed in shapes:
        W = synth.q8_0_weights(rows, K, synth.stream(900 + seed, 0))
        Wp = packed(oracle.FORMAT_Q8_0, W, rows, K)
        x = dev(synth.normal(K, synth.stream(900 + seed, 1)))
        fresh = gpu_logits_topk(Wp, x, rows, K, k, 30.0, with_logits=False)
        idx = t.empty(k, dtype=t.int32, device="cuda")
        val = t.empty(k, dtype=t.float32, device="cuda")
        gq.gq_logits_topk(Wp, x, 30.0, k, idx, val, None, shared, big, rows, K)
        t.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), fresh[0])
        assert np.array_equal(val.cpu().numpy(), fresh[1])
        # the counter (first 4 bytes) is zero again
        assert int(shared[:4].view(t.int32).item()) == 0
    assert gq.gq_device_status() == gq.GQ_OK
