"""GPU parity of the GELU-gated Q4_0 down projection (gq_q4_0_geglu_down):
y = W_down (gelu_tanh(g) * u), the gate applied while the input is staged.

Bound per row (written in gq_geglu.h):
  |y - y_ref| <= 1e-5 sum_j |w_ij h_j| + 2^-20 sum_j |w_ij| (|g_j u_j| + |h_j|)
with h_j the exact gelu_tanh(g_j) u_j; the second term covers the f32
evaluation of h (tanhf and three roundings stay below 2^-22 of |g u| + |h|).
"""

import numpy as np
import pytest

import block_quantized_matvec_gq_gb300 as gq
import oracle
import synth
from gpu_util import dev, guarded, packed, torch

pytestmark = pytest.mark.gpu


def run(Wd, g, u, rows, K):
    t = torch()
    wp = packed(oracle.FORMAT_Q4_0, Wd, rows, K)
    fy, y, cy = guarded(rows, t.float32)
    gq.gq_q4_0_geglu_down(wp, dev(g), dev(u), y, rows, K)
    t.cuda.synchronize()
    cy()
    return y.cpu().numpy().astype(np.float64)


def check(y, Wd, g, u, rows, K, row_idx=None):
    yr, a, b = oracle.geglu_down(oracle.FORMAT_Q4_0, Wd, g, u, rows, K, row_idx=row_idx)
    bound = 1e-5 * a + 2.0 ** -20 * b
    err = np.abs(y - yr)
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, (bad[:5], y[bad[:5]], yr[bad[:5]], bound[bad[:5]])
    return float(np.max(err / np.where(bound > 0, bound, 1.0)))


def inputs(rows, K, seed, gate_scale=2.0):
    Wd = synth.q4_0_weights(rows, K, synth.stream(seed, 0))
    g = (synth.normal(K, synth.stream(seed, 1)) * gate_scale).astype(np.float32)
    u = synth.normal(K, synth.stream(seed, 2))
    return Wd, g, u


# shapes: single block, ragged rows, block counts that are and are not
# multiples of 32 (the two lane-group widths), the model's down shape
@pytest.mark.parametrize("rows,K", [(1, 32), (5, 96), (32, 256), (97, 512), (544, 2048), (300, 4192),
                                    (1024, 5376), (5376, 21504), (131, 49152)])
def test_geglu_down_matches_oracle(rows, K):
    Wd, g, u = inputs(rows, K, 700 + rows + K)
    y = run(Wd, g, u, rows, K)
    check(y, Wd, g, u, rows, K)


def test_geglu_down_large_gates_stay_finite():
    """Gate values up to 1e4 (finding F1: an unclamped tanh gave NaN there)."""
    rows, K = 64, 1024
    Wd, _, u = inputs(rows, K, 720)
    rng = np.random.default_rng(721)
    g = (rng.choice([-1.0, 1.0], K) * 10.0 ** rng.uniform(0, 4, K)).astype(np.float32)
    y = run(Wd, g, u, rows, K)
    assert np.all(np.isfinite(y))
    check(y, Wd, g, u, rows, K)


def test_geglu_down_one_hot_up_pairs_gate_and_up_by_index():
    """u = e_j with every gate value distinct: y must be column j times
    gelu(g_j), within the bound, for several j (a gate value taken from
    another index, or GELU applied to u, is far outside it)."""
    rows, K = 40, 1024
    Wd, g, _ = inputs(rows, K, 730)
    for j in (0, 7, 31, 32, 128, 255, 256, 1023):
        u = np.zeros(K, np.float32)
        u[j] = 1.5
        y = run(Wd, g, u, rows, K)
        check(y, Wd, g, u, rows, K)


def test_geglu_down_on_gpu_gate_and_up_outputs():
    """The path as a model runs it: g and u from the GPU Q4_0 matvecs of the
    gate and up matrices (21504 x 5376), then the fused down projection
    (5376 x 21504), checked against the oracle on the GPU's g and u."""
    t = torch()
    rows, K = 5376, 21504
    Wg = synth.q4_0_weights(K, rows, synth.stream(740, 0))
    Wu = synth.q4_0_weights(K, rows, synth.stream(740, 1))
    Wd = synth.q4_0_weights(rows, K, synth.stream(740, 2))
    x = synth.normal(rows, synth.stream(740, 3))
    gp = packed(oracle.FORMAT_Q4_0, Wg, K, rows)
    up = packed(oracle.FORMAT_Q4_0, Wu, K, rows)
    wp = packed(oracle.FORMAT_Q4_0, Wd, rows, K)
    xd = dev(x)
    g = t.empty(K, dtype=t.float32, device="cuda")
    u = t.empty(K, dtype=t.float32, device="cuda")
    y = t.empty(rows, dtype=t.float32, device="cuda")
    gq.gq_q4_0_matvec(gp, xd, g, K, rows)
    gq.gq_q4_0_matvec(up, xd, u, K, rows)
    gq.gq_q4_0_geglu_down(wp, g, u, y, rows, K)
    t.cuda.synchronize()
    check(y.cpu().numpy().astype(np.float64), Wd, g.cpu().numpy(), u.cpu().numpy(), rows, K)


def test_geglu_down_repeat_runs_bitwise_identical():
    rows, K = 5376, 21504
    Wd, g, u = inputs(rows, K, 750)
    y1 = run(Wd, g, u, rows, K)
    y2 = run(Wd, g, u, rows, K)
    assert np.array_equal(y1, y2)
