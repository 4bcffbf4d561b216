"""GPU parity of the gated GELU FFN (gate/up pair, then the Q4_0 down matvec).

h bound (per row), with eps = 1e-5 * sum|w x| of each matvec:
  |h - h_ref| <= 1.13 eps_g (|u| + eps_u) + |gelu(g)| eps_u + 2^-20 (|g u| + |h|)
(1.13 bounds |gelu'|; the last term covers the f32 GELU evaluation).
The down projection is checked against the oracle applied to the GPU's own h
(the plain matvec bound) and, at small sizes, end to end against the oracle's
h with the extra term sum_j |w_ij| |h_j - h_ref_j|.
"""

import numpy as np
import pytest

import block_quantized_matvec_gq_gb300 as gq
import oracle
import synth
from gpu_util import assert_within, dev, guarded, packed, torch

pytestmark = pytest.mark.gpu


def run_ffn(Wg, Wu, Wd, x, rows, K):
    t = torch()
    gp = packed(oracle.FORMAT_Q4_0, Wg, rows, K)
    up = packed(oracle.FORMAT_Q4_0, Wu, rows, K)
    dp = packed(oracle.FORMAT_Q4_0, Wd, K, rows)
    fh, h, ch = guarded(rows, t.float32)
    fy, y, cy = guarded(K, t.float32)
    gq.gq_ffn_gate_up_gelu(gp, up, dev(x), h, rows, K)
    gq.gq_q4_0_matvec(dp, h, y, K, rows)
    t.cuda.synchronize()
    ch()
    cy()
    return h.cpu().numpy(), y.cpu().numpy()


def h_bound(ref):
    eg = 1e-5 * ref["ag"]
    eu = 1e-5 * ref["au"]
    gel = np.array([oracle.gelu_tanh(v) for v in ref["g"]])
    return 1.13 * eg * (np.abs(ref["u"]) + eu) + np.abs(gel) * eu + 2.0 ** -20 * (
        np.abs(ref["g"] * ref["u"]) + np.abs(ref["h"]))


@pytest.mark.parametrize("rows,K", [(32, 32), (96, 256), (320, 512), (1024, 5376), (544, 2048), (160, 21504)])
def test_ffn_small_end_to_end(rows, K):
    seed = 300 + rows + K
    Wg = synth.q4_0_weights(rows, K, synth.stream(seed, 0))
    Wu = synth.q4_0_weights(rows, K, synth.stream(seed, 1))
    Wd = synth.q4_0_weights(K, rows, synth.stream(seed, 2))
    x = synth.normal(K, synth.stream(seed, 3))
    h, y = run_ffn(Wg, Wu, Wd, x, rows, K)
    ref = oracle.ffn_gate_up(Wg, Wu, x, rows, K)
    hb = h_bound(ref)
    err = np.abs(h.astype(np.float64) - ref["h"])
    assert np.all(err <= hb), (np.argmax(err - hb), float(np.max(err / np.where(hb > 0, hb, 1))))
    # down on the GPU's own h
    yd, ad = oracle.matvec(oracle.FORMAT_Q4_0, Wd, h, K, rows)
    assert_within(y, yd, ad, what="down(h_gpu)")
    # end to end against the oracle's h
    Wd_dense = oracle.dequant(oracle.FORMAT_Q4_0, Wd, rows)
    y_e2e = Wd_dense @ ref["h"]
    a_e2e = np.abs(Wd_dense) @ np.abs(ref["h"])
    extra = np.abs(Wd_dense) @ np.abs(h.astype(np.float64) - ref["h"])
    assert np.all(np.abs(y - y_e2e) <= 1e-5 * a_e2e + extra + 1e-5 * ad)


def test_ffn_full_21504x5376_workload():
    rows, K = 21504, 5376
    Wg, Wu, Wd, x = synth.ffn_inputs()
    h, y = run_ffn(Wg, Wu, Wd, x, rows, K)
    ref = oracle.ffn_gate_up(Wg, Wu, x, rows, K)
    hb = h_bound(ref)
    assert np.all(np.abs(h.astype(np.float64) - ref["h"]) <= hb)
    yd, ad = oracle.matvec(oracle.FORMAT_Q4_0, Wd, h, K, rows)
    assert_within(y, yd, ad, what="down 5376x21504")


def test_gelu_large_arguments_stay_finite():
    """Gate rows built to give |g| in the thousands: the clamped tanh keeps h finite."""
    import blockenc as be
    rows, K = 64, 64
    q_hi = np.full(32, 15)
    q_lo = np.zeros(32, int)
    blocks_g = [[be.enc_q4_0(q_hi if r % 2 else q_lo, 60000.0)] * 2 for r in range(rows)]
    Wg = be.rows_from_blocks(blocks_g)
    Wu = synth.q4_0_weights(rows, K, synth.stream(9, 1))
    Wd = synth.q4_0_weights(K, rows, synth.stream(9, 2))
    x = np.ones(K, np.float32) * 0.125
    h, y = run_ffn(Wg, Wu, Wd, x, rows, K)
    assert np.all(np.isfinite(h)) and np.all(np.isfinite(y))
    ref = oracle.ffn_gate_up(Wg, Wu, x, rows, K)
    hb = h_bound(ref)
    assert np.all(np.abs(h.astype(np.float64) - ref["h"]) <= hb)
    assert np.all(h[0::2] == 0.0) or np.all(np.abs(h[0::2]) <= hb[0::2])   # gelu(-large) -> 0
