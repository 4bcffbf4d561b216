"""GPU parity of the decode matvecs (Q4_0, Q8_0, Q4_K, Q6_K) against the fp64 oracle.

Bound (per row): |y - y_ref| <= 1e-5 * sum_j |w_ij x_j|.  Cases span several
tiles and a ragged row tail, K at the block minimum, the lane-group widths
(blocks per row divisible by 32, by 8 only, by none), the full 4096 x 4096
Q4_0 and 21504 x 5376 Q4_K workloads, and the degenerate inputs of each
format (all-8 nibbles, one-hot x, zero scales).
"""

import numpy as np
import pytest

import block_quantized_matvec_gq_gb300 as gq
import oracle
import synth
from gpu_util import assert_same_specials, assert_within, dev, guarded, packed, torch

pytestmark = pytest.mark.gpu

FMT_FN = {
    oracle.FORMAT_Q4_0: gq.gq_q4_0_matvec,
    oracle.FORMAT_Q8_0: gq.gq_q8_0_matvec,
    oracle.FORMAT_Q4_K: gq.gq_q4k_matvec,
    oracle.FORMAT_Q6_K: gq.gq_q6k_matvec,
}


def run_matvec(fmt, W_canon, x, rows, K):
    t = torch()
    Wp = packed(fmt, W_canon, rows, K)
    full, y, check = guarded(rows, t.float32)
    FMT_FN[fmt](Wp, dev(x), y, rows, K)
    t.cuda.synchronize()
    check()
    return y.cpu().numpy()


SHAPES = [(1, 32), (3, 64), (37, 96), (257, 256), (1000, 512), (129, 4096), (515, 5376), (77, 21504),
          (33, 2304), (250, 800), (8, 49152), (256, 21504), (5, 2048), (600, 1024), (2048, 49152),
          (1000, 5376), (1213, 8192),  # the ring at four to eight rows per SM
          (1216, 5376)]  # the register streams just past the ring's limit (eight rows per SM)


@pytest.mark.parametrize("fmt", [oracle.FORMAT_Q4_0, oracle.FORMAT_Q8_0, oracle.FORMAT_Q4_K, oracle.FORMAT_Q6_K])
@pytest.mark.parametrize("rows,K", SHAPES)
def test_matvec_matches_oracle(fmt, rows, K):
    if fmt in (oracle.FORMAT_Q4_K, oracle.FORMAT_Q6_K) and K % 256:
        pytest.skip("K-quants need K % 256 == 0")
    seed = 1000 + rows + K
    W = synth.weights(fmt, rows, K, synth.stream(seed, 0))
    x = synth.normal(K, synth.stream(seed, 1))
    y = run_matvec(fmt, W, x, rows, K)
    y_ref, a_ref = oracle.matvec(fmt, W, x, rows, K)
    assert_within(y, y_ref, a_ref, what=f"fmt{fmt} {rows}x{K}")


def test_q4_0_full_4096x4096_workload():
    W, x = synth.q4_0_matvec_inputs()
    y = run_matvec(oracle.FORMAT_Q4_0, W, x, 4096, 4096)
    y_ref, a_ref = oracle.matvec(oracle.FORMAT_Q4_0, W, x, 4096, 4096)
    assert_within(y, y_ref, a_ref, what="q4_0 4096x4096")


def test_q6_k_21504x5376_sampled_rows():
    rows, K = 21504, 5376
    W = synth.q6_k_weights(rows, K, synth.stream(70, 0))
    x = synth.normal(K, synth.stream(70, 1))
    y = run_matvec(oracle.FORMAT_Q6_K, W, x, rows, K)
    sel = np.concatenate([[0, 1, 2, 3, rows - 1], np.random.default_rng(0).choice(rows, 400, replace=False)])
    y_ref, a_ref = oracle.matvec(oracle.FORMAT_Q6_K, W, x, rows, K, row_idx=sel)
    assert_within(y[sel], y_ref, a_ref, what="q6_k 21504x5376")


def test_q4_k_full_21504x5376_workload():
    W, x = synth.q4_k_matvec_inputs()
    y = run_matvec(oracle.FORMAT_Q4_K, W, x, 21504, 5376)
    y_ref, a_ref = oracle.matvec(oracle.FORMAT_Q4_K, W, x, 21504, 5376)
    assert_within(y, y_ref, a_ref, what="q4_k 21504x5376")


@pytest.mark.parametrize("fmt", [oracle.FORMAT_Q4_0, oracle.FORMAT_Q8_0, oracle.FORMAT_Q4_K, oracle.FORMAT_Q6_K])
def test_one_hot_x_is_bit_exact(fmt):
    rows, K = 70, 512
    W = synth.weights(fmt, rows, K, synth.stream(5, fmt))
    Wp = packed(fmt, W, rows, K)
    dense = oracle.dequant(fmt, W, K)
    t = torch()
    y = t.empty(rows, dtype=t.float32, device="cuda")
    for j in (0, 1, 16, 17, 31, 32, 255, 256, 511):
        x = np.zeros(K, np.float32)
        x[j] = 1.0
        FMT_FN[fmt](Wp, dev(x), y, rows, K)
        got = y.cpu().numpy().astype(np.float64)
        assert np.array_equal(got, dense[:, j]), (fmt, j)


def test_q4_0_all_eight_rows_are_exactly_zero():
    import blockenc as be
    rows, K = 40, 256
    W = synth.q4_0_weights(rows, K, synth.stream(6, 0))
    zero_blk = np.frombuffer(be.enc_q4_0(np.full(32, 8), 1.75), np.uint8)
    Wb = W.reshape(rows, K // 32, 18)
    for r in (0, 7, 39):
        Wb[r, :, :] = zero_blk
    x = synth.normal(K, synth.stream(6, 1)) * 50
    y = run_matvec(oracle.FORMAT_Q4_0, W, x, rows, K)
    for r in (0, 7, 39):
        assert y[r] == 0.0
    y_ref, a_ref = oracle.matvec(oracle.FORMAT_Q4_0, W, x, rows, K)
    assert_within(y, y_ref, a_ref, what="q4_0 with zero rows")


def test_q4_k_zero_scales_and_mins():
    import blockenc as be
    rows, K = 16, 512
    rng = np.random.default_rng(0)
    blocks = []
    for r in range(rows):
        row = []
        for s in range(2):
            q = rng.integers(0, 16, 256)
            sc = [0] * 8 if r % 2 == 0 else list(rng.integers(0, 64, 8))
            m = [0] * 8 if r % 3 == 0 else list(rng.integers(0, 64, 8))
            row.append(be.enc_q4_k(q, sc, m, 0.01, 0.02))
        blocks.append(row)
    W = be.rows_from_blocks(blocks)
    x = synth.normal(K, synth.stream(7, 1))
    y = run_matvec(oracle.FORMAT_Q4_K, W, x, rows, K)
    y_ref, a_ref = oracle.matvec(oracle.FORMAT_Q4_K, W, x, rows, K)
    assert_within(y, y_ref, a_ref, what="q4_k special scales")
    assert y[0] == 0.0 and y[6] == 0.0     # sc = 0 and m = 0


@pytest.mark.parametrize("rows,K", [(515, 5376), (3000, 2048)])
def test_q4_k_power_of_two_scaling_of_x_is_exact(rows, K):
    """The Q4_K kernel stages x with power-of-two scales taken from max|x|,
    so multiplying x by 2^k must multiply every y by exactly 2^k (no result
    under- or overflows here)."""
    W = synth.q4_k_weights(rows, K, synth.stream(8, 0))
    x = synth.normal(K, synth.stream(8, 1))
    y0 = run_matvec(oracle.FORMAT_Q4_K, W, x, rows, K)
    for k in (-100, -37, 50, 90):
        xk = (x.astype(np.float64) * 2.0 ** k).astype(np.float32)
        yk = run_matvec(oracle.FORMAT_Q4_K, W, xk, rows, K)
        assert np.array_equal(yk.astype(np.float64), y0.astype(np.float64) * 2.0 ** k), k


def test_q4_k_x_with_wide_dynamic_range():
    """Elements of x spread over 2^-60 .. 2^60 (and some zeros): every
    product stays a normal number in the scaled domain, so the bound holds."""
    rows, K = 600, 4096
    W = synth.q4_k_weights(rows, K, synth.stream(9, 0))
    rng = np.random.default_rng(9)
    x = (synth.normal(K, synth.stream(9, 1)).astype(np.float64)
         * np.exp2(rng.integers(-60, 61, K))).astype(np.float32)
    x[rng.integers(0, K, 40)] = 0.0
    y = run_matvec(oracle.FORMAT_Q4_K, W, x, rows, K)
    y_ref, a_ref = oracle.matvec(oracle.FORMAT_Q4_K, W, x, rows, K)
    assert_within(y, y_ref, a_ref, what="q4_k wide-range x")


@pytest.mark.parametrize("fmt", [oracle.FORMAT_Q4_0, oracle.FORMAT_Q8_0, oracle.FORMAT_Q4_K, oracle.FORMAT_Q6_K])
def test_repeat_runs_are_bitwise_identical(fmt):
    rows, K = 3001, 5376 if fmt != oracle.FORMAT_Q4_0 else 4096
    W = synth.weights(fmt, rows, K, synth.stream(8, 0))
    t = torch()
    Wp = packed(fmt, W, rows, K)
    x = dev(synth.normal(K, synth.stream(8, 1)))
    ys = []
    for _ in range(5):
        y = t.empty(rows, dtype=t.float32, device="cuda")
        FMT_FN[fmt](Wp, x, y, rows, K)
        ys.append(y)
    for y in ys[1:]:
        assert t.equal(y, ys[0])


@pytest.mark.parametrize("fmt", [oracle.FORMAT_Q4_0, oracle.FORMAT_Q4_K])
@pytest.mark.parametrize("rows,K", [(8, 49152), (77, 21504), (256, 21504), (600, 4096)])
def test_split_k_repeat_runs_are_bitwise_identical(fmt, rows, K):
    """Short, wide shapes split K across the CTAs of a cluster; the partial
    sums are added in a fixed order, so repeated runs agree bit for bit."""
    W = synth.weights(fmt, rows, K, synth.stream(9, rows))
    t = torch()
    Wp = packed(fmt, W, rows, K)
    x = dev(synth.normal(K, synth.stream(9, rows + 1)))
    ys = []
    for _ in range(4):
        y = t.empty(rows, dtype=t.float32, device="cuda")
        FMT_FN[fmt](Wp, x, y, rows, K)
        ys.append(y)
    for y in ys[1:]:
        assert t.equal(y, ys[0])
    y_ref, a_ref = oracle.matvec(fmt, W, x.cpu().numpy(), rows, K)
    assert_within(ys[0].cpu().numpy(), y_ref, a_ref, what=f"fmt{fmt} {rows}x{K} split-K")


def test_argument_errors_launch_nothing():
    t = torch()
    W = t.zeros(1024, dtype=t.uint8, device="cuda")
    x = t.zeros(64, dtype=t.float32, device="cuda")
    y = t.full((4,), 3.0, dtype=t.float32, device="cuda")
    with pytest.raises(gq.GQError) as e:
        gq.gq_q4_0_matvec(W, x, y, 4, 48)          # partial block
    assert e.value.status == gq.GQ_ERR_SHAPE
    with pytest.raises(gq.GQError) as e:
        gq.gq_q4_0_matvec(W, x, y, 4, 64, M=2)      # batched decode not offered
    assert e.value.status == gq.GQ_ERR_SHAPE
    with pytest.raises(gq.GQError) as e:
        gq.gq_q4k_matvec(W, x, y, 1, 64)            # Q4_K needs K % 256
    assert e.value.status == gq.GQ_ERR_SHAPE
    with pytest.raises(gq.GQError) as e:
        gq.gq_q8_0_matvec(W, x.data_ptr() + 4, y, 4, 32)
    assert e.value.status == gq.GQ_ERR_ALIGN
    t.cuda.synchronize()
    assert t.equal(y, t.full((4,), 3.0, dtype=t.float32, device="cuda"))


@pytest.mark.parametrize("fmt", [oracle.FORMAT_Q4_0, oracle.FORMAT_Q8_0, oracle.FORMAT_Q4_K, oracle.FORMAT_Q6_K])
@pytest.mark.parametrize("rows,K", [(300, 2048), (256, 21504)])  # register streams; short-wide split-K rings
def test_non_finite_x_propagates_as_in_the_definition(fmt, rows, K):
    """x holding +inf and -inf (rows get +-inf, or NaN where the two meet or
    a weight is zero) and, separately, a NaN (every row NaN): the same
    pattern of non-finite results as the fp64 definition, the bound on the
    rest.  Q4_K forms each sub-block as d sc sum(q x) - dmin m sum(x), so an
    infinity that meets a zero code or the min term can give NaN where the
    per-weight definition gives an infinity: there the set of non-finite
    rows is the definition's."""
    W = synth.weights(fmt, rows, K, synth.stream(31, fmt))
    x = synth.normal(K, synth.stream(31, 1))
    xi = x.copy()
    xi[3] = np.inf
    xi[K - 40] = -np.inf
    y = run_matvec(fmt, W, xi, rows, K)
    y_ref, a_ref = oracle.matvec(fmt, W, xi, rows, K)
    n_nan, n_inf = assert_same_specials(y, y_ref, a_ref, what=f"fmt{fmt} {rows}x{K} inf",
                                        exact=fmt != oracle.FORMAT_Q4_K)
    assert n_nan > 0 and n_inf > 0  # both kinds occur on these inputs
    xn = x.copy()
    xn[K // 2 + 1] = np.nan
    y = run_matvec(fmt, W, xn, rows, K)
    assert np.all(np.isnan(y))


@pytest.mark.parametrize("fmt", [oracle.FORMAT_Q4_0, oracle.FORMAT_Q4_K, oracle.FORMAT_Q6_K])
@pytest.mark.parametrize("rows,K", [(7296, 16384), (7168, 4096)])
def test_matvec_between_one_and_two_tasks_per_warp(fmt, rows, K):
    """Shapes with 1.25 to 1.75 row tasks per resident warp (on 152 SMs): long
    rows take the balanced schedule (leftover rows split along K across a
    CTA's warps, partial sums added in warp order), short rows round-robin.
    Sampled rows against the oracle, and repeat runs bitwise identical."""
    W = synth.weights(fmt, rows, K, synth.stream(60, fmt))
    x = synth.normal(K, synth.stream(60, 1))
    t = torch()
    Wp = packed(fmt, W, rows, K)
    xd = dev(x)
    ys = []
    for _ in range(2):
        y = t.empty(rows, dtype=t.float32, device="cuda")
        FMT_FN[fmt](Wp, xd, y, rows, K)
        ys.append(y)
    t.cuda.synchronize()
    assert t.equal(ys[0], ys[1])
    sel = np.concatenate([[0, 1, rows - 2, rows - 1], np.random.default_rng(fmt).choice(rows, 600, replace=False)])
    y_ref, a_ref = oracle.matvec(fmt, W, x, rows, K, row_idx=sel)
    assert_within(ys[0].cpu().numpy()[sel], y_ref, a_ref, what=f"fmt{fmt} {rows}x{K}")
