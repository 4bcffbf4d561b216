"""GPU parity of the Q8_0 activation quantizer (bit-exact) and the Q4_0 x Q8_0
prefill contraction.

Two bounds for Y[t][r]:
  element level  |Y - Y_ref| <= 1e-5 * sum_k |d_w (q_w - 8)| * |dx Xq|
                 (the matvec bound, on the dequantized operands): guaranteed
                 for any inputs, and the one the scale-folded path (operands
                 dx*Xq and d_w*(q_w-8) rounded per element) is built to;
  block level    |Y - Y_ref| <= 1e-5 * sum_b |d_w dx D_b|, tighter when a
                 block's integer dot cancels; it holds on the pages-shaped
                 inputs and is asserted there, but no f32 evaluation that
                 rounds dx*Xq per element can promise it under heavy
                 cancellation inside a block (the spread-scale test below).
"""

import numpy as np
import pytest

import block_quantized_matvec_gq_gb300 as gq
import oracle
import synth
from gpu_util import assert_same_specials, dev, guarded, packed, torch

pytestmark = pytest.mark.gpu


def gpu_quantize(X, M, K):
    t = torch()
    Xq = t.empty((M, K), dtype=t.int8, device="cuda")
    dx = t.empty((M, K // 32), dtype=t.float32, device="cuda")
    gq.gq_quantize_q8_0(dev(X), Xq, dx, K, M)
    t.cuda.synchronize()
    return Xq, dx


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (512, 5376), (7, 21504)])
def test_quantize_bit_exact(M, K):
    X = synth.normal((M, K), synth.stream(400 + M, K))
    X[0, :32] = 0.0                                  # a zero block
    if K >= 64:
        X[0, 32:64] = np.arange(32, dtype=np.float32) - 15.5   # half-way quotients
    Xq, dx = gpu_quantize(X, M, K)
    q_ref, d_ref = oracle.quantize_q8_0(X, M, K)
    assert np.array_equal(dx.cpu().numpy().view(np.uint32), d_ref.view(np.uint32))
    assert np.array_equal(Xq.cpu().numpy(), q_ref)


def test_quantize_half_integer_window_and_extreme_scales():
    """Blocks built so that x/d lands on half-integers (d = 1 exactly, and an
    inexact d = RN(100/127)), within 2^-16 of them on both sides, at the
    clamp, and at extreme scales (a largest value near FLT_MAX, and one so
    small that 1/d overflows): every code takes the reciprocal form or the
    division the rule keeps for such quotients, and all must equal the
    oracle's division and roundf bit for bit."""
    K, M = 256, 2
    X = np.zeros((M, K), dtype=np.float32)
    k = np.arange(-15, 16, dtype=np.float32)            # 31 half-integers k + 0.5 (|q| <= 15.5)
    X[0, 0] = 127.0                                     # d = 1
    X[0, 1:32] = k + 0.5
    X[0, 32] = 127.0
    X[0, 33:64] = k + np.float32(0.5) + np.float32(2.0 ** -16)
    X[0, 64] = 127.0
    X[0, 65:96] = k + np.float32(0.5) - np.float32(2.0 ** -16)
    d = np.float32(np.float32(100.0) / np.float32(127.0))
    X[0, 96] = 100.0                                    # d = RN(100/127), 1/d inexact
    X[0, 97:128] = ((k + np.float32(0.5)) * d).astype(np.float32)
    X[0, 128] = -127.0                                  # codes at the clamp, both signs
    X[0, 129:160] = np.linspace(-127.0, 127.0, 31, dtype=np.float32)
    X[0, 160] = np.float32(3.0e38)                      # near FLT_MAX
    X[0, 161:192] = np.float32(3.0e38) * np.linspace(-1.0, 1.0, 31, dtype=np.float32)
    X[0, 192] = np.float32(1.0e-41)                     # subnormal: 1/d overflows
    X[0, 193:224] = np.float32(1.0e-41) * np.linspace(-1.0, 1.0, 31, dtype=np.float32)
    X[1] = synth.normal(K, synth.stream(444, 0)) * np.float32(1e-30)
    Xq, dx = gpu_quantize(X, M, K)
    q_ref, d_ref = oracle.quantize_q8_0(X, M, K)
    assert np.array_equal(dx.cpu().numpy().view(np.uint32), d_ref.view(np.uint32))
    assert np.array_equal(Xq.cpu().numpy(), q_ref)


def workspace(K, M):
    t = torch()
    n = gq.gq_q4_0_gemm_workspace_bytes(K, M)
    # stale contents must not matter: the pre-pass overwrites every byte the GEMM reads
    return t.full((n,), 0x7B, dtype=t.uint8, device="cuda"), n


def element_bound(W, Xq, dx, K):
    """sum_k |w[r][k]| * |x[t][k]| with w = d_w (q_w - 8) (the oracle's dequantization)
    and x = dx * Xq, as (tokens, rows)."""
    w = np.abs(oracle.dequant(oracle.FORMAT_Q4_0, W, K))
    x = np.abs(np.repeat(dx.astype(np.float64), 32, axis=1) * Xq.astype(np.float64))
    return x @ w.T


def run_gemm(W, Xq_np, dx_np, rows, K, M):
    t = torch()
    Wp = packed(oracle.FORMAT_Q4_0, W, rows, K)
    full, Y, check = guarded(M * rows, t.float32)
    ws, n = workspace(K, M)
    gq.gq_q4_0_gemm_q8act(Wp, dev(Xq_np), dev(dx_np), Y, ws, n, rows, K, M)
    t.cuda.synchronize()
    check()
    return Y.view(M, rows).cpu().numpy()


@pytest.mark.parametrize("M,rows,K", [(1, 1, 32), (37, 100, 256), (64, 64, 64), (130, 257, 544),
                                      (5, 3000, 5376),
                                      # several tiles per CTA, each of fewer blocks than operand stages
                                      (260, 40000, 64),
                                      # scale tiles (K % 256 == 0), several tiles per CTA, one group each
                                      (300, 30000, 256)])
def test_gemm_matches_oracle(M, rows, K):
    W = synth.q4_0_weights(rows, K, synth.stream(500 + M, 0))
    X = synth.normal((M, K), synth.stream(500 + M, 1))
    Xq, dx = oracle.quantize_q8_0(X, M, K)
    Y = run_gemm(W, Xq, dx, rows, K, M)
    Y_ref, A = oracle.gemm_q8act(W, Xq, dx, rows, K, M)
    err = np.abs(Y.astype(np.float64) - Y_ref)
    assert np.all(err <= 1e-5 * A), float(np.max(err / np.maximum(A, 1e-300)))


# Shapes for the CTA-pair kernel (K % 256 == 0, M > 128): the peer CTA's half of
# B entirely past the last row (rows <= 96), its tokens all padding but one
# (M = 129), one 8-block chunk per tile (K = 256), ragged row and token tiles,
# and more tiles than CTA pairs.
@pytest.mark.parametrize("M,rows,K", [(129, 50, 256), (129, 96, 512), (257, 200, 768), (384, 97, 256),
                                      (1000, 193, 512), (300, 31000, 256)])
def test_gemm_cta_pair_shapes(M, rows, K):
    W = synth.q4_0_weights(rows, K, synth.stream(800 + M, rows))
    X = synth.normal((M, K), synth.stream(800 + M, K))
    Xq, dx = oracle.quantize_q8_0(X, M, K)
    Y = run_gemm(W, Xq, dx, rows, K, M)
    Y_ref, A = oracle.gemm_q8act(W, Xq, dx, rows, K, M)
    err = np.abs(Y.astype(np.float64) - Y_ref)
    assert np.all(err <= 1e-5 * A), float(np.max(err / np.maximum(A, 1e-300)))


# Small batches: K % 256 == 0 runs on the register-operand kernel (exact
# block dots, passes of up to 64 tokens); other K with M <= 24 in passes of
# up to 8 tokens whose staged codes fit in shared memory on the CUDA-core
# kernel: odd rows, one block, the largest K an 8-token pass still stages,
# several passes with a short last one; just past those limits the
# tensor-memory tiles take over.
@pytest.mark.parametrize("M,rows,K", [(2, 1, 32), (3, 77, 96), (4, 100, 21504), (8, 300, 5376), (13, 1001, 256),
                                      (16, 3001, 5376), (17, 77, 96), (24, 300, 5376), (6, 50, 15744),
                                      # staging too large or too many tokens: tensor cores
                                      (8, 50, 15872), (8, 40, 21504), (25, 200, 256), (32, 300, 5376)])
def test_gemm_small_batches(M, rows, K):
    W = synth.q4_0_weights(rows, K, synth.stream(1000 + M, rows))
    X = synth.normal((M, K), synth.stream(1000 + M, K))
    Xq, dx = oracle.quantize_q8_0(X, M, K)
    Y = run_gemm(W, Xq, dx, rows, K, M)
    Y_ref, A = oracle.gemm_q8act(W, Xq, dx, rows, K, M)
    err = np.abs(Y.astype(np.float64) - Y_ref)
    assert np.all(err <= 1e-5 * A), float(np.max(err / np.maximum(A, 1e-300)))


def test_gemm_full_512x21504x5376_sampled():
    rows, K, M = 21504, 5376, 512
    W, X = synth.gemm_inputs()
    Xq_g, dx_g = gpu_quantize(X, M, K)
    q_ref, d_ref = oracle.quantize_q8_0(X, M, K)
    assert np.array_equal(Xq_g.cpu().numpy(), q_ref)
    t = torch()
    Wp = packed(oracle.FORMAT_Q4_0, W, rows, K)
    Y = t.empty((M, rows), dtype=t.float32, device="cuda")
    ws, n = workspace(K, M)
    gq.gq_q4_0_gemm_q8act(Wp, Xq_g, dx_g, Y, ws, n, rows, K, M)
    t.cuda.synchronize()
    rng = np.random.default_rng(0)
    toks = np.concatenate([[0, 1, 127, 128, 511], rng.choice(M, 27, replace=False)])
    rws = np.concatenate([[0, 1, 255, 256, 21503], rng.choice(rows, 123, replace=False)])
    Y_ref, A = oracle.gemm_q8act(W, q_ref, d_ref, rows, K, M, tok_idx=toks, row_idx=rws)
    Yg = Y.cpu().numpy()[np.ix_(toks, rws)].astype(np.float64)
    assert np.all(np.abs(Yg - Y_ref) <= 1e-5 * A)


@pytest.mark.parametrize("M", [40, 200])  # exact block dots in registers; scale-folded f16 pieces (CTA pairs)
def test_gemm_scales_spread_over_many_octaves(M):
    """Block scales spread over many octaves inside each 8-block chunk (weight
    scales down to f16 subnormals, activation blocks 2^-12..2^12 apart, an
    all-zero block and an all-zero chunk): the power-of-two chunk factors of
    the f16 operand pieces, and the per-block fold of the exact block dots,
    keep every output within the bound."""
    rows, K = 200, 512
    nb = K // 32
    rng = np.random.default_rng(77)
    W = synth.q4_0_weights(rows, K, synth.stream(77, 0))
    e = rng.integers(-24, 9, size=(rows, nb))
    d = np.ldexp(rng.uniform(0.5, 1.0, size=(rows, nb)), e).astype(np.float16)
    d[7, :] = np.float16(2.0 ** -24)  # a row of the smallest subnormal scale
    W.reshape(rows, nb, 18)[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    X = synth.normal((M, K), synth.stream(77, 1)).astype(np.float64)
    X *= np.repeat(np.ldexp(1.0, rng.integers(-12, 13, size=(M, nb))), 32, axis=1)
    X[3, 64:96] = 0.0
    X[5, 256:512] = 0.0
    X = X.astype(np.float32)
    Xq, dx = oracle.quantize_q8_0(X, M, K)
    Y = run_gemm(W, Xq, dx, rows, K, M)
    Y_ref, A_blk = oracle.gemm_q8act(W, Xq, dx, rows, K, M)
    err = np.abs(Y.astype(np.float64) - Y_ref)
    A_el = element_bound(W, Xq, dx, K)
    assert np.all(err <= 1e-5 * A_el), float(np.max(err / np.maximum(A_el, 1e-300)))
    if M <= 112:  # exact integer block dots: the block-level bound holds under any cancellation
        assert np.all(err <= 1e-5 * A_blk), float(np.max(err / np.maximum(A_blk, 1e-300)))


# per-block fold (one CTA); small batches; exact block dots on CTA pairs
@pytest.mark.parametrize("K,M", [(128, 130), (256, 9), (256, 200)])
def test_gemm_all_eight_weights_exact_zero(K, M):
    import blockenc as be
    rows = 70
    blk = be.enc_q4_0(np.full(32, 8), 0.5)
    W = be.rows_from_blocks([[blk] * (K // 32)] * rows)
    X = synth.normal((M, K), synth.stream(501, 1))
    Xq, dx = oracle.quantize_q8_0(X, M, K)
    Y = run_gemm(W, Xq, dx, rows, K, M)
    assert np.all(Y == 0.0)


@pytest.mark.parametrize("M,rows,K", [(1, 1, 32), (128, 192, 64), (130, 200, 96), (37, 385, 256),
                                      (260, 40000, 64)])
def test_tensor_core_block_dots_are_bit_exact(M, rows, K):
    """The integer block dot products computed on the tensor cores (f16
    operands holding exact small integers, f32 accumulation) equal the int32
    brute force exactly."""
    t = torch()
    W = synth.q4_0_weights(rows, K, synth.stream(700 + M, rows))
    Xq = np.random.default_rng(M + rows).integers(-127, 128, size=(M, K)).astype(np.int8)
    Xq[0, :32] = 127
    Xq[-1, -32:] = -127
    Wp = packed(oracle.FORMAT_Q4_0, W, rows, K)
    D = t.full((M, rows, K // 32), -999999, dtype=t.int32, device="cuda")
    ws, n = workspace(K, M)
    gq.gq_q4_0_gemm_block_dots(Wp, dev(Xq), D, ws, n, rows, K, M)
    t.cuda.synchronize()
    assert gq.gq_device_status() == gq.GQ_OK
    ref = oracle.block_dots(W, Xq, rows, K, M, 0, M, 0, rows)
    assert np.array_equal(D.cpu().numpy(), ref)


def test_gemm_extreme_block_dots_exact():
    """All-15 nibbles against all-127 codes: the largest block dot (32 * 7 * 127)."""
    import blockenc as be
    rows, K, M = 5, 64, 3
    W = be.rows_from_blocks([[be.enc_q4_0(np.full(32, 15), 1.0), be.enc_q4_0(np.zeros(32, int), 1.0)]] * rows)
    Xq = np.full((M, K), 127, np.int8)
    Xq[1] = -127
    t = torch()
    D = t.empty((M, rows, 2), dtype=t.int32, device="cuda")
    ws, n = workspace(K, M)
    gq.gq_q4_0_gemm_block_dots(packed(oracle.FORMAT_Q4_0, W, rows, K), dev(Xq), D, ws, n, rows, K, M)
    t.cuda.synchronize()
    got = D.cpu().numpy()
    assert np.all(got[0, :, 0] == 32 * 7 * 127) and np.all(got[0, :, 1] == -32 * 8 * 127)
    assert np.all(got[1, :, 0] == -32 * 7 * 127) and np.all(got[1, :, 1] == 32 * 8 * 127)


# register operands (one pass; four passes); single-CTA tensor-memory tiles; CTA pairs
@pytest.mark.parametrize("M,rows,K", [(8, 2000, 5376), (100, 2000, 5376), (120, 2000, 5376), (512, 3000, 5376)])
def test_gemm_repeat_runs_bitwise_identical(M, rows, K):
    """Partial sums are added in a fixed order on every path (K quarters,
    chunk read-outs): the same inputs give the same bits."""
    t = torch()
    W = synth.q4_0_weights(rows, K, synth.stream(900 + M, 0))
    X = synth.normal((M, K), synth.stream(900 + M, 1))
    Xq, dx = oracle.quantize_q8_0(X, M, K)
    Wp = packed(oracle.FORMAT_Q4_0, W, rows, K)
    ws, n = workspace(K, M)
    outs = []
    for _ in range(3):
        Y = t.full((M, rows), float("nan"), dtype=t.float32, device="cuda")
        gq.gq_q4_0_gemm_q8act(Wp, dev(Xq), dev(dx), Y, ws, n, rows, K, M)
        t.cuda.synchronize()
        outs.append(Y.cpu().numpy().view(np.uint32))
    assert gq.gq_device_status() == gq.GQ_OK
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


# The register-operand kernel (K % 256 == 0, M <= 112): one row and fewer
# than 16 rows, ragged 16-row tiles, every pass width (1, 2 and 4 token
# tiles, a last pass of 3 tiles padded to 4), passes of 32 tokens with a
# short last one, a single 16-block stage half past the end of the row
# (K = 256) and many stages, more row groups than CTAs (each CTA then takes
# two groups).
@pytest.mark.parametrize("M,rows,K", [(1, 1, 256), (3, 17, 512), (9, 5, 256), (20, 1000, 768), (33, 130, 2048),
                                      (64, 300, 5376), (65, 300, 512), (75, 257, 256), (112, 2000, 5376),
                                      (32, 40000, 256), (100, 25000, 256), (7, 61, 21504)])
def test_gemm_register_path_shapes(M, rows, K):
    W = synth.q4_0_weights(rows, K, synth.stream(1100 + M, rows))
    X = synth.normal((M, K), synth.stream(1100 + M, K))
    Xq, dx = oracle.quantize_q8_0(X, M, K)
    Y = run_gemm(W, Xq, dx, rows, K, M)
    assert gq.gq_device_status() == gq.GQ_OK
    Y_ref, A = oracle.gemm_q8act(W, Xq, dx, rows, K, M)
    err = np.abs(Y.astype(np.float64) - Y_ref)
    assert np.all(err <= 1e-5 * A), float(np.max(err / np.maximum(A, 1e-300)))


@pytest.mark.parametrize("M,rows,K", [(1, 40, 5376), (8, 33, 5376), (13, 100, 2048), (64, 50, 5376),
                                      (100, 70, 5376)])
def test_gemm_register_path_block_dots_exact(M, rows, K):
    """With every block scale 1 (d_w and dx), Y is the plain sum of the
    integer block dots, an integer below 2^24: the register-operand kernel
    must return it exactly, for codes over the whole int8 range (-128
    included) and nibble blocks of all 0 and all 15 (the largest products)."""
    nb = K // 32
    W = synth.q4_0_weights(rows, K, synth.stream(1200 + M, rows))
    Wb = W.reshape(rows, nb, 18)
    Wb[:, :, 0:2] = np.full((rows, nb), 1.0, np.float16).view(np.uint8).reshape(rows, nb, 2)
    Wb[0, :, 2:] = 0x00          # q = 0 everywhere: w = -8
    Wb[1 % rows, ::2, 2:] = 0xFF  # q = 15 in every other block: w = 7
    rng = np.random.default_rng(1200 + M)
    Xq = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    Xq[0, :] = -128
    Xq[-1, ::2] = 127
    dx = np.ones((M, nb), np.float32)
    Y = run_gemm(W, Xq, dx, rows, K, M)
    D = oracle.block_dots(W, Xq, rows, K, M, 0, M, 0, rows).astype(np.int64)
    ref = D.sum(axis=2)
    assert np.abs(ref).max() < 2 ** 24
    assert np.array_equal(Y.astype(np.float64), ref.astype(np.float64))


# register-operand path (two shapes); CUDA-core dp4a (K % 256 != 0, M <= 24);
# per-block tcgen05 read-out (K % 256 != 0, M > 24); scale-folded pieces (M > 112)
@pytest.mark.parametrize("M,rows,K", [(16, 300, 2048), (40, 97, 5376), (8, 77, 544), (30, 50, 544),
                                      (200, 97, 5376)])
def test_gemm_non_finite_scales(M, rows, K):
    """Non-finite block scales: an activation scale of NaN makes its token's
    row of Y NaN; an infinite activation scale or weight scale gives
    +-inf, or NaN where it meets a zero block dot or another infinity of
    the other sign, exactly as in the fp64 definition on the register-operand
    path (exact block dots, then (d_w dx) D in f32).  The scale-folded path
    (M > 112) splits d_w (q - 8) into two f16 pieces, whose difference of
    infinities is NaN: there every non-finite result is NaN, on the same
    set of outputs."""
    nb = K // 32
    W = synth.q4_0_weights(rows, K, synth.stream(1300 + M, rows))
    Wb = W.reshape(rows, nb, 18)
    d16 = Wb[:, :, 0:2].copy().view(np.float16).reshape(rows, nb)
    d16[11 % rows, 3] = np.float16(np.inf)
    d16[5 % rows, nb - 1] = np.float16(-np.inf)
    Wb[:, :, 0:2] = d16.view(np.uint8).reshape(rows, nb, 2)
    X = synth.normal((M, K), synth.stream(1300 + M, K))
    Xq, dx = oracle.quantize_q8_0(X, M, K)
    dx = dx.copy()
    dx[2, 5] = np.nan
    dx[7, 10] = np.inf
    dx[M - 1, 0] = -np.inf
    Y = run_gemm(W, Xq, dx, rows, K, M)
    Y_ref, A = oracle.gemm_q8act(W, Xq, dx, rows, K, M)
    folded = K % 256 == 0 and M > 112
    n_nan, n_inf = assert_same_specials(Y.reshape(-1), Y_ref.reshape(-1), A.reshape(-1), what=f"{M}x{rows}x{K}",
                                        exact=not folded)
    assert n_nan > 0 and n_inf > 0
    assert np.all(np.isnan(Y[2]))


# The single-CTA tensor-memory tiles (K % 256 == 0, 112 < M <= 128): ragged
# rows, one 8-block chunk, the full row width; and both sides of the 112-token
# boundary with the register-operand kernel.
@pytest.mark.parametrize("M,rows,K", [(113, 1000, 512), (120, 300, 5376), (128, 97, 256), (112, 33, 768),
                                      (113, 33, 768)])
def test_gemm_single_cta_tiles_and_the_register_boundary(M, rows, K):
    W = synth.q4_0_weights(rows, K, synth.stream(1400 + M, rows))
    X = synth.normal((M, K), synth.stream(1400 + M, K))
    Xq, dx = oracle.quantize_q8_0(X, M, K)
    Y = run_gemm(W, Xq, dx, rows, K, M)
    assert gq.gq_device_status() == gq.GQ_OK
    Y_ref, A = oracle.gemm_q8act(W, Xq, dx, rows, K, M)
    err = np.abs(Y.astype(np.float64) - Y_ref)
    assert np.all(err <= 1e-5 * A), float(np.max(err / np.maximum(A, 1e-300)))
