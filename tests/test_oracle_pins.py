"""Pins of the CPU oracle against what the block definitions and mathematics fix.

None of these checks compares the oracle with a retyped copy of itself:
  * hand-built blocks (tests/golden) whose expected weights are derived by
    hand from the block definitions;
  * test-side ENCODERS (blockenc.py) that build blocks from intended integer
    codes, so a decoding slip in the oracle shows as a mismatch;
  * closed forms (all-ones x gives row sums from the raw bytes; all-8 nibbles
    give 0), one-hot x (reproduces one dequantized column);
  * brute force with exact rational arithmetic on 2 x 64 / 2 x 256 inputs;
  * special cases that reduce to a library routine (numpy fp16 decoding,
    Python's sorted, numpy integer matmul, erf-based GELU).
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import blockenc as be
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    data = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, rest = line.split(" ", 1)
            data[key] = rest.strip()
    return bytes.fromhex(data["bytes"]), np.array([float(v) for v in data["weights"].split()])


# ---------------------------------------------------------------- fp16 decode

def test_half_to_double_matches_numpy_for_every_finite_pattern():
    pats = np.arange(1 << 16, dtype=np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    lib = oracle.lib()
    got = np.array([lib.gqo_half_to_double(int(p)) for p in pats[::7]])
    r = ref[::7]
    fin = np.isfinite(r)
    assert np.array_equal(got[fin], r[fin])
    assert np.array_equal(np.isnan(got), np.isnan(r))
    assert np.array_equal(np.isinf(got), np.isinf(r))


# ---------------------------------------------------------------- golden blocks

@pytest.mark.parametrize("fmt,name,K", [
    (oracle.FORMAT_Q4_0, "q4_0_handbuilt.txt", 32),
    (oracle.FORMAT_Q8_0, "q8_0_handbuilt.txt", 32),
    (oracle.FORMAT_Q4_K, "q4_k_handbuilt.txt", 256),
    (oracle.FORMAT_Q6_K, "q6_k_handbuilt.txt", 256),
])
def test_golden_handbuilt_blocks(fmt, name, K):
    blk, expect = _golden(name)
    got = oracle.dequant(fmt, np.frombuffer(blk, dtype=np.uint8).reshape(1, -1), K)[0]
    assert np.array_equal(got, expect)


# ---------------------------------------------------------------- Q4_0 special blocks

def test_q4_0_all_eight_is_zero_for_any_x():
    rng = np.random.default_rng(11)
    blk = be.enc_q4_0(np.full(32, 8), 0.75)
    W = be.rows_from_blocks([[blk] * 4, [blk] * 4])
    x = rng.standard_normal(128).astype(np.float32) * 100
    y, a = oracle.matvec(oracle.FORMAT_Q4_0, W, x, 2, 128)
    assert np.all(y == 0.0) and np.all(a == 0.0)


def test_q4_0_extreme_codes():
    d = 0.375
    hi = oracle.dequant(oracle.FORMAT_Q4_0, np.frombuffer(be.enc_q4_0(np.full(32, 15), d), np.uint8), 32)
    lo = oracle.dequant(oracle.FORMAT_Q4_0, np.frombuffer(be.enc_q4_0(np.zeros(32, int), d), np.uint8), 32)
    assert np.all(hi == 7 * d) and np.all(lo == -8 * d)


def test_q8_0_extreme_codes():
    d = 0.125
    q = np.array([127, -127] * 16)
    w = oracle.dequant(oracle.FORMAT_Q8_0, np.frombuffer(be.enc_q8_0(q, d), np.uint8), 32)[0]
    assert np.array_equal(w, q * d)


def test_q4_k_special_sub_blocks():
    # sc = 0 -> w = -dmin*m ; m = 0 -> w = d*sc*q ; q = 0 with m = 63 -> -63 dmin
    q = np.tile(np.arange(32) % 16, 8)
    q[7 * 32:] = 0
    sc = [0, 5, 0, 40, 1, 63, 17, 9]
    m = [3, 0, 63, 0, 48, 0, 33, 63]
    d, dmin = 0.5, 0.25
    w = oracle.dequant(oracle.FORMAT_Q4_K,
                       np.frombuffer(be.enc_q4_k(q, sc, m, d, dmin), np.uint8), 256)[0]
    for s in range(8):
        seg = w[32 * s:32 * s + 32]
        qs = q[32 * s:32 * s + 32]
        assert np.array_equal(seg, d * sc[s] * qs - dmin * m[s]), s
    assert np.all(w[7 * 32:] == -63 * dmin)
    assert np.all(w[0:32] == -dmin * 3)


def test_q6_k_special_codes_and_scales():
    # q = 32 -> 0 for any scale; q = 63 -> 31 d sc; q = 0 -> -32 d sc; sc = 0, -128, 127
    d = 0.25
    q = np.full(256, 32)
    q[16:32] = 63
    q[32:48] = 0
    q[48:64] = 63
    q[64:80] = 0
    sc = [7, -3, 5, -128, 127, 0] + [1] * 10
    w = oracle.dequant(oracle.FORMAT_Q6_K, np.frombuffer(be.enc_q6_k(q, sc, d), np.uint8), 256)[0]
    assert np.all(w[0:16] == 0.0) and np.all(w[80:] == 0.0)
    assert np.all(w[16:32] == 31 * d * -3) and np.all(w[32:48] == -32 * d * 5)
    assert np.all(w[48:64] == 31 * d * -128) and np.all(w[64:80] == -32 * d * 127)
    q[80:96] = 63
    w = oracle.dequant(oracle.FORMAT_Q6_K, np.frombuffer(be.enc_q6_k(q, sc, d), np.uint8), 256)[0]
    assert np.all(w[80:96] == 0.0)  # sc = 0


def test_q4_k_scale_min_unpacking_every_field():
    rng = np.random.default_rng(3)
    for _ in range(200):
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        packed = be.pack_q4_k_scales(sc, m)
        for s in range(8):
            assert oracle.q4_k_scale_min(packed, s) == (sc[s], m[s])


# ---------------------------------------------------------------- encoder round trips

@pytest.mark.parametrize("rows,K", [(3, 64), (2, 256)])
def test_q4_0_decode_matches_intended_values(rows, K):
    W, dense, _, _ = be.random_q4_0_matrix(rows, K, np.random.default_rng(5))
    assert np.array_equal(oracle.dequant(oracle.FORMAT_Q4_0, W, K), dense)


def test_q8_0_decode_matches_intended_values():
    W, dense = be.random_q8_0_matrix(3, 96, np.random.default_rng(6))
    assert np.array_equal(oracle.dequant(oracle.FORMAT_Q8_0, W, 96), dense)


def test_q4_k_decode_matches_intended_values():
    W, dense = be.random_q4_k_matrix(2, 512, np.random.default_rng(7))
    assert np.array_equal(oracle.dequant(oracle.FORMAT_Q4_K, W, 512), dense)


def test_q6_k_decode_matches_intended_values():
    W, dense = be.random_q6_k_matrix(3, 512, np.random.default_rng(17))
    assert np.array_equal(oracle.dequant(oracle.FORMAT_Q6_K, W, 512), dense)


# ---------------------------------------------------------------- one-hot / all-ones

@pytest.mark.parametrize("fmt", [oracle.FORMAT_Q4_0, oracle.FORMAT_Q8_0, oracle.FORMAT_Q4_K, oracle.FORMAT_Q6_K])
def test_one_hot_x_reproduces_a_column(fmt):
    rng = np.random.default_rng(8)
    rows, K = 3, 512
    if fmt == oracle.FORMAT_Q4_0:
        W, dense, _, _ = be.random_q4_0_matrix(rows, K, rng)
    elif fmt == oracle.FORMAT_Q8_0:
        W, dense = be.random_q8_0_matrix(rows, K, rng)
    elif fmt == oracle.FORMAT_Q4_K:
        W, dense = be.random_q4_k_matrix(rows, K, rng)
    else:
        W, dense = be.random_q6_k_matrix(rows, K, rng)
    for j in (0, 1, 15, 16, 17, 31, 33, 255, 256, 300, 511):
        x = np.zeros(K, np.float32)
        x[j] = 1.0
        y, a = oracle.matvec(fmt, W, x, rows, K)
        assert np.array_equal(y, dense[:, j])
        assert np.array_equal(a, np.abs(dense[:, j]))


def test_q4_0_all_ones_x_closed_form_from_raw_bytes():
    # sum_j w_j = sum_b d_b * (sum of the 32 nibbles - 256): independent of nibble order
    from synth import q4_0_weights, stream
    rows, K = 16, 4096
    W = q4_0_weights(rows, K, stream(99, 0))
    y, _ = oracle.matvec(oracle.FORMAT_Q4_0, W, np.ones(K, np.float32), rows, K)
    blk = W.reshape(rows, K // 32, 18)
    d = blk[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    nib = (blk[:, :, 2:] & 15).astype(np.int64).sum(-1) + (blk[:, :, 2:] >> 4).astype(np.int64).sum(-1)
    ref = (d * (nib - 256)).sum(-1)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- exact brute force

def _exact_dot(dense_row, x):
    return sum(Fraction(float(w)) * Fraction(float(v)) for w, v in zip(dense_row, x))


@pytest.mark.parametrize("fmt,K", [(oracle.FORMAT_Q4_0, 64), (oracle.FORMAT_Q8_0, 64),
                                   (oracle.FORMAT_Q4_K, 256), (oracle.FORMAT_Q6_K, 256)])
def test_brute_force_exact_rational_2xK(fmt, K):
    rng = np.random.default_rng(21 + fmt)
    if fmt == oracle.FORMAT_Q4_0:
        W, dense, _, _ = be.random_q4_0_matrix(2, K, rng)
    elif fmt == oracle.FORMAT_Q8_0:
        W, dense = be.random_q8_0_matrix(2, K, rng)
    elif fmt == oracle.FORMAT_Q4_K:
        W, dense = be.random_q4_k_matrix(2, K, rng)
    else:
        W, dense = be.random_q6_k_matrix(2, K, rng)
    x = rng.standard_normal(K).astype(np.float32)
    y, a = oracle.matvec(fmt, W, x, 2, K)
    for r in range(2):
        exact = _exact_dot(dense[r], x)
        absum = sum(abs(Fraction(float(w)) * Fraction(float(v))) for w, v in zip(dense[r], x))
        # double accumulation of K terms: |err| <= K * 2^-53 * sum|w x|
        assert abs(Fraction(y[r]) - exact) <= Fraction(K) * Fraction(2) ** -52 * absum
        assert abs(Fraction(a[r]) - absum) <= Fraction(K) * Fraction(2) ** -52 * absum


def test_matvec_rejects_partial_blocks():
    with pytest.raises(ValueError):
        oracle.matvec(oracle.FORMAT_Q4_0, np.zeros(18, np.uint8), np.zeros(48, np.float32), 1, 48)
    with pytest.raises(ValueError):
        oracle.matvec(oracle.FORMAT_Q4_K, np.zeros(144, np.uint8), np.zeros(128, np.float32), 1, 128)
    with pytest.raises(ValueError):
        oracle.matvec(oracle.FORMAT_Q6_K, np.zeros(210, np.uint8), np.zeros(128, np.float32), 1, 128)


def test_row_selection_matches_full_rows():
    from synth import q8_0_weights, stream
    W = q8_0_weights(40, 256, stream(5, 0))
    x = np.random.default_rng(0).standard_normal(256).astype(np.float32)
    y, a = oracle.matvec(oracle.FORMAT_Q8_0, W, x, 40, 256)
    idx = np.array([39, 0, 17, 17, 5])
    ys, as_ = oracle.matvec(oracle.FORMAT_Q8_0, W, x, 40, 256, row_idx=idx)
    assert np.array_equal(ys, y[idx]) and np.array_equal(as_, a[idx])


# ---------------------------------------------------------------- GELU and soft-cap

def test_gelu_tanh_special_values():
    assert oracle.gelu_tanh(0.0) == 0.0
    # large |a|: the clamped tanh argument (+-15) leaves 1 - tanh(15) ~ 1.9e-13
    assert abs(oracle.gelu_tanh(10.0) - 10.0) <= 10.0 * 1e-12
    assert abs(oracle.gelu_tanh(-10.0)) <= 10.0 * 1e-12
    # slope 1/2 at the origin
    h = 1e-6
    assert abs((oracle.gelu_tanh(h) - oracle.gelu_tanh(-h)) / (2 * h) - 0.5) < 1e-9
    for a in (-1e4, -50.0, -15.0, 15.0, 50.0, 1e4):
        assert math.isfinite(oracle.gelu_tanh(a))


def test_gelu_tanh_approximates_erf_gelu():
    # The tanh form is a published approximation of x * Phi(x); a wrong constant
    # (sqrt(2/pi) or 0.044715) moves it far outside this band.
    xs = np.linspace(-8, 8, 4001)
    err = max(abs(oracle.gelu_tanh(v) - 0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0)))) for v in xs)
    assert err < 5e-4
    assert err > 1e-6   # and it is not the erf form itself


def test_softcap_closed_forms():
    c = 30.0
    assert oracle.softcap(0.0, c) == 0.0
    assert oracle.softcap(1e6, c) == 30.0 and oracle.softcap(-1e6, c) == -30.0
    v = c * math.atanh(0.5)
    assert abs(oracle.softcap(v, c) - 15.0) < 1e-12
    for t in (0.1, 3.0, 29.0, 100.0):
        assert oracle.softcap(-t, c) == -oracle.softcap(t, c)
    xs = np.linspace(-200, 200, 1001)
    ys = [oracle.softcap(v, c) for v in xs]
    assert all(b >= a for a, b in zip(ys, ys[1:]))
    assert oracle.softcap(12.5, 0.0) == 12.5   # no cap


# ---------------------------------------------------------------- top-k

def _ref_topk(v, k):
    order = sorted(range(len(v)), key=lambda i: (math.isnan(v[i]), -v[i] if not math.isnan(v[i]) else 0.0, i))
    return np.array(order[:k]), np.array([v[i] for i in order[:k]])


@pytest.mark.parametrize("n,k,kind", [(1, 1, "rand"), (10, 10, "rand"), (1000, 10, "rand"),
                                      (4096, 64, "ties"), (5000, 40, "nan"), (1 << 18, 10, "rand"),
                                      (300, 30, "allnan"), (777, 7, "zeros")])
def test_topk_matches_full_sort(n, k, kind):
    rng = np.random.default_rng(n + k)
    if kind == "rand":
        v = rng.standard_normal(n)
    elif kind == "ties":
        v = rng.integers(0, 5, n).astype(np.float64)
    elif kind == "nan":
        v = rng.standard_normal(n)
        v[rng.random(n) < 0.3] = np.nan
        v[rng.random(n) < 0.1] = 1.0
    elif kind == "allnan":
        v = np.full(n, np.nan)
        v[[5, 17]] = -3.0
    else:
        v = np.where(rng.random(n) < 0.5, 0.0, -0.0)
    idx, val = oracle.topk(v, k)
    ridx, rval = _ref_topk(list(v), k)
    assert np.array_equal(idx, ridx)
    assert np.array_equal(np.isnan(val), np.isnan(rval))
    assert np.array_equal(val[~np.isnan(val)], rval[~np.isnan(rval)])


# ---------------------------------------------------------------- Q8_0 activation quantization

def _round_half_away(fr: Fraction) -> int:
    s = 1 if fr >= 0 else -1
    a = abs(fr)
    n = int(a)
    return s * (n + 1 if a - n >= Fraction(1, 2) else n)


def _f32(v):
    return np.float32(v)


def test_quantize_reproduces_integer_multiples():
    rng = np.random.default_rng(4)
    for _ in range(50):
        k = rng.integers(-127, 128, 32)
        k[rng.integers(0, 32)] = 127 * (1 if rng.random() < 0.5 else -1)   # amax = 127 d
        d = np.float32(2.0) ** int(rng.integers(-10, 5))                   # power of two: k*d exact
        x = (k * d).astype(np.float32)
        q, dd = oracle.quantize_q8_0(x.reshape(1, 32), 1, 32)
        assert dd[0, 0] == d
        assert np.array_equal(q[0], k)


def test_quantize_amax_maps_to_127_and_zero_block():
    x = np.zeros((2, 64), np.float32)
    x[0, 5] = -3.7
    x[0, 40] = 2.2
    q, d = oracle.quantize_q8_0(x, 2, 64)
    assert q[0, 5] == -127 and q[0, 40] == 127
    assert np.all(q[1] == 0) and np.all(d[1] == 0)
    assert d[0, 0] == np.float32(np.float32(3.7) / np.float32(127.0))


def test_quantize_half_way_rounds_away_from_zero():
    # d = 1 exactly (amax 127); x = +-(n + 0.5) must round away from zero
    x = np.zeros(32, np.float32)
    x[0] = 127.0
    x[1:9] = [0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 100.5, -126.5]
    q, d = oracle.quantize_q8_0(x.reshape(1, 32), 1, 32)
    assert d[0, 0] == 1.0
    assert list(q[0, 1:9]) == [1, -1, 2, -2, 3, -3, 101, -127]


def test_quantize_brute_force_exact_rounding():
    rng = np.random.default_rng(12)
    X = rng.standard_normal((3, 96)).astype(np.float32)
    q, d = oracle.quantize_q8_0(X, 3, 96)
    for t in range(3):
        for b in range(3):
            blk = X[t, 32 * b:32 * b + 32]
            amax = np.max(np.abs(blk))
            dd = np.float32(amax) / np.float32(127.0)          # numpy f32 division is IEEE
            assert d[t, b] == dd
            for j in range(32):
                r = np.float32(blk[j]) / dd                    # f32 quotient, then exact rounding
                ref = max(-127, min(127, _round_half_away(Fraction(float(r)))))
                assert q[t, 32 * b + j] == ref


# ---------------------------------------------------------------- block dots and the GEMM

def test_block_dots_brute_force_int64():
    rng = np.random.default_rng(13)
    rows, K, M = 5, 128, 3
    W, _, qw, _ = be.random_q4_0_matrix(rows, K, rng)
    Xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    D = oracle.block_dots(W, Xq, rows, K, M, 0, M, 0, rows)
    for b in range(K // 32):
        ref = Xq[:, 32 * b:32 * b + 32].astype(np.int64) @ (qw[:, b, :] - 8).astype(np.int64).T
        assert np.array_equal(D[:, :, b], ref)


def test_gemm_all_eight_weights_give_zero():
    blk = be.enc_q4_0(np.full(32, 8), 1.5)
    W = be.rows_from_blocks([[blk] * 2] * 3)
    Xq = np.random.default_rng(1).integers(-127, 128, size=(4, 64)).astype(np.int8)
    dx = np.ones((4, 2), np.float32)
    Y, A = oracle.gemm_q8act(W, Xq, dx, 3, 64, 4)
    assert np.all(Y == 0) and np.all(A == 0)


def test_gemm_matches_dense_dequantized_product():
    # Y[t, r] = sum_j (q_x d_x)[t, j] * w[r, j]: the block form against a plain dense product
    rng = np.random.default_rng(14)
    rows, K, M = 6, 160, 4
    W, dense, _, _ = be.random_q4_0_matrix(rows, K, rng)
    X = rng.standard_normal((M, K)).astype(np.float32)
    Xq, dx = oracle.quantize_q8_0(X, M, K)
    Y, A = oracle.gemm_q8act(W, Xq, dx, rows, K, M)
    xhat = Xq.astype(np.float64) * np.repeat(dx.astype(np.float64), 32, axis=1)
    ref = xhat @ dense.T
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12 * np.abs(A).max())


def test_gemm_m1_equals_matvec_of_dequantized_activation():
    rng = np.random.default_rng(15)
    rows, K = 7, 256
    W, dense, _, _ = be.random_q4_0_matrix(rows, K, rng)
    Xq = rng.integers(-127, 128, size=(1, K)).astype(np.int8)
    dx = (np.float32(2.0) ** rng.integers(-8, -2, size=(1, K // 32))).astype(np.float32)
    xhat = (Xq.astype(np.float32) * np.repeat(dx, 32, axis=1))[0]    # exact: power-of-two scales
    Y, _ = oracle.gemm_q8act(W, Xq, dx, rows, K, 1)
    y, a = oracle.matvec(oracle.FORMAT_Q4_0, W, xhat, rows, K)
    np.testing.assert_allclose(Y[0], y, rtol=0, atol=1e-13 * a.max())


def test_gemm_token_and_row_selection():
    from synth import q4_0_weights, stream
    W = q4_0_weights(9, 64, stream(1, 2))
    X = np.random.default_rng(2).standard_normal((5, 64)).astype(np.float32)
    Xq, dx = oracle.quantize_q8_0(X, 5, 64)
    Y, A = oracle.gemm_q8act(W, Xq, dx, 9, 64, 5)
    Ys, As = oracle.gemm_q8act(W, Xq, dx, 9, 64, 5, tok_idx=[4, 0], row_idx=[8, 3, 3])
    assert np.array_equal(Ys, Y[np.ix_([4, 0], [8, 3, 3])])
    assert np.array_equal(As, A[np.ix_([4, 0], [8, 3, 3])])


# ---------------------------------------------------------------- FFN

def test_ffn_gate_up_combines_two_matvecs():
    from synth import q4_0_weights, stream
    rows, K = 12, 128
    Wg = q4_0_weights(rows, K, stream(2, 0))
    Wu = q4_0_weights(rows, K, stream(2, 1))
    x = np.random.default_rng(9).standard_normal(K).astype(np.float32)
    out = oracle.ffn_gate_up(Wg, Wu, x, rows, K)
    g, ag = oracle.matvec(oracle.FORMAT_Q4_0, Wg, x, rows, K)
    u, au = oracle.matvec(oracle.FORMAT_Q4_0, Wu, x, rows, K)
    assert np.array_equal(out["g"], g) and np.array_equal(out["u"], u)
    assert np.array_equal(out["ag"], ag) and np.array_equal(out["au"], au)
    # gate (not up) goes through GELU: swap the matrices and the result changes
    for i in range(rows):
        assert out["h"][i] == oracle.gelu_tanh(g[i]) * u[i]


# ---------------------------------------------------------------- GELU-gated down projection

def _matrix(fmt, rows, K, seed):
    rng = np.random.default_rng(seed)
    if fmt == oracle.FORMAT_Q4_0:
        W, dense, _, _ = be.random_q4_0_matrix(rows, K, rng)
    elif fmt == oracle.FORMAT_Q4_K:
        W, dense = be.random_q4_k_matrix(rows, K, rng)
    else:
        W, dense = be.random_q6_k_matrix(rows, K, rng)
    return W, dense


def test_geglu_down_zero_gate_or_zero_up_gives_zero():
    rows, K = 5, 256
    W, _ = _matrix(oracle.FORMAT_Q4_0, rows, K, 40)
    rng = np.random.default_rng(41)
    v = rng.standard_normal(K).astype(np.float32)
    z = np.zeros(K, np.float32)
    for g, u in ((v, z), (z, v)):
        y, a, b = oracle.geglu_down(oracle.FORMAT_Q4_0, W, g, u, rows, K)
        assert np.all(y == 0.0) and np.all(a == 0.0)


@pytest.mark.parametrize("fmt", [oracle.FORMAT_Q4_0, oracle.FORMAT_Q4_K, oracle.FORMAT_Q6_K])
def test_geglu_down_one_hot_up_gives_a_gated_column(fmt):
    # u = e_j: one nonzero term, y_i = w_ij gelu(g_j) exactly.  The gate, not
    # the up value, goes through GELU (gelu(2.5) * 1 != gelu(1) * 2.5), and
    # the other gate values must not leak in.
    rows, K = 3, 512
    W, dense = _matrix(fmt, rows, K, 42 + fmt)
    g = np.random.default_rng(43).standard_normal(K).astype(np.float32) * 4
    for j in (0, 1, 31, 32, 255, 256, 511):
        for c in (2.5, -0.75, 9.0):
            gg = g.copy()
            gg[j] = c
            u = np.zeros(K, np.float32)
            u[j] = 1.0
            y, a, b = oracle.geglu_down(fmt, W, gg, u, rows, K)
            gel = oracle.gelu_tanh(c)
            assert np.array_equal(y, dense[:, j] * gel)
            assert np.array_equal(a, np.abs(dense[:, j] * gel))
            assert np.array_equal(b, np.abs(dense[:, j]) * (abs(c) + abs(gel)))


def test_geglu_down_clamped_gate_is_a_scaled_matvec():
    # For a >= 6 the clamp holds the tanh argument at 15, so
    # gelu(a) = a (1 + tanh(15)) / 2 and y = gelu(a) * (W u).
    rows, K = 7, 1024
    W, _ = _matrix(oracle.FORMAT_Q4_0, rows, K, 44)
    u = np.random.default_rng(45).standard_normal(K).astype(np.float32)
    g = np.full(K, 8.0, np.float32)
    y, a, _ = oracle.geglu_down(oracle.FORMAT_Q4_0, W, g, u, rows, K)
    ymv, amv = oracle.matvec(oracle.FORMAT_Q4_0, W, u, rows, K)
    s = 8.0 * (1.0 + math.tanh(15.0)) / 2.0
    assert np.all(np.abs(y - s * ymv) <= 1e-13 * s * amv)
    assert np.all(np.abs(a - s * amv) <= 1e-13 * s * amv)


@pytest.mark.parametrize("fmt,K", [(oracle.FORMAT_Q4_0, 64), (oracle.FORMAT_Q4_K, 256), (oracle.FORMAT_Q6_K, 256)])
def test_geglu_down_brute_force_exact_rational(fmt, K):
    # h_j = gelu(g_j) u_j as one double product; the sum over j then checked
    # exactly with rationals.
    W, dense = _matrix(fmt, 2, K, 46 + fmt)
    rng = np.random.default_rng(47)
    g = (rng.standard_normal(K) * 3).astype(np.float32)
    u = rng.standard_normal(K).astype(np.float32)
    y, a, _ = oracle.geglu_down(fmt, W, g, u, 2, K)
    h = [oracle.gelu_tanh(float(gv)) * float(uv) for gv, uv in zip(g, u)]
    for r in range(2):
        exact = sum(Fraction(float(w)) * Fraction(hv) for w, hv in zip(dense[r], h))
        absum = sum(abs(Fraction(float(w)) * Fraction(hv)) for w, hv in zip(dense[r], h))
        assert abs(Fraction(y[r]) - exact) <= Fraction(K) * Fraction(2) ** -52 * absum
        assert abs(Fraction(a[r]) - absum) <= Fraction(K) * Fraction(2) ** -52 * absum


def test_geglu_down_row_selection_and_partial_blocks():
    rows, K = 9, 256
    W, _ = _matrix(oracle.FORMAT_Q4_0, rows, K, 48)
    rng = np.random.default_rng(49)
    g, u = (rng.standard_normal(K).astype(np.float32) for _ in range(2))
    y, a, b = oracle.geglu_down(oracle.FORMAT_Q4_0, W, g, u, rows, K)
    idx = np.array([8, 0, 3, 3])
    ys, as_, bs = oracle.geglu_down(oracle.FORMAT_Q4_0, W, g, u, rows, K, row_idx=idx)
    assert np.array_equal(ys, y[idx]) and np.array_equal(as_, a[idx]) and np.array_equal(bs, b[idx])
    with pytest.raises(ValueError):
        oracle.geglu_down(oracle.FORMAT_Q4_0, np.zeros(18, np.uint8), np.zeros(48, np.float32),
                          np.zeros(48, np.float32), 1, 48)


# ---------------------------------------------------------------- RMS norm (Q8 prologue)

def _wide_rows(K, rng):
    normal = rng.standard_normal(K)
    wide = rng.standard_normal(K) * 2.0 ** rng.integers(-140, 120, K)
    sub = rng.integers(1, 1 << 23, K).astype(np.uint32).view(np.float32).astype(np.float64)   # subnormals
    spike = np.concatenate([[1.0 + 2.0 ** -23 * rng.integers(0, 1 << 23)], 2.0 ** rng.integers(-149, -20, K - 1)])
    return [r.astype(np.float32) for r in (normal, wide, sub, spike)]


def test_rmsnorm_sum_of_squares_is_the_exact_sum_rounded_once():
    rng = np.random.default_rng(60)
    K = 256
    for x in _wide_rows(K, rng):
        _, ss, _ = oracle.rmsnorm(x[None], np.zeros(K, np.float32), 1.0, 1e-6, 1, K)
        exact = sum((Fraction(float(v)) ** 2 for v in x), Fraction(0))
        assert ss[0] == float(exact)   # float(Fraction) rounds to nearest


def test_rmsnorm_closed_form_perfect_square():
    # x = 3 everywhere and eps = 7: ss / K = 9, r = sqrt(16) = 4, inv = 1/4,
    # y = 0.75 (w + offset)
    K = 256
    X = np.full((1, K), 3.0, np.float32)
    w = (np.arange(K) % 5 - 2).astype(np.float32)
    y, ss, r = oracle.rmsnorm(X, w, 1.0, 7.0, 1, K)
    assert ss[0] == 9.0 * K and r[0] == 4.0
    assert np.array_equal(y[0], (0.75 * (w + 1.0)).astype(np.float32))


def test_rmsnorm_power_of_two_scale_invariance():
    # eps far below the rounding of ss / K: scaling x by 4 scales ss by 16 and
    # r by 4 exactly, so y is unchanged bit for bit
    rng = np.random.default_rng(61)
    M, K = 3, 512
    X = rng.standard_normal((M, K)).astype(np.float32)
    w = rng.standard_normal(K).astype(np.float32)
    y1, _, r1 = oracle.rmsnorm(X, w, 1.0, 1e-30, M, K)
    y2, _, r2 = oracle.rmsnorm(X * np.float32(4), w, 1.0, 1e-30, M, K)
    assert np.array_equal(r2, 4 * r1) and np.array_equal(y1, y2)


def test_rmsnorm_against_high_precision_formula():
    # y_j against x_j (w_j + offset) / sqrt(mean x^2 + eps) in 50-digit
    # decimals: the fixed roundings (four f32, a few double) stay below
    # 5 * 2^-24 relative, plus the f32 underflow step (2^-149) of the two
    # products for elements far below the RMS
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    rng = np.random.default_rng(62)
    K = 256
    w = rng.standard_normal(K).astype(np.float32)
    for x in _wide_rows(K, rng)[:2]:
        y, _, _ = oracle.rmsnorm(x[None], w, 1.0, 1e-6, 1, K)
        mean = sum((Decimal(float(v)) ** 2 for v in x), Decimal(0)) / K
        rms = (mean + Decimal(float(np.float32(1e-6)))).sqrt()
        for j in range(K):
            exact = Decimal(float(x[j])) * (Decimal(float(w[j])) + 1) / rms
            tiny = Decimal(2) ** -149 * (1 + abs(Decimal(float(w[j])) + 1))
            assert abs(Decimal(float(y[0, j])) - exact) <= abs(exact) * Decimal(5) / Decimal(2 ** 24) + tiny


def test_rmsnorm_quantize_is_the_quantizer_on_the_normalized_row():
    rng = np.random.default_rng(63)
    M, K = 4, 128
    X = rng.standard_normal((M, K)).astype(np.float32)
    w = rng.standard_normal(K).astype(np.float32)
    q, d = oracle.rmsnorm_quantize_q8_0(X, w, 1.0, 1e-6, M, K)
    y, _, _ = oracle.rmsnorm(X, w, 1.0, 1e-6, M, K)
    q2, d2 = oracle.quantize_q8_0(y, M, K)
    assert np.array_equal(q, q2) and np.array_equal(d, d2)
    assert np.all(np.abs(q) <= 127) and np.any(np.abs(q) == 127)


# ---------------------------------------------------------------- planted mistakes are caught

def test_planted_nibble_order_mistake_is_caught_by_golden_fixture():
    """A decoder that reads the GGUF nibbles in sequential order (element 2j
    low, 2j+1 high) must disagree with the hand-built fixture."""
    blk, expect = _golden("q4_0_handbuilt.txt")
    qs = blk[2:]
    wrong = []
    for j in range(16):
        wrong += [(qs[j] & 15) - 8, (qs[j] >> 4) - 8]
    assert not np.array_equal(np.array(wrong, float), expect)


def test_planted_q6_k_bit_placement_mistakes_are_caught_by_golden_fixture():
    """Decoders that take a weight's top bits from the wrong qh bit pair, or
    its low bits from the other nibble, must disagree with the hand-built
    fixture (whose weights were derived from the intended codes)."""
    blk, expect = _golden("q6_k_handbuilt.txt")
    ql, qh = blk[:128], blk[128:192]
    sc = np.frombuffer(blk[192:208], dtype=np.int8).astype(int)
    d = float(np.frombuffer(blk[208:210], dtype=np.float16)[0])

    def decode(hi_shift, lo_high):
        out = []
        for e in range(256):
            half, c, l = e // 128, (e % 128) // 32, e % 32
            b = ql[64 * half + l + 32 * (c % 2)]
            lo = (b >> 4) if lo_high(c) else (b & 15)
            hi = (qh[32 * half + l] >> hi_shift(c)) & 3
            out.append(d * sc[e // 16] * ((lo | (hi << 4)) - 32))
        return np.array(out)

    assert np.array_equal(decode(lambda c: 2 * c, lambda c: c >= 2), expect)  # the reading itself
    assert not np.array_equal(decode(lambda c: 6 - 2 * c, lambda c: c >= 2), expect)  # qh pairs reversed
    assert not np.array_equal(decode(lambda c: 2 * c, lambda c: c % 2 == 1), expect)  # nibble by c parity
