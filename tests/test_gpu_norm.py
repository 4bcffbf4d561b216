"""GPU parity of the RMS norm fused with Q8_0 quantization
(gq_rmsnorm_quantize_q8_0): the codes Xq and the block scales dx must equal
the oracle's bit for bit, since every rounding of the path is fixed (the
sum of squares is the exact sum rounded once)."""

import numpy as np
import pytest

import block_quantized_matvec_gq_gb300 as gq
import oracle
import synth
from gpu_util import dev, guarded, torch

pytestmark = pytest.mark.gpu


def run(X, w, offset, eps, M, K):
    t = torch()
    fq, q, cq = guarded(M * K, t.int8, fill=-7)
    fd, d, cd = guarded(M * (K // 32), t.float32)
    gq.gq_rmsnorm_quantize_q8_0(dev(X), dev(w), offset, eps, q, d, K, M)
    t.cuda.synchronize()
    cq()
    cd()
    return q.cpu().numpy().reshape(M, K), d.cpu().numpy().reshape(M, K // 32)


def check(X, w, offset, eps, M, K):
    q, d = run(X, w, offset, eps, M, K)
    qr, dr = oracle.rmsnorm_quantize_q8_0(X, w, offset, eps, M, K)
    assert np.array_equal(q, qr), np.argwhere(q != qr)[:5]
    assert np.array_equal(d.view(np.uint32), dr.view(np.uint32)), np.argwhere(d != dr)[:5]


def special_rows(K, rng):
    """Rows that stress the exact sum: wide exponents, subnormals, one large
    value over many tiny ones, zeros, a constant, alternating signs."""
    wide = rng.standard_normal(K) * 2.0 ** rng.integers(-140, 120, K)
    sub = rng.integers(1, 1 << 23, K).astype(np.uint32).view(np.float32).astype(np.float64)
    spike = np.concatenate([[1.0 + 2.0 ** -23 * rng.integers(0, 1 << 23)], 2.0 ** rng.integers(-149, -20, K - 1)])
    zero = np.zeros(K)
    const = np.full(K, 3.0)
    alt = np.where(np.arange(K) % 2 == 0, 1.0, -1.0) * 2.0 ** 60
    return np.stack([wide, sub, spike, zero, const, alt]).astype(np.float32)


# M = 512, K = 5376 is the prefill activation; K = 49152 the largest row
@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (7, 256), (64, 5376), (512, 5376), (2, 49152)])
def test_rmsnorm_q8_matches_oracle_bitwise(M, K):
    X = synth.normal((M, K), synth.stream(800 + M, K))
    w = (synth.normal(K, synth.stream(801, K)) * 0.1).astype(np.float32)
    check(X, w, 1.0, 1e-6, M, K)


@pytest.mark.parametrize("K", [256, 5376])
def test_rmsnorm_q8_special_rows(K):
    rng = np.random.default_rng(810 + K)
    X = special_rows(K, rng)
    w = (rng.standard_normal(K) * 0.1).astype(np.float32)
    check(X, w, 1.0, 1e-6, X.shape[0], K)


def test_rmsnorm_q8_offset_and_eps():
    """offset 0 with w = 0 gives zero codes and scales; a large eps and
    another offset move the codes the same way on both sides."""
    M, K = 5, 512
    X = synth.normal((M, K), synth.stream(820, 0))
    q, d = run(X, np.zeros(K, np.float32), 0.0, 1e-6, M, K)
    assert np.all(q == 0) and np.all(d == 0.0)
    w = synth.normal(K, synth.stream(820, 1))
    check(X, w, 0.0, 1e-6, M, K)
    check(X, w, 1.0, 10.0, M, K)
    check(X * np.float32(1e-20), w, 1.0, np.float32(1e-38), M, K)


def gpu_sum_squares(X, M, K):
    t = torch()
    fs, ss, cs = guarded(M, t.float64, fill=-7.25)
    gq.gq_rmsnorm_sum_squares(dev(X), ss, K, M)
    t.cuda.synchronize()
    cs()
    return ss.cpu().numpy()


def midpoint_rows(K):
    """Rows whose exact sum of squares lies on or next to a rounding boundary
    of the double: 1 + 2^-53 (an exact tie: stays 1), the same plus a square
    far below the fixed-point window (the tie broken upward), 1 + 3 2^-53
    (a tie rounding up to even), and the tie plus a square just inside the
    window."""
    rows = []
    base = np.zeros(K, np.float64)
    r = base.copy(); r[0] = 1.0; r[1] = r[2] = 2.0 ** -27; rows.append(r)                   # 1 + 2^-53
    r = rows[0].copy(); r[3] = 2.0 ** -100; rows.append(r)                                  # + 2^-200
    r = base.copy(); r[0] = 1.0; r[1] = r[2] = 2.0 ** -27; r[3] = 2.0 ** -26.0; rows.append(r)  # 1 + 3 2^-53
    r = rows[0].copy(); r[3] = 2.0 ** -50; rows.append(r)                                   # + 2^-100
    r = base.copy(); r[0] = 2.0 ** 60; r[1] = r[2] = 2.0 ** 33; r[K - 1] = 2.0 ** -140; rows.append(r)
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("K", [32, 256, 5376, 49152])
def test_sum_of_squares_is_the_correctly_rounded_sum(K):
    """The statistic itself against math.fsum (the oracle's), bit for bit, on
    normal rows, the special rows and rows on rounding boundaries."""
    rng = np.random.default_rng(830 + K)
    X = np.concatenate([synth.normal((3, K), synth.stream(830, K)), special_rows(K, rng), midpoint_rows(K)])
    M = X.shape[0]
    ss = gpu_sum_squares(X, M, K)
    _, ss_ref, _ = oracle.rmsnorm(X, np.ones(K, np.float32), 0.0, 1e-6, M, K)
    assert np.array_equal(ss.view(np.uint64), ss_ref.view(np.uint64)), (ss, ss_ref)


def test_sum_of_squares_non_finite_rows():
    K = 64
    X = synth.normal((3, K), synth.stream(840, 0))
    X[0, 5] = np.inf
    X[1, 7] = np.nan
    X[2, 9] = -np.inf
    X[2, 10] = np.nan
    ss = gpu_sum_squares(X, 3, K)
    assert ss[0] == np.inf and np.isnan(ss[1]) and np.isnan(ss[2])
