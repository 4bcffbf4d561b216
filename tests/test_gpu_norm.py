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
