"""The Q8_0 code rule the quantizer kernels use, checked on the CPU against
the oracle's definition.

"Metal kernel capability table (Phase B ground truth)", section 2
(quantize_q8): q = clamp(round_half_away(x / d), -127, 127), d = amax / 127,
the division IEEE-rounded.  The kernels avoid the per-code division: with
r = RN(1/d) and y = RN(x r), the nearest integer is read from the bits of
m = RN(y + 1.5 * 2^23), and only quotients within 2^-15 of a half-integer
(or a reciprocal that overflowed) take the division itself.  This test
replays that sequence of correctly rounded f32 operations in numpy (each
numpy float32 operation rounds to nearest, with no fused multiply-add) and
requires the codes to equal the oracle's on millions of values: random
blocks over many octaves, quotients placed on half-integers and within
2^-16, 2^-15 and 2^-14 of them, values at the clamp, and extreme scales."""

import numpy as np

import oracle
import synth

MAGIC = np.float32(12582912.0)  # 1.5 * 2^23
WINDOW = np.float32(0.5) - np.float32(2.0 ** -15)


def rule_codes(X):
    """The kernels' codes for X (M x K, f32), by the reciprocal rule."""
    M, K = X.shape
    B = X.reshape(M, K // 32, 32)
    with np.errstate(all="ignore"):
        amax = np.max(np.abs(B), axis=2).astype(np.float32)
        d = (amax / np.float32(127.0)).astype(np.float32)
        r = (np.float32(1.0) / d).astype(np.float32)
        y = (B * r[..., None]).astype(np.float32)
        m = (y + MAGIC).astype(np.float32)
        f = (y - (m - MAGIC).astype(np.float32)).astype(np.float32)
        slow = ~(np.abs(y) <= np.float32(128.0)) | (np.abs(f) >= WINDOW)
        fast_q = m.view(np.int32).astype(np.int64) - 0x4B400000
        # the division itself: t = RN(x / d) in f32, then roundf (half away
        # from zero; exact in double), then fmaxf / fminf, which return -127
        # for a NaN quotient
        t = (B / d[..., None]).astype(np.float32).astype(np.float64)
        rt = np.sign(t) * np.floor(np.abs(t) + 0.5)
        exact = np.where(np.isnan(rt), -127.0, np.clip(rt, -127.0, 127.0))
        q = np.where(slow, exact, np.clip(fast_q, -127, 127))
        q = np.where(d[..., None] == 0, 0, q)
    return q.reshape(M, K).astype(np.int8), d


def check(X):
    M, K = X.shape
    q_ref, d_ref = oracle.quantize_q8_0(X, M, K)
    q, d = rule_codes(X)
    assert np.array_equal(d.view(np.uint32), d_ref.view(np.uint32))
    bad = np.nonzero(q != q_ref)
    assert bad[0].size == 0, (bad[0][:5], bad[1][:5], X[bad][:5], q[bad][:5], q_ref[bad][:5])


def test_random_blocks_over_many_octaves():
    M, K = 4096, 1024
    X = synth.normal((M, K), synth.stream(901, 0))
    scale = np.exp2(synth.stream(901, 1).integers(-60, 60, size=(M, K // 32))).astype(np.float32)
    X = (X.reshape(M, K // 32, 32) * scale[..., None]).reshape(M, K).astype(np.float32)
    check(X)


def test_quotients_on_and_next_to_half_integers():
    rng = synth.stream(902, 0)
    M, K = 2048, 1024
    X = np.empty((M, K), dtype=np.float32)
    B = X.reshape(M, K // 32, 32)
    amax = (rng.uniform(0.5, 2.0, size=(M, K // 32)) * np.exp2(rng.integers(-20, 20, size=(M, K // 32)))
            ).astype(np.float32)
    d = (amax / np.float32(127.0)).astype(np.float32)
    k = rng.integers(-127, 127, size=(M, K // 32, 31)).astype(np.float32)
    off = rng.choice(np.array([0.0, 2.0 ** -16, -2.0 ** -16, 2.0 ** -15, -2.0 ** -15, 2.0 ** -14, -2.0 ** -14],
                              dtype=np.float32), size=(M, K // 32, 31))
    B[..., 0] = amax
    B[..., 1:] = ((k + np.float32(0.5) + off) * d[..., None]).astype(np.float32)
    over = np.abs(B[..., 1:]) > amax[..., None]       # keep amax the block's largest value
    B[..., 1:][over] = np.copysign(amax[..., None], B[..., 1:])[over]
    check(X)


def test_clamp_zero_blocks_and_extreme_scales():
    K = 256
    rows = []
    for amax in (np.float32(3.0e38), np.float32(1.0e-38), np.float32(1.0e-41), np.float32(1.0), np.float32(0.0)):
        v = np.linspace(-1.0, 1.0, K, dtype=np.float32) * amax
        v[0] = amax
        rows.append(v)
    rows.append(np.linspace(-127.5, 127.5, K, dtype=np.float32))
    check(np.stack(rows).astype(np.float32))
