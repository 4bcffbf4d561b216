"""Test-side block ENCODERS: intended integer codes and scales -> canonical bytes.

They run in the opposite direction to the oracle's decoders, written from the
format definitions alone, so a decoding mistake in the oracle (nibble order,
offset, sign, the 6-bit packing) shows up as a mismatch between the values a
test intended and the values the oracle decodes.

Layouts (the GGUF conventions):
  Q4_0: fp16 d | 16 bytes, byte j = element j (low nibble) + element j+16 (high)
  Q8_0: fp16 d | 32 int8
  Q4_K: fp16 d | fp16 dmin | 12 bytes 6-bit sc/m | 128 bytes: chunk c (32 B)
        holds sub-block 2c (low nibbles) and sub-block 2c+1 (high nibbles)
  Q6_K: 128 bytes ql | 64 bytes qh | 16 int8 sub-scales | fp16 d; in each
        128-weight half, weight 32c + l keeps its low 4 bits in ql byte
        l + 32 (c % 2) of the half's 64 (low nibble for c < 2) and its top 2
        bits at bit 2c of qh byte l of the half's 32
"""

from __future__ import annotations

import numpy as np


def fp16_bytes(v: float) -> bytes:
    return np.array([v], dtype=np.float16).tobytes()


def enc_q4_0(q: np.ndarray, d: float) -> bytes:
    """q: 32 integers 0..15 (element order)."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (32,) and q.min() >= 0 and q.max() <= 15
    payload = bytes(int(q[j]) | (int(q[j + 16]) << 4) for j in range(16))
    return fp16_bytes(d) + payload


def enc_q8_0(q: np.ndarray, d: float) -> bytes:
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (32,) and q.min() >= -128 and q.max() <= 127
    return fp16_bytes(d) + q.astype(np.int8).tobytes()


def pack_q4_k_scales(sc, m) -> bytes:
    """8 six-bit scales and 8 six-bit mins -> 12 bytes."""
    sc = [int(v) for v in sc]
    m = [int(v) for v in m]
    assert all(0 <= v < 64 for v in sc + m)
    b = [0] * 12
    for s in range(4):
        b[s] = (sc[s] & 63) | ((sc[s + 4] >> 4) << 6)
        b[s + 4] = (m[s] & 63) | ((m[s + 4] >> 4) << 6)
        b[s + 8] = (sc[s + 4] & 15) | ((m[s + 4] & 15) << 4)
    return bytes(b)


def enc_q4_k(q: np.ndarray, sc, m, d: float, dmin: float) -> bytes:
    """q: 256 integers 0..15 (element order); sc, m: 8 integers 0..63."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() <= 15
    qs = bytearray(128)
    for c in range(4):
        for l in range(32):
            qs[32 * c + l] = int(q[64 * c + l]) | (int(q[64 * c + 32 + l]) << 4)
    return fp16_bytes(d) + fp16_bytes(dmin) + pack_q4_k_scales(sc, m) + bytes(qs)


def enc_q6_k(q: np.ndarray, sc, d: float) -> bytes:
    """q: 256 integers 0..63 (element order); sc: 16 integers -128..127."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() <= 63
    sc = [int(v) for v in sc]
    assert len(sc) == 16 and all(-128 <= v <= 127 for v in sc)
    ql = bytearray(128)
    qh = bytearray(64)
    for half in range(2):
        for c in range(4):
            for l in range(32):
                v = int(q[128 * half + 32 * c + l])
                ql[64 * half + l + 32 * (c % 2)] |= (v & 15) << (4 if c >= 2 else 0)
                qh[32 * half + l] |= (v >> 4) << (2 * c)
    return bytes(ql) + bytes(qh) + np.array(sc, dtype=np.int8).tobytes() + fp16_bytes(d)


def rows_from_blocks(blocks_per_row) -> np.ndarray:
    """List of rows (each a list of block byte strings) -> uint8 (rows, bytes)."""
    return np.frombuffer(b"".join(b"".join(r) for r in blocks_per_row), dtype=np.uint8).reshape(
        len(blocks_per_row), -1).copy()


def random_q4_0_matrix(rows, K, rng, dvals=None):
    """Canonical Q4_0 rows plus the intended dense float64 weights."""
    nb = K // 32
    q = rng.integers(0, 16, size=(rows, nb, 32))
    d = (dvals if dvals is not None else
         np.float16(2.0 ** -6) * (0.5 + rng.random((rows, nb))).astype(np.float16)).astype(np.float16)
    blocks = [[enc_q4_0(q[r, b], float(d[r, b])) for b in range(nb)] for r in range(rows)]
    dense = ((q - 8) * d.astype(np.float64)[:, :, None]).reshape(rows, K)
    return rows_from_blocks(blocks), dense, q, d


def random_q8_0_matrix(rows, K, rng):
    nb = K // 32
    q = rng.integers(-127, 128, size=(rows, nb, 32))
    d = (np.float16(2.0 ** -9) * (0.5 + rng.random((rows, nb))).astype(np.float16)).astype(np.float16)
    blocks = [[enc_q8_0(q[r, b], float(d[r, b])) for b in range(nb)] for r in range(rows)]
    dense = (q * d.astype(np.float64)[:, :, None]).reshape(rows, K)
    return rows_from_blocks(blocks), dense


def random_q4_k_matrix(rows, K, rng):
    ns = K // 256
    q = rng.integers(0, 16, size=(rows, ns, 256))
    sc = rng.integers(0, 64, size=(rows, ns, 8))
    m = rng.integers(0, 64, size=(rows, ns, 8))
    d = (np.float16(2.0 ** -8) * (0.5 + rng.random((rows, ns))).astype(np.float16)).astype(np.float16)
    dmin = (np.float16(2.0 ** -8) * (0.5 + rng.random((rows, ns))).astype(np.float16)).astype(np.float16)
    blocks = [[enc_q4_k(q[r, s], sc[r, s], m[r, s], float(d[r, s]), float(dmin[r, s]))
               for s in range(ns)] for r in range(rows)]
    dense = np.empty((rows, ns, 256))
    for r in range(rows):
        for s in range(ns):
            for sb in range(8):
                dense[r, s, 32 * sb:32 * sb + 32] = (
                    float(d[r, s]) * sc[r, s, sb] * q[r, s, 32 * sb:32 * sb + 32]
                    - float(dmin[r, s]) * m[r, s, sb])
    return rows_from_blocks(blocks), dense.reshape(rows, K)


def random_q6_k_matrix(rows, K, rng):
    ns = K // 256
    q = rng.integers(0, 64, size=(rows, ns, 256))
    sc = rng.integers(-128, 128, size=(rows, ns, 16))
    d = (np.float16(2.0 ** -10) * (0.5 + rng.random((rows, ns))).astype(np.float16)).astype(np.float16)
    blocks = [[enc_q6_k(q[r, s], sc[r, s], float(d[r, s])) for s in range(ns)] for r in range(rows)]
    dense = np.empty((rows, ns, 256))
    for r in range(rows):
        for s in range(ns):
            dense[r, s] = float(d[r, s]) * np.repeat(sc[r, s], 16) * (q[r, s] - 32)
    return rows_from_blocks(blocks), dense.reshape(rows, K)
