"""The packing is lossless (gq_unpack restores the canonical bytes exactly) and
the packed planes hold what the header documents."""

import numpy as np
import pytest

import block_quantized_matvec_gq_gb300 as gq
import oracle
import synth
from gpu_util import dev, packed, torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,rows,K", [(0, 1, 32), (0, 37, 4096), (1, 5, 96), (1, 300, 5376),
                                        (2, 1, 256), (2, 77, 5376), (3, 1, 256), (3, 77, 5376)])
def test_pack_unpack_round_trip(fmt, rows, K):
    t = torch()
    W = synth.weights(fmt, rows, K, synth.stream(600 + fmt, rows))
    Wp = packed(fmt, W, rows, K)
    back = t.empty(W.size, dtype=t.uint8, device="cuda")
    gq.gq_unpack(fmt, Wp, back, rows, K)
    t.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), W.reshape(-1))
    assert Wp.numel() == W.size


def _decode_packed_host(fmt, P, rows, K):
    """Decode the packed planes on the host from the documented layout."""
    if fmt == oracle.FORMAT_Q4_0:
        nb = K // 32
        nib = P[:rows * nb * 16].reshape(rows, nb, 16)
        d = P[rows * nb * 16:].copy().view(np.float16).reshape(rows, nb).astype(np.float64)
        q = np.empty((rows, nb, 32), np.int64)
        q[:, :, 0::2] = nib & 15
        q[:, :, 1::2] = nib >> 4
        return ((q - 8) * d[:, :, None]).reshape(rows, K)
    if fmt == oracle.FORMAT_Q8_0:
        nb = K // 32
        u = P[:rows * nb * 32].reshape(rows, nb, 32).astype(np.int64)
        d = P[rows * nb * 32:].copy().view(np.float16).reshape(rows, nb).astype(np.float64)
        return ((u - 128) * d[:, :, None]).reshape(rows, K)
    if fmt == oracle.FORMAT_Q6_K:
        ns = K // 256
        lo = P[:rows * ns * 128].reshape(rows, ns, 128)
        hw = P[rows * ns * 128:rows * ns * 192].copy().view("<u4").reshape(rows, ns, 16).astype(np.int64)
        scp = P[rows * ns * 192:rows * ns * 208].reshape(rows, ns, 16)
        dp = P[rows * ns * 208:].reshape(rows, ns, 2)
        q = np.empty((rows, ns, 256), np.int64)
        q[:, :, 0::2] = lo & 15
        q[:, :, 1::2] = lo >> 4
        for j in range(16):               # element j of every 16-element word
            a, i = j // 4, j % 4
            p = 4 * i + (2 if a & 1 else 0) + (16 if a & 2 else 0)
            q[:, :, j::16] |= ((hw >> p) & 3) << 4
        sc = scp.copy().view(np.int8).astype(np.float64)
        d = dp.copy().view(np.float16).reshape(rows, ns).astype(np.float64)
        return (d[:, :, None] * np.repeat(sc, 16, axis=2) * (q - 32)).reshape(rows, K)
    raise ValueError(fmt)


@pytest.mark.parametrize("fmt", [oracle.FORMAT_Q4_0, oracle.FORMAT_Q8_0, oracle.FORMAT_Q6_K])
def test_packed_layout_is_as_documented(fmt):
    rows, K = 9, (512 if fmt == oracle.FORMAT_Q6_K else 160)
    W = synth.weights(fmt, rows, K, synth.stream(610, fmt))
    P = packed(fmt, W, rows, K).cpu().numpy()
    assert np.array_equal(_decode_packed_host(fmt, P, rows, K), oracle.dequant(fmt, W, K))


def test_packed_q4_k_records_keep_canonical_scale_bytes():
    rows, K = 3, 512
    W = synth.q4_k_weights(rows, K, synth.stream(611, 0))
    P = packed(oracle.FORMAT_Q4_K, W, rows, K).cpu().numpy()
    ns = K // 256
    rec = P[rows * ns * 128:].reshape(rows, ns, 16)
    assert np.array_equal(rec, W.reshape(rows, ns, 144)[:, :, :16])
