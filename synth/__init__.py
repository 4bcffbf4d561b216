"""Seeded synthetic inputs for the block-quantized matvec workloads.

This module is shared by the oracle side (tests, the CPU baseline) and the
CUDA side (tests, bench, smoke).  It holds no arithmetic of the method: it
draws random bytes and random floats and lays them out as whole canonical
blocks, and it never decodes a block.

Canonical block byte sizes follow the quant-matvec table of "Metal kernel
capability table (Phase B ground truth)", section 1 (Q4_0 = 18 B per 32
weights, Q4_K = 144 B per 256 weights) and the Q8_0 record of 34 B per 32
weights (a 2-byte fp16 scale followed by 32 signed bytes).

How each field is drawn:

* Q4_0 payload: 16 uniform random bytes per block.  Every nibble of a
  uniform byte is an independent uniform integer 0..15, whatever order the
  format gives the nibbles, so no knowledge of the nibble order is needed.
* Q8_0 payload: 32 independent integers uniform on -127..127.
* Q4_K: 12 uniform random bytes for the packed 6-bit sub-scales and mins
  (every 6-bit field is then an independent uniform integer 0..63, whatever
  the bit packing) and 128 uniform random bytes of nibbles.
* Q6_K: 192 uniform random bytes for the low and high code bits (every 6-bit
  code is then an independent uniform integer 0..63, whatever the bit
  placement), 16 sub-scales uniform on -128..127, and the fp16 scale in the
  last two bytes.
* fp16 scales: the f32 value 2**e * U(0.5, 1.5), rounded to nearest-even
  fp16, stored little-endian in the first bytes of the block.
* Activations: standard normal f32.

Every tensor of a workload draws from its own stream,
``numpy.random.Generator(PCG64(seed * 2**32 + tensor_id))``.
"""

from __future__ import annotations

import dataclasses

import numpy as np

Q4_0_BYTES = 18
Q8_0_BYTES = 34
Q4_K_BYTES = 144
Q6_K_BYTES = 210
QK = 32  # weights per Q4_0 / Q8_0 block
QK_K = 256  # weights per Q4_K super-block

FORMAT_Q4_0 = 0
FORMAT_Q8_0 = 1
FORMAT_Q4_K = 2
FORMAT_Q6_K = 3

_BLOCK_BYTES = {FORMAT_Q4_0: Q4_0_BYTES, FORMAT_Q8_0: Q8_0_BYTES, FORMAT_Q4_K: Q4_K_BYTES,
                FORMAT_Q6_K: Q6_K_BYTES}
_BLOCK_WEIGHTS = {FORMAT_Q4_0: QK, FORMAT_Q8_0: QK, FORMAT_Q4_K: QK_K, FORMAT_Q6_K: QK_K}


def block_bytes(fmt: int) -> int:
    return _BLOCK_BYTES[fmt]


def block_weights(fmt: int) -> int:
    return _BLOCK_WEIGHTS[fmt]


def canonical_bytes(fmt: int, rows: int, K: int) -> int:
    return rows * (K // _BLOCK_WEIGHTS[fmt]) * _BLOCK_BYTES[fmt]


def stream(seed: int, tensor_id: int) -> np.random.Generator:
    """Independent random stream for one tensor of one workload."""
    return np.random.Generator(np.random.PCG64(seed * (1 << 32) + tensor_id))


def _fp16_scales(rng: np.random.Generator, n: int, exp2: int) -> np.ndarray:
    """n fp16 values 2**exp2 * U(0.5, 1.5), drawn in f32 then rounded to fp16."""
    u = rng.random(n, dtype=np.float32) + np.float32(0.5)
    v = u * np.float32(2.0 ** exp2)
    return v.astype(np.float16)


def q4_0_weights(rows: int, K: int, rng: np.random.Generator, d_exp2: int = -6) -> np.ndarray:
    """Canonical Q4_0 rows: uint8 array (rows, K//32*18)."""
    assert K % QK == 0
    nb = K // QK
    out = np.empty((rows, nb, Q4_0_BYTES), dtype=np.uint8)
    d = _fp16_scales(rng, rows * nb, d_exp2).reshape(rows, nb)
    out[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:] = rng.integers(0, 256, size=(rows, nb, 16), dtype=np.uint8)
    return out.reshape(rows, nb * Q4_0_BYTES)


def q8_0_weights(rows: int, K: int, rng: np.random.Generator, d_exp2: int = -9) -> np.ndarray:
    """Canonical Q8_0 rows: uint8 array (rows, K//32*34)."""
    assert K % QK == 0
    nb = K // QK
    out = np.empty((rows, nb, Q8_0_BYTES), dtype=np.uint8)
    d = _fp16_scales(rng, rows * nb, d_exp2).reshape(rows, nb)
    out[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    q = rng.integers(-127, 128, size=(rows, nb, 32), dtype=np.int8)
    out[:, :, 2:] = q.view(np.uint8)
    return out.reshape(rows, nb * Q8_0_BYTES)


def q4_k_weights(rows: int, K: int, rng: np.random.Generator, d_exp2: int = -8) -> np.ndarray:
    """Canonical Q4_K rows: uint8 array (rows, K//256*144).

    Bytes 0..1 hold d, bytes 2..3 hold dmin (independent draws), bytes 4..15
    the packed 6-bit sub-scales and mins, bytes 16..143 the nibbles.
    """
    assert K % QK_K == 0
    ns = K // QK_K
    out = np.empty((rows, ns, Q4_K_BYTES), dtype=np.uint8)
    d = _fp16_scales(rng, rows * ns, d_exp2).reshape(rows, ns)
    dmin = _fp16_scales(rng, rows * ns, d_exp2).reshape(rows, ns)
    out[:, :, 0:2] = d.view(np.uint8).reshape(rows, ns, 2)
    out[:, :, 2:4] = dmin.view(np.uint8).reshape(rows, ns, 2)
    out[:, :, 4:] = rng.integers(0, 256, size=(rows, ns, 140), dtype=np.uint8)
    return out.reshape(rows, ns * Q4_K_BYTES)


def q6_k_weights(rows: int, K: int, rng: np.random.Generator, d_exp2: int = -10) -> np.ndarray:
    """Canonical Q6_K rows: uint8 array (rows, K//256*210).

    Bytes 0..191 hold the code bits, 192..207 the int8 sub-scales, 208..209 d.
    """
    assert K % QK_K == 0
    ns = K // QK_K
    out = np.empty((rows, ns, Q6_K_BYTES), dtype=np.uint8)
    out[:, :, 0:192] = rng.integers(0, 256, size=(rows, ns, 192), dtype=np.uint8)
    out[:, :, 192:208] = rng.integers(-128, 128, size=(rows, ns, 16), dtype=np.int8).view(np.uint8)
    d = _fp16_scales(rng, rows * ns, d_exp2).reshape(rows, ns)
    out[:, :, 208:210] = d.view(np.uint8).reshape(rows, ns, 2)
    return out.reshape(rows, ns * Q6_K_BYTES)


def weights(fmt: int, rows: int, K: int, rng: np.random.Generator) -> np.ndarray:
    if fmt == FORMAT_Q4_0:
        return q4_0_weights(rows, K, rng)
    if fmt == FORMAT_Q8_0:
        return q8_0_weights(rows, K, rng)
    if fmt == FORMAT_Q4_K:
        return q4_k_weights(rows, K, rng)
    if fmt == FORMAT_Q6_K:
        return q6_k_weights(rows, K, rng)
    raise ValueError(fmt)


def normal(shape, rng: np.random.Generator) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32)


# --------------------------------------------------------------------------
# The five workloads.  Names say what each one is; sizes are the Gemma-4 31B
# shapes the source pages measure on (5376 embedding, 21504 FFN, 262,144
# vocabulary) plus a 4096-square Q4_0 case small enough for the oracle.
# --------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    description: str


WORKLOADS = {
    "q4_0_matvec_4096x4096": Workload(
        "q4_0_matvec_4096x4096", 0,
        "Q4_0 x f32 matvec, rows=4096, K=4096, batch 1"),
    "q8_0_logits_topk_262144x5376": Workload(
        "q8_0_logits_topk_262144x5376", 1,
        "Q8_0 x f32 tied-embedding logits, rows=262144, K=5376, soft-cap 30, top-10"),
    "q4_0_ffn_gelu_21504x5376": Workload(
        "q4_0_ffn_gelu_21504x5376", 2,
        "Q4_0 FFN decode: gate/up 21504x5376 + GELU gating, down 5376x21504"),
    "q4_k_matvec_21504x5376": Workload(
        "q4_k_matvec_21504x5376", 3,
        "Q4_K x f32 matvec, rows=21504, K=5376"),
    "q4_0_gemm_q8act_512x21504x5376": Workload(
        "q4_0_gemm_q8act_512x21504x5376", 4,
        "Q4_0 W 21504x5376 x Q8_0-quantized X 512x5376 -> Y 512x21504"),
}


def q4_0_matvec_inputs(rows=4096, K=4096, seed=0):
    """Q4_0 matvec: W (canonical), x."""
    return q4_0_weights(rows, K, stream(seed, 0)), normal(K, stream(seed, 1))


def q8_0_logits_inputs(rows=262144, K=5376, seed=1):
    """Tied-embedding logits: W (canonical Q8_0), x."""
    return q8_0_weights(rows, K, stream(seed, 0)), normal(K, stream(seed, 1))


def ffn_inputs(rows=21504, K=5376, seed=2):
    """FFN: W_gate, W_up (rows x K), W_down (K x rows), x (K)."""
    wg = q4_0_weights(rows, K, stream(seed, 0))
    wu = q4_0_weights(rows, K, stream(seed, 1))
    wd = q4_0_weights(K, rows, stream(seed, 2))
    return wg, wu, wd, normal(K, stream(seed, 3))


def q4_k_matvec_inputs(rows=21504, K=5376, seed=3):
    return q4_k_weights(rows, K, stream(seed, 0)), normal(K, stream(seed, 1))


def gemm_inputs(rows=21504, K=5376, M=512, seed=4):
    """Prefill contraction: W (canonical Q4_0, rows x K), X (M x K) f32."""
    return q4_0_weights(rows, K, stream(seed, 0)), normal((M, K), stream(seed, 1))
