"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/*.h declares, and rejects bad arguments before
launching."""

import ctypes
import os
import re

import pytest

import block_quantized_matvec_gq_gb300 as gq
from block_quantized_matvec_gq_gb300 import build as gqbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gqbuild.build()
    return gq.lib()


def declared_functions():
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, n)).read() for n in sorted(os.listdir(inc)) if n.endswith(".h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gq_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    so = ctypes.CDLL(gq.LIB_PATH)
    for n in names:
        assert hasattr(so, n), n


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5, -6, -7):
        s = gq.status_string(st)
        assert s.startswith("GQ_")
    assert "unknown" in gq.status_string(12345)


def test_packed_bytes(lib):
    assert gq.gq_packed_bytes(0, 4096, 4096) == 9437184
    assert gq.gq_packed_bytes(1, 262144, 5376) == 1497366528
    assert gq.gq_packed_bytes(2, 21504, 5376) == 65028096
    assert gq.gq_packed_bytes(3, 21504, 5376) == 21504 * 21 * 210
    assert gq.gq_packed_bytes(3, 1, 512 + 32) == 0
    assert gq.gq_packed_bytes(0, 21504, 5376) == 65028096
    assert gq.gq_packed_bytes(0, 1, 48) == 0
    assert gq.gq_packed_bytes(2, 1, 512 + 32) == 0
    assert gq.gq_packed_bytes(7, 1, 32) == 0
    assert gq.gq_packed_bytes(0, 0, 32) == 0


def test_workspace_bytes(lib):
    assert gq.gq_logits_topk_workspace_bytes(262144, 5376, 10) > 0
    assert gq.gq_logits_topk_workspace_bytes(262144, 5376, 65) == 0
    assert gq.gq_logits_topk_workspace_bytes(262144, 5376, 0) == 0
    assert gq.gq_logits_topk_workspace_bytes(1, 32, 1) >= 8


# Fake, never-dereferenced addresses: validation must reject before any CUDA call.
A = 1 << 20          # 16-byte aligned
U = (1 << 20) + 4    # misaligned


def call(name, *args):
    return getattr(gq.lib(), name)(*args)


def test_matvec_argument_validation(lib):
    for name in ("gq_q4_0_matvec", "gq_q8_0_matvec", "gq_q4k_matvec", "gq_q6k_matvec"):
        assert call(name, None, A, A, 4, 256, 1, None) == gq.GQ_ERR_NULL
        assert call(name, A, None, A, 4, 256, 1, None) == gq.GQ_ERR_NULL
        assert call(name, A, A, None, 4, 256, 1, None) == gq.GQ_ERR_NULL
        assert call(name, U, A, A, 4, 256, 1, None) == gq.GQ_ERR_ALIGN
        assert call(name, A, U, A, 4, 256, 1, None) == gq.GQ_ERR_ALIGN
        assert call(name, A, A, U, 4, 256, 1, None) == gq.GQ_ERR_ALIGN
        assert call(name, A, A, A, 0, 256, 1, None) == gq.GQ_ERR_SHAPE
        assert call(name, A, A, A, 4, 0, 1, None) == gq.GQ_ERR_SHAPE
        assert call(name, A, A, A, 4, 256 + 16, 1, None) == gq.GQ_ERR_SHAPE
        assert call(name, A, A, A, 4, 256, 2, None) == gq.GQ_ERR_SHAPE
        assert call(name, A, A, A, 4, 256, 0, None) == gq.GQ_ERR_SHAPE
        assert call(name, A, A, A, 4, gq.GQ_MAX_K + 256, 1, None) == gq.GQ_ERR_SHAPE
    assert call("gq_q4k_matvec", A, A, A, 4, 288, 1, None) == gq.GQ_ERR_SHAPE
    assert call("gq_q6k_matvec", A, A, A, 4, 288, 1, None) == gq.GQ_ERR_SHAPE
    assert call("gq_q8_0_matvec", A + 16, A, A, 4, 256, 1, None) == gq.GQ_ERR_ALIGN   # needs 32 B
    assert call("gq_q4_0_matvec", A + 16, None, A, 4, 256, 1, None) == gq.GQ_ERR_NULL


def test_geglu_down_validation(lib):
    name = "gq_q4_0_geglu_down"
    assert call(name, None, A, A, A, 4, 256, 1, None) == gq.GQ_ERR_NULL
    assert call(name, A, None, A, A, 4, 256, 1, None) == gq.GQ_ERR_NULL
    assert call(name, A, A, None, A, 4, 256, 1, None) == gq.GQ_ERR_NULL
    assert call(name, A, A, A, None, 4, 256, 1, None) == gq.GQ_ERR_NULL
    assert call(name, U, A, A, A, 4, 256, 1, None) == gq.GQ_ERR_ALIGN
    assert call(name, A, U, A, A, 4, 256, 1, None) == gq.GQ_ERR_ALIGN
    assert call(name, A, A, U, A, 4, 256, 1, None) == gq.GQ_ERR_ALIGN
    assert call(name, A, A, A, U, 4, 256, 1, None) == gq.GQ_ERR_ALIGN
    assert call(name, A, A, A, A, 0, 256, 1, None) == gq.GQ_ERR_SHAPE
    assert call(name, A, A, A, A, 4, 256 + 16, 1, None) == gq.GQ_ERR_SHAPE   # not whole blocks (F16)
    assert call(name, A, A, A, A, 4, 256, 2, None) == gq.GQ_ERR_SHAPE
    assert call(name, A, A, A, A, 4, gq.GQ_MAX_K + 32, 1, None) == gq.GQ_ERR_SHAPE


def test_rmsnorm_quantize_validation(lib):
    name = "gq_rmsnorm_quantize_q8_0"
    f = ctypes.c_float
    one, eps = f(1.0), f(1e-6)
    assert call(name, None, A, one, eps, A, A, 64, 2, None) == gq.GQ_ERR_NULL
    assert call(name, A, None, one, eps, A, A, 64, 2, None) == gq.GQ_ERR_NULL
    assert call(name, A, A, one, eps, None, A, 64, 2, None) == gq.GQ_ERR_NULL
    assert call(name, A, A, one, eps, A, None, 64, 2, None) == gq.GQ_ERR_NULL
    for i in range(4):
        p = [A, A, A, A]
        p[i] = U
        assert call(name, p[0], p[1], one, eps, p[2], p[3], 64, 2, None) == gq.GQ_ERR_ALIGN
    assert call(name, A, A, one, eps, A, A, 65, 2, None) == gq.GQ_ERR_SHAPE
    assert call(name, A, A, one, eps, A, A, 0, 2, None) == gq.GQ_ERR_SHAPE
    assert call(name, A, A, one, eps, A, A, 64, 0, None) == gq.GQ_ERR_SHAPE
    assert call(name, A, A, one, eps, A, A, gq.GQ_MAX_K + 32, 2, None) == gq.GQ_ERR_SHAPE
    for bad in (0.0, -1e-6, float("nan"), float("inf")):
        assert call(name, A, A, one, f(bad), A, A, 64, 2, None) == gq.GQ_ERR_SHAPE
    for bad in (float("nan"), float("inf")):
        assert call(name, A, A, f(bad), eps, A, A, 64, 2, None) == gq.GQ_ERR_SHAPE


def test_ffn_logits_quant_gemm_pack_validation(lib):
    assert call("gq_ffn_gate_up_gelu", A, None, A, A, 4, 64, 1, None) == gq.GQ_ERR_NULL
    assert call("gq_ffn_gate_up_gelu", A, U, A, A, 4, 64, 1, None) == gq.GQ_ERR_ALIGN
    assert call("gq_ffn_gate_up_gelu", A, A, A, A, 4, 40, 1, None) == gq.GQ_ERR_SHAPE
    ws = gq.gq_logits_topk_workspace_bytes(100, 64, 10)
    f = ctypes.c_float(30.0)
    assert call("gq_logits_topk", A, A, f, 10, None, A, None, A, ws, 100, 64, 1, None) == gq.GQ_ERR_NULL
    assert call("gq_logits_topk", A + 16, A, f, 10, A, A, None, A, ws, 100, 64, 1, None) == gq.GQ_ERR_ALIGN
    assert call("gq_logits_topk", A, A, f, 10, A, A, U, A, ws, 100, 64, 1, None) == gq.GQ_ERR_ALIGN
    assert call("gq_logits_topk", A, A, f, 0, A, A, None, A, ws, 100, 64, 1, None) == gq.GQ_ERR_SHAPE
    assert call("gq_logits_topk", A, A, f, 65, A, A, None, A, ws, 100, 64, 1, None) == gq.GQ_ERR_SHAPE
    assert call("gq_logits_topk", A, A, f, 10, A, A, None, A, ws, 5, 64, 1, None) == gq.GQ_ERR_SHAPE
    assert call("gq_logits_topk", A, A, ctypes.c_float(float("nan")), 10, A, A, None, A, ws, 100, 64, 1,
                None) == gq.GQ_ERR_SHAPE
    assert call("gq_logits_topk", A, A, f, 10, A, A, None, None, ws, 100, 64, 1, None) == gq.GQ_ERR_WORKSPACE
    assert call("gq_logits_topk", A, A, f, 10, A, A, None, A, ws - 1, 100, 64, 1, None) == gq.GQ_ERR_WORKSPACE
    assert call("gq_quantize_q8_0", A, A, None, 64, 2, None) == gq.GQ_ERR_NULL
    assert call("gq_quantize_q8_0", A, U, A, 64, 2, None) == gq.GQ_ERR_ALIGN
    assert call("gq_quantize_q8_0", A, A, A, 65, 2, None) == gq.GQ_ERR_SHAPE
    assert call("gq_quantize_q8_0", A, A, A, 64, 0, None) == gq.GQ_ERR_SHAPE
    gws = gq.gq_q4_0_gemm_workspace_bytes(64, 4)
    assert gws == 8192 * 2  # one 128-token tile x two 32-blocks of f16 codes (K % 256 != 0: per-block fold)
    # two 128-token tiles (an even count: 256-token tiles for CTA pairs) x 8 blocks
    # x two f16 operand pieces, then one chunk factor per padded token
    assert gq.gq_q4_0_gemm_workspace_bytes(256, 4) == 2 * 8 * 2 * 8192 + 256 * 4
    assert gq.gq_q4_0_gemm_workspace_bytes(48, 4) == 0 and gq.gq_q4_0_gemm_workspace_bytes(64, 0) == 0
    assert call("gq_q4_0_gemm_q8act", A, A, A, None, A, gws, 8, 64, 4, None) == gq.GQ_ERR_NULL
    assert call("gq_q4_0_gemm_q8act", A, A, A, A, None, gws, 8, 64, 4, None) == gq.GQ_ERR_NULL
    assert call("gq_q4_0_gemm_q8act", A, A, U, A, A, gws, 8, 64, 4, None) == gq.GQ_ERR_ALIGN
    assert call("gq_q4_0_gemm_q8act", A, A, A, A, U, gws, 8, 64, 4, None) == gq.GQ_ERR_ALIGN
    assert call("gq_q4_0_gemm_q8act", A, A, A, A, A, gws, 8, 48, 4, None) == gq.GQ_ERR_SHAPE
    assert call("gq_q4_0_gemm_q8act", A, A, A, A, A, gws, 8, 64, 0, None) == gq.GQ_ERR_SHAPE
    assert call("gq_q4_0_gemm_q8act", A, A, A, A, A, gws - 16, 8, 64, 4, None) == gq.GQ_ERR_WORKSPACE
    assert call("gq_q4_0_gemm_block_dots", A, A, A, A, gws - 16, 8, 64, 4, None) == gq.GQ_ERR_WORKSPACE
    assert call("gq_q4_0_gemm_block_dots", A, A, None, A, gws, 8, 64, 4, None) == gq.GQ_ERR_NULL
    assert call("gq_pack", 9, A, A, 1, 32, None) == gq.GQ_ERR_FORMAT
    assert call("gq_pack", 0, A, None, 1, 32, None) == gq.GQ_ERR_NULL
    assert call("gq_pack", 0, A, U, 1, 32, None) == gq.GQ_ERR_ALIGN
    assert call("gq_unpack", 2, A, A, 1, 128, None) == gq.GQ_ERR_SHAPE


def test_binding_fails_loudly_without_cuda_tensors(lib):
    import torch
    x = torch.zeros(32)
    with pytest.raises(ValueError):
        gq.gq_q4_0_matvec(x, x, x, 1, 32)
