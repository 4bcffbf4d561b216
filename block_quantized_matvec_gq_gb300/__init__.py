"""Python binding of libgq (block-quantized matvec kernels for GB300, sm_103a).

Argument marshalling only: every function here checks that it got CUDA
tensors (or raw device addresses), passes pointers, sizes and the current
CUDA stream to the C entry point of the same name in libgq.so, and raises
GQError on a non-zero status.  All arithmetic runs in the library's CUDA
kernels; there is no fallback.  If libgq.so is missing or cannot be
loaded, importing this package succeeds but every call raises.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgq.so")

GQ_FORMAT_Q4_0 = 0
GQ_FORMAT_Q8_0 = 1
GQ_FORMAT_Q4_K = 2
GQ_FORMAT_Q6_K = 3
GQ_MAX_K = 49152
GQ_MAX_TOPK = 64

GQ_OK = 0
GQ_ERR_NULL = -1
GQ_ERR_ALIGN = -2
GQ_ERR_SHAPE = -3
GQ_ERR_WORKSPACE = -4
GQ_ERR_CUDA = -5
GQ_ERR_TIMEOUT = -6
GQ_ERR_FORMAT = -7

_lib = None
_load_error = None


class GQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def _declare(L):
    P = ctypes.c_void_p
    I = ctypes.c_int
    S = ctypes.c_size_t
    sig = {
        "gq_status_string": ([I], ctypes.c_char_p),
        "gq_packed_bytes": ([I, I, I], S),
        "gq_pack": ([I, P, P, I, I, P], I),
        "gq_unpack": ([I, P, P, I, I, P], I),
        "gq_q4_0_matvec": ([P, P, P, I, I, I, P], I),
        "gq_q8_0_matvec": ([P, P, P, I, I, I, P], I),
        "gq_q4k_matvec": ([P, P, P, I, I, I, P], I),
        "gq_q6k_matvec": ([P, P, P, I, I, I, P], I),
        "gq_ffn_gate_up_gelu": ([P, P, P, P, I, I, I, P], I),
        "gq_q4_0_geglu_down": ([P, P, P, P, I, I, I, P], I),
        "gq_logits_topk_workspace_bytes": ([I, I, I], S),
        "gq_logits_topk": ([P, P, ctypes.c_float, I, P, P, P, P, S, I, I, I, P], I),
        "gq_logits_topk_noalloc": ([P, P, ctypes.c_float, I, P, P, P, I, I, I, P], I),
        "gq_quantize_q8_0": ([P, P, P, I, I, P], I),
        "gq_rmsnorm_quantize_q8_0": ([P, P, ctypes.c_float, ctypes.c_float, P, P, I, I, P], I),
        "gq_rmsnorm_sum_squares": ([P, P, I, I, P], I),
        "gq_q4_0_gemm_workspace_bytes": ([I, I], S),
        "gq_q4_0_gemm_q8act": ([P, P, P, P, P, S, I, I, I, P], I),
        "gq_q4_0_gemm_block_dots": ([P, P, P, P, S, I, I, I, P], I),
        "gq_device_status": ([I], I),
        "gq_selftest_bounded_wait": ([P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res


def lib():
    """The loaded libgq.so (raises if it is missing: there is no fallback)."""
    global _lib, _load_error
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libgq.so is not built ({LIB_PATH}); run "
                               "block_quantized_matvec_gq_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        _declare(L)
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gq_status_string(int(status)).decode()


# ---------------------------------------------------------------- marshalling

def _ptr(t):
    """Device address of a CUDA tensor (or an int address / None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libgq takes CUDA tensors (device memory)")
    if not t.is_contiguous():
        raise ValueError("libgq takes contiguous tensors")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != GQ_OK:
        raise GQError(status, what)


# ---------------------------------------------------------------- entry points (same names as include/*.h)

def gq_packed_bytes(format: int, rows: int, K: int) -> int:
    return int(lib().gq_packed_bytes(format, rows, K))


def gq_pack(format, W_canon, W_packed, rows, K, stream=None):
    _check(lib().gq_pack(format, _ptr(W_canon), _ptr(W_packed), rows, K, _stream(stream)), "gq_pack")


def gq_unpack(format, W_packed, W_canon, rows, K, stream=None):
    _check(lib().gq_unpack(format, _ptr(W_packed), _ptr(W_canon), rows, K, _stream(stream)), "gq_unpack")


def gq_q4_0_matvec(W, x, y, rows, K, M=1, stream=None):
    _check(lib().gq_q4_0_matvec(_ptr(W), _ptr(x), _ptr(y), rows, K, M, _stream(stream)), "gq_q4_0_matvec")


def gq_q8_0_matvec(W, x, y, rows, K, M=1, stream=None):
    _check(lib().gq_q8_0_matvec(_ptr(W), _ptr(x), _ptr(y), rows, K, M, _stream(stream)), "gq_q8_0_matvec")


def gq_q4k_matvec(W, x, y, rows, K, M=1, stream=None):
    _check(lib().gq_q4k_matvec(_ptr(W), _ptr(x), _ptr(y), rows, K, M, _stream(stream)), "gq_q4k_matvec")


def gq_q6k_matvec(W, x, y, rows, K, M=1, stream=None):
    _check(lib().gq_q6k_matvec(_ptr(W), _ptr(x), _ptr(y), rows, K, M, _stream(stream)), "gq_q6k_matvec")


def gq_ffn_gate_up_gelu(W_gate, W_up, x, h, rows, K, M=1, stream=None):
    _check(lib().gq_ffn_gate_up_gelu(_ptr(W_gate), _ptr(W_up), _ptr(x), _ptr(h), rows, K, M,
                                     _stream(stream)), "gq_ffn_gate_up_gelu")


def gq_q4_0_geglu_down(W_down, g, u, y, rows, K, M=1, stream=None):
    _check(lib().gq_q4_0_geglu_down(_ptr(W_down), _ptr(g), _ptr(u), _ptr(y), rows, K, M, _stream(stream)),
           "gq_q4_0_geglu_down")


def gq_logits_topk_workspace_bytes(rows, K, k) -> int:
    return int(lib().gq_logits_topk_workspace_bytes(rows, K, k))


def gq_logits_topk(W, x, softcap, k, idx, val, logits_or_null, workspace, workspace_bytes, rows, K,
                   M=1, stream=None):
    _check(lib().gq_logits_topk(_ptr(W), _ptr(x), float(softcap), k, _ptr(idx), _ptr(val),
                                _ptr(logits_or_null), _ptr(workspace), int(workspace_bytes), rows, K, M,
                                _stream(stream)), "gq_logits_topk")


def gq_logits_topk_noalloc(W, x, softcap, k, idx, val, logits_or_null, rows, K, M=1, stream=None):
    """gq_logits_topk with the key lists in the library's own fixed device array
    (for callers that cannot allocate; calls that may overlap on the GPU race)."""
    _check(lib().gq_logits_topk_noalloc(_ptr(W), _ptr(x), float(softcap), k, _ptr(idx), _ptr(val),
                                        _ptr(logits_or_null), rows, K, M, _stream(stream)), "gq_logits_topk_noalloc")


def gq_quantize_q8_0(X, Xq, dx, K, M, stream=None):
    _check(lib().gq_quantize_q8_0(_ptr(X), _ptr(Xq), _ptr(dx), K, M, _stream(stream)), "gq_quantize_q8_0")


def gq_rmsnorm_quantize_q8_0(X, w, offset, eps, Xq, dx, K, M, stream=None):
    _check(lib().gq_rmsnorm_quantize_q8_0(_ptr(X), _ptr(w), float(offset), float(eps), _ptr(Xq), _ptr(dx), K, M,
                                          _stream(stream)), "gq_rmsnorm_quantize_q8_0")


def gq_rmsnorm_sum_squares(X, ss, K, M, stream=None):
    _check(lib().gq_rmsnorm_sum_squares(_ptr(X), _ptr(ss), K, M, _stream(stream)), "gq_rmsnorm_sum_squares")


def gq_q4_0_gemm_workspace_bytes(K, M) -> int:
    return int(lib().gq_q4_0_gemm_workspace_bytes(K, M))


def gq_q4_0_gemm_q8act(W, Xq, dx, Y, workspace, workspace_bytes, rows, K, M, stream=None):
    _check(lib().gq_q4_0_gemm_q8act(_ptr(W), _ptr(Xq), _ptr(dx), _ptr(Y), _ptr(workspace), int(workspace_bytes),
                                    rows, K, M, _stream(stream)), "gq_q4_0_gemm_q8act")


def gq_q4_0_gemm_block_dots(W, Xq, D, workspace, workspace_bytes, rows, K, M, stream=None):
    _check(lib().gq_q4_0_gemm_block_dots(_ptr(W), _ptr(Xq), _ptr(D), _ptr(workspace), int(workspace_bytes),
                                         rows, K, M, _stream(stream)), "gq_q4_0_gemm_block_dots")


def gq_selftest_bounded_wait(stream=None):
    _check(lib().gq_selftest_bounded_wait(_stream(stream)), "gq_selftest_bounded_wait")


def gq_device_status(reset: bool = True) -> int:
    """Synchronizes; GQ_ERR_TIMEOUT if a bounded in-kernel wait gave up."""
    return int(lib().gq_device_status(1 if reset else 0))


# ---------------------------------------------------------------- conveniences (allocation only)

def pack(format: int, W_canon, rows: int, K: int, stream=None):
    """Allocate a packed copy (torch uint8 on W_canon's device) and fill it with gq_pack."""
    import torch
    out = torch.empty(gq_packed_bytes(format, rows, K), dtype=torch.uint8, device=W_canon.device)
    gq_pack(format, W_canon, out, rows, K, stream)
    return out
