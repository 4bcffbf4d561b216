"""ctypes wrapper for the plain-C fp64 oracle (gq_oracle.c), and the RMS
norm, written here in numpy: its sum of squares is math.fsum, the correctly
rounded sum, and its other steps are single IEEE operations.

TEST INFRASTRUCTURE: only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package.  It shares no code with the CUDA
library and reads canonical (GGUF-order) block bytes only.

Functions without a pin against something other than the oracle itself:
none ("parity unpinned" applies only to bit compatibility with real GGUF
files, which no function here can be checked against).
"""

from __future__ import annotations

import ctypes
import math
import os
import shutil
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gq_oracle.c")
_LIB = os.path.join(_HERE, "libgq_oracle.so")

FORMAT_Q4_0 = 0
FORMAT_Q8_0 = 1
FORMAT_Q4_K = 2
FORMAT_Q6_K = 3
_SUPER = (FORMAT_Q4_K, FORMAT_Q6_K)  # 256-weight super-block formats
_BLOCK_BYTES = {0: 18, 1: 34, 2: 144, 3: 210}

_lib = None


def build(force: bool = False) -> str:
    """Compile gq_oracle.c into libgq_oracle.so (OpenMP when available).

    -ffp-contract=off keeps every f32/f64 operation separately rounded, so
    the oracle gives the same bits on x86-64 and aarch64 hosts.
    """
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found to build the oracle")
    base = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    tmp = _LIB + f".tmp{os.getpid()}"
    for extra in (["-fopenmp"], []):
        cmd = base + extra + [_SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, _LIB)
            return _LIB
    raise RuntimeError("oracle build failed:\n" + r.stderr)


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        L.gqo_half_to_double.argtypes = [ctypes.c_uint16]
        L.gqo_half_to_double.restype = ctypes.c_double
        for name in ("gqo_dequant_q4_0", "gqo_dequant_q8_0", "gqo_dequant_q4_k", "gqo_dequant_q6_k"):
            getattr(L, name).argtypes = [P, I64, P]
            getattr(L, name).restype = None
        L.gqo_q4_k_scale_min.argtypes = [P, ctypes.c_int, P, P]
        L.gqo_matvec.argtypes = [ctypes.c_int, P, I64, I64, P, P, I64, P, P]
        L.gqo_matvec.restype = ctypes.c_int
        L.gqo_gelu_tanh.argtypes = [ctypes.c_double]
        L.gqo_gelu_tanh.restype = ctypes.c_double
        L.gqo_softcap.argtypes = [ctypes.c_double, ctypes.c_double]
        L.gqo_softcap.restype = ctypes.c_double
        L.gqo_ffn_gate_up.argtypes = [P, P, I64, I64, P, P, I64, P, P, P, P, P]
        L.gqo_ffn_gate_up.restype = ctypes.c_int
        L.gqo_geglu_down.argtypes = [ctypes.c_int, P, I64, I64, P, P, P, I64, P, P, P]
        L.gqo_geglu_down.restype = ctypes.c_int
        L.gqo_topk.argtypes = [P, I64, I64, P, P]
        L.gqo_topk.restype = ctypes.c_int
        L.gqo_quantize_q8_0.argtypes = [P, I64, I64, P, P]
        L.gqo_quantize_q8_0.restype = ctypes.c_int
        L.gqo_block_dots.argtypes = [P, P, I64, I64, I64, I64, I64, I64, I64, P]
        L.gqo_block_dots.restype = ctypes.c_int
        L.gqo_gemm_q8act.argtypes = [P, P, P, I64, I64, I64, P, I64, P, I64, P, P]
        L.gqo_gemm_q8act.restype = ctypes.c_int
        L.gqo_set_threads.argtypes = [ctypes.c_int]
        L.gqo_set_threads.restype = None
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def half_to_double(h: int) -> float:
    return lib().gqo_half_to_double(int(h))


def dequant(fmt: int, blocks: np.ndarray, K: int) -> np.ndarray:
    """Decode canonical rows (rows x row_bytes uint8) to float64 (rows x K)."""
    blocks = _c(blocks, np.uint8)
    rows = blocks.size // (K // (256 if fmt in _SUPER else 32) * _BLOCK_BYTES[fmt])
    out = np.empty((rows, K), dtype=np.float64)
    fn = {0: lib().gqo_dequant_q4_0, 1: lib().gqo_dequant_q8_0, 2: lib().gqo_dequant_q4_k,
          3: lib().gqo_dequant_q6_k}[fmt]
    nblk = rows * K // (256 if fmt in _SUPER else 32)
    fn(_ptr(blocks), nblk, _ptr(out))
    return out


def q4_k_scale_min(sc12: bytes, s: int):
    a = np.frombuffer(bytes(sc12), dtype=np.uint8).copy()
    sc = ctypes.c_int()
    m = ctypes.c_int()
    lib().gqo_q4_k_scale_min(_ptr(a), s, ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def matvec(fmt: int, W: np.ndarray, x: np.ndarray, rows: int, K: int, row_idx=None):
    """(y, a) in float64 for the selected rows: y = W x, a = sum |w x|."""
    W = _c(W, np.uint8)
    x = _c(x, np.float32)
    idx = None if row_idx is None else _c(row_idx, np.int64)
    n = rows if idx is None else idx.size
    y = np.empty(n, dtype=np.float64)
    a = np.empty(n, dtype=np.float64)
    rc = lib().gqo_matvec(fmt, _ptr(W), rows, K, _ptr(x), _ptr(idx), n, _ptr(y), _ptr(a))
    if rc != 0:
        raise ValueError("oracle matvec rejected the shape")
    return y, a


def gelu_tanh(a: float) -> float:
    return lib().gqo_gelu_tanh(float(a))


def softcap(v: float, cap: float) -> float:
    return lib().gqo_softcap(float(v), float(cap))


def ffn_gate_up(Wg, Wu, x, rows: int, K: int, row_idx=None):
    """dict with g, u, ag, au, h (float64) for the selected rows."""
    Wg = _c(Wg, np.uint8)
    Wu = _c(Wu, np.uint8)
    x = _c(x, np.float32)
    idx = None if row_idx is None else _c(row_idx, np.int64)
    n = rows if idx is None else idx.size
    out = {k: np.empty(n, dtype=np.float64) for k in ("g", "u", "ag", "au", "h")}
    rc = lib().gqo_ffn_gate_up(_ptr(Wg), _ptr(Wu), rows, K, _ptr(x), _ptr(idx), n,
                               _ptr(out["g"]), _ptr(out["u"]), _ptr(out["ag"]),
                               _ptr(out["au"]), _ptr(out["h"]))
    if rc != 0:
        raise ValueError("oracle ffn rejected the shape")
    return out


def geglu_down(fmt: int, W, g, u, rows: int, K: int, row_idx=None):
    """(y, a, b) float64 for the selected rows: y = W h with h = gelu_tanh(g) * u,
    a = sum |w h|, b = sum |w| (|g u| + |h|)."""
    W = _c(W, np.uint8)
    g = _c(g, np.float32)
    u = _c(u, np.float32)
    idx = None if row_idx is None else _c(row_idx, np.int64)
    n = rows if idx is None else idx.size
    y, a, b = (np.empty(n, dtype=np.float64) for _ in range(3))
    rc = lib().gqo_geglu_down(fmt, _ptr(W), rows, K, _ptr(g), _ptr(u), _ptr(idx), n, _ptr(y), _ptr(a), _ptr(b))
    if rc != 0:
        raise ValueError("oracle geglu_down rejected the shape")
    return y, a, b


def topk(values: np.ndarray, k: int):
    v = _c(values, np.float64)
    idx = np.empty(k, dtype=np.int64)
    val = np.empty(k, dtype=np.float64)
    rc = lib().gqo_topk(_ptr(v), v.size, k, _ptr(idx), _ptr(val))
    if rc != 0:
        raise ValueError("oracle topk: k out of range")
    return idx, val


def quantize_q8_0(X: np.ndarray, M: int, K: int):
    X = _c(X, np.float32)
    q = np.empty((M, K), dtype=np.int8)
    d = np.empty((M, K // 32), dtype=np.float32)
    rc = lib().gqo_quantize_q8_0(_ptr(X), M, K, _ptr(q), _ptr(d))
    if rc != 0:
        raise ValueError("oracle quantize rejected the shape")
    return q, d


def rmsnorm(X, w, offset: float, eps: float, M: int, K: int):
    """RMS normalization of each token's row ("Metal kernel capability table
    (Phase B ground truth)", section 6: rms_norm scales by the inverse RMS
    and by (w + offset)), with every rounding fixed so that the Q8 codes
    that follow are a function of the inputs alone:
      ss  = sum_j x_j^2 rounded once to double (each x_j^2 is exact in
            double; math.fsum returns the correctly rounded sum),
      r   = sqrt(ss / K + eps), in double, each operation rounded,
      inv = f32(1 / r),
      y_j = f32(f32(x_j * inv) * f32(w_j + offset)).
    Returns (y f32[M][K], ss float64[M], r float64[M])."""
    X = np.ascontiguousarray(X, dtype=np.float32).reshape(M, K)
    wo = np.ascontiguousarray(w, dtype=np.float32) + np.float32(offset)   # f32 addition
    y = np.empty((M, K), dtype=np.float32)
    ss = np.empty(M, dtype=np.float64)
    r = np.empty(M, dtype=np.float64)
    for t in range(M):
        x64 = X[t].astype(np.float64)
        ss[t] = math.fsum((x64 * x64).tolist())
        r[t] = math.sqrt(ss[t] / K + float(np.float32(eps)))
        inv = np.float32(1.0 / r[t])
        y[t] = (X[t] * inv) * wo        # two f32 multiplications, each rounded
    return y, ss, r


def rmsnorm_quantize_q8_0(X, w, offset: float, eps: float, M: int, K: int):
    """rmsnorm, then the Q8_0 quantization of its f32 output: (q, d)."""
    y, _, _ = rmsnorm(X, w, offset, eps, M, K)
    return quantize_q8_0(y, M, K)


def block_dots(W, Xq, rows: int, K: int, M: int, t0: int, nt: int, r0: int, nr: int):
    W = _c(W, np.uint8)
    Xq = _c(Xq, np.int8)
    D = np.empty((nt, nr, K // 32), dtype=np.int32)
    rc = lib().gqo_block_dots(_ptr(W), _ptr(Xq), rows, K, M, t0, nt, r0, nr, _ptr(D))
    if rc != 0:
        raise ValueError("oracle block_dots rejected the range")
    return D


def gemm_q8act(W, Xq, dx, rows: int, K: int, M: int, tok_idx=None, row_idx=None):
    """(Y, A) float64 of shape (n_tok, n_row)."""
    W = _c(W, np.uint8)
    Xq = _c(Xq, np.int8)
    dx = _c(dx, np.float32)
    ti = None if tok_idx is None else _c(tok_idx, np.int64)
    ri = None if row_idx is None else _c(row_idx, np.int64)
    nt = M if ti is None else ti.size
    nr = rows if ri is None else ri.size
    Y = np.empty((nt, nr), dtype=np.float64)
    A = np.empty((nt, nr), dtype=np.float64)
    rc = lib().gqo_gemm_q8act(_ptr(W), _ptr(Xq), _ptr(dx), rows, K, M, _ptr(ti), nt,
                              _ptr(ri), nr, _ptr(Y), _ptr(A))
    if rc != 0:
        raise ValueError("oracle gemm rejected the shape")
    return Y, A


def set_threads(n: int) -> None:
    """Threads for the oracle's row-parallel loops from now on (n >= 1)."""
    lib().gqo_set_threads(int(n))


def threads() -> int:
    """OpenMP threads the oracle will use (1 when built without OpenMP)."""
    try:
        n = int(os.environ.get("OMP_NUM_THREADS", "0"))
    except ValueError:
        n = 0
    build()
    r = subprocess.run(["nm", "-D", _LIB], capture_output=True, text=True)
    if "omp_" not in r.stdout and "GOMP" not in r.stdout:
        return 1
    return n if n > 0 else (os.cpu_count() or 1)
