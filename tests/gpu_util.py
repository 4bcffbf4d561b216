"""Helpers shared by the GPU parity tests (device transfer, packing, bounds)."""

from __future__ import annotations

import numpy as np

import block_quantized_matvec_gq_gb300 as gq


def torch():
    import torch as _t
    return _t


def dev(a: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a)).cuda()


def packed(fmt: int, W_canon: np.ndarray, rows: int, K: int):
    t = torch()
    Wc = dev(W_canon.reshape(-1))
    out = t.empty(gq.gq_packed_bytes(fmt, rows, K), dtype=t.uint8, device="cuda")
    gq.gq_pack(fmt, Wc, out, rows, K)
    return out


def guarded(n: int, dtype, guard: int = 64, fill=-7.25):
    """Device buffer with guard bands: returns (full, view, check_fn)."""
    t = torch()
    full = t.full((n + 2 * guard,), fill, dtype=dtype, device="cuda")
    view = full[guard:guard + n]
    ref = full.clone()

    def check():
        f = full.cpu()
        r = ref.cpu()
        assert t.equal(f[:guard], r[:guard]), "write before the output buffer"
        assert t.equal(f[guard + n:], r[guard + n:]), "write after the output buffer"

    return full, view, check


def assert_within(y_gpu: np.ndarray, y_ref: np.ndarray, a_ref: np.ndarray, rel: float = 1e-5, what=""):
    """|y - y_ref| <= rel * sum|w x| per row (the matvec acceptance bound)."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bound = rel * a_ref
    bad = np.nonzero(~(err <= bound))[0]
    if bad.size:
        i = bad[0]
        raise AssertionError(
            f"{what}: {bad.size} rows outside the bound; first row {i}: gpu={y_gpu[i]!r} "
            f"ref={y_ref[i]!r} err={err[i]:.3e} bound={bound[i]:.3e} (A={a_ref[i]:.3e})")
    return float(np.max(err / np.where(bound > 0, bound, 1.0))) if err.size else 0.0


def assert_same_specials(y_gpu, y_ref, a_ref, rel: float = 1e-5, what="", exact: bool = True):
    """Non-finite results exactly where the oracle's are (with exact: NaN
    where it is NaN and the same infinity where it is infinite; else any
    non-finite value), and the acceptance bound everywhere else."""
    y = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    nan_ref, inf_ref = np.isnan(y_ref), np.isinf(y_ref)
    if exact:
        assert np.array_equal(np.isnan(y), nan_ref), f"{what}: NaN pattern differs"
        assert np.array_equal(y[inf_ref], y_ref[inf_ref]), f"{what}: infinities differ"
    else:
        assert np.array_equal(~np.isfinite(y), nan_ref | inf_ref), f"{what}: non-finite set differs"
    fin = ~(nan_ref | inf_ref)
    if fin.any():
        assert_within(y[fin], y_ref[fin], np.asarray(a_ref)[fin], rel=rel, what=what)
    return int(nan_ref.sum()), int(inf_ref.sum())
