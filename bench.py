"""Benchmark of the block-quantized decode path on GB300.

Default workload (one JSON line): the Q8_0 tied-embedding logit projection
with soft-cap and top-k over the 262,144 x 5376 vocabulary matrix (1.5 GB of
weights, far larger than L2).  One step = one gq_logits_topk call: stage x,
stream every weight row, soft-cap, per-CTA top-k, final merge.  The metric is
effective weight GB/s: the algorithmic bytes of a step (weights + x + the
k (index, value) pairs written) divided by the device time of the step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--config NAME | --suite]

Other workloads (--config / --suite) print one line each with the same keys:
q4_0_matvec_4096x4096, q4_k_matvec_21504x5376, q4_0_ffn_gelu_21504x5376,
q4_0_gemm_q8act_512x21504x5376.  Small matrices rotate over enough
independent copies that the working set exceeds 4x the L2 size.

--impl reference times the fp64 C oracle on the host cores on a bounded
sample of the same workload (the oracle is the reference of this project).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

DEFAULT_WORKLOAD = "q8_0_logits_topk_262144x5376"
METRIC = "quant matvec effective weight GB/s (% of GB300 HBM peak); M=512 int8 GEMM TOPS"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------- environment

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


_CSRC = os.path.join(ROOT, "block_quantized_matvec_gq_gb300", "csrc")
_INCLUDE = os.path.join(ROOT, "include")


def _kernel_unit(kernel: str):
    """The csrc translation unit that defines the __global__ function `kernel`
    (or, for a kernel template defined in a header, the unit that includes
    that header and instantiates it)."""
    pat = re.compile(r"__global__[^;{]*?\b" + re.escape(kernel) + r"\s*\(", re.S)
    names = sorted(os.listdir(_CSRC))
    for name in names:
        if name.endswith(".cu"):
            with open(os.path.join(_CSRC, name)) as f:
                if pat.search(f.read()):
                    return os.path.join(_CSRC, name)
    for header in names:
        if header.endswith(".cuh"):
            with open(os.path.join(_CSRC, header)) as f:
                if not pat.search(f.read()):
                    continue
            inc = re.compile(r'^\s*#\s*include\s*"' + re.escape(header) + '"', re.M)
            for name in names:
                if name.endswith(".cu"):
                    with open(os.path.join(_CSRC, name)) as f:
                        if inc.search(f.read()):
                            return os.path.join(_CSRC, name)
    return None


def kernel_source_hash(kernel: str):
    """Digest of the sources a kernel's machine code depends on: its
    translation unit and every file it includes, transitively, from csrc/
    and include/ (None if no unit defines it)."""
    unit = _kernel_unit(kernel)
    if unit is None:
        return None
    seen, todo = set(), [unit]
    while todo:
        p = todo.pop()
        if p in seen:
            continue
        seen.add(p)
        with open(p) as f:
            for inc in re.findall(r'^\s*#\s*include\s*"([^"]+)"', f.read(), re.M):
                for d in (os.path.dirname(p), _CSRC, _INCLUDE):
                    q = os.path.join(d, inc)
                    if os.path.exists(q):
                        todo.append(os.path.normpath(q))
                        break
    h = hashlib.sha256()
    for p in sorted(seen):
        h.update(os.path.relpath(p, ROOT).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    sources are unchanged since the capture; otherwise None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    h = kernel_source_hash(kernel)
    if not e or e.get("kernel") != kernel or h is None or e.get("source_hash") != h:
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem,clocks.max.mem")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        def window(a, b):
            return [p for (t, p) in self.samples if a <= t <= b]
        sel = window(t0, t1)
        where = "timed"
        if not sel:  # timed region shorter than the sampling period: use the second before it
            sel = window(t0 - 1.5, t1 + 0.3)
            where = "timed+preceding load"
        if not sel:
            return None
        sm = [float(p[1]) for p in sel if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for p in sel if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in sel for n, v in zip(names, p[5:9]) if v.lower() == "active"})
        mem = [float(p[9]) for p in sel if len(p) > 9 and p[9].replace(".", "").isdigit()]
        mem_mx = [float(p[10]) for p in sel if len(p) > 10 and p[10].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sel), "window": where,
                "mem_mhz": statistics.median(mem) if mem else None, "mem_max_mhz": max(mem_mx) if mem_mx else None}


# ---------------------------------------------------------------- workloads

class Workload:
    name = ""
    kernel = ""           # dominant kernel (for the roofline)
    bound = "hbm"
    cpu_unit, cpu_scale = "GB/s", 1e9   # unit of the oracle's timing (cpu_reference amounts per second)

    def setup(self, torch, gq):
        raise NotImplementedError

    def step(self, i):
        raise NotImplementedError

    # End to end through the public API: every step copies the step's inputs
    # from pinned host memory, runs the step, and reads its outputs back.
    def e2e_inputs(self):
        return []

    def e2e_outputs(self):
        return []

    def e2e_targets(self, i):
        """The device tensors step i reads its host inputs into (the
        e2e_inputs, unless the step rotates its input copies)."""
        return self.e2e_inputs()

    def e2e_setup(self, torch):
        self._e2e_in = [(d, d.cpu().pin_memory()) for d in self.e2e_inputs()]
        self._e2e_out = [(d, torch.empty(d.shape, dtype=d.dtype).pin_memory()) for d in self.e2e_outputs()]
        self.h2d = sum(h.numel() * h.element_size() for _, h in self._e2e_in)
        self.d2h = sum(h.numel() * h.element_size() for _, h in self._e2e_out)

    def e2e_body(self, torch, i):
        """Step i end to end, without the final wait: the inputs' copy from
        pinned host memory, the API call, the outputs' copy back."""
        for d, (_, h) in zip(self.e2e_targets(i), self._e2e_in):
            d.copy_(h, non_blocking=True)
        self.step(i)
        for d, h in self._e2e_out:
            h.copy_(d, non_blocking=True)


def _to_dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class LogitsTopK(Workload):
    name = "q8_0_logits_topk_262144x5376"
    kernel = "k_q8_0_logits_topk"
    rows, K, k, cap = 262144, 5376, 10, 30.0
    launches_per_step = 1  # the top-k merge runs inside the logits kernel

    def setup(self, torch, gq):
        W, x = synth.q8_0_logits_inputs(self.rows, self.K)
        self.x_host = x
        Wc = _to_dev(torch, W.reshape(-1))
        del W
        self.Wp = gq.pack(gq.GQ_FORMAT_Q8_0, Wc, self.rows, self.K)
        del Wc
        self.x = _to_dev(torch, x)
        self.wsb = gq.gq_logits_topk_workspace_bytes(self.rows, self.K, self.k)
        self.ws = torch.zeros(self.wsb, dtype=torch.uint8, device="cuda")  # zero-filled once before first use
        # idx and val in one device buffer (16-byte aligned halves), so the
        # end-to-end step reads the result back with one copy
        self.kpad = -(-self.k // 4) * 4
        self.out = torch.empty(2 * self.kpad * 4, dtype=torch.uint8, device="cuda")
        self.idx = self.out[:self.k * 4].view(torch.int32)
        self.val = self.out[self.kpad * 4:self.kpad * 4 + self.k * 4].view(torch.float32)
        self.gq = gq
        self.bytes_per_step = gq.gq_packed_bytes(1, self.rows, self.K) + 4 * self.K + 8 * self.k
        self.weight_bytes = gq.gq_packed_bytes(1, self.rows, self.K)
        self.working_set = self.weight_bytes
        self.l2_policy = "inputs larger than L2 (1.5 GB weight matrix)"

    def step(self, i):
        self.gq.gq_logits_topk(self.Wp, self.x, self.cap, self.k, self.idx, self.val, None, self.ws,
                               self.wsb, self.rows, self.K)

    def e2e_setup(self, torch):
        self.xh = torch.from_numpy(self.x_host.copy()).pin_memory()
        self.out_h = torch.empty(self.out.numel(), dtype=torch.uint8).pin_memory()
        self.h2d, self.d2h = self.xh.numel() * 4, self.out.numel()

    def e2e_body(self, torch, i):
        self.x.copy_(self.xh, non_blocking=True)
        self.step(i)
        self.out_h.copy_(self.out, non_blocking=True)  # idx and val

    def cpu_reference(self, oracle, rows_sample):
        W, x = synth.q8_0_logits_inputs(self.rows, self.K)
        n = min(rows_sample, self.rows)
        sel = np.arange(n, dtype=np.int64)

        def run():
            y, _ = oracle.matvec(oracle.FORMAT_Q8_0, W, x, self.rows, self.K, row_idx=sel)
            c = np.array([oracle.softcap(v, self.cap) for v in y])
            oracle.topk(c, self.k)
        return run, n * (self.K // 32) * 34, f"{n} of {self.rows} rows (fp64 decode, soft-cap, full-sort top-{self.k})"


class Rotating(Workload):
    """A matvec-like workload over R independent weight copies (working set > 4x L2)."""
    launches_per_step = 1

    def _matvec_reference(self, oracle, fmt, W, x, rows_sample):
        n = min(rows_sample, self.rows)
        sel = np.arange(n, dtype=np.int64)
        row_bytes = W.shape[1]

        def run():
            oracle.matvec(fmt, W, x, self.rows, self.K, row_idx=sel)
        return run, n * row_bytes + 4 * self.K + 4 * n, f"{n} of {self.rows} rows (fp64 decode and dot)"

    def _rotate(self, torch, one_copy_bytes):
        l2 = torch.cuda.get_device_properties(0).L2_cache_size
        need = max(4 * l2, 256 << 20)
        return max(1, -(-need // one_copy_bytes))


class Q40Matvec(Rotating):
    name = "q4_0_matvec_4096x4096"
    kernel = "k_q4_0_matvec"
    rows, K = 4096, 4096

    def setup(self, torch, gq):
        W, x = synth.q4_0_matvec_inputs(self.rows, self.K)
        nbytes = gq.gq_packed_bytes(0, self.rows, self.K)
        R = self._rotate(torch, nbytes)
        Wp = gq.pack(0, _to_dev(torch, W.reshape(-1)), self.rows, self.K)
        self.copies = [Wp] + [Wp.clone() for _ in range(R - 1)]
        self.x = _to_dev(torch, x)
        self.y = torch.empty(self.rows, dtype=torch.float32, device="cuda")
        self.gq = gq
        self.bytes_per_step = nbytes + 4 * self.K + 4 * self.rows
        self.weight_bytes = nbytes
        self.working_set = nbytes * R
        self.l2_policy = f"{R} rotating weight copies ({nbytes * R / 2**20:.0f} MiB > 4x L2)"

    def step(self, i):
        self.gq.gq_q4_0_matvec(self.copies[i % len(self.copies)], self.x, self.y, self.rows, self.K)

    def e2e_inputs(self):
        return [self.x]

    def e2e_outputs(self):
        return [self.y]

    def cpu_reference(self, oracle, rows_sample):
        W, x = synth.q4_0_matvec_inputs(self.rows, self.K)
        return self._matvec_reference(oracle, oracle.FORMAT_Q4_0, W, x, rows_sample)


class Q40MatvecShortWide(Q40Matvec):
    """A short, wide Q4_0 matvec (256 rows, K = 21504: the FFN down
    projection's width with few rows): too few rows to fill the GPU, so K is
    split across the CTAs of a cluster (the shared-memory ring kernel)."""
    name = "q4_0_matvec_256x21504"
    kernel = "k_ring_matvec"
    rows, K = 256, 21504


class Q4KMatvec(Rotating):
    name = "q4_k_matvec_21504x5376"
    kernel = "k_q4k_matvec"
    rows, K = 21504, 5376

    def setup(self, torch, gq):
        W, x = synth.q4_k_matvec_inputs(self.rows, self.K)
        nbytes = gq.gq_packed_bytes(2, self.rows, self.K)
        R = self._rotate(torch, nbytes)
        Wp = gq.pack(2, _to_dev(torch, W.reshape(-1)), self.rows, self.K)
        self.copies = [Wp] + [Wp.clone() for _ in range(R - 1)]
        self.x = _to_dev(torch, x)
        self.y = torch.empty(self.rows, dtype=torch.float32, device="cuda")
        self.gq = gq
        self.bytes_per_step = nbytes + 4 * self.K + 4 * self.rows
        self.weight_bytes = nbytes
        self.working_set = nbytes * R
        self.l2_policy = f"{R} rotating weight copies ({nbytes * R / 2**20:.0f} MiB > 4x L2)"

    def step(self, i):
        self.gq.gq_q4k_matvec(self.copies[i % len(self.copies)], self.x, self.y, self.rows, self.K)

    def e2e_inputs(self):
        return [self.x]

    def e2e_outputs(self):
        return [self.y]

    def cpu_reference(self, oracle, rows_sample):
        W, x = synth.q4_k_matvec_inputs(self.rows, self.K)
        return self._matvec_reference(oracle, oracle.FORMAT_Q4_K, W, x, rows_sample)


class Q6KMatvec(Rotating):
    """Q6_K at the FFN shape (21 super-blocks per row, 4410 B per row)."""
    name = "q6_k_matvec_21504x5376"
    kernel = "k_q6k_matvec"
    rows, K = 21504, 5376

    def setup(self, torch, gq):
        W = synth.q6_k_weights(self.rows, self.K, synth.stream(6, 0))
        x = synth.normal(self.K, synth.stream(6, 1))
        nbytes = gq.gq_packed_bytes(3, self.rows, self.K)
        R = self._rotate(torch, nbytes)
        Wp = gq.pack(3, _to_dev(torch, W.reshape(-1)), self.rows, self.K)
        self.copies = [Wp] + [Wp.clone() for _ in range(R - 1)]
        self.x = _to_dev(torch, x)
        self.y = torch.empty(self.rows, dtype=torch.float32, device="cuda")
        self.gq = gq
        self.bytes_per_step = nbytes + 4 * self.K + 4 * self.rows
        self.weight_bytes = nbytes
        self.working_set = nbytes * R
        self.l2_policy = f"{R} rotating weight copies ({nbytes * R / 2**20:.0f} MiB > 4x L2)"

    def step(self, i):
        self.gq.gq_q6k_matvec(self.copies[i % len(self.copies)], self.x, self.y, self.rows, self.K)

    def e2e_inputs(self):
        return [self.x]

    def e2e_outputs(self):
        return [self.y]

    def cpu_reference(self, oracle, rows_sample):
        W = synth.q6_k_weights(self.rows, self.K, synth.stream(6, 0))
        x = synth.normal(self.K, synth.stream(6, 1))
        return self._matvec_reference(oracle, oracle.FORMAT_Q6_K, W, x, rows_sample)


class GegluDown(Rotating):
    """The FFN's down projection (5376 x 21504, Q4_0) taking the gate and up
    outputs, with gelu_tanh(g) * u formed while the input is staged."""
    name = "q4_0_geglu_down_5376x21504"
    kernel = "k_q4_0_matvec"
    rows, K = 5376, 21504

    def setup(self, torch, gq):
        W = synth.q4_0_weights(self.rows, self.K, synth.stream(7, 0))
        g = (synth.normal(self.K, synth.stream(7, 1)) * 2).astype(np.float32)
        u = synth.normal(self.K, synth.stream(7, 2))
        nbytes = gq.gq_packed_bytes(0, self.rows, self.K)
        R = self._rotate(torch, nbytes)
        Wp = gq.pack(0, _to_dev(torch, W.reshape(-1)), self.rows, self.K)
        self.copies = [Wp] + [Wp.clone() for _ in range(R - 1)]
        self.g = _to_dev(torch, g)
        self.u = _to_dev(torch, u)
        self.y = torch.empty(self.rows, dtype=torch.float32, device="cuda")
        self.gq = gq
        self.bytes_per_step = nbytes + 2 * 4 * self.K + 4 * self.rows
        self.weight_bytes = nbytes
        self.working_set = nbytes * R
        self.l2_policy = f"{R} rotating weight copies ({nbytes * R / 2**20:.0f} MiB > 4x L2)"

    def step(self, i):
        self.gq.gq_q4_0_geglu_down(self.copies[i % len(self.copies)], self.g, self.u, self.y, self.rows, self.K)

    def e2e_inputs(self):
        return [self.g, self.u]

    def e2e_outputs(self):
        return [self.y]

    def cpu_reference(self, oracle, rows_sample):
        W = synth.q4_0_weights(self.rows, self.K, synth.stream(7, 0))
        g = (synth.normal(self.K, synth.stream(7, 1)) * 2).astype(np.float32)
        u = synth.normal(self.K, synth.stream(7, 2))
        n = min(rows_sample, self.rows)
        sel = np.arange(n, dtype=np.int64)

        def run():
            oracle.geglu_down(oracle.FORMAT_Q4_0, W, g, u, self.rows, self.K, row_idx=sel)
        return run, n * W.shape[1] + 8 * self.K + 4 * n, f"{n} of {self.rows} rows (fp64 gated input, decode, dot)"


class RMSNormQ8(Rotating):
    """The prefill activations (512 tokens x 5376) normalized and quantized to
    Q8_0 in one kernel: X is read, Xq and dx are written."""
    name = "rmsnorm_q8_0_512x5376"
    kernel = "k_rmsnorm_q8_0"
    M, K = 512, 5376
    rows = M   # the rows of X

    def setup(self, torch, gq):
        X = synth.normal((self.M, self.K), synth.stream(8, 0))
        w = (synth.normal(self.K, synth.stream(8, 1)) * 0.1).astype(np.float32)
        xbytes = 4 * self.M * self.K
        R = self._rotate(torch, xbytes)
        X0 = _to_dev(torch, X)
        self.copies = [X0] + [X0.clone() for _ in range(R - 1)]
        self.w = _to_dev(torch, w)
        self.Xq = torch.empty((self.M, self.K), dtype=torch.int8, device="cuda")
        self.dx = torch.empty((self.M, self.K // 32), dtype=torch.float32, device="cuda")
        self.gq = gq
        self.bytes_per_step = xbytes + 4 * self.K + self.M * self.K + 4 * self.M * (self.K // 32)
        self.weight_bytes = xbytes
        self.working_set = xbytes * R
        self.l2_policy = f"{R} rotating activation copies ({xbytes * R / 2**20:.0f} MiB > 4x L2)"

    def step(self, i):
        self.gq.gq_rmsnorm_quantize_q8_0(self.copies[i % len(self.copies)], self.w, 1.0, 1e-6, self.Xq, self.dx,
                                         self.K, self.M)

    def e2e_inputs(self):
        return [self.copies[0]]

    def e2e_targets(self, i):
        return [self.copies[i % len(self.copies)]]   # the copy step(i) reads

    def e2e_outputs(self):
        return [self.Xq, self.dx]

    def cpu_reference(self, oracle, rows_sample):
        X = synth.normal((self.M, self.K), synth.stream(8, 0))
        w = (synth.normal(self.K, synth.stream(8, 1)) * 0.1).astype(np.float32)
        n = min(rows_sample, self.M)
        Xs = np.ascontiguousarray(X[:n])

        def run():
            oracle.rmsnorm_quantize_q8_0(Xs, w, 1.0, 1e-6, n, self.K)
        amount = n * (4 * self.K + self.K + 4 * (self.K // 32)) + 4 * self.K
        return run, amount, f"{n} of {self.M} tokens (exact sum of squares by math.fsum, f32 scaling, Q8_0)"


class Q8Quantize(Rotating):
    """The prefill activations (512 tokens x 5376, ~N(0,1)) quantized to
    Q8_0, the contraction's prologue: X is read, Xq and dx are written."""
    name = "q8_0_quantize_512x5376"
    kernel = "k_quantize_q8_0"
    M, K = 512, 5376
    rows = M   # the rows of X

    def setup(self, torch, gq):
        X = synth.normal((self.M, self.K), synth.stream(9, 0))
        xbytes = 4 * self.M * self.K
        R = self._rotate(torch, xbytes)
        X0 = _to_dev(torch, X)
        self.copies = [X0] + [X0.clone() for _ in range(R - 1)]
        self.Xq = torch.empty((self.M, self.K), dtype=torch.int8, device="cuda")
        self.dx = torch.empty((self.M, self.K // 32), dtype=torch.float32, device="cuda")
        self.gq = gq
        self.bytes_per_step = xbytes + self.M * self.K + 4 * self.M * (self.K // 32)
        self.weight_bytes = xbytes
        self.working_set = xbytes * R
        self.l2_policy = f"{R} rotating activation copies ({xbytes * R / 2**20:.0f} MiB > 4x L2)"

    def step(self, i):
        self.gq.gq_quantize_q8_0(self.copies[i % len(self.copies)], self.Xq, self.dx, self.K, self.M)

    def e2e_inputs(self):
        return [self.copies[0]]

    def e2e_targets(self, i):
        return [self.copies[i % len(self.copies)]]   # the copy step(i) reads

    def e2e_outputs(self):
        return [self.Xq, self.dx]

    def cpu_reference(self, oracle, rows_sample):
        X = synth.normal((self.M, self.K), synth.stream(9, 0))
        n = min(rows_sample, self.M)
        Xs = np.ascontiguousarray(X[:n])

        def run():
            oracle.quantize_q8_0(Xs, n, self.K)
        amount = n * (4 * self.K + self.K + 4 * (self.K // 32))
        return run, amount, f"{n} of {self.M} tokens (f32 division and rounding, Q8_0)"


class FFN(Rotating):
    name = "q4_0_ffn_gelu_21504x5376"
    kernel = "k_ffn_gate_up"
    rows, K = 21504, 5376
    launches_per_step = 2

    def setup(self, torch, gq):
        Wg, Wu, Wd, x = synth.ffn_inputs(self.rows, self.K)
        nb = gq.gq_packed_bytes(0, self.rows, self.K)
        R = self._rotate(torch, 3 * nb)
        g = gq.pack(0, _to_dev(torch, Wg.reshape(-1)), self.rows, self.K)
        u = gq.pack(0, _to_dev(torch, Wu.reshape(-1)), self.rows, self.K)
        d = gq.pack(0, _to_dev(torch, Wd.reshape(-1)), self.K, self.rows)
        self.copies = [(g, u, d)] + [(g.clone(), u.clone(), d.clone()) for _ in range(R - 1)]
        self.x = _to_dev(torch, x)
        self.h = torch.empty(self.rows, dtype=torch.float32, device="cuda")
        self.y = torch.empty(self.K, dtype=torch.float32, device="cuda")
        self.gq = gq
        self.bytes_per_step = 3 * nb + 4 * self.K + 2 * 4 * self.rows + 4 * self.K
        self.weight_bytes = 3 * nb
        self.working_set = 3 * nb * R
        self.l2_policy = f"{R} rotating weight sets ({3 * nb * R / 2**20:.0f} MiB > 4x L2)"

    def step(self, i):
        g, u, d = self.copies[i % len(self.copies)]
        self.gq.gq_ffn_gate_up_gelu(g, u, self.x, self.h, self.rows, self.K)
        self.gq.gq_q4_0_matvec(d, self.h, self.y, self.K, self.rows)

    def e2e_inputs(self):
        return [self.x]

    def e2e_outputs(self):
        return [self.y]

    def cpu_reference(self, oracle, rows_sample):
        Wg, Wu, Wd, x = synth.ffn_inputs(self.rows, self.K)
        nb = Wg.shape[1]

        def run():
            h = oracle.ffn_gate_up(Wg, Wu, x, self.rows, self.K)["h"]
            oracle.matvec(oracle.FORMAT_Q4_0, Wd, h.astype(np.float32), self.K, self.rows)
        amount = 3 * self.rows * nb + 4 * self.K + 2 * 4 * self.rows + 4 * self.K
        return run, amount, "the whole step (fp64 gate/up with GELU, then the down matvec)"


class Gemm(Workload):
    name = "q4_0_gemm_q8act_512x21504x5376"
    kernel = "k_gemm_pair"  # K % 256 == 0 and M > 128: f16 operand pieces on CTA pairs
    bound = "tensor"
    rows, K, M = 21504, 5376, 512
    launches_per_step = 3

    def setup(self, torch, gq):
        W, X = synth.gemm_inputs(self.rows, self.K, self.M)
        self.ws_bytes = gq.gq_q4_0_gemm_workspace_bytes(self.K, self.M)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        self.Wp = gq.pack(0, _to_dev(torch, W.reshape(-1)), self.rows, self.K)
        self.X = _to_dev(torch, X)
        self.Xq = torch.empty((self.M, self.K), dtype=torch.int8, device="cuda")
        self.dx = torch.empty((self.M, self.K // 32), dtype=torch.float32, device="cuda")
        self.Y = torch.empty((self.M, self.rows), dtype=torch.float32, device="cuda")
        self.gq = gq
        self.ops_per_step = 2 * self.M * self.rows * self.K
        self.bytes_per_step = gq.gq_packed_bytes(0, self.rows, self.K) + 4 * self.M * self.K + 4 * self.M * self.rows
        self.weight_bytes = gq.gq_packed_bytes(0, self.rows, self.K)
        self.working_set = self.bytes_per_step
        self.l2_policy = "compute-bound contraction (inputs stay resident)"

    def step(self, i):
        self.gq.gq_quantize_q8_0(self.X, self.Xq, self.dx, self.K, self.M)
        self.gq.gq_q4_0_gemm_q8act(self.Wp, self.Xq, self.dx, self.Y, self.ws, self.ws_bytes, self.rows, self.K,
                                   self.M)

    def e2e_inputs(self):
        return [self.X]

    def e2e_outputs(self):
        return [self.Y]

    cpu_unit, cpu_scale = "TOPS", 1e12
    cpu_tokens = 16   # the oracle's bounded sample: this many tokens against every row

    def cpu_reference(self, oracle, rows_sample):
        W, X = synth.gemm_inputs(self.rows, self.K, self.M)
        nt = min(self.M, self.cpu_tokens)
        Xs = np.ascontiguousarray(X[:nt])

        def run():
            q, d = oracle.quantize_q8_0(Xs, nt, self.K)
            oracle.gemm_q8act(W, q, d, self.rows, self.K, nt)
        if self.cpu_unit == "TOPS":
            amount = 2 * nt * self.rows * self.K
        else:
            amount = W.size + 4 * nt * self.K + 4 * nt * self.rows
        return run, amount, (f"{nt} of {self.M} tokens against all {self.rows} rows (Q8_0 quantization, "
                             "fp64 block-scaled contraction)")


class GemmSmallBatch8(Gemm, Rotating):
    """The same contraction at a small batch (a verifier's eight tokens): the
    register-operand tensor-core kernel (exact integer block dots, every
    weight streamed once per step).  The 65 MB weight matrix fits in L2, so
    the step rotates over independent copies (working set > 4x L2)."""
    name = "q4_0_gemm_q8act_8x21504x5376"
    kernel = "k_gemm_mma"
    bound = "hbm"  # reported as bytes per step (weights, X, Y) over the step time
    M = 8
    launches_per_step = 3  # quantizer, activation image, contraction
    cpu_unit, cpu_scale = "GB/s", 1e9
    cpu_tokens = 32

    def setup(self, torch, gq):
        super().setup(torch, gq)
        R = self._rotate(torch, self.weight_bytes)
        self.copies = [self.Wp] + [self.Wp.clone() for _ in range(R - 1)]
        self.working_set = self.weight_bytes * R
        self.l2_policy = f"{R} rotating weight copies ({self.weight_bytes * R / 2**20:.0f} MiB > 4x L2)"

    def step(self, i):
        self.gq.gq_quantize_q8_0(self.X, self.Xq, self.dx, self.K, self.M)
        self.gq.gq_q4_0_gemm_q8act(self.copies[i % len(self.copies)], self.Xq, self.dx, self.Y, self.ws,
                                   self.ws_bytes, self.rows, self.K, self.M)


class GemmSmallBatch32(GemmSmallBatch8):
    """32 tokens (a short prompt): the same kernel with four 8-token tiles."""
    name = "q4_0_gemm_q8act_32x21504x5376"
    kernel = "k_gemm_mma"
    M = 32


WORKLOADS = {w.name: w for w in (LogitsTopK, Q40Matvec, Q40MatvecShortWide, Q4KMatvec, Q6KMatvec, FFN, GegluDown,
                                  RMSNormQ8, Q8Quantize, Gemm, GemmSmallBatch8, GemmSmallBatch32)}


# ---------------------------------------------------------------- timing

def run_gpu(wl_cls, args, rank, world, torch, dist):
    import block_quantized_matvec_gq_gb300 as gq
    gq.lib()
    wl = wl_cls()
    wl.setup(torch, gq)
    stream = torch.cuda.current_stream()
    use_graph = True   # replay a captured graph of exactly K steps (no host launch cost in the timing)

    for i in range(args.warmup):
        wl.step(i)
    torch.cuda.synchronize()

    graph = None
    if use_graph:
        # capture exactly K steps; the timed region replays them once
        s = torch.cuda.Stream()
        s.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                for i in range(args.steps):
                    wl.step(i)
        torch.cuda.synchronize()
        graph.replay()  # one untimed replay (warm)
        torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        # load the GPU for ~1.5 s so the clock samples reflect a busy GPU
        t_end = time.time() + 1.5
        j = 0
        while time.time() < t_end:
            if graph is not None:
                graph.replay()
            else:
                wl.step(j)
                j += 1
            torch.cuda.synchronize()

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    e0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            wl.step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    clocks = None
    if sampler:
        time.sleep(0.25)
        sampler.stop()
        clocks = sampler.summary(t0, t1)

    ms = max_over_ranks(ms, dist, "cuda")

    # Per-call spread: five more replays of the same K steps, each timed alone,
    # with the timed run's own figure (rank 0; no collective in between).
    per_call = None
    if graph is not None and rank == 0:
        vals = [ms * 1000.0 / args.steps]
        for _ in range(5):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(stream)
            graph.replay()
            b.record(stream)
            torch.cuda.synchronize()
            vals.append(a.elapsed_time(b) * 1000.0 / args.steps)
        per_call = {"samples": len(vals), "steps_per_sample": args.steps,
                    "median_us": round(statistics.median(vals), 3), "min_us": round(min(vals), 3)}

    # End to end through the public API with host buffers (every workload).
    # Each step copies its inputs from pinned host memory, makes the API call
    # on the weight copy the device timing would use, copies the outputs back
    # into pinned host memory and waits for them.  The three are captured as
    # one CUDA graph per weight copy (a serving loop's form); each timed step
    # replays one and synchronizes.  Eager launches if capture fails.
    e2e = None
    if hasattr(wl, "e2e_setup") and rank == 0:
        wl.e2e_setup(torch)
        nrot = len(getattr(wl, "copies", [None]))
        s2 = torch.cuda.Stream()
        s2.wait_stream(torch.cuda.current_stream())
        graphs = None
        with torch.cuda.stream(s2):
            for i in range(3):
                wl.e2e_body(torch, i)
            s2.synchronize()
            try:
                graphs = []
                for i in range(nrot):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=s2):
                        wl.e2e_body(torch, i)
                    graphs.append(g)
            except RuntimeError:
                graphs = None
                torch.cuda.synchronize()

            def e2e_step(i):
                if graphs is not None:
                    graphs[i % nrot].replay()
                else:
                    wl.e2e_body(torch, i)
                s2.synchronize()
            for i in range(3):
                e2e_step(i)
            n = args.steps
            t_a = time.perf_counter()
            for i in range(n):
                e2e_step(i)
            t_b = time.perf_counter()
        torch.cuda.current_stream().wait_stream(s2)
        e2e_ms = (t_b - t_a) * 1e3 / n
        if wl.bound == "tensor":
            ev, eu = wl.ops_per_step / (e2e_ms * 1e-3) / 1e12, "TOPS"
        else:
            ev, eu = wl.bytes_per_step / (e2e_ms * 1e-3) / 1e9, "GB/s"
        e2e = {"value": round(ev, 3), "unit": eu,
               "h2d_bytes_per_step": wl.h2d, "d2h_bytes_per_step": wl.d2h,
               "ms_per_step": round(e2e_ms, 4), "launch": "graph" if graphs is not None else "eager"}
    return wl, ms, clocks, e2e, per_call


def max_over_ranks(ms, dist, device):
    """The slowest rank's time: the job ends when its last rank does."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step, ms_per_step, world):
    """Whole-job rate (weak scaling): the units every rank processed in one
    step, over the slowest rank's step time."""
    return units_per_rank_step * world / (ms_per_step * 1e-3)


def cpu_baseline(wl_cls, sample_rows):
    import oracle
    oracle.build()
    wl = wl_cls()
    if not hasattr(wl, "cpu_reference"):
        return None
    run, amount, desc = wl.cpu_reference(oracle, sample_rows)
    cores = oracle.threads()
    t = time.perf_counter()
    run()
    dt = time.perf_counter() - t
    out = {"value": round(amount / dt / wl.cpu_scale, 4), "unit": wl.cpu_unit, "cores": cores,
           "kind": "oracle", "sample": desc, "seconds": round(dt, 3), "cpu_model": cpu_model()}
    if cores > 1:
        # the same sample on one core (the row loops are the only parallel part)
        oracle.set_threads(1)
        try:
            t = time.perf_counter()
            run()
            d1 = time.perf_counter() - t
        finally:
            oracle.set_threads(cores)
        out["single_core"] = {"value": round(amount / d1 / wl.cpu_scale, 4), "seconds": round(d1, 3)}
    return out


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine() or "unknown"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--suite", action="store_true", help="every workload, one line each")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tensor-peaks", action="store_true",
                    help="build and run the tensor-path peak probes and print their JSON (no bench line)")
    ap.add_argument("--rows", type=int, default=0,
                    help="logits workload only: vocabulary rows (default 262144; smaller for profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.impl == "reference":
        return run_reference(args, rank)
    if args.tensor_peaks:
        sys.exit(tensor_peaks())

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    hbm, bf16, bf16_sus, peak_src = peaks()
    names = sorted(WORKLOADS) if args.suite else [args.config]
    if args.rows:
        LogitsTopK.rows = args.rows
        LogitsTopK.name = f"q8_0_logits_topk_{args.rows}x5376"
    for name in names:
        wl, ms, clocks, e2e, per_call = run_gpu(WORKLOADS[name], args, rank, world, torch, dist)
        if rank != 0:
            continue
        ms_step = ms / args.steps
        sec = ms_step * 1e-3
        if wl.bound == "tensor":
            value = job_throughput(wl.ops_per_step, ms_step, world) / 1e12
            unit = "TOPS"
            achieved = wl.ops_per_step / sec / 1e12
            roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": bf16, "unit": "TFLOP/s",
                    "frac": round(achieved / bf16, 4), "traffic": recorded_traffic(wl.kernel, wl.name),
                    "peak_source": f"{peak_src} bf16 dense (f16 MMAs run at the same rate; achieved counts "
                                   "useful ops, the exact f16-piece products make the tensor pipe do 3x that)"}
        else:
            value = job_throughput(wl.bytes_per_step, ms_step, world) / 1e9
            unit = "GB/s"
            roof = {"bound": "hbm", "achieved": round(wl.bytes_per_step / sec / 1e9, 2), "peak": hbm,
                    "unit": "GB/s", "frac": round(wl.bytes_per_step / sec / 1e9 / hbm, 4),
                    "traffic": recorded_traffic(wl.kernel, wl.name),
                    "peak_source": f"{peak_src} HBM copy bandwidth",
                    "timing": "events bracket every launch of the step (the dominant kernel plus "
                              "any small follow-up kernel), so achieved is a lower bound"}
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": {"workload": wl.name, "bytes_per_step": wl.bytes_per_step,
                       "weight_bytes": wl.weight_bytes, "working_set_bytes": wl.working_set,
                       "l2": wl.l2_policy, "parallelism": f"replicas x{world}"},
            "roofline": roof, "clocks": clocks, "per_call_us": per_call, "e2e": e2e,
            "gpu_launches": wl.launches_per_step * args.steps,
        }
        if not args.no_cpu_baseline and world == 1 and hasattr(wl, "cpu_reference"):
            line["cpu_baseline"] = cpu_baseline(WORKLOADS[name], sample_rows=wl.rows)
        else:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def tensor_peaks():
    """Build and run the tensor-path peak probes (block_quantized_matvec_gq_gb300/peaks/tensor_peaks.cu):
    tcgen05 kind::f16, tcgen05.ld read-out, mma.sync f16 and s8, f32 FMA (scalar and packed).
    Prints the probe's JSON object."""
    from block_quantized_matvec_gq_gb300 import build as gqbuild
    src = os.path.join(ROOT, "block_quantized_matvec_gq_gb300", "peaks", "tensor_peaks.cu")
    os.makedirs(gqbuild.BUILD, exist_ok=True)
    exe = os.path.join(gqbuild.BUILD, "tensor_peaks")
    cmd = [gqbuild.nvcc()] + gqbuild.ARCH + ["-O3", "-std=c++17", "-I", gqbuild.INCLUDE, "-I", gqbuild.CSRC,
                                             "--expt-relaxed-constexpr", "-o", exe, src]
    subprocess.run(cmd, check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    sys.stdout.write(r.stdout)
    return r.returncode


def run_reference(args, rank):
    """The oracle (fp64 C, OpenMP) on the host cores: rank 0 only."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl_cls = WORKLOADS[args.config]
    wl = wl_cls()
    if not hasattr(wl, "cpu_reference"):
        print(json.dumps({"impl": "reference", "unavailable": f"no oracle timing for {wl.name}"}))
        return
    sample = 32768
    run, amount, desc = wl.cpu_reference(oracle, sample)
    for _ in range(args.warmup):
        run()
    t = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t) / args.steps
    value = amount / dt / wl.cpu_scale
    unit = wl.cpu_unit
    cores = oracle.threads()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": unit, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name},
        "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


if __name__ == "__main__":
    main()
