"""Host-side logic of bench.py that needs no GPU: the staleness check of the
recorded DRAM traffic (a kernel's digest covers its translation unit and
every file it includes, so a change to another kernel leaves it valid and a
change to a shared header does not)."""

import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_every_workload_kernel_has_a_unit():
    for wl in bench.WORKLOADS.values():
        assert bench._kernel_unit(wl.kernel) is not None, wl.kernel
        assert bench.kernel_source_hash(wl.kernel) == bench.kernel_source_hash(wl.kernel)


def test_unknown_kernel_has_no_digest_and_no_traffic():
    assert bench.kernel_source_hash("k_not_a_kernel") is None
    assert bench.recorded_traffic("k_not_a_kernel", "q4_0_matvec_4096x4096") is None


def test_digest_follows_the_include_graph(tmp_path, monkeypatch):
    src = os.path.join(ROOT, "block_quantized_matvec_gq_gb300", "csrc")
    csrc = tmp_path / "csrc"
    inc = tmp_path / "include"
    shutil.copytree(src, csrc, ignore=shutil.ignore_patterns("*.o"))
    shutil.copytree(os.path.join(ROOT, "include"), inc)
    monkeypatch.setattr(bench, "_CSRC", str(csrc))
    monkeypatch.setattr(bench, "_INCLUDE", str(inc))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h_q4 = bench.kernel_source_hash("k_q4_0_matvec")
    h_gemm = bench.kernel_source_hash("k_gemm_pair")
    # another kernel's unit: no effect
    with open(csrc / "gq_gemm_small.cu", "a") as f:
        f.write("\n// edit\n")
    assert bench.kernel_source_hash("k_q4_0_matvec") == h_q4
    assert bench.kernel_source_hash("k_gemm_pair") == h_gemm
    # a header only the matvec family includes
    with open(csrc / "gq_matvec.cuh", "a") as f:
        f.write("\n// edit\n")
    assert bench.kernel_source_hash("k_q4_0_matvec") != h_q4
    assert bench.kernel_source_hash("k_gemm_pair") == h_gemm
    # the public header reaches every kernel
    h_q4 = bench.kernel_source_hash("k_q4_0_matvec")
    with open(inc / "gq.h", "a") as f:
        f.write("\n/* edit */\n")
    assert bench.kernel_source_hash("k_q4_0_matvec") != h_q4
    assert bench.kernel_source_hash("k_gemm_pair") != h_gemm


def test_reference_arm_runs_for_every_workload(capsys):
    """--impl reference: the oracle, timed on the host for each workload (the
    1.5 GB logits matrix aside), prints one line in the workload's unit."""
    import argparse
    import json
    for name, wl in sorted(bench.WORKLOADS.items()):
        if name == bench.DEFAULT_WORKLOAD:
            continue
        bench.run_reference(argparse.Namespace(config=name, steps=1, warmup=1), rank=0)
        line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
        assert line["impl"] == "reference" and line["config"]["workload"] == name
        assert line["unit"] == wl.cpu_unit and line["value"] > 0
        assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    bench.run_reference(argparse.Namespace(config=bench.DEFAULT_WORKLOAD, steps=1, warmup=1), rank=1)
    assert capsys.readouterr().out == ""   # ranks other than 0 print nothing


def test_cpu_baseline_reports_one_core_and_the_model():
    """The oracle baseline of a bench line: the sample on all host cores, the
    same sample on one core (whenever the oracle has more than one thread),
    and the CPU model; the thread count is restored afterwards."""
    import oracle
    cores = oracle.threads()
    b = bench.cpu_baseline(bench.WORKLOADS["q4_0_matvec_4096x4096"], 512)
    assert b["kind"] == "oracle" and b["cores"] == cores and b["value"] > 0
    assert isinstance(b["cpu_model"], str) and b["cpu_model"]
    if cores > 1:
        assert b["single_core"]["value"] > 0 and b["single_core"]["seconds"] > 0
    else:
        assert "single_core" not in b
    assert oracle.threads() == cores
