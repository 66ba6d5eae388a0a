"""The JSON line bench.py prints: keys, types and internal consistency.

The GPU case runs a short bench of the 4096^3 workload through the library;
the CPU case runs the reference arm (the fp64 oracle) on the 256^3 workload.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=600):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                         capture_output=True, text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [x for x in out.stdout.strip().splitlines() if x.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _check_common(d, steps, warmup):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "dtype", "data", "config", "e2e"):
        assert k in d, k
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == steps and d["warmup"] == warmup and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert isinstance(d["config"], dict) and "workload" in d["config"]
    assert set(d["e2e"]) >= {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}


@pytest.mark.gpu
def test_gpu_bench_line_has_the_contract_keys():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    steps, warmup = 5, 3
    d = _run(["--workload", "gemm_4096_f16", "--steps", str(steps), "--warmup", str(warmup),
              "--e2e-steps", "2", "--dist-reps", "0", "--cpu-seconds", "1",
              "--sustained-seconds", "0.3"])
    _check_common(d, steps, warmup)
    assert d["scaling"] == "weak" and d["data"].startswith("synthetic")
    assert d["vs_baseline"] is None or d["vs_baseline"] > 0
    # roofline of the dominant kernel
    r = d["roofline"]
    assert r["bound"] in ("tensor", "hbm") and r["unit"] in ("TFLOP/s", "GB/s")
    assert 0 < r["frac"] < 1.5 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-6
    # the DRAM bytes of the committed ncu summary, whenever it was taken on the
    # current kernel code (the digest must not depend on where the repository sits)
    sys.path.insert(0, ROOT)
    import bench
    from software_pipelined_tiled_gemm_gb300 import _build
    assert r["traffic"] == bench.traffic_from_profiles("gemm_4096_f16", _build.kernel_digest())
    # one GEMM launch per step (the operands are aligned: no padding copy)
    assert d["gpu_launches"] == steps
    # the oracle timed on the host cores
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    # end to end through host buffers: A and B in, C out, every step
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] == 2 * 2 * 4096 * 4096
    assert e["d2h_bytes_per_step"] == 2 * 4096 * 4096
    assert 0 < e["value"] <= d["value"] * 1.05
    c = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(c)
    # the timed C and the end-to-end call's C, on the oracle's sample rows
    p = d["parity"]
    assert p["ok"] and p["elements"] >= 4096 and p["elements"] % 4096 == 0, p
    assert e["parity"]["ok"] and e["parity"]["elements"] == p["elements"], e["parity"]
    # the sustained window, with its own clock record
    s = d["sustained"]
    assert s["value"] > 0 and s["steps"] >= 10 and 0 < s["frac"] < 1.5
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(s["clocks"])
    # the fractions beside the measured one
    assert r["frac_of_nominal"] == pytest.approx(r["achieved"] / r["nominal_peak"])
    assert r["frac_of_clock_peak"] == pytest.approx(r["achieved"] / r["clock_peak"])
    assert r["clock_peak"] > r["nominal_peak"] * 0.8


def test_reference_arm_times_the_oracle_on_cpu():
    steps, warmup = 1, 1
    d = _run(["--impl", "reference", "--workload", "gemm_256_f16", "--steps", str(steps),
              "--warmup", str(warmup)], timeout=300)
    _check_common(d, steps, warmup)
    assert d["impl"] == "reference"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_lookup_follows_the_kernel_digest(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from software_pipelined_tiled_gemm_gb300 import _build
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k.md").write_text(
        "# summary\n"
        "bench-traffic: kernel=k<1> workload=w source_digest=abc dram_bytes_per_launch=123\n"
        "bench-traffic: kernel=k<1> workload=w:nn source_digest=abc dram_bytes_per_launch=456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profiles("w", "abc") == 123
    assert bench.traffic_from_profiles("w:nn", "abc") == 456
    assert bench.traffic_from_profiles("w", "other") is None      # kernel changed since
    assert bench.traffic_from_profiles("x", "abc") is None        # no summary
    monkeypatch.undo()
    # the committed summaries: each line's figure is found for its own workload
    digest = _build.kernel_digest()
    for fn in os.listdir(os.path.join(ROOT, "profiles")):
        for line in open(os.path.join(ROOT, "profiles", fn)):
            if line.startswith("bench-traffic:"):
                kv = dict(x.split("=", 1) for x in line.split()[1:])
                want = int(kv["dram_bytes_per_launch"]) if kv["source_digest"] == digest else None
                assert bench.traffic_from_profiles(kv["workload"], digest) == want


def test_cpu_baseline_sample_reaches_both_ends_and_checks_parity():
    # The oracle block the bench times is the first and the last rows of the
    # output; the same rows are the parity check of the GPU result.
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import gemm_inputs
    import oracle
    w = gemm_inputs.WORKLOADS["mosaic_16896x512x640_f16"]
    A, B = gemm_inputs.make(w)
    cpu, idx, ref = bench.cpu_baseline(A, B, w, seconds=0.05)
    rows = len(idx)
    assert 2 <= rows < w.M and idx[0] == 0 and idx[-1] == w.M - 1
    assert idx == sorted(set(idx)) and ref.shape == (rows, w.N)
    assert np.array_equal(ref, oracle.gemm_nt_entries(
        A, B, "f16", np.repeat(idx, w.N), np.tile(np.arange(w.N), rows)).reshape(rows, w.N))
    assert cpu["kind"] == "oracle" and "first" in cpu["sample"] and "last" in cpu["sample"]
    C = torch.from_numpy(oracle.round_to(ref, "f16").view(np.int16)).view(torch.float16)
    assert bench.parity_of_rows(C, ref, "f16", False)["ok"]
    bad = C.clone()
    bad[rows - 1, 7] = float(bad[rows - 1, 7]) + 0.5
    st = bench.parity_of_rows(bad, ref, "f16", False)
    assert not st["ok"] and st["bad"] == 1


@pytest.mark.gpu
def test_gpu_bench_headline_line_carries_the_other_configurations():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _run(["--steps", "3", "--warmup", "3", "--other-steps", "2", "--cpu-seconds", "1",
              "--e2e-steps", "1", "--dist-reps", "0", "--sustained-seconds", "0.1"], timeout=900)
    assert d["config"]["workload"] == "gemm_8192_f16" and d["parity"]["ok"]
    o = d["other_configs"]
    assert set(o) == {"gemm_256_f16", "gemm_4096_f16", "gemm_8192_f16:single_buffer",
                      "gelu_3072x16384x4096_bf16", "ragged_4095x4097x8191_f16",
                      "skinny_64x8192x8192_f16"}
    for name, r in o.items():
        assert r["value"] > 0 and r["ms_per_step"] > 0 and r["steps"] == 2, name
        assert r["roofline"]["bound"] in ("tensor", "hbm") and r["roofline"]["frac"] > 0, name
    assert o["skinny_64x8192x8192_f16"]["roofline"]["bound"] == "hbm"
    assert o["ragged_4095x4097x8191_f16"]["kernels_per_step"] == 2
    assert o["gemm_8192_f16:single_buffer"]["stages"] == 1
    assert "cublas_context" in o["gemm_4096_f16"] and "cublas_context" not in o[
        "gelu_3072x16384x4096_bf16"]
