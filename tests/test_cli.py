"""The planning CLI (python -m software_pipelined_tiled_gemm_gb300 budget):
runs without a GPU on the GB300 description."""
from __future__ import annotations

import os
import subprocess
import sys

import software_pipelined_tiled_gemm_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _budget(*args):
    res = subprocess.run([sys.executable, "-m", "software_pipelined_tiled_gemm_gb300", "budget",
                          *args], capture_output=True, text=True, cwd=ROOT, timeout=120)
    assert res.returncode == 0, res.stderr
    rows = {}
    for line in res.stdout.splitlines()[3:]:
        f = line.split()
        rows[f[0]] = f
    return res.stdout, rows


def test_budget_marks_depths_that_do_not_fit():
    out, rows = _budget("--m", "8192", "--n", "8192", "--k", "8192", "--tile-n", "256",
                        "--cta-group", "1")
    assert "GB300 description" in out
    # 128 x 256 single-CTA tiles: 48 KiB of ring per slice, so 4 fit and 5 do not
    # columns: stages, tile, grid, ring bytes, CTA total, fits, last wave
    assert rows["4"][5] == "ok" and rows["5"][5] == "OVER"
    assert int(rows["5"][3]) == sg.gemm_smem_bytes(128, 256, 64, 2, 5)
    for s in ("1", "2", "3", "4"):
        d = sg.describe(8192, 8192, 8192, "f16", stages=int(s), tile_n=256, cta_group=1,
                        variant="single_buffer" if s == "1" else "pipelined", device=sg.GB300)
        assert int(rows[s][4]) == d["smem_bytes"] and int(rows[s][2]) == d["grid"]


def test_budget_default_problem_and_ring_cap():
    out, rows = _budget("--k", "256", "--stages", "2", "6")
    assert rows["2"][5] == "ok" and rows["6->4"][5] == "ok"     # K = 256 has 4 slices
    _, rows = _budget("--k", "256", "--stages", "4", "--smem-limit", "100000")
    assert rows["4"][1:3] == ["none", "-"] and rows["4"][5] == "OVER"
