"""The bounds-checked build (libspgemm_checked.so, SPGEMM_BOUNDS_CHECKS=1).

Its kernels range-check every tile index, K slot, copy coordinate (the K
coordinate of a tiled copy must be 16-byte aligned), TMEM column, ring slot,
staging buffer, C block and stream-K workspace slot before using it.  A
failed check records GEMM_ERR_BOUNDS and the check's identity in the plan's
status word and skips the access; nothing traps.  These checks guard the
shared-memory ring whose reuse the Mosaic GPU pipelining guide's
delay_release discussion is about.

CPU tests: both builds load, name the new status and checks, and only the
checked build accepts the test hook that forces a check to fail.  GPU test:
in a child process that loads the checked build, every kernel instance and
path runs bit-exact against the oracle with no check firing, and the forced
failure is reported as GEMM_ERR_BOUNDS (GEMM_CHECK_TMA_COORD), after which a
normal GEMM on the same context is exact.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys
import textwrap

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _child(code, timeout=900):
    env = dict(os.environ, SPGEMM_BOUNDS_CHECKS="1")
    out = subprocess.run([sys.executable, "-c", textwrap.dedent(code)], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-4000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_checked_build_loads_and_names_its_codes():
    r = _child("""
        import json, software_pipelined_tiled_gemm_gb300 as sg
        lib = sg.load_library()
        print(json.dumps({"checked": sg.gemm_bounds_checked(), "path": sg.library_path(),
                          "status": sg.gemm_status_string(sg.GEMM_ERR_BOUNDS),
                          "coord": sg.gemm_wait_detail_string((1 << 16) | 18),
                          "slot": sg.gemm_wait_detail_string((2 << 16) | 17)}))
    """)
    assert r["checked"] == 1 and r["path"].endswith("libspgemm_checked.so")
    assert r["status"] == "GEMM_ERR_BOUNDS"
    assert "coordinate" in r["coord"] and "slot" in r["slot"]


def test_only_the_checked_build_accepts_the_forced_check_failure():
    import software_pipelined_tiled_gemm_gb300 as sg
    if sg.bounds_checked_requested():
        pytest.skip("this process already loads the checked build")
    assert sg.gemm_bounds_checked() == 0
    assert sg.gemm_status_string(sg.GEMM_ERR_BOUNDS) == "GEMM_ERR_BOUNDS"
    with pytest.raises(sg.GemmError) as e:
        sg.describe(512, 512, 512, "f16", device=sg.GB300, debug_fault=2)
    assert e.value.status == sg.GEMM_ERR_INVALID_ARG
    assert "bounds-checked" in sg.gemm_last_error()
    r = _child("""
        import json, software_pipelined_tiled_gemm_gb300 as sg
        info = sg.describe(512, 512, 512, "f16", device=sg.GB300, debug_fault=2)
        print(json.dumps({"tile_n": info["tile_n"]}))
    """)
    assert r["tile_n"] > 0


_GPU_CHILD = """
    import json, time
    import numpy as np, torch
    import gemm_inputs, oracle
    import software_pipelined_tiled_gemm_gb300 as sg
    from tests import gpu_util as gu
    assert sg.gemm_bounds_checked() == 1
    cases = [
        # (M, N, K, dtype, epilogue, stages, variant, tuning)
        (256, 256, 256, "f16", None, 4, "pipelined", {}),
        (512, 512, 512, "f16", None, 4, "pipelined", {"cta_group": 1, "tile_n": 256}),
        (512, 512, 512, "bf16", None, 3, "pipelined", {"cta_group": 1, "tile_n": 128}),
        (768, 1024, 1024, "f16", None, 6, "pipelined", {"cta_group": 2, "tile_n": 256}),
        (768, 1024, 1024, "f16", "relu", 4, "pipelined", {"cta_group": 2, "tile_n": 128}),
        (768, 1024, 4096, "f16", None, 4, "pipelined",
         {"cta_group": 2, "tile_n": 256, "max_ctas": 10, "tail_split": 1}),
        (384, 1024, 2048, "f16", None, 4, "pipelined",
         {"cta_group": 1, "tile_n": 256, "max_ctas": 5, "tail_split": 1}),
        (128, 512, 2048, "f16", None, 4, "pipelined", {}),
        (64, 1024, 2048, "f16", None, 6, "pipelined", {}),
        (512, 512, 768, "f16", "relu", 6, "pipelined", {"b_kn": 1, "cta_group": 2}),
        (384, 1024, 1024, "f16", None, 4, "pipelined",
         {"cta_group": 1, "tile_n": 256, "max_ctas": 5, "tail_split": 2}),
        (256, 512, 512, "f16", None, 1, "single_buffer", {}),
        (256, 384, 512, "f16", None, 4, "pipelined", {"out_f32": 1}),
        (300, 520, 1001, "f16", None, 4, "pipelined", {}),
        (512, 768, 1024, "f16", None, 6, "pipelined", {"cta_group": 2, "k_serpentine": 1,
                                                      "max_ctas": 4, "epi_groups": 2}),
        # M <= 64: 64-row A slices, 8 slices in flight (K halves in clusters;
        # whole K on 64-wide tiles; B stored K x N)
        (64, 4096, 2048, "f16", None, 8, "pipelined", {}),
        (33, 8192, 2048, "f16", None, 8, "pipelined", {"tile_n": 64}),
        (64, 2048, 1024, "f16", None, 8, "pipelined", {"b_kn": 1}),
    ]
    results = []
    for i, (M, N, K, dt, epi, stages, variant, tuning) in enumerate(cases):
        lim = 2 if dt == "f16" else 1
        A, B = gemm_inputs.custom(M, N, K, dtype=dt, dist="int", lo=-lim, hi=lim, seed=900 + i)
        Bdev = B.t().contiguous() if tuning.get("b_kn") else B
        C, info, canary = gu.run_device(A, Bdev, dt, epilogue=epi, stages=stages,
                                        variant=variant, **tuning)
        ref = oracle.gemm_nt(A, B, dt, epilogue=epi)
        if tuning.get("out_f32"):
            exact = bool(np.array_equal(C.numpy().astype(np.float64), ref))
        else:
            exact = bool(np.array_equal(gu.bits(C), oracle.round_to(ref, dt)))
        results.append({"case": i, "exact": exact, "canary": canary,
                        "stream_k": info["stream_k"], "sk_cluster": info["sk_cluster"],
                        "tail_splits": info["tail_splits"], "cta_group": info["cta_group"]})
    # The forced failure: CTA 0's first copy fails its check (run_device
    # asserts a clean status, so the plan is driven by hand here).
    forced = []
    for cg in (1, 2):
        A, B = gemm_inputs.custom(512, 512, 512, dist="int", lo=-2, hi=2, seed=77)
        a, b = A.cuda(), B.cuda()
        c = torch.zeros(512, 512, dtype=torch.float16, device="cuda")
        plan = sg.Plan(512, 512, 512, "f16", stages=4, cta_group=cg, tile_n=256,
                       timeout_ns=20_000_000, debug_fault=2)
        t0 = time.perf_counter()
        plan.run(a, b, c)
        status, detail = plan.check()
        el = time.perf_counter() - t0
        plan.close()
        C, _, canary = gu.run_device(A, B, "f16", cta_group=cg, tile_n=256)
        after = bool(np.array_equal(gu.bits(C), oracle.round_to(oracle.gemm_nt(A, B, "f16"), "f16")))
        forced.append({"cg": cg, "status": status, "detail": detail, "seconds": el,
                       "after_exact": after and canary})
    print(json.dumps({"results": results, "forced": forced}))
"""


@pytest.mark.gpu
def test_checked_build_runs_every_path_exactly_and_reports_a_forced_failure():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = _child(_GPU_CHILD, timeout=1200)
    for c in r["results"]:
        assert c["exact"] and c["canary"], c
    paths = r["results"]
    assert any(c["stream_k"] and not c["sk_cluster"] for c in paths)
    assert any(c["sk_cluster"] for c in paths)
    assert any(c["tail_splits"] > 1 for c in paths)
    assert {c["cta_group"] for c in paths} == {1, 2}
    for f in r["forced"]:
        assert f["status"] == 7, f                           # GEMM_ERR_BOUNDS
        assert f["detail"] == (1 << 16) | 18, f              # GEMM_CHECK_TMA_COORD
        assert f["seconds"] < 10.0 and f["after_exact"], f
