"""gemm_plan_describe against the plans the device builds: the host-only
planner tests rest on these two facts."""
from __future__ import annotations

import numpy as np
import pytest

import software_pipelined_tiled_gemm_gb300 as sg
from tests.test_planner_host import GB300

pytestmark = pytest.mark.gpu


def test_device_query_is_the_description_the_host_tests_use():
    st, desc = sg.gemm_device_query(0)
    assert st == sg.GEMM_OK, sg.gemm_last_error()
    assert desc.as_dict() == GB300


def _cases():
    named = [
        (8192, 8192, 8192, "f16", dict(stages=6)),
        (4096, 4096, 4096, "f16", dict(stages=6)),
        (3072, 16384, 4096, "bf16", dict(stages=6, epilogue="gelu")),
        (4095, 4097, 8191, "f16", dict(stages=6)),
        (64, 8192, 8192, "f16", dict(stages=6)),
        (16896, 512, 640, "f16", dict(stages=6)),
        (256, 256, 256, "f16", dict(stages=6)),
        (8192, 8192, 8192, "f16", dict(stages=1, variant="single_buffer")),
        (8192, 8192, 8192, "f16", dict(stages=6, b_kn=1)),
        (0, 512, 512, "f16", dict(stages=4)),
        (512, 512, 0, "f16", dict(stages=4)),
    ]
    rng = np.random.default_rng(2024)
    drawn = []
    for i in range(48):
        M = int(rng.choice([1, 64, 100, 128, 300, 512, 1000, 2048, 3000, 8192, 12000]))
        N = int(rng.choice([8, 64, 200, 256, 1000, 2048, 4096, 9000, 16384]))
        K = int(rng.choice([8, 64, 72, 256, 640, 1000, 2048, 4096, 8192]))
        kw = dict(stages=int(rng.integers(2, 9)))
        for name, choices in (("cta_group", [0, 0, 1, 2]), ("tile_n", [0, 0, 64, 128, 256]),
                              ("tail_split", [0, 0, -1, 1, 2]), ("epi_groups", [0, 1, 2]),
                              ("k_serpentine", [0, -1, 1]), ("max_ctas", [0, 0, 8, 64]),
                              ("b_kn", [0, 0, 1]), ("out_f32", [0, 0, 1])):
            v = int(rng.choice(choices))
            if v:
                kw[name] = v
        drawn.append((M, N, K, "bf16" if i % 3 == 0 else "f16", kw))
    return named + drawn


def _outcome(fn):
    try:
        return "ok", fn()
    except sg.GemmError as e:
        return "error", e.status


@pytest.mark.parametrize("M,N,K,dtype,kw", _cases())
def test_describe_equals_the_plan_the_device_builds(M, N, K, dtype, kw):
    want = _outcome(lambda: sg.describe(M, N, K, dtype, device=0, **kw))

    def build():
        p = sg.Plan(M, N, K, dtype, **kw)
        try:
            return p.info()
        finally:
            p.close()

    got = _outcome(build)
    assert got == want
