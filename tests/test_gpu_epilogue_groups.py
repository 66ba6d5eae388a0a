"""GPU parity with four and with eight epilogue warps.

With one column group (epi_groups=1) warps 2-5 each read one TMEM lane
quarter across the whole tile; with two (epi_groups=2) warps 2-9 split each
quarter's columns in two halves, and stream-K partials, flags and the cluster
split's exchange are per warp over its half.  Both are forced here on the
paths whose partitioning changes: whole tiles, stream-K on single CTAs and
on pairs, narrow tail tiles (whose 64-wide units leave the second group
idle), 64-wide tiles, the cluster split, and the bias.  Small-integer inputs
must match the oracle bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_inputs
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import software_pipelined_tiled_gemm_gb300 as sg
    sg.load_library()


def _bits_equal(A, B, dtype, C, epilogue=None, bias=None):
    want = oracle.round_to(oracle.gemm_nt(A, B, dtype, epilogue=epilogue, bias=bias), dtype)
    got = gu.bits(C)
    mism = np.argwhere(want != got)
    assert mism.size == 0, "first mismatch at %s (%d mismatches)" % (tuple(mism[0]), len(mism))


CASES = {
    # name: (M, N, K, tuning, stages)
    "pairs_whole": (768, 1024, 512, dict(cta_group=2, tile_n=256, tail_split=-1), 6),
    "pairs_stream_k": (768, 1024, 1024, dict(cta_group=2, tile_n=256, max_ctas=10, tail_split=1), 6),
    "single_stream_k": (384, 1024, 1024, dict(cta_group=1, tile_n=256, max_ctas=5, tail_split=1), 4),
    "narrow_tail": (640, 896, 512, dict(cta_group=1, tile_n=128, max_ctas=6, tail_split=2), 6),
    "tile_64": (300, 520, 264, dict(cta_group=1, tile_n=64), 6),
    "cluster_split": (128, 1024, 2048, dict(cta_group=1, tile_n=128), 6),
    "cluster_split_256": (128, 512, 2048, dict(cta_group=1, tile_n=256), 4),
    "nn_pairs": (512, 768, 640, dict(cta_group=2, tile_n=256, b_kn=1), 6),
}


@pytest.mark.parametrize("groups", [1, 2])
@pytest.mark.parametrize("name", sorted(CASES))
def test_epilogue_groups_bit_exact_on_integers(name, groups):
    M, N, K, tuning, stages = CASES[name]
    A, B = gemm_inputs.custom(M, N, K, dist="int", lo=-2, hi=2, seed=1800 + len(name))
    Bd = B.t().contiguous() if tuning.get("b_kn") else B
    C, info, canary = gu.run_device(A, Bd, "f16", stages=stages, epi_groups=groups, **tuning)
    assert canary and info["epi_groups"] == groups, info
    if name.startswith("cluster_split"):
        assert info["sk_cluster"] == 1, info
    if "stream_k" in name:
        assert info["stream_k"] == 1, info
    if name == "narrow_tail":
        assert info["tail_splits"] == 2, info
    _bits_equal(A, B, "f16", C)


@pytest.mark.parametrize("groups", [1, 2])
def test_epilogue_groups_bias_gelu_bf16(groups):
    # 3 x 6 pair tiles on 5 clusters: 3 whole tiles each, the rest stream-K
    M, N, K = 768, 1536, 1024
    A, B = gemm_inputs.custom(M, N, K, dtype="bf16", dist="normal_scaled", seed=1850)
    bias = gemm_inputs.bias(N, "bf16", seed=1851)
    C, info, canary = gu.run_device(A, B, "bf16", epilogue="gelu", stages=6, cta_group=2,
                                    tile_n=256, max_ctas=10, tail_split=1, bias=bias,
                                    epi_groups=groups)
    assert canary and info["epi_groups"] == groups and info["stream_k"] == 1
    st, _, _ = gu.check_full(A, B, "bf16", C, epilogue="gelu", bias=bias)
    assert st["ok"], st


def test_epilogue_groups_planner_choice():
    import software_pipelined_tiled_gemm_gb300 as sg

    def groups(M, N, K):
        p = sg.Plan(M, N, K, "f16", None, 6, "pipelined", 0)
        try:
            return p.info()["epi_groups"]
        finally:
            p.close()

    assert groups(8192, 8192, 8192) == 1       # the epilogue hides behind 128 K slices
    assert groups(4096, 4096, 4096) == 1
    assert groups(8192, 8192, 512) == 2        # 8 K slices: the epilogue is exposed
    assert groups(16896, 512, 640) == 2
    assert groups(64, 8192, 8192) == 2         # a single row of tiles
