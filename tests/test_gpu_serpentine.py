"""GPU parity with serpentine K order: a walker's odd-numbered tiles copy
their K slices in descending order (the MMA loop is unchanged).

The sum over K is then taken in the opposite order on alternate tiles, so
floating-point results may differ from the ascending order by rounding (the
usual 2 ulp + 1e-3 / Frobenius 1e-3 bar applies), while small-integer inputs,
whose partial sums are all exact in fp32, must match the oracle bit for bit.
Small plans force the order on (k_serpentine=1) with few CTAs so that every
CTA walks several tiles; the planner's automatic choice is checked on the
large shapes it is meant for.
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


def _bits_equal(A, B, dtype, C, epilogue=None):
    want = oracle.round_to(oracle.gemm_nt(A, B, dtype, epilogue=epilogue), dtype)
    got = gu.bits(C)
    mism = np.argwhere(want != got)
    assert mism.size == 0, "first mismatch at %s (%d mismatches)" % (tuple(mism[0]), len(mism))


@pytest.mark.parametrize("cta_group,b_kn,stages,tile_n", [(1, 0, 4, 256), (2, 0, 6, 256),
                                                          (1, 1, 4, 256), (2, 1, 6, 256),
                                                          (2, 0, 4, 256), (1, 0, 6, 128)])
def test_serpentine_bit_exact_on_integers(cta_group, b_kn, stages, tile_n):
    # 4 x 4 tiles of 256 rows (pairs) or 8 x 4+ of 128 rows on 3 walkers:
    # every walker alternates direction several times.  K = 1000 leaves a
    # ragged last slice, which a descending walk copies first.
    M, N, K = 1024, 1024, 1000
    A, B = gemm_inputs.custom(M, N, K, dist="int", lo=-2, hi=2, seed=1300 + 10 * cta_group + b_kn)
    Bd = B.t().contiguous() if b_kn else B
    C, info, canary = gu.run_device(A, Bd, "f16", stages=stages, cta_group=cta_group,
                                    b_kn=b_kn, tile_n=tile_n, max_ctas=3 * cta_group,
                                    tail_split=-1, k_serpentine=1)
    assert canary and info["k_serpentine"] == 1 and info["stream_k"] == 0
    _bits_equal(A, B, "f16", C)


@pytest.mark.parametrize("cta_group", [1, 2])
def test_serpentine_with_stream_k_tail_bit_exact(cta_group):
    # whole tiles alternate; the stream-K pieces of the last wave stay ascending
    M = 1280 if cta_group == 2 else 640
    A, B = gemm_inputs.custom(M, 1024, 1024, dist="int", lo=-2, hi=2, seed=1400 + cta_group)
    C, info, canary = gu.run_device(A, B, "f16", stages=6 if cta_group == 2 else 4,
                                    cta_group=cta_group, tile_n=256, max_ctas=3 * cta_group,
                                    tail_split=1, k_serpentine=1)
    assert canary and info["k_serpentine"] == 1 and info["stream_k"] == 1
    _bits_equal(A, B, "f16", C)


@pytest.mark.parametrize("dtype,epilogue", [("f16", None), ("bf16", "gelu"), ("f16", "relu")])
def test_serpentine_within_tolerance(dtype, epilogue):
    M, N, K = 1000, 1300, 1500
    A, B = gemm_inputs.custom(M, N, K, dtype=dtype, dist="normal_scaled", seed=1500)
    C, info, canary = gu.run_device(A, B, dtype, epilogue=epilogue, stages=6, cta_group=2,
                                    max_ctas=8, k_serpentine=1)
    assert canary and info["k_serpentine"] == 1
    st, _, _ = gu.check_full(A, B, dtype, C, epilogue=epilogue)
    assert st["ok"], st


def test_serpentine_planner_choice():
    import software_pipelined_tiled_gemm_gb300 as sg

    def serp(M, N, K, **t):
        p = sg.Plan(M, N, K, "f16", None, 6, "pipelined", 0, **t)
        try:
            return p.info()["k_serpentine"]
        finally:
            p.close()

    # one wave of 76 pair tiles reads (8 + 10) x 256 rows x K: ~73 MB at K = 8192
    assert serp(8192, 8192, 8192) == 1
    assert serp(4096, 4096, 4096) == 0          # ~37 MB: fits in L2 as it is
    assert serp(8192, 8192, 8192, k_serpentine=-1) == 0
    assert serp(512, 512, 512, k_serpentine=1) == 1
    assert serp(128, 8192, 8192, k_serpentine=1) == 0   # one tile row: staggered K instead
    with pytest.raises(sg.GemmError):
        serp(512, 512, 512, k_serpentine=2)


def test_l2_prefetch_planner_choice():
    # the first ring's slices are prefetched into L2 only for operands that do
    # not stay in L2 (above 3/4 of it: GB300 reports 135.5 MB)
    import software_pipelined_tiled_gemm_gb300 as sg

    def pf(M, N, K):
        p = sg.Plan(M, N, K, "f16", None, 6, "pipelined", 0)
        try:
            return p.info()["l2_prefetch_first"]
        finally:
            p.close()

    assert pf(64, 8192, 8192) == 1        # 135 MB of operands
    assert pf(8192, 8192, 8192) == 1
    assert pf(4096, 4096, 4096) == 0      # 64 MB: L2-resident
    assert pf(16896, 512, 640) == 0


def test_serpentine_order_is_deterministic():
    # same plan, same inputs: identical bits on every run
    import software_pipelined_tiled_gemm_gb300 as sg
    A, B = gemm_inputs.custom(1536, 1536, 2048, dist="normal_scaled", seed=1600)
    a, b = A.cuda(), B.cuda()
    p = sg.Plan(1536, 1536, 2048, "f16", None, 6, "pipelined", 0, cta_group=2, max_ctas=6,
                k_serpentine=1)
    outs = []
    for _ in range(3):
        c = torch.empty(1536, 1536, dtype=torch.float16, device="cuda")
        p.run_ptr(a.data_ptr(), b.data_ptr(), c.data_ptr(), torch.cuda.current_stream().cuda_stream)
        outs.append(c)
    torch.cuda.synchronize()
    assert p.check()[0] == 0
    p.close()
    assert all(torch.equal(outs[0].view(torch.int16), o.view(torch.int16)) for o in outs[1:])
