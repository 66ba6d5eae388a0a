"""Failure detection without a GPU fault.

Every wait inside the GEMM kernel has a wall-clock limit.  With the test
hook debug_fault=1 the first CTA's copies of its first K slice are announced
but never issued, so the MMA issuer's wait on that ring slot, the producer's
wait for the slot to be released and the epilogue's wait for the accumulator
all run out (here after 20 ms each).  The kernel must record
GEMM_ERR_TIMEOUT in the plan's status word, finish by itself (draining the
copies it did issue and freeing its tensor memory), and leave the context
usable: a normal GEMM right after must be exact.
"""
from __future__ import annotations

import time

import pytest
import torch

import gemm_inputs
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

TIMEOUT_NS = 20_000_000   # 20 ms per wait


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("cta_group", [1, 2])
def test_wait_timeout_is_reported_and_context_survives(cta_group):
    import software_pipelined_tiled_gemm_gb300 as sg
    M, N, K = 512, 512, 512
    A, B = gemm_inputs.custom(M, N, K, dist="int", lo=-2, hi=2, seed=77)
    a, b = A.cuda(), B.cuda()
    c = torch.zeros(M, N, dtype=torch.float16, device="cuda")
    plan = sg.Plan(M, N, K, "f16", stages=4, cta_group=cta_group, tile_n=256,
                   timeout_ns=TIMEOUT_NS, debug_fault=1)
    t0 = time.perf_counter()
    plan.run(a, b, c)
    status, detail = plan.check()          # synchronises
    elapsed = time.perf_counter() - t0
    plan.close()
    assert status == sg.GEMM_ERR_TIMEOUT, (status, hex(detail))
    assert (detail >> 16) in (1, 2, 3)      # producer, MMA issuer or epilogue
    assert sg.gemm_wait_detail_string(detail) not in ("", "unknown wait")
    assert elapsed < 10.0
    # The context is still usable and the status word was cleared.
    C, info, canary = gu.run_device(A, B, "f16", cta_group=cta_group, tile_n=256)
    want = oracle.round_to(oracle.gemm_nt(A, B, "f16"), "f16")
    assert canary and (gu.bits(C) == want).all()
