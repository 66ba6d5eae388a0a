"""gemm_run_noalloc: the GEMM for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc or anything that
allocates -- code running under an allocator it does not control, or a
runtime that forbids allocations once it has started.  gemm_run needs a plan,
and a plan allocates (its status word, and scratch for padded operand copies
when a row pitch is not 16-byte aligned).  gemm_run_noalloc takes no plan and
uses a static device array for that scratch instead.

These tests call it through the C ABI and compare its output with
gemm_run's, within the tolerance the parity tests use, on two calls in a row
(the second call reuses the static scratch the first one left behind).  The
file is named so pytest collects it last.
"""
from __future__ import annotations

import pytest
import torch

import gemm_inputs
import oracle
from tests import gpu_util as gu
from tests import tolerance

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 32 * 1024 * 1024   # GEMM_NOALLOC_SCRATCH_BYTES in include/gemm.h


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _with_plan(sg, a, b, M, N, K, dtype, epi):
    c = torch.full((M, N), float("nan"), dtype=a.dtype, device=a.device)
    plan = sg.Plan(M, N, K, dtype, epi, stages=4)
    plan.run(a, b, c)
    torch.cuda.synchronize()
    assert plan.check()[0] == 0
    plan.close()
    return c.cpu()


def _no_alloc(sg, a, b, M, N, K, dt_code, epi_code):
    c = torch.full((M, N), float("nan"), dtype=a.dtype, device=a.device)
    stream = torch.cuda.current_stream()
    st = sg.gemm_run_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, dt_code,
                             epi_code, 4, stream.cuda_stream)
    assert st == sg.GEMM_OK, sg.gemm_status_string(st)
    torch.cuda.synchronize()
    return c.cpu()


@pytest.mark.parametrize("dtype,epi,shape", [
    ("f16", None, (300, 520, 1001)),        # K % 8 != 0: both operands staged in the scratch
    ("bf16", "gelu", (257, 384, 771)),
    ("f16", None, (256, 512, 512)),         # aligned: no scratch needed
])
def test_no_alloc_matches_gemm_run_on_two_calls(dtype, epi, shape):
    import software_pipelined_tiled_gemm_gb300 as sg
    M, N, K = shape
    dt_code = sg.GEMM_BF16 if dtype == "bf16" else sg.GEMM_F16
    epi_code = sg.GEMM_EPI_GELU_TANH if epi else sg.GEMM_EPI_NONE
    for call, seed in enumerate((41, 42)):           # two calls in a row, different data
        A, B = gemm_inputs.custom(M, N, K, dtype=dtype, dist="normal_scaled", seed=seed + M)
        a, b = A.cuda(), B.cuda()
        want = _with_plan(sg, a, b, M, N, K, dtype, epi)
        got = _no_alloc(sg, a, b, M, N, K, dt_code, epi_code)
        st = tolerance.compare(oracle.decode(gu.bits(got), dtype),
                               oracle.decode(gu.bits(want), dtype), dtype)
        assert st["ok"], (call, st)


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    import software_pipelined_tiled_gemm_gb300 as sg
    # K % 8 != 0 forces padded copies of (M + N) rows of round_up(K, 8) elements.
    M, N, K = 4096, 4096, 4095
    assert (M + N) * 4096 * 2 > SCRATCH_LIMIT
    a = torch.empty(M * K, dtype=torch.float16, device="cuda")
    b = torch.empty(N * K, dtype=torch.float16, device="cuda")
    c = torch.empty(M * N, dtype=torch.float16, device="cuda")
    st = sg.gemm_run_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, sg.GEMM_F16,
                             sg.GEMM_EPI_NONE, 4, 0)
    assert st == sg.GEMM_ERR_INVALID_ARG
