"""gemm_run_noalloc: the GEMM for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc or anything that
allocates -- code running under an allocator it does not control, or a
runtime that forbids allocations once it has started.  gemm_run needs a plan,
and a plan allocates (its status word, and scratch for padded operand copies
when a row pitch is not 16-byte aligned).  gemm_run_noalloc takes no plan and
uses a static device array for that scratch instead.

These tests call it through the C ABI, two calls in a row on different data
(the second call reuses the static scratch the first one left behind), and
check every output element against the fp64 oracle -- bit for bit on
small-integer inputs, whose products and sums are exact in any order -- and
against gemm_run's output on the same inputs.  The shapes reach each path
the entry point can take: both operands padded (K % 8 != 0), only A padded
(A's base one element off a 16-byte boundary), no padding, row-wise stores
of C (N % 8 != 0), and the tile widths 256, 128 and 64 (its rule: the widest
tile whose tiles keep every SM busy, else the narrowest).  The file is named
so pytest collects it last.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_inputs
import oracle
from tests import gpu_util as gu
from tests import tolerance

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 32 * 1024 * 1024   # GEMM_NOALLOC_SCRATCH_BYTES in include/gemm.h
_TD = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _place(x, offset):
    """x copied to the device `offset` elements into a larger allocation."""
    buf = torch.zeros(x.numel() + offset + 64, dtype=x.dtype, device="cuda")
    view = buf[offset:offset + x.numel()]
    view.copy_(x.reshape(-1).cuda())
    return buf, view


def _with_plan(sg, a, b, M, N, K, dtype, epi):
    c = torch.full((M, N), float("nan"), dtype=_TD[dtype], device="cuda")
    plan = sg.Plan(M, N, K, dtype, epi, stages=4)
    plan.run_ptr(a.data_ptr(), b.data_ptr(), c.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert plan.check()[0] == 0
    plan.close()
    return c.cpu()


def _no_alloc(sg, a, b, M, N, K, dtype, epi):
    c = torch.full((M, N), float("nan"), dtype=_TD[dtype], device="cuda")
    stream = torch.cuda.current_stream()
    st = sg.gemm_run_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                             sg.GEMM_BF16 if dtype == "bf16" else sg.GEMM_F16,
                             sg.GEMM_EPI_GELU_TANH if epi else sg.GEMM_EPI_NONE, 4,
                             stream.cuda_stream)
    assert st == sg.GEMM_OK, sg.gemm_status_string(st)
    torch.cuda.synchronize()
    return c.cpu()


@pytest.mark.parametrize("dtype,epi,shape", [
    ("f16", None, (300, 520, 1001)),        # K % 8 != 0: both operands staged in the scratch
    ("bf16", "gelu", (257, 384, 771)),
    ("f16", None, (256, 512, 512)),         # aligned: no scratch needed
])
def test_no_alloc_matches_oracle_and_gemm_run_on_two_calls(dtype, epi, shape):
    import software_pipelined_tiled_gemm_gb300 as sg
    M, N, K = shape
    for call, seed in enumerate((41, 42)):           # two calls in a row, different data
        A, B = gemm_inputs.custom(M, N, K, dtype=dtype, dist="normal_scaled", seed=seed + M)
        a, b = A.cuda(), B.cuda()
        got = _no_alloc(sg, a, b, M, N, K, dtype, epi)
        st, _, _ = gu.check_full(A, B, dtype, got, epilogue=epi)       # the oracle decides
        assert st["ok"], (call, st)
        want = _with_plan(sg, a, b, M, N, K, dtype, epi)
        st = tolerance.compare(oracle.decode(gu.bits(got), dtype),
                               oracle.decode(gu.bits(want), dtype), dtype)
        assert st["ok"], (call, st)


@pytest.mark.parametrize("dtype,shape,a_offset,path", [
    ("f16", (2048, 4096, 256), 0, "tile 256 (512 TMEM columns), no padding"),
    ("f16", (2048, 1536, 256), 0, "tile 128"),
    ("f16", (300, 520, 1000), 1, "A alone padded (base off 16 B), tile 64"),
    ("bf16", (256, 250, 256), 0, "row-wise stores (N % 8 != 0)"),
    ("bf16", (257, 384, 251), 0, "both operands padded (K % 8 != 0)"),
])
def test_no_alloc_bit_exact_on_integers(dtype, shape, a_offset, path):
    # Small-integer entries (fp16 {-2..2}, bf16 {-1, 0, 1}) keep every
    # partial sum an integer far below 2^24, exact in the fp32 accumulator in
    # any order; the one rounding at the end then gives the oracle's value,
    # rounded once, bit for bit.
    import software_pipelined_tiled_gemm_gb300 as sg
    M, N, K = shape
    lim = 2 if dtype == "f16" else 1
    for call, seed in enumerate((51, 52)):
        A, B = gemm_inputs.custom(M, N, K, dtype=dtype, dist="int", lo=-lim, hi=lim,
                                  seed=seed + N)
        _, a = _place(A, a_offset)
        _, b = _place(B, 0)
        want = oracle.round_to(oracle.gemm_nt(A, B, dtype), dtype)
        got = _no_alloc(sg, a, b, M, N, K, dtype, None)
        assert np.array_equal(gu.bits(got), want), (path, call)
        assert np.array_equal(gu.bits(_with_plan(sg, a, b, M, N, K, dtype, None)), want), path


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
