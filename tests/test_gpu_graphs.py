"""gemm_run inside CUDA graphs, and GEMMs that consume each other's output.

A plan's launch is captured into a CUDA graph (torch.cuda.graph, global
capture mode) and replayed on new contents of the same buffers: each replay
must compute the GEMM of the buffers' current contents (the tensor maps
captured in the launch hold addresses, not data; the stream-K flags reset
themselves between launches).  Plans whose operands need padded copies
allocate that scratch on their first run, so they run once before capture.

The chained tests feed one GEMM's C into the next GEMM as an operand on the
same stream, eagerly and in a graph: the second kernel may be launched early
(programmatic dependent launch), so this checks that it still reads the
first one's finished output."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_inputs
import oracle
import software_pipelined_tiled_gemm_gb300 as sg
from tests import gpu_util as gu
from tests import tolerance

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
_TD = {"f16": torch.float16, "bf16": torch.bfloat16}

# (M, N, K, dtype, integer span, feature the plan must use); the spans keep
# every sum exact in the output type (|C| < 2048 in fp16, < 256 in bf16)
CASES = [
    (4096, 4096, 4096, "f16", 2, "stream_k"),       # CTA pairs, stream-K last wave
    (128, 8192, 2048, "f16", 2, "sk_cluster"),      # few tiles: K halves in 2-CTA clusters
    (1024, 2048, 4096, "f16", 2, None),             # 256 x 128 pair tiles
    (300, 500, 1001, "f16", 2, "pads_operands"),    # K pitch not 16-byte aligned: padded copies
    (384, 640, 2048, "bf16", 1, None),
]


def _ints(M, N, K, dtype, seed, span=2):
    return gemm_inputs.custom(M, N, K, dtype=dtype, dist="int", seed=seed, lo=-span, hi=span)


def _assert_bit_exact(A, B, dtype, C):
    ref = oracle.gemm_nt(A, B, dtype)
    assert np.all(np.abs(ref) < (2048 if dtype == "f16" else 256))
    want = oracle.round_to(ref, dtype)
    got = gu.bits(C)
    mism = np.argwhere(want != got)
    assert mism.size == 0, "first mismatch at %s" % (mism[0],)


@pytest.mark.parametrize("M,N,K,dtype,span,feature", CASES)
def test_captured_gemm_replays_on_new_inputs(M, N, K, dtype, span, feature):
    A0, B0 = _ints(M, N, K, dtype, seed=1, span=span)
    A, B = A0.to(DEV), B0.to(DEV)
    C = torch.empty(M, N, dtype=_TD[dtype], device=DEV)
    plan = sg.Plan(M, N, K, dtype, stages=6)
    try:
        plan.run(A, B, C)                        # first run: allocates any scratch
        torch.cuda.synchronize(DEV)
        info = plan.info()
        if feature:
            assert info[feature], info
        _assert_bit_exact(A0, B0, dtype, C)

        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.run(A, B, C)
        for seed in (2, 3, 4):
            An, Bn = _ints(M, N, K, dtype, seed=seed, span=span)
            A.copy_(An)
            B.copy_(Bn)
            C.view(torch.int16).fill_(-1)        # NaN pattern: every element must be rewritten
            g.replay()
            torch.cuda.synchronize(DEV)
            _assert_bit_exact(An, Bn, dtype, C)
        ds, detail = plan.check()
        assert ds == 0, (ds, hex(detail))
    finally:
        plan.close()


def _chain_inputs(dtype):
    # C1 = A . B^T is exact (|C1| <= 64 * 4 = 256); E = C1 . D^T is compared
    # with the oracle of (C1, D) within the tolerance.
    M, N1, K1, N2 = 512, 640, 64, 384
    A, B = _ints(M, N1, K1, dtype, seed=11)
    g = torch.Generator().manual_seed(12)
    D = (torch.rand(N2, N1, generator=g) * 2 - 1).to(_TD[dtype])
    return A, B, D


def _check_chain(A, B, D, dtype, C1, E):
    _assert_bit_exact(A, B, dtype, C1)
    ref = oracle.gemm_nt(C1.cpu(), D, dtype)
    got = oracle.decode(gu.bits(E), dtype)
    st = tolerance.compare(got, ref, dtype)
    assert st["ok"], st


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("captured", [False, True])
def test_second_gemm_reads_the_first_ones_output(dtype, captured):
    A0, B0, D0 = _chain_inputs(dtype)
    A, B, D = A0.to(DEV), B0.to(DEV), D0.to(DEV)
    M, N1 = A.shape[0], B.shape[0]
    N2 = D.shape[0]
    C1 = torch.empty(M, N1, dtype=_TD[dtype], device=DEV)
    E = torch.empty(M, N2, dtype=_TD[dtype], device=DEV)
    first = sg.Plan(M, N1, A.shape[1], dtype, stages=6)
    second = sg.Plan(M, N2, N1, dtype, stages=6)
    try:
        if captured:
            first.run(A, B, C1)
            second.run(C1, D, E)
            torch.cuda.synchronize(DEV)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                first.run(A, B, C1)
                second.run(C1, D, E)
            for _ in range(3):
                C1.view(torch.int16).fill_(-1)
                E.view(torch.int16).fill_(-1)
                g.replay()
                torch.cuda.synchronize(DEV)
                _check_chain(A0, B0, D0, dtype, C1, E)
        else:
            for _ in range(3):
                C1.view(torch.int16).fill_(-1)
                E.view(torch.int16).fill_(-1)
                first.run(A, B, C1)
                second.run(C1, D, E)
                torch.cuda.synchronize(DEV)
                _check_chain(A0, B0, D0, dtype, C1, E)
        for p in (first, second):
            ds, detail = p.check()
            assert ds == 0, (ds, hex(detail))
    finally:
        first.close()
        second.close()
