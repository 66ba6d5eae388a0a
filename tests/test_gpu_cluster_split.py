"""GPU parity for tiles split in two K halves inside a 2-CTA cluster.

With few tiles (at most half a wave) on single CTAs, the planner splits every
tile into two K halves: walker 2t owns K slices [0, k/2) and walker 2t+1
contributes [k/2, k).  The two walkers are launched as one cluster and the
contributor bulk-copies its fp32 partial from its own shared memory into the
owner's (the owner signals first that its ring is free); the owner adds it,
its own slices first, in a fixed order.  Small-integer inputs, whose partial sums are
exact in fp32, must match the oracle bit for bit; other inputs meet the usual
2 ulp + 1e-3 / Frobenius 1e-3 bar.
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


@pytest.mark.parametrize("M,N,K,tile_n,b_kn", [
    (128, 1024, 2048, 128, 0),    # every epilogue warp exchanges its rows
    (64, 1024, 2048, 128, 0),     # rows 64..127 are never stored: two warps exchange
    (100, 1000, 1100, 128, 0),    # ragged M, N, K (padded copies): 18 slices in 9 slots
    (128, 512, 2048, 256, 0),     # 256-wide tiles: 32 KiB partial per warp
    (128, 1024, 2048, 128, 1),    # K x N B
])
def test_cluster_split_bit_exact_on_integers(M, N, K, tile_n, b_kn):
    A, B = gemm_inputs.custom(M, N, K, dist="int", lo=-2, hi=2, seed=1700 + M + N + K + b_kn)
    Bd = B.t().contiguous() if b_kn else B
    stages = 6 if tile_n == 128 else 4
    C, info, canary = gu.run_device(A, Bd, "f16", stages=stages, cta_group=1, tile_n=tile_n,
                                    b_kn=b_kn)
    assert canary and info["sk_cluster"] == 1 and info["stream_k"] == 1, info
    assert info["grid"] == 2 * info["num_tiles"], info
    _bits_equal(A, B, "f16", C)


def test_cluster_split_gelu_bias_bf16_within_tolerance():
    M, N, K = 64, 2048, 4096
    A, B = gemm_inputs.custom(M, N, K, dtype="bf16", dist="normal_scaled", seed=1750)
    bias = gemm_inputs.bias(N, "bf16", seed=1751)
    C, info, canary = gu.run_device(A, B, "bf16", epilogue="gelu", stages=6, cta_group=1,
                                    tile_n=128, bias=bias)
    assert canary and info["sk_cluster"] == 1
    st, _, _ = gu.check_full(A, B, "bf16", C, epilogue="gelu", bias=bias)
    assert st["ok"], st


def test_cluster_split_integer_bias_and_relu_bit_exact():
    M, N, K = 128, 768, 1536
    A, B = gemm_inputs.custom(M, N, K, dist="int", lo=-2, hi=2, seed=1760)
    bias = gemm_inputs.bias(N, "f16", seed=1761, dist="int", lo=-30, hi=30)
    C, info, canary = gu.run_device(A, B, "f16", epilogue="relu", stages=6, cta_group=1,
                                    tile_n=128, bias=bias)
    assert canary and info["sk_cluster"] == 1
    _bits_equal(A, B, "f16", C, epilogue="relu", bias=bias)


def test_cluster_split_repeatable_bits():
    import software_pipelined_tiled_gemm_gb300 as sg
    M, N, K = 64, 8192, 8192       # the skinny workload's shape
    A, B = gemm_inputs.custom(M, N, K, dist="normal_scaled", seed=1770)
    a, b = A.cuda(), B.cuda()
    p = sg.Plan(M, N, K, "f16", None, 6, "pipelined", 0)
    assert p.info()["sk_cluster"] == 1
    outs = []
    for _ in range(3):
        c = torch.empty(M, N, dtype=torch.float16, device="cuda")
        p.run_ptr(a.data_ptr(), b.data_ptr(), c.data_ptr(), torch.cuda.current_stream().cuda_stream)
        outs.append(c)
    torch.cuda.synchronize()
    assert p.check()[0] == 0
    p.close()
    assert all(torch.equal(outs[0].view(torch.int16), o.view(torch.int16)) for o in outs[1:])
    st, _, _ = gu.check_full(A, B, "f16", outs[0].cpu())
    assert st["ok"], st
