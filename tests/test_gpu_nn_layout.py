"""GPU parity for the NN layout: B stored (K, N), N contiguous, C = epi(A.B).

This is the [M, K] @ [K, N] form of the Mosaic GPU pipelining guide's Hopper
example; the MMA reads B MN-major.  Inputs are the same seeded draws as the
NT tests, B drawn (N, K) and handed to the kernel transposed (K, N); the
oracle gets the (N, K) copy, so it computes the same C = A.B^T definition.
Bit-exact on small integers (order-independent sums), otherwise the usual
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


def _int_inputs(M, N, K, dtype, seed):
    lo, hi = (-2, 2) if dtype == "f16" else (-1, 1)
    return gemm_inputs.custom(M, N, K, dtype=dtype, dist="int", seed=seed, lo=lo, hi=hi)


def _kn(B):
    return B.t().contiguous()


def _assert_bit_exact(A, B, dtype, C):
    ref = oracle.gemm_nt(A, B, dtype)
    want = oracle.round_to(ref, dtype)
    got = gu.bits(C)
    mism = np.argwhere(want != got)
    assert mism.size == 0, "first mismatch at %s: got %r want %r (%d mismatches)" % (
        tuple(mism[0]), oracle.decode(got[tuple(mism[0])], dtype), ref[tuple(mism[0])],
        len(mism))


@pytest.mark.parametrize("tile_n", [64, 128, 256])
def test_nn_single_cta_bit_exact(tile_n):
    # 8 x 4 tiles of 128 rows over 3 CTAs, 9 K slices: the ring wraps and
    # every accumulator changes hands.
    A, B = _int_inputs(1024, 4 * tile_n, 576, "f16", seed=700 + tile_n)
    C, info, canary = gu.run_device(A, _kn(B), "f16", stages=4, cta_group=1, tile_n=tile_n,
                                    max_ctas=3, b_kn=1)
    assert canary and info["b_kn"] == 1 and info["tile_n"] == tile_n
    _assert_bit_exact(A, B, "f16", C)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("stages", [1, 3, 6])
def test_nn_cta_pair_bit_exact(tile_n, stages):
    if tile_n == 256 and stages > 6:
        pytest.skip("ring does not fit")
    A, B = _int_inputs(768, 1024, 512, "f16", seed=710 + stages + tile_n)
    C, info, canary = gu.run_device(A, _kn(B), "f16", stages=stages, cta_group=2,
                                    tile_n=tile_n, max_ctas=4, b_kn=1)
    assert canary and info["cta_group"] == 2 and info["b_kn"] == 1
    _assert_bit_exact(A, B, "f16", C)


def test_nn_bf16_bit_exact():
    A, B = _int_inputs(512, 768, 1024, "bf16", seed=720)
    C, info, canary = gu.run_device(A, _kn(B), "bf16", b_kn=1)
    assert canary
    _assert_bit_exact(A, B, "bf16", C)


@pytest.mark.parametrize("shape", [(1, 8, 8), (129, 130, 72), (255, 257, 136), (300, 203, 8),
                                   (257, 385, 263), (513, 1001, 1000), (64, 66, 4096),
                                   (200, 256, 100), (256, 512, 1000), (130, 192, 72)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_nn_edge_shapes(shape, dtype):
    # B (K x N) is read in 64-column blocks and 8-row groups: N % 64 != 0 or
    # K % 8 != 0 stage it in padded scratch (K % 8 != 0 also pads A); N and K
    # multiples of 64 and 8 but not of the tile read it in place, the
    # partial K slice and column tiles zero-filled by the copy engine.
    M, N, K = shape
    A, B = gemm_inputs.custom(M, N, K, dtype=dtype, seed=M * 7 + N * 3 + K)
    C, info, canary = gu.run_device(A, _kn(B), dtype, b_kn=1)
    st, _, _ = gu.check_full(A, B, dtype, C)
    assert canary and st["ok"], (shape, st, info)


@pytest.mark.parametrize("offsets", [(0, 3, 0), (1, 0, 5), (0, 8, 0)])
def test_nn_unaligned_base_addresses(offsets):
    a_off, b_off, c_off = offsets
    A, B = gemm_inputs.custom(300, 520, 264, seed=731 + sum(offsets))
    C, info, canary = gu.run_device(A, _kn(B), "f16", a_offset=a_off, b_offset=b_off,
                                    c_offset=c_off, b_kn=1)
    st, _, _ = gu.check_full(A, B, "f16", C)
    assert canary and st["ok"], (offsets, st, info)


@pytest.mark.parametrize("cta_group", [1, 2])
def test_nn_gelu_and_relu(cta_group):
    A, B = gemm_inputs.make("gelu_3072x16384x4096_bf16", M=512, N=1024, K=1024)
    for epi in ("gelu", "relu"):
        C, info, canary = gu.run_device(A, _kn(B), "bf16", epilogue=epi, cta_group=cta_group,
                                        b_kn=1)
        st, _, _ = gu.check_full(A, B, "bf16", C, epilogue=epi)
        assert canary and st["ok"], (epi, st, info)


@pytest.mark.parametrize("cta_group", [1, 2])
def test_nn_stream_k_bit_exact(cta_group):
    M = 768 if cta_group == 2 else 384
    A, B = _int_inputs(M, 1024, 1024, "f16", seed=740 + cta_group)
    C, info, canary = gu.run_device(A, _kn(B), "f16", cta_group=cta_group, tile_n=256,
                                    max_ctas=5 * cta_group, tail_split=1, b_kn=1)
    assert canary and info["stream_k"] == 1
    _assert_bit_exact(A, B, "f16", C)


def test_nn_few_tiles_split_k_and_skinny():
    # Few tiles: the planner cuts K in two (stream-K over every tile).
    A, B = gemm_inputs.custom(64, 2048, 4096, seed=750)
    C, info, canary = gu.run_device(A, _kn(B), "f16", b_kn=1)
    st, _, _ = gu.check_full(A, B, "f16", C)
    assert canary and st["ok"], (st, info)


def test_nn_narrow_tail_rejected():
    import software_pipelined_tiled_gemm_gb300 as sg
    with pytest.raises(sg.GemmError):
        sg.Plan(512, 512, 512, "f16", tail_split=2, b_kn=1)


def test_nn_fp32_output_exact_on_integers():
    import software_pipelined_tiled_gemm_gb300 as sg
    A, B = _int_inputs(300, 520, 264, "f16", seed=760)
    C = sg.matmul_nn(A.cuda(), _kn(B).cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle.gemm_nt(A, B, "f16")
    assert np.array_equal(C.cpu().double().numpy(), ref)


def test_matmul_nn_matches_matmul_nt_bits():
    import software_pipelined_tiled_gemm_gb300 as sg
    A, B = gemm_inputs.custom(1000, 1500, 700, seed=770)
    a, b = A.cuda(), B.cuda()
    c_nt = sg.matmul_nt(a, b)
    c_nn = sg.matmul_nn(a, b.t().contiguous())
    torch.cuda.synchronize()
    st, _, _ = gu.check_full(A, B, "f16", c_nn.cpu())
    assert st["ok"], st
    # Same tiles, same K order, same fp32 accumulation: identical bits.
    assert torch.equal(c_nt.view(torch.int16), c_nn.view(torch.int16))


def test_nn_full_size_8192_sampled():
    w = gemm_inputs.WORKLOADS["gemm_8192_f16"]
    A, B = gemm_inputs.make(w)
    C, info, canary = gu.run_device(A, _kn(B), "f16", stages=6, b_kn=1)
    assert canary and info["b_kn"] == 1
    assert torch.isfinite(C.float()).all()
    r, c = gu.sample_positions(w.M, w.N, 2000, seed=w.seed, tile_n=info["tile_n"])
    st = gu.check_sampled(A, B, "f16", C, r, c)
    assert st["ok"], (st, info)
