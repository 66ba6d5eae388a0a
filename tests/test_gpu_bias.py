"""GPU parity for the per-column bias: C = epi(A . B^T + bias).

The pages define no bias; the reading (a Linear layer's, one value per
output column, added to the fp32 accumulator before the epilogue) is the
oracle's.  Bit-exact on small-integer inputs with an integer bias (every
partial sum and the bias are exact in fp32); otherwise the usual 2 ulp + 1e-3
/ Frobenius 1e-3 bar.
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


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import software_pipelined_tiled_gemm_gb300 as sg
    sg.load_library()


def _assert_bit_exact(A, B, dtype, C, bias, epilogue=None):
    ref = oracle.gemm_nt(A, B, dtype, epilogue=epilogue, bias=bias)
    want = oracle.round_to(ref, dtype)
    got = gu.bits(C)
    mism = np.argwhere(want != got)
    assert mism.size == 0, "first mismatch at %s (%d mismatches)" % (tuple(mism[0]), len(mism))


@pytest.mark.parametrize("cta_group,b_kn", [(1, 0), (2, 0), (1, 1), (2, 1)])
def test_bias_bit_exact_on_integers(cta_group, b_kn):
    A, B = gemm_inputs.custom(512, 1024, 576, dist="int", lo=-2, hi=2, seed=900 + cta_group)
    bias = gemm_inputs.bias(1024, "f16", seed=9, dist="int", lo=-40, hi=40)
    Bd = B.t().contiguous() if b_kn else B
    C, info, canary = gu.run_device(A, Bd, "f16", stages=6, cta_group=cta_group, b_kn=b_kn,
                                    max_ctas=6 * cta_group, bias=bias)
    assert canary and info["b_kn"] == b_kn
    _assert_bit_exact(A, B, "f16", C, bias)
    # ReLU sees s + b: the integer bias moves sums across zero both ways
    C, _, _ = gu.run_device(A, Bd, "f16", epilogue="relu", stages=6, cta_group=cta_group,
                            b_kn=b_kn, bias=bias)
    _assert_bit_exact(A, B, "f16", C, bias, epilogue="relu")


@pytest.mark.parametrize("cta_group", [1, 2])
def test_bias_with_stream_k_bit_exact(cta_group):
    # the owner adds the partner's partial, then the bias: a fixed order
    M = 768 if cta_group == 2 else 384
    A, B = gemm_inputs.custom(M, 1024, 1024, dist="int", lo=-2, hi=2, seed=910 + cta_group)
    bias = gemm_inputs.bias(1024, "f16", seed=10, dist="int", lo=-64, hi=64)
    C, info, canary = gu.run_device(A, B, "f16", stages=6 if cta_group == 2 else 4,
                                    cta_group=cta_group, tile_n=256, max_ctas=5 * cta_group,
                                    tail_split=1, bias=bias)
    assert canary and info["stream_k"] == 1
    _assert_bit_exact(A, B, "f16", C, bias)


@pytest.mark.parametrize("epilogue", [None, "gelu", "relu"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_bias_with_each_epilogue(epilogue, dtype):
    A, B = gemm_inputs.make("gelu_3072x16384x4096_bf16", M=384, N=1536, K=1024)
    if dtype == "f16":
        A, B = A.float().half(), B.float().half()
    bias = gemm_inputs.bias(1536, dtype, seed=11)
    C, info, canary = gu.run_device(A, B, dtype, epilogue=epilogue, stages=6, bias=bias)
    st, _, _ = gu.check_full(A, B, dtype, C, epilogue=epilogue, bias=bias)
    assert canary and st["ok"], (epilogue, dtype, st, info)


@pytest.mark.parametrize("shape,offsets", [((300, 1001, 264), (0, 0, 0)),
                                           ((257, 385, 263), (1, 3, 5)),
                                           ((64, 2048, 4096), (0, 0, 0))])
def test_bias_ragged_unaligned_and_skinny(shape, offsets):
    # N not a multiple of the tile (bias columns >= N are never read), C
    # unaligned (row-wise stores), and a 64-row problem (K halves, B streamed)
    M, N, K = shape
    A, B = gemm_inputs.custom(M, N, K, seed=M + N + K)
    bias = gemm_inputs.bias(N, "f16", seed=12)
    a_off, b_off, c_off = offsets
    C, info, canary = gu.run_device(A, B, "f16", epilogue="gelu", stages=6, a_offset=a_off,
                                    b_offset=b_off, c_offset=c_off, bias=bias)
    st, _, _ = gu.check_full(A, B, "f16", C, epilogue="gelu", bias=bias)
    assert canary and st["ok"], (shape, st, info)


def test_bias_fp32_output_exact_on_integers():
    import software_pipelined_tiled_gemm_gb300 as sg
    A, B = gemm_inputs.custom(300, 520, 264, dist="int", lo=-2, hi=2, seed=920)
    bias = gemm_inputs.bias(520, "bf16", seed=13, dist="int", lo=-100, hi=100)
    A, B = A.float().to(torch.bfloat16), B.float().to(torch.bfloat16)
    C = sg.matmul_nt(A.cuda(), B.cuda(), out_dtype=torch.float32, bias=bias.cuda())
    torch.cuda.synchronize()
    ref = oracle.gemm_nt(A, B, "bf16", bias=bias)
    assert np.array_equal(C.cpu().double().numpy(), ref)


@pytest.mark.parametrize("epilogue", [None, "gelu", "relu"])
@pytest.mark.parametrize("out_f32", [0, 1])
def test_k_zero_with_bias_broadcasts_epi_of_bias(epilogue, out_f32):
    M, N = 70, 130
    A = torch.zeros(M, 0, dtype=torch.float16)
    B = torch.zeros(N, 0, dtype=torch.float16)
    bias = gemm_inputs.bias(N, "f16", seed=14, lo=-3.0, hi=3.0)
    import software_pipelined_tiled_gemm_gb300 as sg
    plan = sg.Plan(M, N, 0, "f16", epilogue, 4, "pipelined", 0, out_f32=out_f32)
    c = torch.full((M, N), float("nan"), dtype=torch.float32 if out_f32 else torch.float16,
                   device="cuda")
    dummy = torch.zeros(8, dtype=torch.float16, device="cuda")
    plan.run_ptr(dummy.data_ptr(), dummy.data_ptr(), c.data_ptr(),
                 torch.cuda.current_stream().cuda_stream, bias.cuda().data_ptr())
    torch.cuda.synchronize()
    assert plan.check()[0] == 0
    plan.close()
    ref = oracle.gemm_nt(A, B, "f16", epilogue=epilogue, bias=bias)   # = epi(bias) per row
    if out_f32:
        st = tolerance.compare(c.cpu().double().numpy(), ref, "f32")
    else:
        st = tolerance.compare(oracle.decode(gu.bits(c.cpu()), "f16"), ref, "f16")
    assert st["ok"], st


def test_matmul_nn_with_bias_matches_matmul_nt_bits():
    import software_pipelined_tiled_gemm_gb300 as sg
    A, B = gemm_inputs.custom(1000, 1500, 700, seed=930)
    bias = gemm_inputs.bias(1500, "f16", seed=15).cuda()
    a, b = A.cuda(), B.cuda()
    c_nt = sg.matmul_nt(a, b, epilogue="relu", bias=bias)
    c_nn = sg.matmul_nn(a, b.t().contiguous(), epilogue="relu", bias=bias)
    torch.cuda.synchronize()
    assert torch.equal(c_nt.view(torch.int16), c_nn.view(torch.int16))
    st, _, _ = gu.check_full(A, B, "f16", c_nt.cpu(), epilogue="relu", bias=bias.cpu())
    assert st["ok"], st


def test_bias_argument_errors():
    import software_pipelined_tiled_gemm_gb300 as sg
    M, N, K = 128, 256, 128
    a = torch.zeros(M, K, dtype=torch.float16, device="cuda")
    b = torch.zeros(N, K, dtype=torch.float16, device="cuda")
    buf = torch.zeros(M * N + 8, dtype=torch.float16, device="cuda")
    c = buf[:M * N]
    plan = sg.Plan(M, N, K, "f16", None, 4, "pipelined", 0)
    s = torch.cuda.current_stream().cuda_stream
    with pytest.raises(sg.GemmError) as ei:           # odd address
        plan.run_ptr(a.data_ptr(), b.data_ptr(), c.data_ptr(), s, buf[M * N:].data_ptr() + 1)
    assert ei.value.status == sg.GEMM_ERR_INVALID_ARG
    with pytest.raises(sg.GemmError) as ei:           # bias inside C
        plan.run_ptr(a.data_ptr(), b.data_ptr(), c.data_ptr(), s, c.data_ptr())
    assert ei.value.status == sg.GEMM_ERR_INVALID_ARG
    plan.close()
    with pytest.raises(ValueError):
        sg.matmul_nt(a, b, bias=torch.zeros(N + 1, dtype=torch.float16, device="cuda"))


def test_gelu_layer_with_bias_full_size_sampled():
    w = gemm_inputs.WORKLOADS["gelu_3072x16384x4096_bf16"]
    A, B = gemm_inputs.make(w)
    bias = gemm_inputs.bias(w.N, "bf16", seed=w.seed)
    C, info, canary = gu.run_device(A, B, "bf16", epilogue="gelu", stages=6, bias=bias)
    assert canary and torch.isfinite(C.float()).all()
    r, c = gu.sample_positions(w.M, w.N, 2000, seed=w.seed, tile_n=info["tile_n"])
    st = gu.check_sampled(A, B, "bf16", C, r, c, epilogue="gelu", bias=bias)
    assert st["ok"], (st, info)
