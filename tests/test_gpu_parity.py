"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar: bit-exact on small-integer inputs (every partial sum is exact in fp32,
so the result is independent of summation order); otherwise every element
within 2 ulps of the output type plus 1e-3 and a relative Frobenius error of
at most 1e-3.  Small shapes are compared in full; the full-size workloads at
sampled positions (random plus every tile boundary and the ragged edges),
with every other element checked to be written and finite.
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


def _int_inputs(M, N, K, dtype, seed):
    lo, hi = (-2, 2) if dtype == "f16" else (-1, 1)
    return gemm_inputs.custom(M, N, K, dtype=dtype, dist="int", seed=seed, lo=lo, hi=hi)


def _assert_bit_exact(A, B, dtype, C):
    ref = oracle.gemm_nt(A, B, dtype)
    assert np.all(np.abs(ref) < (2048 if dtype == "f16" else 256))
    want = oracle.round_to(ref, dtype)
    got = gu.bits(C)
    mism = np.argwhere(want != got)
    assert mism.size == 0, "first mismatch at %s: got %r want %r" % (
        tuple(mism[0]), oracle.decode(got[tuple(mism[0])], dtype), ref[tuple(mism[0])])


# ---------------------------------------------------------- exactness --

def test_small_integer_config_bit_exact():
    A, B = gemm_inputs.make("gemm_256_f16_int")
    C, info, canary = gu.run_device(A, B, "f16")
    assert canary
    _assert_bit_exact(A, B, "f16", C)


@pytest.mark.parametrize("stages", [1, 2, 3, 4, 5, 6, 7, 8])
def test_every_ring_depth_bit_exact_with_persistent_tiles(stages):
    # 9 K slices so the ring wraps; 16 tiles over 2 CTAs so each CTA walks 8
    # tiles and both accumulators change hands several times.
    A, B = _int_inputs(512, 1024, 576, "f16", seed=100 + stages)
    C, info, canary = gu.run_device(A, B, "f16", stages=stages, max_ctas=2, cta_group=1)
    assert canary and info["grid"] == 2 and info["stages"] == stages
    _assert_bit_exact(A, B, "f16", C)


@pytest.mark.parametrize("stages", [1, 2, 3, 4, 5, 6, 7, 8])
def test_cta_pair_every_ring_depth_bit_exact(stages):
    # CTA pairs (256-row tiles): 8 K slices, 12 pair tiles over 2 clusters.
    tile_n = 256 if stages <= 6 else 128
    A, B = _int_inputs(768, 1024, 512, "f16", seed=200 + stages)
    C, info, canary = gu.run_device(A, B, "f16", stages=stages, cta_group=2, tile_n=tile_n,
                                    max_ctas=4)
    assert canary and info["cta_group"] == 2 and info["grid"] == 4
    # even rings of >= 6 slices run as stages / 2 slots of two K slices
    assert info["k_sub"] == (2 if stages % 2 == 0 and stages >= 6 else 1)
    _assert_bit_exact(A, B, "f16", C)


@pytest.mark.parametrize("shape", [(1, 8, 8), (129, 130, 72), (255, 257, 136), (256, 256, 64),
                                   (257, 384, 264), (513, 1000, 1000), (300, 200, 8)])
@pytest.mark.parametrize("tile_n", [128, 256])
def test_cta_pair_edge_shapes(shape, tile_n):
    M, N, K = shape
    A, B = gemm_inputs.custom(M, N, K, seed=M + 3 * N + 5 * K + tile_n)
    C, info, canary = gu.run_device(A, B, "f16", cta_group=2, tile_n=tile_n)
    st, _, _ = gu.check_full(A, B, "f16", C)
    assert canary and st["ok"] and info["cta_group"] == 2, (shape, st, info)


def test_cta_pair_bf16_gelu_and_single_buffer():
    A, B = gemm_inputs.make("gelu_3072x16384x4096_bf16", M=512, N=768, K=512)
    C, info, canary = gu.run_device(A, B, "bf16", epilogue="gelu", cta_group=2, stages=5)
    st, _, _ = gu.check_full(A, B, "bf16", C, epilogue="gelu")
    assert canary and st["ok"] and info["cta_group"] == 2, st
    A, B = _int_inputs(512, 512, 384, "f16", seed=33)
    C, info, canary = gu.run_device(A, B, "f16", cta_group=2, stages=1, variant="single_buffer")
    assert canary and info["cta_group"] == 2 and info["accumulators"] == 1
    _assert_bit_exact(A, B, "f16", C)


@pytest.mark.parametrize("tile_n", [64, 128, 256])
def test_each_tile_width_bit_exact(tile_n):
    A, B = _int_inputs(384, 640, 320, "f16", seed=7)
    C, info, canary = gu.run_device(A, B, "f16", tile_n=tile_n, max_ctas=3, cta_group=1)
    assert canary and info["tile_n"] == tile_n
    _assert_bit_exact(A, B, "f16", C)


def test_bf16_integer_bit_exact():
    A, B = _int_inputs(256, 512, 256, "bf16", seed=9)
    C, _, canary = gu.run_device(A, B, "bf16")
    assert canary
    _assert_bit_exact(A, B, "bf16", C)


def test_single_buffer_variant_bit_exact():
    A, B = _int_inputs(384, 512, 640, "f16", seed=11)
    C, info, canary = gu.run_device(A, B, "f16", stages=1, variant="single_buffer", max_ctas=4,
                                    cta_group=1)
    assert canary and info["accumulators"] == 1 and info["stages"] == 1
    _assert_bit_exact(A, B, "f16", C)


def test_repeated_runs_identical_bits():
    A, B = gemm_inputs.custom(512, 768, 1024, dist="normal_scaled", seed=12)
    C1, _, _ = gu.run_device(A, B, "f16")
    C2, _, _ = gu.run_device(A, B, "f16")
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


# ------------------------------------------------------- small configs --

def test_config_256_uniform_f16():
    A, B = gemm_inputs.make("gemm_256_f16")
    C, _, canary = gu.run_device(A, B, "f16")
    st, _, _ = gu.check_full(A, B, "f16", C)
    assert canary and st["ok"], st


@pytest.mark.parametrize("shape", [
    (1, 1, 1), (1, 8, 8), (7, 3, 5), (63, 65, 64), (64, 64, 64), (65, 63, 72), (127, 129, 136),
    (128, 256, 64), (129, 257, 128), (200, 300, 520), (257, 513, 1000), (300, 200, 8),
    (1, 1024, 4096), (1000, 1, 64), (333, 999, 77),
])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_edge_shapes(shape, dtype):
    M, N, K = shape
    A, B = gemm_inputs.custom(M, N, K, dtype=dtype, seed=M * 7 + N * 3 + K)
    C, info, canary = gu.run_device(A, B, dtype)
    st, _, _ = gu.check_full(A, B, dtype, C)
    assert canary, "wrote outside C"
    assert st["ok"], (shape, st, info)
    assert info["pads_operands"] == (1 if K % 8 else 0)
    assert info["tma_store"] == (0 if N % 8 else 1)


@pytest.mark.parametrize("shape,dtype", [((70001, 24, 40), "f16"), ((5, 70001, 48), "f16"),
                                         ((40000, 130, 8), "bf16"), ((3000, 3000, 3), "f16")])
def test_many_tiles_along_one_dimension_bit_exact(shape, dtype):
    # Hundreds of tiles along one dimension with the other two tiny: many
    # raster groups (or one row of hundreds of tiles), single-slice K, ragged
    # edges on every side.
    M, N, K = shape
    A, B = _int_inputs(M, N, K, dtype, seed=M + 3 * N + 7 * K)
    C, info, canary = gu.run_device(A, B, dtype)
    assert canary and info["num_tiles"] >= 128, info
    _assert_bit_exact(A, B, dtype, C)


@pytest.mark.parametrize("stages", [1, 2, 4])
def test_gelu_bf16_small(stages):
    A, B = gemm_inputs.make("gelu_3072x16384x4096_bf16", M=192, N=640, K=512)
    C, _, canary = gu.run_device(A, B, "bf16", epilogue="gelu", stages=stages)
    st, _, _ = gu.check_full(A, B, "bf16", C, epilogue="gelu")
    assert canary and st["ok"], st


def test_gelu_extreme_values_no_nan():
    # Large |x| must give x (positive) or -0/tiny (negative), never NaN.
    K = 64
    A = torch.zeros(128, K, dtype=torch.bfloat16)
    B = torch.zeros(256, K, dtype=torch.bfloat16)
    A[:, 0] = torch.linspace(-300, 300, 128).to(torch.bfloat16)
    B[:, 0] = torch.linspace(-2, 2, 256).to(torch.bfloat16)
    C, _, _ = gu.run_device(A, B, "bf16", epilogue="gelu")
    assert torch.isfinite(C.float()).all()
    st, _, _ = gu.check_full(A, B, "bf16", C, epilogue="gelu")
    assert st["ok"], st


def test_gelu_f16():
    A, B = gemm_inputs.custom(256, 384, 256, dtype="f16", dist="normal_scaled", seed=5)
    C, _, _ = gu.run_device(A, B, "f16", epilogue="gelu")
    st, _, _ = gu.check_full(A, B, "f16", C, epilogue="gelu")
    assert st["ok"], st


# ------------------------------------------------ alignment / fallbacks --

@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 3, 0), (0, 0, 1), (8, 8, 8), (5, 7, 3)])
def test_unaligned_base_addresses(offsets):
    a_off, b_off, c_off = offsets
    A, B = gemm_inputs.custom(200, 264, 192, seed=sum(offsets))
    C, info, canary = gu.run_device(A, B, "f16", a_offset=a_off, b_offset=b_off, c_offset=c_off)
    st, _, _ = gu.check_full(A, B, "f16", C)
    assert canary and st["ok"], (offsets, st)
    assert info["pads_operands"] == (1 if (a_off % 8 or b_off % 8) else 0)
    assert info["tma_store"] == (0 if c_off % 8 else 1)


def test_k_zero_writes_zeros_and_empty_is_noop():
    import software_pipelined_tiled_gemm_gb300 as sg
    A = torch.zeros(100, 0, dtype=torch.float16)
    B = torch.zeros(70, 0, dtype=torch.float16)
    C, info, canary = gu.run_device(A, B, "f16", epilogue="gelu")
    assert canary and (C.view(torch.int16) == 0).all() and info["kernels_per_run"] == 0
    for M, N in ((0, 5), (5, 0)):
        plan = sg.Plan(M, N, 16, "f16")
        c = torch.empty(max(M * N, 1), dtype=torch.float16, device="cuda")
        a = torch.empty(max(M * 16, 1), dtype=torch.float16, device="cuda")
        b = torch.empty(max(N * 16, 1), dtype=torch.float16, device="cuda")
        plan.run_ptr(a.data_ptr(), b.data_ptr(), c.data_ptr(), 0)
        plan.close()


def test_plan_mismatch_and_aliasing_rejected():
    import software_pipelined_tiled_gemm_gb300 as sg
    plan = sg.Plan(128, 128, 64, "f16")
    a = torch.zeros(128 * 64, dtype=torch.float16, device="cuda")
    c = torch.zeros(128 * 128, dtype=torch.float16, device="cuda")
    st = sg.gemm_run(plan.handle, a.data_ptr(), a.data_ptr(), c.data_ptr(), 128, 128, 32, 0, 0, 4, 0)
    assert st == sg.GEMM_ERR_PLAN_MISMATCH
    st = sg.gemm_run(plan.handle, a.data_ptr(), a.data_ptr(), c.data_ptr(), 128, 128, 64, 1, 0, 4, 0)
    assert st == sg.GEMM_ERR_PLAN_MISMATCH
    st = sg.gemm_run(plan.handle, c.data_ptr(), a.data_ptr(), c.data_ptr(), 128, 128, 64, 0, 0, 4, 0)
    assert st == sg.GEMM_ERR_INVALID_ARG
    st = sg.gemm_run(plan.handle, a.data_ptr() + 1, a.data_ptr(), c.data_ptr(), 128, 128, 64, 0, 0, 4, 0)
    assert st == sg.GEMM_ERR_INVALID_ARG      # odd address
    plan.close()


def test_smem_budget_reported_not_clamped():
    import software_pipelined_tiled_gemm_gb300 as sg
    with pytest.raises(sg.GemmError) as ei:
        sg.Plan(4096, 4096, 4096, "f16", stages=5, tile_n=256, cta_group=1)
    assert ei.value.status == sg.GEMM_ERR_SMEM_BUDGET
    with pytest.raises(sg.GemmError) as ei:
        sg.Plan(4096, 4096, 4096, "f16", stages=7, tile_n=256, cta_group=2)
    assert ei.value.status == sg.GEMM_ERR_SMEM_BUDGET
    p = sg.Plan(4096, 4096, 4096, "f16", stages=6)      # auto: 256x256 CTA pairs fit 6 slots
    assert p.info()["stages"] == 6 and p.info()["cta_group"] == 2 and p.info()["tile_n"] == 256
    p.close()
    p = sg.Plan(4096, 4096, 4096, "f16", stages=6, cta_group=1)   # single CTA: narrower tile
    assert p.info()["tile_n"] < 256
    p.close()


def test_run_host_end_to_end():
    import software_pipelined_tiled_gemm_gb300 as sg
    A, B = gemm_inputs.custom(300, 520, 264, seed=21)
    C = torch.empty(300, 520, dtype=torch.float16).pin_memory()
    Ap, Bp = A.pin_memory(), B.pin_memory()
    plan = sg.Plan(300, 520, 264, "f16")
    stream = torch.cuda.current_stream()
    for _ in range(2):
        C.zero_()
        plan.run_host(Ap.data_ptr(), Bp.data_ptr(), C.data_ptr(), stream.cuda_stream)
        st, _, _ = gu.check_full(A, B, "f16", C)
        assert st["ok"], st
    plan.close()


@pytest.mark.parametrize("shape,tuning,blocks", [
    ((6144, 6144, 1024), {}, 16),                      # 4 x 4 blocks of 1536 x 1536
    ((4096, 2048, 2048), {}, 2),                       # 2 row panels, whole rows of C
    ((3000, 3072, 2000), {}, 2),                       # 1 x 2, ragged rows
    ((4096, 4001, 2048), {}, 4),                       # 2 x 2, C rows not 16-byte aligned
    ((3072, 4096, 2050), {"b_kn": 1}, 2),              # K x N B, padded K: whole rows of C
    ((3072, 4096, 2050), {}, 2),                       # K needs padding: whole rows of C
    ((2048, 3072, 1024), {"out_f32": 1, "cta_group": 1}, 2),
])
def test_run_host_blocks(shape, tuning, blocks):
    # Problems with >= 32 MiB of copies run in blocks of C: A's and B's panels
    # in on one copy stream in turn, each block's GEMM (a plan writing into
    # the whole C) as soon as its panels are in, each block of C back by a 2-D
    # copy on a second stream.  Checked at sampled positions (every row and
    # column panel's first and last rows / columns included), twice on the
    # same plan.
    import software_pipelined_tiled_gemm_gb300 as sg
    M, N, K = shape
    A, B = gemm_inputs.custom(M, N, K, seed=M + N + K)
    f32 = tuning.get("out_f32", 0) == 1
    Bh = (B.t().contiguous() if tuning.get("b_kn") else B).pin_memory()
    C = torch.empty(M, N, dtype=torch.float32 if f32 else torch.float16).pin_memory()
    plan = sg.Plan(M, N, K, "f16", stages=6, **tuning)
    stream = torch.cuda.current_stream()
    rows = [0, M - 1] + [r for i in range(1, 8) for r in (i * M // 8 - 1, i * M // 8)]
    cols = [0, N - 1] + [x for j in range(1, 12) for x in (j * 256 - 1, j * 256) if x < N]
    r = np.array(rows * 40 + list(np.random.default_rng(N).integers(0, M, len(cols))), dtype=np.int64)
    c = np.concatenate([np.random.default_rng(M).integers(0, N, len(rows) * 40),
                        np.array(cols, dtype=np.int64)]).astype(np.int64)
    ref = oracle.gemm_nt_entries(A, B, "f16", r, c)
    for _ in range(2):
        C.fill_(float("nan"))
        plan.run_host(A.pin_memory().data_ptr(), Bh.data_ptr(), C.data_ptr(), stream.cuda_stream)
        assert plan.check()[0] == 0
        assert torch.isfinite(C).all()
        got = C.numpy()[r, c].astype(np.float64) if f32 else \
            oracle.decode(gu.bits(C)[r, c], "f16")
        st = tolerance.compare(got, ref, "f32" if f32 else "f16")
        assert st["ok"], st
    assert plan.info()["host_panels"] == blocks, plan.info()["host_panels"]
    plan.close()


def test_matmul_nt_torch_layer_on_current_stream():
    import software_pipelined_tiled_gemm_gb300 as sg
    A, B = gemm_inputs.custom(256, 512, 320, dtype="bf16", seed=22)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C = sg.matmul_nt(A.cuda(), B.cuda(), epilogue="gelu", stages=3)
    s.synchronize()
    st, _, _ = gu.check_full(A, B, "bf16", C.cpu(), epilogue="gelu")
    assert st["ok"], st


# ---------------------------------------------- full-size workloads --

def _full_size(name, stages=4, variant="pipelined", count=3000, **tuning):
    w = gemm_inputs.WORKLOADS[name]
    A, B = gemm_inputs.make(w)
    C, info, canary = gu.run_device(A, B, w.dtype, epilogue=None if w.epilogue == "none" else "gelu",
                                    stages=stages, variant=variant, **tuning)
    assert canary
    assert torch.isfinite(C.float()).all(), "unwritten (NaN-filled) or non-finite outputs"
    r, c = gu.sample_positions(w.M, w.N, count, seed=w.seed, tile_n=info["tile_n"])
    st = gu.check_sampled(A, B, w.dtype, C, r, c,
                          epilogue=None if w.epilogue == "none" else "gelu")
    assert st["ok"], (name, st, info)
    return A, B, C, info


@pytest.mark.parametrize("stages", [2, 3, 4, 5, 6])
def test_config_4096_stage_sweep(stages):
    _full_size("gemm_4096_f16", stages=stages)


def test_config_4096_single_cta_tiles():
    _full_size("gemm_4096_f16", stages=4, cta_group=1)


def test_config_8192_pipelined():
    A, B, C, info = _full_size("gemm_8192_f16", stages=4)
    # Row-sum property over every output: sum_j C[i,j] ~= a_i . (sum_j b_j)
    a = A.double().cuda()
    bs = B.double().cuda().sum(0)
    want = (a @ bs).cpu()
    got = C.cuda().double().sum(1).cpu()
    # each C element carries <= 2 ulp(fp16) rounding; 8192 of them per row
    assert torch.max(torch.abs(got - want)).item() < 8192 * 2 ** -11 * 0.05 + 1e-3


def test_config_8192_single_buffer():
    _full_size("gemm_8192_f16", stages=1, variant="single_buffer", count=1500)


def test_config_gelu_layer_bf16():
    _full_size("gelu_3072x16384x4096_bf16", stages=4)


def test_config_ragged():
    A, B, C, info = _full_size("ragged_4095x4097x8191_f16", stages=4)
    assert info["pads_operands"] == 1 and info["tma_store"] == 0
    # the whole last row and last column (partial tiles on every dimension)
    M, N = 4095, 4097
    r = np.concatenate([np.full(N, M - 1), np.arange(M)])
    c = np.concatenate([np.arange(N), np.full(M, N - 1)])
    st = gu.check_sampled(A, B, "f16", C, r, c)
    assert st["ok"], st


def test_config_skinny():
    _full_size("skinny_64x8192x8192_f16", stages=4)


def test_mosaic_guide_shape_full_compare():
    w = gemm_inputs.WORKLOADS["mosaic_16896x512x640_f16"]
    A, B = gemm_inputs.make(w)
    C, _, canary = gu.run_device(A, B, "f16")
    st, _, _ = gu.check_full(A, B, "f16", C)
    assert canary and st["ok"], st


def test_plans_with_different_rings_coexist():
    # Creating a plan with a small ring after one with a large ring must not
    # break the large one (the shared-memory limit is per kernel function).
    import software_pipelined_tiled_gemm_gb300 as sg
    A, B = _int_inputs(256, 512, 256, "f16", seed=31)
    big = sg.Plan(256, 512, 256, "f16", stages=4, tile_n=256)
    small = sg.Plan(256, 512, 256, "f16", stages=1, tile_n=256)
    a, b = A.cuda(), B.cuda()
    for plan in (big, small, big):
        c = torch.full((256, 512), float("nan"), dtype=torch.float16, device="cuda")
        plan.run(a, b, c)
        torch.cuda.synchronize()
        _assert_bit_exact(A, B, "f16", c.cpu())
    big.close()
    small.close()


# ------------------------------------- narrow tail tiles (last wave) --

@pytest.mark.parametrize("cta_group,splits", [(2, 2), (2, 4), (1, 2), (1, 4)])
def test_tail_split_bit_exact_and_reusable(cta_group, splits):
    # 12 tiles over 5 walkers: 10 whole tiles, the last 2 cut along N into
    # `splits` narrow tiles.  The same plan runs three times.
    import software_pipelined_tiled_gemm_gb300 as sg
    M = 768 if cta_group == 2 else 384
    A, B = _int_inputs(M, 1024, 1024, "f16", seed=300 + splits)
    plan = sg.Plan(M, 1024, 1024, "f16", stages=4, cta_group=cta_group, tile_n=256,
                   max_ctas=5 * cta_group, tail_split=splits)
    info = plan.info()
    assert info["tail_tiles"] == 2 and info["tail_splits"] == splits
    assert info["work_units"] == 10 + 2 * splits
    a, b = A.cuda(), B.cuda()
    for _ in range(3):
        c = torch.full((M, 1024), float("nan"), dtype=torch.float16, device="cuda")
        plan.run(a, b, c)
        torch.cuda.synchronize()
        assert plan.check()[0] == 0
        _assert_bit_exact(A, B, "f16", c.cpu())
    plan.close()


@pytest.mark.parametrize("shape", [(700, 1000, 520), (300, 900, 136), (1000, 777, 64)])
def test_tail_split_ragged_edges(shape):
    # Narrow tail tiles that straddle or lie beyond the last column / row.
    M, N, K = shape
    A, B = gemm_inputs.custom(M, N, K, seed=M + N + K)
    for cg in (1, 2):
        C, info, canary = gu.run_device(A, B, "f16", cta_group=cg, tile_n=256, max_ctas=3 * cg,
                                        tail_split=4)
        st, _, _ = gu.check_full(A, B, "f16", C)
        assert canary and st["ok"], (shape, cg, st, info)


def test_tail_split_gelu_bf16():
    A, B = gemm_inputs.make("gelu_3072x16384x4096_bf16", M=512, N=1536, K=2048)
    C1, i1, _ = gu.run_device(A, B, "bf16", epilogue="gelu", cta_group=2, max_ctas=10,
                              tail_split=4)
    assert i1["tail_splits"] == 4 and i1["tail_tiles"] > 0
    st, _, _ = gu.check_full(A, B, "bf16", C1, epilogue="gelu")
    assert st["ok"], st


def test_tail_split_invalid_width_rejected():
    import software_pipelined_tiled_gemm_gb300 as sg
    with pytest.raises(sg.GemmError) as ei:
        sg.Plan(768, 1024, 1024, "f16", cta_group=2, tile_n=256, max_ctas=10, tail_split=3)
    assert ei.value.status == sg.GEMM_ERR_INVALID_ARG


def test_auto_tail_split_choice():
    import software_pipelined_tiled_gemm_gb300 as sg
    # 8192^3: 1024 pair tiles over 76 clusters: 12 whole waves, the K
    # iterations of the last 112 tiles shared out stream-K.
    p = sg.Plan(8192, 8192, 8192, "f16", stages=6)
    info = p.info()
    p.close()
    walkers = info["grid"] // info["cta_group"]
    assert info["cta_group"] == 2 and info["stream_k"] == 1
    assert info["tail_tiles"] == info["num_tiles"] - (info["num_tiles"] // walkers - 1) * walkers
    # a single-buffer plan never splits
    p = sg.Plan(8192, 8192, 8192, "f16", stages=1, variant="single_buffer")
    assert p.info()["stream_k"] == 0 and p.info()["tail_splits"] == 1
    p.close()
    # short K (the Mosaic guide's 16896 x 512 x 640: 10 K slices per tile):
    # no automatic stream-K, whose partial exchange would cost more than the
    # idle part of the last wave; forced stream-K still works there.
    p = sg.Plan(16896, 512, 640, "f16", stages=6)
    assert p.info()["stream_k"] == 0 and p.info()["tail_splits"] == 1
    p.close()
    p = sg.Plan(16896, 512, 640, "f16", stages=6, cta_group=2, tail_split=1)
    assert p.info()["stream_k"] == 1
    p.close()


def test_ring_depth_capped_at_the_k_slices_of_short_problems():
    # a ring deeper than K has slices only takes shared memory; runs still
    # pass the requested stages
    import software_pipelined_tiled_gemm_gb300 as sg
    A, B = _int_inputs(256, 256, 256, "f16", seed=1900)          # 4 K slices
    C, info, canary = gu.run_device(A, B, "f16", stages=6)
    assert canary and info["stages"] == 4, info
    _assert_bit_exact(A, B, "f16", C)
    p = sg.Plan(256, 256, 256, "f16", stages=6, tail_split=-1)   # a forced tail mode keeps the ring
    assert p.info()["stages"] == 6
    p.close()
    p = sg.Plan(512, 512, 2048, "f16", stages=6)                 # 32 slices: not capped
    assert p.info()["stages"] == 6
    p.close()


def test_auto_tile_and_stream_k_choice_for_mid_sizes():
    # Half a wave of 256 x 256 pair tiles is taken over one to two waves of
    # 256 x 128 ones; stream-K only when the last wave leaves each walker at
    # least 24 idle K slices.
    import software_pipelined_tiled_gemm_gb300 as sg

    def info(M, N, K):
        p = sg.Plan(M, N, K, "f16", stages=6)
        try:
            return p.info()
        finally:
            p.close()

    for shape in [(2048, 2048, 2048), (4096, 1024, 8192), (512, 8192, 4096)]:
        i = info(*shape)         # 64 pair tiles on 76 clusters
        assert i["cta_group"] == 2 and i["tile_n"] == 256 and i["stream_k"] == 0, (shape, i)
    assert info(3072, 3072, 3072)["stream_k"] == 0    # 68 of 76 in the last wave: 5 idle slices
    assert info(6144, 6144, 2048)["stream_k"] == 0    # 44 of 76, K = 32 slices: 13.5
    assert info(4096, 4096, 4096)["stream_k"] == 1    # 28 of 76, K = 64 slices: 40
    i = info(128, 16384, 2048)      # 128 single-CTA tiles 128 wide keep 84 % of the SMs busy
    assert i["cta_group"] == 1 and i["tile_n"] == 128, i


# ------------------------------------------------------------ stream-K --

@pytest.mark.parametrize("cta_group", [1, 2])
def test_stream_k_bit_exact_and_reusable(cta_group):
    # 12 tiles over 5 walkers: 5 whole tiles, then the 7 x 16 K iterations of
    # the other 7 tiles shared out (22-23 per walker), so 4-5 tiles are split
    # between two walkers.  Three runs of the same plan: flags must reset.
    import software_pipelined_tiled_gemm_gb300 as sg
    M = 768 if cta_group == 2 else 384
    A, B = _int_inputs(M, 1024, 1024, "f16", seed=400 + cta_group)
    plan = sg.Plan(M, 1024, 1024, "f16", stages=4, cta_group=cta_group, tile_n=256,
                   max_ctas=5 * cta_group, tail_split=1)
    info = plan.info()
    assert info["stream_k"] == 1 and info["tail_tiles"] == 7 and info["grid"] == 5 * cta_group
    a, b = A.cuda(), B.cuda()
    for _ in range(3):
        c = torch.full((M, 1024), float("nan"), dtype=torch.float16, device="cuda")
        plan.run(a, b, c)
        torch.cuda.synchronize()
        assert plan.check()[0] == 0
        _assert_bit_exact(A, B, "f16", c.cpu())
    plan.close()


@pytest.mark.parametrize("shape", [(700, 1000, 520), (1000, 777, 264), (513, 1290, 1000)])
def test_stream_k_ragged_edges(shape):
    M, N, K = shape
    A, B = gemm_inputs.custom(M, N, K, seed=M + 2 * N + K)
    for cg in (1, 2):
        C, info, canary = gu.run_device(A, B, "f16", cta_group=cg, tile_n=256, max_ctas=7 * cg,
                                        tail_split=1)
        st, _, _ = gu.check_full(A, B, "f16", C)
        assert info["stream_k"] == 1, info
        assert canary and st["ok"], (shape, cg, st, info)


def test_stream_k_gelu_bf16_and_deterministic():
    A, B = gemm_inputs.make("gelu_3072x16384x4096_bf16", M=512, N=1536, K=2048)
    outs = []
    for _ in range(2):
        C, info, _ = gu.run_device(A, B, "bf16", epilogue="gelu", cta_group=2, max_ctas=10,
                                   tail_split=1)
        assert info["stream_k"] == 1
        outs.append(C)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    st, _, _ = gu.check_full(A, B, "bf16", outs[0], epilogue="gelu")
    assert st["ok"], st


@pytest.mark.parametrize("shape", [(64, 2048, 1024), (100, 4096, 576), (128, 1000, 200)])
def test_single_tile_row_rotated_k_bit_exact(shape):
    # One row of tiles: each CTA starts its K loop at a different slice.
    M, N, K = shape
    A, B = _int_inputs(M, N, K, "f16", seed=M + N)
    C, info, canary = gu.run_device(A, B, "f16")
    assert canary and info["num_tiles"] > 1
    _assert_bit_exact(A, B, "f16", C)


def test_hundred_runs_bit_identical():
    # Race check: a stale ring slot or accumulator would show up as a
    # changed bit somewhere in 100 repetitions of the same GEMM.
    import software_pipelined_tiled_gemm_gb300 as sg
    A, B = gemm_inputs.custom(1024, 1024, 2048, dist="normal_scaled", seed=99)
    a, b = A.cuda(), B.cuda()
    plan = sg.Plan(1024, 1024, 2048, "f16", stages=6)
    outs = torch.empty(100, 1024, 1024, dtype=torch.float16, device="cuda")
    for i in range(100):
        plan.run(a, b, outs[i])
    torch.cuda.synchronize()
    assert plan.check()[0] == 0
    plan.close()
    first = outs[0].view(torch.int16)
    assert all(torch.equal(first, outs[i].view(torch.int16)) for i in range(1, 100))
    st, _, _ = gu.check_full(A, B, "f16", outs[0].cpu())
    assert st["ok"], st


@pytest.mark.parametrize("stages", [5, 6, 7, 8])
@pytest.mark.parametrize("M,b_kn", [(1, 0), (33, 0), (64, 0), (64, 1)])
def test_sixty_four_row_a_slices_every_ring_depth_bit_exact(M, b_kn, stages):
    # M <= 64: the ring keeps 64-row A slices, so up to 8 slices of 128-wide
    # B fit; odd depths run one slice per slot, even ones >= 6 two.  Tiles
    # split into K halves (N = 4096) and not (N = 8192, tile_n 64).
    for N, tuning in ((4096, {}), (8192, {"tile_n": 64})):
        K = 2048
        A, B = _int_inputs(M, N, K, "f16", seed=M * 5 + stages + N)
        Bdev = B.t().contiguous() if b_kn else B
        C, info, canary = gu.run_device(A, Bdev, "f16", stages=stages, b_kn=b_kn, **tuning)
        assert canary and info["stages"] == stages, info
        assert info["k_sub"] == (2 if stages % 2 == 0 and stages >= 6 else 1), info
        _assert_bit_exact(A, B, "f16", C)


@pytest.mark.parametrize("shape", [(64, 4096, 2048), (40, 2048, 1024), (128, 2048, 4096),
                                   (200, 1024, 2048), (64, 8192, 1100)])
def test_few_tiles_split_k_in_two_bit_exact(shape):
    # At most half a wave of tiles: each tile runs as two K halves on two
    # CTAs (the first half adds the second's partial); M <= 64 also copies
    # only 64 rows of A per slice.  Two runs of the same plan.
    import software_pipelined_tiled_gemm_gb300 as sg
    M, N, K = shape
    A, B = _int_inputs(M, N, K, "f16", seed=M * 3 + N + K)
    plan = sg.Plan(M, N, K, "f16", stages=6)
    info = plan.info()
    assert info["stream_k"] == 1 and info["grid"] == 2 * info["num_tiles"], info
    # one row of single-CTA tiles streams B: two K slices per ring slot (with
    # K = 1100, 9 slots per tile, so the halves meet inside a slot's range)
    assert info["k_sub"] == (2 if M <= 128 else 1), info
    a, b = A.cuda(), B.cuda()
    for _ in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        plan.run(a, b, c)
        torch.cuda.synchronize()
        assert plan.check()[0] == 0
        _assert_bit_exact(A, B, "f16", c.cpu())
    plan.close()



# ------------------------------------------- ReLU epilogue, fp32 output --

def _run_f32(A, B, dtype, epilogue=None, c_offset=0, **tuning):
    """C = epi(A.B^T) with fp32 C through gemm_run; returns (C_cpu, info, canary_ok)."""
    import software_pipelined_tiled_gemm_gb300 as sg
    M, K = A.shape
    N = B.shape[0]
    cbuf = torch.full((M * N + c_offset + 32,), -7.0, dtype=torch.float32, device="cuda")
    c = cbuf[c_offset:c_offset + M * N]
    plan = sg.Plan(M, N, K, dtype, epilogue, out_f32=1, **tuning)
    a, b = A.cuda(), B.cuda()          # keep the device copies alive during the run
    plan.run_ptr(a.data_ptr(), b.data_ptr(), c.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert plan.check()[0] == 0
    info = plan.info()
    plan.close()
    around = torch.cat([cbuf[:c_offset], cbuf[c_offset + M * N:]])
    return c.view(M, N).cpu(), info, bool((around == -7.0).all())


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("cta_group", [1, 2])
def test_relu_epilogue_bit_exact(dtype, cta_group):
    A, B = _int_inputs(384, 640, 256, dtype, seed=51)
    C, info, canary = gu.run_device(A, B, dtype, epilogue="relu", cta_group=cta_group)
    want = oracle.round_to(oracle.gemm_nt(A, B, dtype, epilogue="relu"), dtype)
    assert canary and (gu.bits(C) == want).all()


def test_relu_epilogue_general_values_and_unaligned_c():
    A, B = gemm_inputs.custom(300, 261, 520, dist="normal_scaled", seed=52)
    for off in (0, 1):
        C, info, canary = gu.run_device(A, B, "f16", epilogue="relu", c_offset=off)
        st, _, _ = gu.check_full(A, B, "f16", C, epilogue="relu")
        assert canary and st["ok"] and (C.float() >= 0).all(), (off, st)


@pytest.mark.parametrize("cta_group", [1, 2])
def test_fp32_output_exact_on_integers(cta_group):
    A, B = _int_inputs(512, 768, 640, "f16", seed=53)
    C, info, canary = _run_f32(A, B, "f16", cta_group=cta_group)
    assert info["out_f32"] == 1 and canary
    exact = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T
    assert np.array_equal(C.numpy().astype(np.float64), exact.astype(np.float64))


@pytest.mark.parametrize("epilogue", [None, "gelu", "relu"])
@pytest.mark.parametrize("shape,c_offset", [((256, 512, 512), 0), ((300, 261, 264), 0),
                                            ((200, 264, 136), 1)])
def test_fp32_output_within_tolerance(epilogue, shape, c_offset):
    M, N, K = shape
    A, B = gemm_inputs.custom(M, N, K, dtype="bf16", dist="normal_xw", seed=M + N)
    C, info, canary = _run_f32(A, B, "bf16", epilogue=epilogue, c_offset=c_offset)
    ref = oracle.gemm_nt(A, B, "bf16", epilogue=epilogue)
    st = tolerance.compare(C.numpy().astype(np.float64), ref, "f32")
    assert canary and st["ok"], (shape, epilogue, st, info)
    assert info["tma_store"] == (1 if (N % 4 == 0 and c_offset % 4 == 0) else 0)


def test_fp32_output_stream_k_and_matmul_nt():
    import software_pipelined_tiled_gemm_gb300 as sg
    A, B = _int_inputs(768, 1024, 1024, "bf16", seed=54)
    C, info, canary = _run_f32(A, B, "bf16", cta_group=2, tile_n=256, max_ctas=10, tail_split=1)
    assert info["stream_k"] == 1 and canary
    exact = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T
    assert np.array_equal(C.numpy().astype(np.float64), exact.astype(np.float64))
    c2 = sg.matmul_nt(A.cuda(), B.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert c2.dtype == torch.float32 and torch.equal(c2.cpu(), C)
