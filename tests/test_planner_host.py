"""The planner on the host, without a GPU: gemm_plan_describe runs the same
code gemm_plan_create_ex runs, from a description of the device.

GB300 below is the description gemm_device_query returns on a GB300 (a GPU
test checks it), so these tests see the choices a real plan makes there.
The strongest pin is the first test: the kernel instances that the committed
ncu summaries name (their template arguments were recorded on the GPU) must
be the instances the planner chooses for those workloads."""
from __future__ import annotations

import os
import re

import pytest

import gemm_inputs
import software_pipelined_tiled_gemm_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# cudaDeviceProp / occupancy figures of a GB300 (sm_103): 152 SMs, 227 KiB of
# opt-in shared memory per block, the L2 size the driver reports, and one
# 2-CTA cluster per SM pair (the package's description; a GPU test checks it).
GB300 = dict(sg.GB300)


def describe(M, N, K, dtype="f16", device=None, **kw):
    return sg.describe(M, N, K, dtype, device=dict(device or GB300), **kw)


def _profiled_instances():
    """(workload key, template arguments) from the summaries' bench-traffic lines."""
    out = []
    pdir = os.path.join(ROOT, "profiles")
    for fn in sorted(os.listdir(pdir)):
        for line in open(os.path.join(pdir, fn)):
            m = re.match(r"bench-traffic: kernel=gemm_tn_kernel<([\d,]+)> workload=(\S+)", line)
            if m:
                out.append((m.group(2), [int(x) for x in m.group(1).split(",")]))
    return out


def test_the_profiles_name_the_headline_instances():
    keys = {k for k, _ in _profiled_instances()}
    assert {"gemm_8192_f16", "gemm_4096_f16", "skinny_64x8192x8192_f16",
            "mosaic_16896x512x640_f16", "gemm_256_f16"} <= keys


@pytest.mark.parametrize("key,args", _profiled_instances())
def test_describe_chooses_the_profiled_kernel_instance(key, args):
    # gemm_tn_kernel<BN, CG, kSplit, kKN, kStream, kSub, kEpiG>, launched by
    # bench.py with its default ring of 6 slices (1 for the single-buffer variant).
    bn, cg, split, kn, _stream, ksub, epig = args
    name, *opts = key.split(":")
    w = gemm_inputs.WORKLOADS[name]
    kw = dict(stages=6, epilogue=None if w.epilogue == "none" else w.epilogue)
    if "single" in opts:
        kw.update(stages=1, variant="single_buffer")
    if "nn" in opts:
        kw["b_kn"] = 1
    d = describe(w.M, w.N, w.K, w.dtype, **kw)
    assert d["tile_n"] == bn and d["cta_group"] == cg, d
    assert int(d["stream_k"] == 1 or d["tail_splits"] > 1) == split, d
    assert d["b_kn"] == kn and d["k_sub"] == ksub and d["epi_groups"] == epig, d


def test_headline_plan():
    d = describe(8192, 8192, 8192, stages=6)
    assert (d["tile_m"], d["tile_n"], d["tile_k"]) == (256, 256, 64)
    assert d["grid"] == 152 and d["num_tiles"] == 1024
    assert d["stages"] == 6 and d["k_sub"] == 2 and d["accumulators"] == 2
    # 1024 tiles on 76 pairs: 12 whole waves of tiles, the last 112 shared out stream-K
    assert d["stream_k"] == 1 and d["tail_tiles"] == 1024 - 12 * 76
    assert d["k_serpentine"] == 1 and d["l2_prefetch_first"] == 1
    assert 6 * 32768 < d["smem_bytes"] <= GB300["smem_optin"]
    assert (d["pads_operands"], d["tma_store"], d["kernels_per_run"], d["host_panels"]) == (0,) * 4


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (3072, 16384, 4096), (8192, 8192, 8192),
                                   (6144, 6144, 8192), (2560, 10240, 4096)])
def test_stream_k_leaves_whole_waves_and_shares_one_to_two(M, N, K):
    d = describe(M, N, K, stages=6)
    walkers = d["grid"] // d["cta_group"]
    if d["stream_k"]:
        whole = d["num_tiles"] - d["tail_tiles"]
        assert whole % walkers == 0
        assert walkers <= d["tail_tiles"] < 2 * walkers
        assert d["work_units"] == whole
    else:
        assert d["num_tiles"] % walkers == 0 or d["tail_splits"] > 1 or K < 32 * 64


def test_stream_k_needs_idle_time_in_the_last_wave():
    # 3072^3: 144 pair tiles, 68 in the last wave on 76 walkers -> only 8
    # idle walkers x 48 slices, below 24 slices per walker: no stream-K.
    d = describe(3072, 3072, 3072, stages=6)
    assert d["cta_group"] == 2 and d["num_tiles"] == 144 and d["stream_k"] == 0


def test_short_k_gets_no_stream_k_and_eight_epilogue_warps():
    d = describe(16896, 512, 640, stages=6)
    assert d["stream_k"] == 0 and d["tail_splits"] == 1
    assert d["epi_groups"] == 2          # K is 10 slices <= 16
    assert describe(8192, 8192, 1024 + 64, stages=6)["epi_groups"] == 1   # 17 slices


def test_row_wise_c_stores_get_eight_epilogue_warps():
    # A C whose rows are not 16-byte multiples is stored row by row (no bulk
    # tensor store), which exposes the epilogue: eight warps.
    assert describe(4095, 4097, 8191, stages=6)["epi_groups"] == 2
    assert describe(4096, 4100, 8192, stages=6)["epi_groups"] == 2      # 8200 B rows
    assert describe(4096, 4100, 8192, stages=6, out_f32=1)["epi_groups"] == 1  # 16400 B rows
    assert describe(4096, 4104, 8192, stages=6)["epi_groups"] == 1      # 8208 B rows
    assert describe(4095, 4097, 8191, stages=6, epi_groups=1)["epi_groups"] == 1


def test_ring_is_capped_at_the_slices_of_short_k():
    assert describe(1024, 1024, 256, stages=6)["stages"] == 4
    assert describe(1024, 1024, 64 * 20, stages=6)["stages"] == 6
    # a forced tail mode (off, or narrow tiles) keeps the requested ring
    for split in (-1, 2):
        assert describe(1024, 1024, 256, stages=6, cta_group=1, tile_n=128,
                        tail_split=split)["stages"] == 6


def test_pairs_need_half_a_wave_of_pair_tiles():
    # 2 * tiles >= 76 pairs: 38 pair tiles of 256 x 256 (M 512, N 4864) take them
    d = describe(512, 19 * 256, 4096, stages=6)
    assert (d["cta_group"], d["tile_n"]) == (2, 256)
    # 36 tiles of 256 x 256 do not, but 72 of 256 x 128 do
    d = describe(512, 18 * 256, 4096, stages=6)
    assert (d["cta_group"], d["tile_n"]) == (2, 128)
    # 18 tiles of 256 x 128 (M 512, N 1152): single CTAs
    assert describe(512, 9 * 128, 4096, stages=6)["cta_group"] == 1
    # a single 128-row tile row never takes pairs automatically
    assert describe(128, 65536, 4096, stages=6)["cta_group"] == 1
    assert describe(128, 65536, 4096, stages=6, cta_group=2)["cta_group"] == 2


def test_few_tiles_split_in_two_k_halves_in_clusters():
    d = describe(64, 8192, 8192, stages=6)
    assert d["sk_cluster"] == 1 and d["stream_k"] == 1
    assert d["tile_n"] == 128 and d["grid"] == 2 * d["num_tiles"] == 128
    # odd K slice count: no split
    assert describe(64, 8192, 8192 - 64, stages=6)["sk_cluster"] == 0


def test_single_tile_row_and_short_k_choices():
    d = describe(128, 16384, 2048, stages=6)
    assert (d["cta_group"], d["tile_n"], d["num_tiles"], d["grid"]) == (1, 128, 128, 128)
    assert d["epi_groups"] == 2 and d["k_serpentine"] == 0
    d = describe(256, 256, 256, stages=6)
    assert (d["tile_n"], d["stages"], d["grid"]) == (64, 4, 8)


def test_single_buffer_variant():
    d = describe(8192, 8192, 8192, stages=1, variant="single_buffer")
    assert d["stages"] == 1 and d["accumulators"] == 1 and d["k_sub"] == 1
    assert d["stream_k"] == 0 and d["tail_splits"] == 1
    with pytest.raises(sg.GemmError):
        describe(8192, 8192, 8192, stages=2, variant="single_buffer")


def test_l2_rules_follow_the_described_cache():
    M = N = K = 4096                      # operands 64 MiB
    ops = (M + N) * K * 2
    assert describe(M, N, K, stages=6, device=dict(GB300, l2_bytes=ops * 4 // 3 + 4096))[
        "l2_prefetch_first"] == 0
    assert describe(M, N, K, stages=6, device=dict(GB300, l2_bytes=ops * 4 // 3 - 4096))[
        "l2_prefetch_first"] == 1
    # serpentine K: a wave's A and B footprint above half of L2
    assert describe(M, N, K, stages=6)["k_serpentine"] == 0
    assert describe(M, N, K, stages=6, device=dict(GB300, l2_bytes=32 << 20))["k_serpentine"] == 1
    assert describe(M, N, K, stages=6, k_serpentine=1)["k_serpentine"] == 1
    assert describe(8192, 8192, 8192, stages=6, k_serpentine=-1)["k_serpentine"] == 0


def test_grid_follows_the_described_device():
    d = describe(8192, 8192, 8192, stages=6, device=dict(GB300, sm_count=148, pair_clusters=74))
    assert d["grid"] == 148 and d["sm_count"] == 148
    d = describe(8192, 8192, 8192, stages=6, cta_group=1)
    assert d["grid"] == 152 and d["tile_m"] == 128


def test_max_ctas_and_explicit_tiles():
    assert describe(8192, 8192, 8192, stages=6, max_ctas=64)["grid"] == 64
    d = describe(8192, 8192, 8192, stages=4, cta_group=1, tile_n=128)
    assert (d["tile_m"], d["tile_n"]) == (128, 128)


def test_narrow_tail_tiles_on_request():
    # 128-row tiles 256 wide: 4 x 40 = 160 tiles on 152 CTAs leave 8 in the last wave
    d = describe(512, 40 * 256, 4096, stages=4, cta_group=1, tile_n=256, tail_split=4)
    assert d["tail_splits"] == 4 and d["tail_tiles"] == 8
    assert d["work_units"] == 152 + 8 * 4


def test_shared_memory_budget():
    with pytest.raises(sg.GemmError) as e:
        describe(4096, 4096, 4096, stages=8, cta_group=1, tile_n=256)
    assert e.value.status == sg.GEMM_ERR_SMEM_BUDGET
    # a smaller budget narrows the automatic tile instead of failing
    d = describe(4096, 4096, 4096, stages=4, device=dict(GB300, smem_optin=120 * 1024))
    assert d["smem_bytes"] <= 120 * 1024


def test_describe_checks_arguments_like_plan_creation():
    for bad in (dict(tile_n=96), dict(cta_group=3), dict(tail_split=5), dict(epi_groups=3),
                dict(k_serpentine=2), dict(b_kn=1, tail_split=2), dict(timeout_ns=-1)):
        with pytest.raises(sg.GemmError) as e:
            describe(1024, 1024, 1024, stages=4, **bad)
        assert e.value.status == sg.GEMM_ERR_INVALID_ARG, bad
    with pytest.raises(sg.GemmError):
        describe(-1, 8, 8, stages=4)
    with pytest.raises(TypeError):
        describe(1024, 1024, 1024, stages=4, no_such_knob=1)


@pytest.mark.parametrize("field,value", [("sm_count", 0), ("smem_optin", 0), ("l2_bytes", -1),
                                         ("pair_clusters", -1)])
def test_describe_rejects_a_bad_device_description(field, value):
    with pytest.raises(sg.GemmError) as e:
        describe(1024, 1024, 1024, stages=4, device=dict(GB300, **{field: value}))
    assert e.value.status == sg.GEMM_ERR_INVALID_ARG


def test_describe_null_pointers_rejected():
    import ctypes
    lib = sg.load_library()
    info = sg.GemmPlanInfo()
    desc = sg.GemmDeviceDesc(**GB300)
    assert lib.gemm_plan_describe(64, 64, 64, 0, 0, 4, 0, None, None,
                                  ctypes.byref(info)) == sg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_plan_describe(64, 64, 64, 0, 0, 4, 0, None, ctypes.byref(desc),
                                  None) == sg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_device_query(0, None) == sg.GEMM_ERR_INVALID_ARG


def test_device_query_without_a_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, _ = sg.gemm_device_query(0)
    assert st in (sg.GEMM_ERR_CUDA, sg.GEMM_ERR_INVALID_ARG, sg.GEMM_ERR_UNSUPPORTED)


def test_stream_k_share_first_unless_serpentine():
    # Stream-K plans take their stream-K share before their whole tiles,
    # except with the serpentine K order (whose alternating waves the
    # reordering disturbs) and the cluster split (no whole tiles).
    d = describe(4096, 4096, 4096, stages=6)
    assert d["stream_k"] == 1 and d["k_serpentine"] == 0 and d["stream_k_first"] == 1
    assert describe(3072, 16384, 4096, "bf16", epilogue="gelu", stages=6)["stream_k_first"] == 1
    d = describe(8192, 8192, 8192, stages=6)
    assert d["stream_k"] == 1 and d["k_serpentine"] == 1 and d["stream_k_first"] == 0
    assert describe(4096, 4096, 4096, stages=6, k_serpentine=1)["stream_k_first"] == 0
    d = describe(128, 8192, 2048, stages=6)
    assert d["sk_cluster"] == 1 and d["stream_k_first"] == 0
    assert describe(2048, 2048, 2048, stages=6)["stream_k"] == 0
    assert describe(2048, 2048, 2048, stages=6)["stream_k_first"] == 0


def test_sixty_four_row_a_slices_leave_room_for_deeper_rings():
    # M <= 64 keeps 64-row A slices (8 KiB instead of 16), so the skinny
    # 64 x 8192 x 8192 plan fits 8 slices of 128-wide B split in K halves;
    # with M = 65 the full 128-row slices leave room for 6 only at that width.
    d64 = describe(64, 8192, 8192, stages=8)
    assert d64["tile_n"] == 128 and d64["sk_cluster"] == 1 and d64["smem_bytes"] <= 232448
    # (at 8 slices the epilogue staging is single-buffered to make room)
    assert describe(64, 8192, 8192, stages=6)["smem_bytes"] < d64["smem_bytes"]
    assert describe(65, 8192, 8192, stages=8)["tile_n"] == 64
    assert describe(65, 8192, 8192, stages=6)["tile_n"] == 128
