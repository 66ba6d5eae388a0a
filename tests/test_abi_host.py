"""Host-only checks of the C ABI: the library loads, exports every function the
header declares, and rejects bad arguments before touching a GPU."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import software_pipelined_tiled_gemm_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(gemm_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_plan_run_destroy_abi():
    names = _declared_functions()
    for n in ("gemm_plan_create", "gemm_run", "gemm_plan_destroy"):
        assert n in names
    assert len(names) >= 10


def test_library_exports_every_declared_symbol():
    lib = sg.load_library()
    for n in _declared_functions():
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings():
    assert sg.gemm_status_string(sg.GEMM_OK) == "GEMM_OK"
    assert sg.gemm_status_string(sg.GEMM_ERR_TIMEOUT) == "GEMM_ERR_TIMEOUT"
    assert sg.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"
    assert re.match(r"^\d+\.\d+\.\d+$", sg.gemm_version())


def test_wait_detail_strings_name_every_device_wait():
    # role << 16 | wait id, as the kernels record them under GEMM_ERR_TIMEOUT
    codes = {(1 << 16) | 1: "producer", (1 << 16) | 2: "producer", (2 << 16) | 1: "MMA",
             (2 << 16) | 2: "MMA", (2 << 16) | 3: "MMA", (3 << 16) | 1: "epilogue",
             (3 << 16) | 2: "stream-K", (3 << 16) | 3: "stream-K", (3 << 16) | 4: "cluster"}
    texts = set()
    for code, word in codes.items():
        t = sg.gemm_wait_detail_string(code)
        assert word in t, (hex(code), t)
        texts.add(t)
    assert len(texts) == len(codes)          # each wait has its own text
    assert sg.gemm_wait_detail_string(0) == ""
    assert sg.gemm_wait_detail_string(12345) == "unknown wait"


def test_smem_bytes_is_the_tutorial_formula():
    # shared_bytes(block_M, block_N, block_K, elem, stages) of the TileLang
    # tutorial: stages * (bM*bK + bN*bK) * elem.  Its CLI defaults (128, 128,
    # 32, fp16) give 16 KiB at one stage and 48 KiB at three.
    assert sg.gemm_smem_bytes(128, 128, 32, 2, 1) == 16384
    assert sg.gemm_smem_bytes(128, 128, 32, 2, 3) == 49152
    assert sg.gemm_smem_bytes(128, 256, 64, 2, 4) == 4 * 48 * 1024
    assert sg.gemm_smem_bytes(0, 128, 32, 2, 3) == 0
    assert sg.gemm_smem_bytes(128, 128, 32, 2, -1) == 0


@pytest.mark.parametrize("args,code", [
    ((-1, 8, 8, 0, 0, 4, 0, 0), sg.GEMM_ERR_INVALID_ARG),        # negative M
    ((8, 8, -3, 0, 0, 4, 0, 0), sg.GEMM_ERR_INVALID_ARG),        # negative K
    ((8, 8, 8, 2, 0, 4, 0, 0), sg.GEMM_ERR_INVALID_ARG),         # dtype out of range
    ((8, 8, 8, 0, 5, 4, 0, 0), sg.GEMM_ERR_INVALID_ARG),         # epilogue out of range
    ((8, 8, 8, 0, 0, 0, 0, 0), sg.GEMM_ERR_INVALID_ARG),         # stages < 1
    ((8, 8, 8, 0, 0, 9, 0, 0), sg.GEMM_ERR_INVALID_ARG),         # stages > 8
    ((8, 8, 8, 0, 0, 2, 1, 0), sg.GEMM_ERR_INVALID_ARG),         # single buffer needs 1 stage
    ((8, 8, 8, 0, 0, 4, 7, 0), sg.GEMM_ERR_INVALID_ARG),         # variant out of range
    ((8, 8, 8, 0, 0, 4, 0, -1), sg.GEMM_ERR_INVALID_ARG),        # device < 0
    ((1 << 31, 8, 8, 0, 0, 4, 0, 0), sg.GEMM_ERR_INVALID_ARG),   # M >= 2^31
])
def test_plan_create_rejects_bad_arguments(args, code):
    st, h = sg.gemm_plan_create(*args)
    assert st == code and h is None
    assert sg.gemm_last_error() != ""


def test_plan_create_ex_rejects_bad_tuning():
    for t in (sg.GemmTuning(96, 0, 0, 0, 0, 0), sg.GemmTuning(0, -1, 0, 0, 0, 0),
              sg.GemmTuning(0, 0, -2, 0, 0, 0), sg.GemmTuning(0, 0, 0, 3, 0, 0),
              sg.GemmTuning(0, 0, 0, -1, 0, 0), sg.GemmTuning(64, 0, 0, 2, 0, 0),
              sg.GemmTuning(0, 0, 0, 0, -2, 0),
              sg.GemmTuning(0, 0, 0, 0, 5, 0), sg.GemmTuning(0, 0, 0, 0, 0, -5),
              sg.GemmTuning(0, 0, 0, 0, 0, 0, 2), sg.GemmTuning(b_kn=-1),
              sg.GemmTuning(out_f32=3), sg.GemmTuning(tail_split=2, b_kn=1),
              sg.GemmTuning(k_serpentine=2), sg.GemmTuning(k_serpentine=-2),
              sg.GemmTuning(epi_groups=3), sg.GemmTuning(epi_groups=-1)):
        st, h = sg.gemm_plan_create_ex(64, 64, 64, 0, 0, 4, 0, 0, t)
        assert st == sg.GEMM_ERR_INVALID_ARG and h is None


def test_null_out_pointer_rejected():
    lib = sg.load_library()
    assert lib.gemm_plan_create(None, 8, 8, 8, 0, 0, 4, 0, 0) == sg.GEMM_ERR_INVALID_ARG


def test_null_plan_rejected_everywhere():
    assert sg.gemm_run(None, 1, 2, 3, 8, 8, 8, 0, 0, 4, None) == sg.GEMM_ERR_INVALID_ARG
    assert sg.gemm_run_host(None, 1, 2, 3, 8, 8, 8, 0, 0, 4, None) == sg.GEMM_ERR_INVALID_ARG
    assert sg.gemm_run_bias(None, 1, 2, 4, 3, 8, 8, 8, 0, 0, 4, None) == sg.GEMM_ERR_INVALID_ARG
    st, _, _ = sg.gemm_plan_check(None)
    assert st == sg.GEMM_ERR_INVALID_ARG
    st, _ = sg.gemm_plan_get_info(None)
    assert st == sg.GEMM_ERR_INVALID_ARG
    sg.gemm_plan_destroy(None)     # allowed, no-op


def test_valid_plan_without_gpu_reports_cuda_or_unsupported():
    # On a machine without a GB300 a well-formed request fails cleanly.
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = sg.gemm_plan_create(256, 256, 256, 0, 0, 4, 0, 0)
    assert st in (sg.GEMM_ERR_CUDA, sg.GEMM_ERR_UNSUPPORTED, sg.GEMM_ERR_INVALID_ARG)
    assert h is None


def test_plan_class_raises_gemm_error():
    with pytest.raises(sg.GemmError) as ei:
        sg.Plan(-1, 4, 4, "f16")
    assert ei.value.status == sg.GEMM_ERR_INVALID_ARG


def test_tuning_field_order_matches_the_header():
    # The ctypes mirror must list gemm_tuning_t's fields in the header's order.
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct \{(.*?)\} gemm_tuning_t;", src, flags=re.S).group(1)
    names = re.findall(r"\b(\w+);", body)
    assert names == [f[0] for f in sg.GemmTuning._fields_]


def test_matmul_nn_checks_shapes_on_cpu_tensors():
    import torch
    a = torch.zeros(4, 8, dtype=torch.float16)
    with pytest.raises(ValueError):
        sg.matmul_nn(a, torch.zeros(4, 8, dtype=torch.float16))   # B must be (K, N)


def test_matmul_nt_checks_arguments_on_cpu_tensors():
    import torch
    a = torch.zeros(4, 8, dtype=torch.float16)
    b = torch.zeros(4, 8, dtype=torch.float16)
    with pytest.raises(ValueError):
        sg.matmul_nt(a, b)


def test_plan_cache_is_lru_and_bounded_on_request(monkeypatch):
    # get_plan's cache logic with a stand-in for Plan (creating a real plan needs a GPU)
    closed = []

    class FakePlan:
        def __init__(self, M, *args, **kw):
            self.M = M

        def close(self):
            closed.append(self.M)

    monkeypatch.setattr(sg, "Plan", FakePlan)
    sg.clear_plan_cache()
    try:
        p1 = sg.get_plan(1, 8, 8, "f16")
        assert sg.get_plan(1, 8, 8, "f16") is p1           # cached
        for m in (2, 3, 4):
            sg.get_plan(m, 8, 8, "f16")
        assert sg.plan_cache_size() == 4 and closed == []  # unbounded by default
        sg.get_plan(1, 8, 8, "f16")                        # 1 becomes the most recent
        sg.set_plan_cache_limit(2)                         # evicts the two least recent: 2, 3
        assert closed == [2, 3] and sg.plan_cache_size() == 2
        sg.get_plan(5, 8, 8, "f16")                        # evicts 4
        assert closed == [2, 3, 4]
        assert sg.get_plan(1, 8, 8, "f16") is p1
        with pytest.raises(ValueError):
            sg.set_plan_cache_limit(-1)
    finally:
        sg.set_plan_cache_limit(0)
        sg.clear_plan_cache()
    assert sorted(closed) == [1, 2, 3, 4, 5] and sg.plan_cache_size() == 0
