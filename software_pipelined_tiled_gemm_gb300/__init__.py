"""GB300 (sm_103a) software-pipelined tiled GEMM: C = epi(A . B^T).

A thin ctypes binding over the C ABI in ``include/gemm.h`` (library
``_lib/libspgemm.so``).  The functions ``gemm_plan_create``,
``gemm_plan_create_ex``, ``gemm_run``, ``gemm_run_host``, ``gemm_plan_check``,
``gemm_plan_get_info``, ``gemm_plan_destroy``, ``gemm_status_string``,
``gemm_smem_bytes`` carry the C names and only marshal arguments; every step of
the GEMM runs in the library's CUDA kernels.  PyTorch is used for device
memory and the current stream only.

There is no fallback: if the library is missing or cannot be loaded, every
call raises.

With the environment variable ``SPGEMM_BOUNDS_CHECKS=1`` the package loads
the bounds-checked build ``_lib/libspgemm_checked.so`` instead (built on
first use): its kernels range-check their indexes and copy coordinates and
report a failed check as ``GEMM_ERR_BOUNDS`` (see ``gemm_check_t`` in
``include/gemm.h``).

Convenience layer: :func:`matmul_nt` takes torch CUDA tensors A (M,K) and
B (N,K), caches a plan per problem, and launches on the current stream --
the operation of the TileLang tutorial's ``matmul_auto`` (A (M,K), B (N,K),
``T.gemm(..., transpose_B=True)``) with an optional tanh-GELU or ReLU
epilogue and fp16/bf16 or fp32 output.  :func:`matmul_nn` takes B as (K,N),
the form of the Mosaic GPU guide's matmul example.  :func:`describe` reports
what a plan would choose, for this GPU or for a device described by its
properties (no GPU needed).
"""
from __future__ import annotations

import collections
import ctypes
import os
import threading
from typing import Optional

__all__ = [
    "GemmError", "Plan", "matmul_nt", "matmul_nn", "load_library", "library_path",
    "gemm_plan_create", "gemm_plan_create_ex", "gemm_run", "gemm_run_bias", "gemm_run_host",
    "gemm_plan_check",
    "gemm_plan_get_info", "gemm_plan_destroy", "gemm_status_string", "gemm_smem_bytes",
    "gemm_last_error", "gemm_version", "gemm_run_noalloc", "GemmTuning", "GemmPlanInfo",
    "gemm_device_query", "gemm_plan_describe", "GemmDeviceDesc", "describe", "GB300",
    "get_plan", "set_plan_cache_limit", "clear_plan_cache", "plan_cache_size",
    "GEMM_OK", "GEMM_ERR_INVALID_ARG", "GEMM_ERR_UNSUPPORTED", "GEMM_ERR_SMEM_BUDGET",
    "GEMM_ERR_PLAN_MISMATCH", "GEMM_ERR_CUDA", "GEMM_ERR_TIMEOUT", "GEMM_ERR_BOUNDS",
    "gemm_bounds_checked", "bounds_checked_requested",
    "GEMM_F16", "GEMM_BF16", "GEMM_EPI_NONE", "GEMM_EPI_GELU_TANH", "GEMM_EPI_RELU",
    "GEMM_PIPELINED", "GEMM_SINGLE_BUFFER",
]

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(HERE, "_lib", "libspgemm.so")

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED = 2
GEMM_ERR_SMEM_BUDGET = 3
GEMM_ERR_PLAN_MISMATCH = 4
GEMM_ERR_CUDA = 5
GEMM_ERR_TIMEOUT = 6
GEMM_ERR_BOUNDS = 7

GEMM_F16 = 0
GEMM_BF16 = 1
GEMM_EPI_NONE = 0
GEMM_EPI_GELU_TANH = 1
GEMM_EPI_RELU = 2
GEMM_PIPELINED = 0
GEMM_SINGLE_BUFFER = 1


class GemmTuning(ctypes.Structure):
    _fields_ = [("tile_n", ctypes.c_int), ("raster_group", ctypes.c_int),
                ("max_ctas", ctypes.c_int), ("cta_group", ctypes.c_int),
                ("tail_split", ctypes.c_int), ("timeout_ns", ctypes.c_int64),
                ("b_kn", ctypes.c_int), ("out_f32", ctypes.c_int), ("debug_fault", ctypes.c_int),
                ("k_serpentine", ctypes.c_int), ("epi_groups", ctypes.c_int)]


class GemmPlanInfo(ctypes.Structure):
    _fields_ = [("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int), ("tile_k", ctypes.c_int),
                ("stages", ctypes.c_int), ("accumulators", ctypes.c_int),
                ("raster_group", ctypes.c_int), ("grid", ctypes.c_int),
                ("num_tiles", ctypes.c_int64), ("smem_bytes", ctypes.c_size_t),
                ("pads_operands", ctypes.c_int), ("tma_store", ctypes.c_int),
                ("kernels_per_run", ctypes.c_int), ("sm_count", ctypes.c_int),
                ("cta_group", ctypes.c_int), ("tail_tiles", ctypes.c_int64),
                ("tail_splits", ctypes.c_int), ("work_units", ctypes.c_int64),
                ("stream_k", ctypes.c_int), ("out_f32", ctypes.c_int), ("b_kn", ctypes.c_int),
                ("k_sub", ctypes.c_int), ("host_panels", ctypes.c_int),
                ("k_serpentine", ctypes.c_int), ("l2_prefetch_first", ctypes.c_int),
                ("sk_cluster", ctypes.c_int), ("epi_groups", ctypes.c_int),
                ("stream_k_first", ctypes.c_int)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


# What gemm_device_query reports on a GB300 (sm_103): 152 SMs, 227 KiB of
# opt-in shared memory per block, the L2 size the driver reports, 76
# co-resident 2-CTA clusters.  describe() and the planning CLI use it to plan
# for a GB300 on a machine without one.
GB300 = dict(sm_count=152, smem_optin=232448, l2_bytes=135528448, pair_clusters=76)


class GemmDeviceDesc(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int), ("smem_optin", ctypes.c_int),
                ("l2_bytes", ctypes.c_int64), ("pair_clusters", ctypes.c_int)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        name = _status_name(status)
        super().__init__("%s: %s%s" % (where, name, (" -- " + detail) if detail else ""))


_lib = None
_lib_lock = threading.Lock()


def bounds_checked_requested() -> bool:
    """True when SPGEMM_BOUNDS_CHECKS=1 asks for the bounds-checked build."""
    return os.environ.get("SPGEMM_BOUNDS_CHECKS", "0") not in ("", "0")


def library_path() -> str:
    from . import _build
    return _build.LIB_CHECKED if bounds_checked_requested() else _LIB_PATH


def load_library(path: Optional[str] = None):
    """Load libspgemm.so (building it first if the sources are newer)."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        if path is None:
            from . import _build
            checked = bounds_checked_requested()
            if not _build.up_to_date(checked):
                _build.build(checked=checked)
            path = library_path()
        if not os.path.exists(path):
            raise ImportError("libspgemm.so not found at %s; run __graft_entry__.build()" % path)
        lib = ctypes.CDLL(path)
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        pp = ctypes.POINTER(ctypes.c_void_p)
        lib.gemm_plan_create.argtypes = [pp, i64, i64, i64, ci, ci, ci, ci, ci]
        lib.gemm_plan_create.restype = ci
        lib.gemm_plan_create_ex.argtypes = [pp, i64, i64, i64, ci, ci, ci, ci, ci,
                                            ctypes.POINTER(GemmTuning)]
        lib.gemm_plan_create_ex.restype = ci
        lib.gemm_run.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, vp]
        lib.gemm_run.restype = ci
        lib.gemm_run_bias.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, vp]
        lib.gemm_run_bias.restype = ci
        lib.gemm_run_host.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, vp]
        lib.gemm_run_host.restype = ci
        lib.gemm_plan_check.argtypes = [vp, ctypes.POINTER(ctypes.c_int32),
                                        ctypes.POINTER(ctypes.c_int32)]
        lib.gemm_plan_check.restype = ci
        lib.gemm_plan_get_info.argtypes = [vp, ctypes.POINTER(GemmPlanInfo)]
        lib.gemm_plan_get_info.restype = ci
        lib.gemm_plan_destroy.argtypes = [vp]
        lib.gemm_plan_destroy.restype = None
        lib.gemm_status_string.argtypes = [ci]
        lib.gemm_status_string.restype = ctypes.c_char_p
        lib.gemm_wait_detail_string.argtypes = [ctypes.c_int32]
        lib.gemm_wait_detail_string.restype = ctypes.c_char_p
        lib.gemm_last_error.argtypes = []
        lib.gemm_last_error.restype = ctypes.c_char_p
        lib.gemm_smem_bytes.argtypes = [ci, ci, ci, ci, ci]
        lib.gemm_smem_bytes.restype = ctypes.c_size_t
        lib.gemm_version.argtypes = []
        lib.gemm_version.restype = ctypes.c_char_p
        lib.gemm_bounds_checked.argtypes = []
        lib.gemm_bounds_checked.restype = ci
        lib.gemm_run_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, ci, ci, ci, vp]
        lib.gemm_run_noalloc.restype = ci
        lib.gemm_device_query.argtypes = [ci, ctypes.POINTER(GemmDeviceDesc)]
        lib.gemm_device_query.restype = ci
        lib.gemm_plan_describe.argtypes = [i64, i64, i64, ci, ci, ci, ci, ctypes.POINTER(GemmTuning),
                                           ctypes.POINTER(GemmDeviceDesc),
                                           ctypes.POINTER(GemmPlanInfo)]
        lib.gemm_plan_describe.restype = ci
        _lib = lib
        return lib


def _status_name(status: int) -> str:
    try:
        return load_library().gemm_status_string(int(status)).decode()
    except Exception:  # noqa: BLE001 - naming only
        return "status %d" % status


def _check(status: int, where: str):
    if status != GEMM_OK:
        raise GemmError(status, where, load_library().gemm_last_error().decode())


# ------------------------------------------------------- C-named wrappers --

def gemm_status_string(status: int) -> str:
    return load_library().gemm_status_string(int(status)).decode()


def gemm_wait_detail_string(detail: int) -> str:
    """Which device-side wait ran out of time, from a device status detail."""
    return load_library().gemm_wait_detail_string(int(detail)).decode()


def gemm_last_error() -> str:
    return load_library().gemm_last_error().decode()


def gemm_version() -> str:
    return load_library().gemm_version().decode()


def gemm_bounds_checked() -> int:
    """1 when the loaded library is the bounds-checked build."""
    return int(load_library().gemm_bounds_checked())


def gemm_smem_bytes(bm: int, bn: int, bk: int, elem_bytes: int, stages: int) -> int:
    return int(load_library().gemm_smem_bytes(bm, bn, bk, elem_bytes, stages))


def gemm_plan_create(M, N, K, dtype, epi, stages, variant, device):
    """Returns (status, plan_handle_or_None)."""
    h = ctypes.c_void_p()
    st = load_library().gemm_plan_create(ctypes.byref(h), M, N, K, dtype, epi, stages, variant,
                                         device)
    return st, (h.value if st == GEMM_OK else None)


def gemm_plan_create_ex(M, N, K, dtype, epi, stages, variant, device, tuning=None):
    h = ctypes.c_void_p()
    tp = ctypes.byref(tuning) if tuning is not None else None
    st = load_library().gemm_plan_create_ex(ctypes.byref(h), M, N, K, dtype, epi, stages,
                                            variant, device, tp)
    return st, (h.value if st == GEMM_OK else None)


def gemm_run(plan, A, B, C, M, N, K, dtype, epi, stages, stream):
    """A, B, C, stream: integer addresses / handles.  Returns the status."""
    return load_library().gemm_run(plan, A, B, C, M, N, K, dtype, epi, stages, stream)


def gemm_run_bias(plan, A, B, bias, C, M, N, K, dtype, epi, stages, stream):
    """As gemm_run, plus a device pointer to N bias values (or None)."""
    return load_library().gemm_run_bias(plan, A, B, bias, C, M, N, K, dtype, epi, stages, stream)


def gemm_run_host(plan, hA, hB, hC, M, N, K, dtype, epi, stages, stream):
    return load_library().gemm_run_host(plan, hA, hB, hC, M, N, K, dtype, epi, stages, stream)


def gemm_run_noalloc(A, B, C, M, N, K, dtype, epi, stages, stream):
    """Allocation-free GEMM (no plan); see include/gemm.h.  Returns the status."""
    return load_library().gemm_run_noalloc(A, B, C, M, N, K, dtype, epi, stages, stream)


def gemm_plan_check(plan):
    """Returns (status, device_status, detail)."""
    ds, dt = ctypes.c_int32(0), ctypes.c_int32(0)
    st = load_library().gemm_plan_check(plan, ctypes.byref(ds), ctypes.byref(dt))
    return st, ds.value, dt.value


def gemm_plan_get_info(plan):
    info = GemmPlanInfo()
    st = load_library().gemm_plan_get_info(plan, ctypes.byref(info))
    return st, info


def gemm_plan_destroy(plan):
    load_library().gemm_plan_destroy(plan)


def gemm_device_query(device: int):
    desc = GemmDeviceDesc()
    st = load_library().gemm_device_query(int(device), ctypes.byref(desc))
    return st, desc


def gemm_plan_describe(M, N, K, dtype, epi, stages, variant, tuning, desc):
    info = GemmPlanInfo()
    st = load_library().gemm_plan_describe(M, N, K, dtype, epi, stages, variant,
                                           ctypes.byref(tuning) if tuning is not None else None,
                                           ctypes.byref(desc), ctypes.byref(info))
    return st, info


# ------------------------------------------------------------ torch layer --

_DT = {"f16": GEMM_F16, "bf16": GEMM_BF16}
_EPI = {None: GEMM_EPI_NONE, "none": GEMM_EPI_NONE, "gelu": GEMM_EPI_GELU_TANH,
        "gelu_tanh": GEMM_EPI_GELU_TANH, "relu": GEMM_EPI_RELU}
_VAR = {"pipelined": GEMM_PIPELINED, "single_buffer": GEMM_SINGLE_BUFFER}


def _torch_dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return GEMM_F16
    if t.dtype == torch.bfloat16:
        return GEMM_BF16
    raise TypeError("A and B must be float16 or bfloat16, got %s" % t.dtype)


class Plan:
    """Owns one gemm_plan_t."""

    def __init__(self, M, N, K, dtype, epilogue=None, stages=4, variant="pipelined", device=0,
                 tile_n=0, raster_group=0, max_ctas=0, cta_group=0, tail_split=0,
                 timeout_ns=0, b_kn=0, out_f32=0, debug_fault=0, k_serpentine=0, epi_groups=0):
        self.M, self.N, self.K = int(M), int(N), int(K)
        self.dtype = _DT[dtype] if isinstance(dtype, str) else int(dtype)
        self.epi = _EPI[epilogue] if not isinstance(epilogue, int) else int(epilogue)
        self.stages = int(stages)
        self.variant = _VAR[variant] if isinstance(variant, str) else int(variant)
        self.device = int(device)
        self._h = None
        tuning = GemmTuning(int(tile_n), int(raster_group), int(max_ctas), int(cta_group),
                            int(tail_split), int(timeout_ns), int(b_kn), int(out_f32),
                            int(debug_fault), int(k_serpentine), int(epi_groups))
        st, h = gemm_plan_create_ex(self.M, self.N, self.K, self.dtype, self.epi, self.stages,
                                    self.variant, self.device, tuning)
        _check(st, "gemm_plan_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def info(self) -> dict:
        st, info = gemm_plan_get_info(self._h)
        _check(st, "gemm_plan_get_info")
        return info.as_dict()

    def run_ptr(self, A: int, B: int, C: int, stream: int = 0, bias: int = 0):
        """Device addresses; bias: address of N bias values, or 0 for none."""
        if bias:
            _check(gemm_run_bias(self._h, A, B, bias, C, self.M, self.N, self.K, self.dtype,
                                 self.epi, self.stages, stream), "gemm_run_bias")
        else:
            _check(gemm_run(self._h, A, B, C, self.M, self.N, self.K, self.dtype, self.epi,
                            self.stages, stream), "gemm_run")

    def run(self, A, B, C, stream=None, bias=None):
        """A, B, C: torch CUDA tensors (contiguous, shapes (M,K), (N,K) -- or
        (K,N) with b_kn -- and (M,N)); bias: None or a contiguous (N,) tensor
        of A's dtype on the same device."""
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(A.device)
        self.run_ptr(A.data_ptr(), B.data_ptr(), C.data_ptr(), s.cuda_stream,
                     bias.data_ptr() if bias is not None else 0)

    def run_host(self, hA: int, hB: int, hC: int, stream: int = 0):
        _check(gemm_run_host(self._h, hA, hB, hC, self.M, self.N, self.K, self.dtype, self.epi,
                             self.stages, stream), "gemm_run_host")

    def check(self):
        """Synchronise and return (device_status, detail); raises on a device error."""
        st, ds, detail = gemm_plan_check(self._h)
        _check(st, "gemm_plan_check")
        return ds, detail

    def close(self):
        if self._h is not None:
            gemm_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass


def describe(M, N, K, dtype, epilogue=None, stages=4, variant="pipelined", device=0,
             **tuning) -> dict:
    """What ``Plan(M, N, K, dtype, epilogue, stages, variant, device, **tuning)``
    would choose, as :meth:`Plan.info` reports it, without creating the plan.

    ``device``: a CUDA device index (its properties are queried), or a dict
    or :class:`GemmDeviceDesc` with ``sm_count``, ``smem_optin``,
    ``l2_bytes`` and ``pair_clusters`` -- then no CUDA call is made."""
    if isinstance(device, GemmDeviceDesc):
        desc = device
    elif isinstance(device, dict):
        desc = GemmDeviceDesc(**{k: int(device[k]) for k, _ in GemmDeviceDesc._fields_})
    else:
        st, desc = gemm_device_query(int(device))
        _check(st, "gemm_device_query")
    names = [k for k, _ in GemmTuning._fields_]
    unknown = set(tuning) - set(names)
    if unknown:
        raise TypeError("unknown tuning keyword(s): %s" % ", ".join(sorted(unknown)))
    t = GemmTuning(**{k: int(v) for k, v in tuning.items()})
    st, info = gemm_plan_describe(int(M), int(N), int(K),
                                  _DT[dtype] if isinstance(dtype, str) else int(dtype),
                                  _EPI[epilogue] if not isinstance(epilogue, int) else int(epilogue),
                                  int(stages),
                                  _VAR[variant] if isinstance(variant, str) else int(variant), t,
                                  desc)
    _check(st, "gemm_plan_describe")
    return info.as_dict()


# Plans cached by get_plan (and so by matmul_nt / matmul_nn), least recently
# used first.  Each plan holds device memory (its status word; a stream-K
# workspace of up to a few tens of MiB; staging for run_host), so a caller
# with many distinct shapes can bound the cache.  Unbounded by default: a
# plan captured in a CUDA graph must outlive the graph, and closing a plan
# synchronises its device, which is not allowed during stream capture.
_plans: "collections.OrderedDict" = collections.OrderedDict()
_plans_lock = threading.Lock()
_plans_limit = 0


def set_plan_cache_limit(n: int) -> None:
    """Keep at most n cached plans (0: no limit), closing the least recently
    used ones beyond it, now and on later insertions.  Do not use a limit
    while graphs that captured cached plans are alive."""
    global _plans_limit
    if int(n) < 0:
        raise ValueError("the plan cache limit must be >= 0")
    with _plans_lock:
        _plans_limit = int(n)
        _evict_locked()


def clear_plan_cache() -> None:
    """Close every cached plan (synchronises their devices)."""
    with _plans_lock:
        while _plans:
            _plans.popitem(last=False)[1].close()


def plan_cache_size() -> int:
    with _plans_lock:
        return len(_plans)


def _evict_locked() -> None:
    while _plans_limit and len(_plans) > _plans_limit:
        _plans.popitem(last=False)[1].close()


def matmul_nn(A, B, epilogue=None, stages: int = 6, out=None, out_dtype=None, bias=None,
              **tuning):
    """C = epi(A @ B + bias) on the current CUDA stream, B stored (K, N) row-major.

    The [M, K] @ [K, N] form of the Mosaic GPU pipelining guide's example;
    same arguments and checks as :func:`matmul_nt` otherwise."""
    if B.dim() != 2 or A.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("A must be (M, K) and B (K, N) with the same K")
    return matmul_nt(A, B, epilogue=epilogue, stages=stages, out=out, out_dtype=out_dtype,
                     bias=bias, _b_kn=True, **tuning)


def get_plan(M, N, K, dtype, epilogue=None, stages=4, variant="pipelined", device=0,
             **tuning) -> Plan:
    key = (M, N, K, dtype, epilogue, stages, variant, device, tuple(sorted(tuning.items())))
    with _plans_lock:
        p = _plans.get(key)
        if p is None:
            p = Plan(M, N, K, dtype, epilogue, stages, variant, device, **tuning)
            _plans[key] = p
            _evict_locked()
        else:
            _plans.move_to_end(key)
        return p


def matmul_nt(A, B, epilogue=None, stages: int = 6, variant: str = "pipelined", out=None,
              out_dtype=None, bias=None, **tuning):
    """C = epi(A @ B.T + bias) on the current CUDA stream.

    A: (M, K) and B: (N, K) CUDA tensors of the same dtype (float16 or
    bfloat16), contiguous.  epilogue: None, "gelu" or "relu".  bias: None or
    an (N,) tensor of that dtype, added before the epilogue.  Returns C
    (M, N) of that dtype, or of float32 when out_dtype is torch.float32
    (``out`` if given).  ``tuning`` keywords go to :class:`Plan` (tile_n,
    cta_group, raster_group, max_ctas, tail_split, timeout_ns); plans are
    cached per shape, dtype, epilogue and tuning.
    """
    import torch
    b_kn = bool(tuning.pop("_b_kn", False))
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0 if b_kn else 1]:
        raise ValueError("A must be (M, K) and B (N, K) with the same K")
    if A.dtype != B.dtype:
        raise TypeError("A and B must have the same dtype")
    if not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("A and B must be contiguous")
    if A.device != B.device:
        raise ValueError("A and B must be on the same device")
    dt = _torch_dtype_code(A)
    M, K = A.shape
    N = B.shape[1] if b_kn else B.shape[0]
    if b_kn:
        tuning["b_kn"] = 1
    c_dtype = out_dtype if out_dtype is not None else (out.dtype if out is not None else A.dtype)
    if c_dtype not in (A.dtype, torch.float32):
        raise TypeError("C must have A's dtype or float32")
    if out is None:
        out = torch.empty((M, N), dtype=c_dtype, device=A.device)
    elif out.shape != (M, N) or out.dtype != c_dtype or not out.is_contiguous() or out.device != A.device:
        raise ValueError("out must be a contiguous (M, N) tensor of the output dtype on A's device")
    dtype = "bf16" if dt == GEMM_BF16 else "f16"
    if c_dtype == torch.float32:
        tuning["out_f32"] = 1
    if bias is not None and (not bias.is_cuda or bias.dtype != A.dtype or bias.dim() != 1
                             or bias.shape[0] != N or not bias.is_contiguous()
                             or bias.device != A.device):
        raise ValueError("bias must be a contiguous (N,) CUDA tensor of A's dtype and device")
    plan = get_plan(M, N, K, dtype, epilogue, stages, variant, A.device.index or 0, **tuning)
    plan.run(A, B, out, bias=bias)
    return out
