"""CPU oracle for C = epi(A . B^T) -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg (``bench.py --impl reference`` and the ``cpu_baseline`` field) may import
this package.  The product library never links, loads or calls it, and this
package imports nothing from the product: the two share no code.

The arithmetic lives in ``gemm_oracle.c`` (plain C, fp64 accumulation, OpenMP
over output rows).  This wrapper only marshals numpy arrays through ctypes.

Definitions followed (see the C file for the full statement):
  * TileLang tutorial ch. 11, "pipelined_gemm.py", matmul_auto: A (M,K),
    B (N,K), C (M,N), ``T.gemm(..., transpose_B=True)``, fp32 accumulator.
  * ReLU, max(x, 0), the clamp of the Triton lecture notes' matmul example.
  * tanh-GELU as written in the Triton lecture notes ("GeLU") and the
    XLA:GPU emitters page (loop-emitter example, ``@gelu``), constant
    sqrt(2/pi) = 0.7978845608.
  * Bias (no page defines one; the reading is a Linear layer's): one value
    per output column, added to the exact sum before the epilogue.

Every function here has a pin in ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F16 = 0
BF16 = 1
_DTYPES = {"f16": F16, "fp16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16}

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = _open(build())
        return _lib


def _open(path):
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_gemm_nt.argtypes = [u16p, u16p, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                   f64p, ctypes.c_int]
    lib.oracle_gemm_nt.restype = ctypes.c_int
    lib.oracle_gemm_nt_entries.argtypes = [u16p, u16p, i64, i64, i64, ctypes.c_int,
                                           ctypes.c_int, i64p, i64p, i64, f64p, ctypes.c_int]
    lib.oracle_gemm_nt_entries.restype = ctypes.c_int
    lib.oracle_gemm_nt_bias.argtypes = [u16p, u16p, u16p, i64, i64, i64, ctypes.c_int,
                                        ctypes.c_int, f64p, ctypes.c_int]
    lib.oracle_gemm_nt_bias.restype = ctypes.c_int
    lib.oracle_gemm_nt_entries_bias.argtypes = [u16p, u16p, u16p, i64, i64, i64, ctypes.c_int,
                                                ctypes.c_int, i64p, i64p, i64, f64p,
                                                ctypes.c_int]
    lib.oracle_gemm_nt_entries_bias.restype = ctypes.c_int
    lib.oracle_decode_array.argtypes = [u16p, i64, ctypes.c_int, f64p]
    lib.oracle_decode_array.restype = None
    lib.oracle_round_array.argtypes = [f64p, i64, ctypes.c_int, u16p]
    lib.oracle_round_array.restype = None
    lib.oracle_gelu_array.argtypes = [f64p, i64, f64p]
    lib.oracle_gelu_array.restype = None
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


class use_library:
    """Context manager: route this module's calls through another build of the
    oracle (the mutation tests use it to check that the pins catch planted
    mistakes)."""

    def __init__(self, path):
        self._path = path
        self._saved = None

    def __enter__(self):
        global _lib
        _load()
        with _lock:
            self._saved = _lib
            _lib = _open(self._path)
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self._saved
        return False


_EPI = {None: 0, "none": 0, 0: 0, "gelu": 1, "gelu_tanh": 1, 1: 1, "relu": 2, 2: 2}


def _epi(epilogue) -> int:
    return _EPI[epilogue]


def _dt(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    return _DTYPES[str(dtype).replace("torch.", "")]


def _u16(a) -> np.ndarray:
    """Accept a uint16 bit-pattern array, a numpy float16 array or a CPU torch
    tensor of float16/bfloat16, and return contiguous uint16 bit patterns."""
    if hasattr(a, "detach"):  # torch tensor: reinterpret the storage bits
        import torch
        t = a.detach().cpu().contiguous()
        if t.dtype in (torch.float16, torch.bfloat16):
            t = t.view(torch.int16)
        return np.ascontiguousarray(t.numpy().view(np.uint16))
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("expected uint16 bit patterns, float16 or a torch half tensor")
    return np.ascontiguousarray(a)


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _bias(bias, N):
    """Bias bit patterns (N values) as a uint16 array and its pointer, or None."""
    if bias is None:
        return None, None
    v = _u16(bias).reshape(-1)
    if v.size != N:
        raise ValueError("bias must have N = %d values" % N)
    return v, _ptr(v, ctypes.c_uint16)


def gemm_nt(A, B, dtype, epilogue=None, threads: int = 0, bias=None) -> np.ndarray:
    """fp64 C[i,j] = epi(sum_k A[i,k] B[j,k] + bias[j]); A (M,K), B (N,K) and
    bias (N values, optional) as bit patterns."""
    lib = _load()
    a, b = _u16(A), _u16(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError("A must be (M,K) and B (N,K)")
    M, K = a.shape
    N = b.shape[0]
    bias_bits, bp = _bias(bias, N)  # keep the array alive across the call
    C = np.zeros((M, N), dtype=np.float64)
    rc = lib.oracle_gemm_nt_bias(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16), bp, M, N, K,
                                 _dt(dtype), _epi(epilogue), _ptr(C, ctypes.c_double),
                                 int(threads))
    if rc != 0:
        raise RuntimeError("oracle_gemm_nt failed")
    return C


def gemm_nt_entries(A, B, dtype, rows, cols, epilogue=None, threads: int = 0,
                    bias=None) -> np.ndarray:
    """The same definition at chosen (row, col) positions only."""
    lib = _load()
    a, b = _u16(A), _u16(B)
    M, K = a.shape
    N = b.shape[0]
    bias_bits, bp = _bias(bias, N)  # keep the array alive across the call
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    if r.shape != c.shape:
        raise ValueError("rows and cols must have the same shape")
    out = np.zeros(r.shape, dtype=np.float64)
    rc = lib.oracle_gemm_nt_entries_bias(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16), bp,
                                         M, N, K, _dt(dtype), _epi(epilogue),
                                         _ptr(r, ctypes.c_int64), _ptr(c, ctypes.c_int64), r.size,
                                         _ptr(out, ctypes.c_double), int(threads))
    if rc != 0:
        raise RuntimeError("oracle_gemm_nt_entries failed (index out of range?)")
    return out


def decode(bits, dtype) -> np.ndarray:
    """Exact value of each fp16/bf16 bit pattern, as float64."""
    lib = _load()
    a = _u16(bits)
    out = np.empty(a.shape, dtype=np.float64)
    lib.oracle_decode_array(_ptr(a, ctypes.c_uint16), a.size, _dt(dtype), _ptr(out, ctypes.c_double))
    return out


def round_to(x, dtype) -> np.ndarray:
    """Round-to-nearest-even from float64 to fp16/bf16; returns uint16 bit patterns."""
    lib = _load()
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(a.shape, dtype=np.uint16)
    lib.oracle_round_array(_ptr(a, ctypes.c_double), a.size, _dt(dtype), _ptr(out, ctypes.c_uint16))
    return out


def gelu_tanh(x) -> np.ndarray:
    """tanh-GELU in float64."""
    lib = _load()
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(a.shape, dtype=np.float64)
    lib.oracle_gelu_array(_ptr(a, ctypes.c_double), a.size, _ptr(out, ctypes.c_double))
    return out
