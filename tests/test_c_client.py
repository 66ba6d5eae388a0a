"""The C ABI from plain C: include/gemm.h compiles as strict C99, a C program
links the shared library with nothing else, the structs it sees have the
layout the Python binding's ctypes mirrors assume, and (on a GPU) a GEMM run
from C through host buffers matches the oracle bit for bit."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import gemm_inputs
import oracle
import software_pipelined_tiled_gemm_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE = os.path.join(ROOT, "tests", "c_client", "abi_client.c")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = sg.library_path()
    if not os.path.exists(lib):
        sg.load_library()          # raises with the build instructions
    exe = str(tmp_path_factory.mktemp("c_client") / "abi_client")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), SOURCE, lib,
           "-Wl,-rpath," + os.path.dirname(lib), "-o", exe]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def _layout(exe):
    res = subprocess.run([exe, "layout"], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr
    out = {}
    for line in res.stdout.splitlines():
        key, _, rest = line.partition(" ")
        if key in ("offset", "sizeof"):
            name, value = rest.rsplit(" ", 1)
            out[(key, name)] = int(value)
        else:
            out[key] = rest
    return out


def test_c_program_sees_the_documented_host_behaviour(client):
    got = _layout(client)
    assert got["version"] == sg.gemm_version()
    assert got["status_ok"] == "GEMM_OK"
    assert got["status_timeout"] == "GEMM_ERR_TIMEOUT"
    assert int(got["smem"]) == 4 * (128 * 64 + 256 * 64) * 2
    # rejected before any CUDA call, with *out reset to NULL
    assert got["bad_m"] == "%d 1" % sg.GEMM_ERR_INVALID_ARG
    assert got["bad_stages"] == "%d 1" % sg.GEMM_ERR_INVALID_ARG
    assert got["destroy_null"] == "ok"
    assert got["wait_mma_full"] == sg.gemm_wait_detail_string((2 << 16) | 2)


@pytest.mark.parametrize("tag,mirror", [("tuning", sg.GemmTuning), ("info", sg.GemmPlanInfo),
                                        ("device", sg.GemmDeviceDesc)])
def test_struct_layout_matches_the_ctypes_mirror(client, tag, mirror):
    got = _layout(client)
    assert got[("sizeof", tag)] == ctypes.sizeof(mirror)
    c_fields = {key[1].split(".", 1)[1]: off for key, off in got.items()
                if isinstance(key, tuple) and key[0] == "offset" and key[1].startswith(tag + ".")}
    py_fields = {name: getattr(mirror, name).offset for name, _ in mirror._fields_}
    assert c_fields == py_fields


def _write(path, t):
    import torch
    t.contiguous().view(torch.int16).numpy().tofile(path)


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,dtype,epi,span", [
    (200, 136, 264, "f16", None, 3),      # partial tiles in M and N, 4 full K slices + a tail
    (129, 300, 257, "bf16", "relu", 1),   # K pitch not 16-byte aligned: padded staging
])
def test_c_program_runs_a_gemm_from_host_buffers(client, tmp_path, M, N, K, dtype, epi, span):
    # integers small enough that every sum is exact in fp32 and in the output type
    A, B = gemm_inputs.custom(M, N, K, dtype=dtype, dist="int", seed=M + N + K, lo=-span,
                              hi=span)
    a, b, c = (str(tmp_path / n) for n in ("a.bin", "b.bin", "c.bin"))
    _write(a, A)
    _write(b, B)
    code = {None: sg.GEMM_EPI_NONE, "relu": sg.GEMM_EPI_RELU}[epi]
    res = subprocess.run([client, "run", str(M), str(N), str(K),
                          str(1 if dtype == "bf16" else 0), str(code), a, b, c],
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    got = np.fromfile(c, dtype=np.uint16).reshape(M, N)
    ref = oracle.gemm_nt(A, B, dtype, epilogue=epi)
    assert np.all(np.abs(ref) < (2048 if dtype == "f16" else 256))   # exact in the output type
    want = oracle.round_to(ref, dtype)
    mism = np.argwhere(want != got)
    assert mism.size == 0, "first mismatch at %s" % (mism[0],)
