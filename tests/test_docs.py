"""The README's examples stay true: every package function and C entry point
it names exists, and its C example compiles against include/gemm.h."""
from __future__ import annotations

import os
import re
import shutil
import subprocess

import pytest

import software_pipelined_tiled_gemm_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
README = open(os.path.join(ROOT, "README.md")).read()
HEADER = open(os.path.join(ROOT, "include", "gemm.h")).read()


def test_python_names_in_the_readme_exist():
    names = set(re.findall(r"\bsg\.([A-Za-z_]\w*)", README))
    assert {"matmul_nt", "matmul_nn", "Plan", "describe"} <= names
    for n in names:
        assert hasattr(sg, n), n


def test_c_names_in_the_readme_are_declared():
    names = set(re.findall(r"\b(gemm_[a-z_]+)\s*\(", README)) | set(
        re.findall(r"`(gemm_[a-z_]+)`", README))
    assert {"gemm_plan_create", "gemm_run", "gemm_plan_destroy", "gemm_plan_describe"} <= names
    for n in names:
        assert re.search(r"\b%s\b" % n, HEADER), n


def test_readme_c_example_compiles(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    body = re.search(r"```c\n(.*?)```", README, re.S).group(1)
    includes = [ln for ln in body.splitlines() if ln.startswith("#include")]
    code = [ln for ln in body.splitlines() if not ln.startswith("#include")]
    src = "\n".join(["#include <stdio.h>"] + includes + [
        "int example(int64_t M, int64_t N, int64_t K, const void* dA, const void* dB,",
        "            const void* dBias, void* dC, void* stream) {"] + code +
        ["  return (int)s;", "}"])
    (tmp_path / "ex.c").write_text(src)
    res = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                          os.path.join(ROOT, "include"), "-c", str(tmp_path / "ex.c"), "-o",
                          str(tmp_path / "ex.o")], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
