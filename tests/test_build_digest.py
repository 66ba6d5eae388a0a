"""Host-only checks of the kernel-source digest that keys the committed ncu
traffic figures: it must follow the code and ignore comments and layout."""
from __future__ import annotations

from software_pipelined_tiled_gemm_gb300 import _build


def test_comments_and_blank_lines_do_not_count():
    a = "int f(int x) {  // add one\n  return x + 1;\n}\n"
    b = "/* increment */\nint f(int x) {\n\n    return x + 1;   \n}\n"
    assert _build._code_only(a) == _build._code_only(b)


def test_code_changes_count():
    a = "int f(int x) { return x + 1; }"
    b = "int f(int x) { return x + 2; }"
    assert _build._code_only(a) != _build._code_only(b)


def test_comment_markers_inside_literals_are_kept():
    src = 'asm("mov.u32 %0, 1; // not a comment" : "=r"(r)); char c = \'/\'; // gone\n'
    out = _build._code_only(src)
    assert "// not a comment" in out
    assert "'/'" in out
    assert "gone" not in out


def test_escaped_quote_does_not_end_a_literal():
    src = 'const char* s = "a\\"//b"; /* c */ int y;'
    out = _build._code_only(src)
    assert '"a\\"//b"' in out and "int y;" in out and "c */" not in out


def test_digest_is_stable_and_short():
    d = _build.kernel_digest()
    assert d == _build.kernel_digest() and len(d) == 16


def test_digest_does_not_depend_on_the_checkout_directory(tmp_path):
    # The committed ncu figures are looked up by this digest on whatever
    # machine runs the bench, where the repository sits in another directory.
    import importlib.util
    import shutil
    pkg = tmp_path / "elsewhere" / "software_pipelined_tiled_gemm_gb300"
    shutil.copytree(_build.CSRC, pkg / "csrc")
    shutil.copy(_build.__file__, pkg / "_build.py")
    shutil.copytree(_build.INCLUDE, tmp_path / "elsewhere" / "include")
    spec = importlib.util.spec_from_file_location("moved_build", pkg / "_build.py")
    moved = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(moved)
    assert moved.CSRC != _build.CSRC
    assert moved.kernel_digest() == _build.kernel_digest()
