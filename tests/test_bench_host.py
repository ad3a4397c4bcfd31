"""Host-side pieces of bench.py that need no GPU: the code-only source digest
that ties the stored ncu traffic figure to the kernels it was measured on."""
import os
import shutil

import bench


def test_code_only_drops_comments_and_whitespace_keeps_strings():
    src = 'int a = 1;  // note "x"\n/* block\n // */ const char* s = "a // b /* c */";\n  f( x ,y );\n'
    assert bench._code_only(src) == 'inta=1;constchar*s="a // b /* c */";f(x,y);'


def _digest_of(tmp_path, edit=None):
    """Digest of a copy of the library sources, optionally edited."""
    import mx_gemm_gb300 as fg
    pkg = tmp_path / "pkg"
    csrc = pkg / "csrc"
    shutil.copytree(os.path.join(os.path.dirname(fg.__file__), "csrc"), csrc)
    (pkg / "__init__.py").write_text("")
    if edit:
        name, old, new = edit
        p = csrc / name
        text = p.read_text()
        assert old in text
        p.write_text(text.replace(old, new, 1))

    class Fake:
        __file__ = str(pkg / "__init__.py")

    return bench.kernel_sources_digest(Fake)


def test_digest_ignores_comment_edits_and_sees_code_edits(tmp_path):
    import mx_gemm_gb300 as fg
    base = bench.kernel_sources_digest(fg)
    assert _digest_of(tmp_path / "a") == base
    # a comment reworded and re-indented: same code, same digest
    assert _digest_of(tmp_path / "b", ("fg_decode.cu", "// Split-K decode GEMM", "//   Split-K  decode  GEMM")) == base
    # one constant changed: a different kernel, a different digest
    assert _digest_of(tmp_path / "c", ("fg_decode.cu", "constexpr int kSlabBytes = 16384;",
                                       "constexpr int kSlabBytes = 32768;")) != base
    # a change inside a string literal (inline PTX) also counts
    assert _digest_of(tmp_path / "d", ("fg_ptx.cuh", "tcgen05.commit.cta_group::1",
                                       "tcgen05.commit.cta_group::2")) != base
