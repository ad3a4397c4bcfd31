"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function include/fg.h declares, and
reject bad arguments on the host before touching a device.
"""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "fg.h")


@pytest.fixture(scope="module")
def fg():
    from mx_gemm_gb300 import build
    build.build()
    import mx_gemm_gb300
    return mx_gemm_gb300


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FG_API\s+[\w\s\*]+?\b(fg_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("fg_preshuffle_b", "fg_gemm", "fg_gemm_splitk_reduce", "fg_unshuffle_b", "fg_get_error"):
        assert want in names


def test_library_exports_every_declared_symbol(fg):
    L = fg.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    # and ELF-level: each is a defined dynamic symbol
    lib = ctypes.CDLL(fg.LIB_PATH)
    for name in declared_functions():
        ctypes.cast(getattr(lib, name), ctypes.c_void_p)


def test_version_and_status_names(fg):
    assert fg.version() >= 100
    for i, s in enumerate(fg.STATUS):
        assert fg.status_str(i) == s
    assert fg.status_str(99) == "FG_ERR_UNKNOWN"


@pytest.mark.parametrize("mode,N,K,b,sf", [
    ("bf16", 256, 64, 256 * 128, 0),
    ("fp8_tensor", 2048, 7168, 2048 * 7168, 16),
    ("fp8_block128", 16384, 7168, 16384 * 7168, 128 * 56 * 4),
    ("mxfp8", 16384, 7168, 16384 * 7168, 128 * 14 * 512),
    ("mxfp8", 256, 640, 256 * 640, 2 * 2 * 512),
    ("mxfp4", 16384, 7168, 16384 * 3584, 128 * 28 * 1024),
    ("mxfp8_b32", 16384, 7168, 16384 * 7168, 128 * 56 * 512),
    ("mxfp4_fp8a", 16384, 7168, 16384 * 3584, 128 * 56 * 512),
    ("mxfp4_fp8a", 256, 384, 256 * 192, 2 * 3 * 512),
])
def test_preshuffle_sizes(fg, mode, N, K, b, sf):
    assert fg.preshuffle_b_size(mode, N, K) == (b, sf)


@pytest.mark.parametrize("mode,N,K", [
    ("fp8_tensor", 100, 128), ("fp8_tensor", 128, 100), ("fp8_block128", 128, 64),
    ("mxfp4", 128, 128), ("bf16", 128, 32), ("mxfp8", 0, 128),
])
def test_bad_shapes_rejected(fg, mode, N, K):
    with pytest.raises(fg.FgError) as e:
        fg.preshuffle_b_size(mode, N, K)
    assert e.value.status == fg.FG_ERR_SHAPE
    assert "K=" in fg.last_error_message() or "N=" in fg.last_error_message()


def test_bad_mode_rejected(fg):
    with pytest.raises(fg.FgError) as e:
        fg.preshuffle_b_size(7, 128, 128)
    assert e.value.status == fg.FG_ERR_INVALID_ARG


def test_plan_heuristic_and_table(fg):
    p = fg.gemm_plan("fp8_tensor", 1, 2048, 7168)
    assert p["path"] == 0 and p["split_k"] == 8 and p["from_table"]
    p = fg.gemm_plan("fp8_tensor", 1, 16384, 7168)
    assert p["split_k"] == 2 and p["ctas"] == 256 and p["from_table"]
    p = fg.gemm_plan("fp8_tensor", 16, 16384, 7168)
    assert p["split_k"] == 2 and (p["stage_slabs"], p["stages"]) == (2, 3) and p["from_table"]
    p = fg.gemm_plan("fp8_tensor", 8, 4096, 4096)          # heuristic: >= 1.5 CTAs per SM
    assert not p["from_table"] and p["ctas"] >= 1.5 * 148
    # heuristic pipeline: 1 x 5 (two fp8 CTAs to an SM) when the grid needs one
    # to two CTAs per SM and each streams >= 12 slabs, 1 x 4 otherwise
    for mode, M, N, K, cfg in [("fp8_tensor", 16, 8192, 7168, (1, 5)), ("fp8_block128", 1, 8192, 7168, (1, 5)),
                               ("fp8_tensor", 1, 12288, 5120, (1, 4)), ("fp8_tensor", 1, 4096, 4096, (1, 4)),
                               ("fp8_tensor", 16, 16384, 2048, (1, 4)), ("mxfp8", 16, 8192, 7168, (1, 4)),
                               ("fp8_tensor", 20, 8192, 7168, (1, 4))]:
        p = fg.gemm_plan(mode, M, N, K)
        assert not p["from_table"] and (p["stage_slabs"], p["stages"]) == cfg, (mode, M, N, K, p)
    p = fg.gemm_plan("fp8_tensor", 1, 2048, 7168, split_k=4)   # the row for an explicit split of 4
    assert p["split_k"] == 4 and p["from_table"] and (p["stage_slabs"], p["stages"]) == (2, 5)
    p = fg.gemm_plan("fp8_tensor", 1, 2048, 7168, split_k=2)   # a split no row has: the heuristic pipeline
    assert p["split_k"] == 2 and not p["from_table"] and (p["stage_slabs"], p["stages"]) == (1, 4)
    p = fg.gemm_plan("fp8_tensor", 1, 2048, 7168, split_k=8)   # the row's own split
    assert p["from_table"] and (p["stage_slabs"], p["stages"]) == (2, 3)
    assert "sm103a" in p["name"] and "n2048" in p["name"] and "k7168" in p["name"]
    with pytest.raises(fg.FgError) as e:
        fg.gemm_plan("fp8_tensor", 1, 256, 256, split_k=4)  # only 2 slabs
    assert e.value.status == fg.FG_ERR_SHAPE
    with pytest.raises(fg.FgError):
        fg.gemm_plan("fp8_tensor", 1, 256, 7168, split_k=17)
    # splits up to 8 reduce inside a cluster (no workspace); larger ones need one
    assert fg.gemm_workspace_size("fp8_tensor", 1, 2048, 7168, 4) == 0
    assert fg.gemm_workspace_size("fp8_tensor", 3, 2048, 7168, 16) == 16 * 3 * 2048 * 4
    assert fg.gemm_workspace_size("fp8_tensor", 1, 16384, 7168, 1) == 0
    # large-M MX needs room for the per-call A scale image (and nothing more:
    # fp8 x fp4 reads its packed weights directly)
    assert fg.gemm_workspace_size("mxfp4", 4096, 16384, 7168) == 32 * 28 * 2 * 512
    assert fg.gemm_workspace_size("mxfp4_fp8a", 4096, 16384, 7168) == 32 * 56 * 512


def _fake_desc(fg, mode=1, N=128, K=128):
    d = fg.BShuf()
    d.magic, d.version, d.mode, d.tile_rows, d.N, d.K = 0x31424746, 1, mode, 128, N, K
    d.data, d.sf, d.data_bytes, d.sf_bytes, d.check = 16, 16, N * K, 16, 12345
    return d


def test_gemm_rejects_handmade_descriptor(fg):
    """A descriptor not produced by fg_preshuffle_b (e.g. raw or re-shuffled
    weights) is refused before any launch."""
    L = fg.lib()
    d = _fake_desc(fg)
    rc = L.fg_gemm(ctypes.c_void_p(256), ctypes.c_void_p(256), 1, ctypes.byref(d), 1, 1,
                   ctypes.c_void_p(256), None, 0, 0, None)
    assert rc == fg.FG_ERR_LAYOUT
    rc = L.fg_gemm(ctypes.c_void_p(256), ctypes.c_void_p(256), 1, None, 1, 1,
                   ctypes.c_void_p(256), None, 0, 0, None)
    assert rc == fg.FG_ERR_INVALID_ARG
    rc = L.fg_unshuffle_b(ctypes.byref(d), ctypes.c_void_p(256), None, None)
    assert rc == fg.FG_ERR_LAYOUT


def test_preshuffle_argument_checks(fg):
    L = fg.lib()
    out = fg.BShuf()
    # bf16 takes no scales
    rc = L.fg_preshuffle_b(0, ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21), 128, 64,
                           ctypes.c_void_p(1 << 22), 128 * 128, None, 0, ctypes.byref(out), None)
    assert rc == fg.FG_ERR_INVALID_ARG
    # misaligned B
    rc = L.fg_preshuffle_b(1, ctypes.c_void_p((1 << 20) + 8), ctypes.c_void_p(1 << 21), 128, 128,
                           ctypes.c_void_p(1 << 22), 128 * 128, ctypes.c_void_p(1 << 23), 16,
                           ctypes.byref(out), None)
    assert rc == fg.FG_ERR_ALIGN
    # the fp4 image of fp8 x fp4 is read by a tensor copy that needs 32 bytes
    rc = L.fg_preshuffle_b(fg.FG_MXFP4_FP8A, ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21), 128, 128,
                           ctypes.c_void_p((1 << 22) + 16), 128 * 64, ctypes.c_void_p(1 << 23), 512,
                           ctypes.byref(out), None)
    assert rc == fg.FG_ERR_ALIGN
    # image too small
    rc = L.fg_preshuffle_b(1, ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21), 128, 128,
                           ctypes.c_void_p(1 << 22), 100, ctypes.c_void_p(1 << 23), 16,
                           ctypes.byref(out), None)
    assert rc == fg.FG_ERR_WORKSPACE
    # overlapping B and image
    rc = L.fg_preshuffle_b(1, ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21), 128, 128,
                           ctypes.c_void_p((1 << 20) + 4096), 128 * 128, ctypes.c_void_p(1 << 23), 16,
                           ctypes.byref(out), None)
    assert rc == fg.FG_ERR_INVALID_ARG


def test_reduce_argument_checks(fg):
    L = fg.lib()
    p = ctypes.c_void_p(1 << 20)
    assert L.fg_gemm_splitk_reduce(None, 2, 1, 128, None, None, p, None) == fg.FG_ERR_INVALID_ARG
    assert L.fg_gemm_splitk_reduce(p, 0, 1, 128, None, None, p, None) == fg.FG_ERR_SHAPE
    assert L.fg_gemm_splitk_reduce(p, 2, 1, 100, None, None, p, None) == fg.FG_ERR_SHAPE
    assert L.fg_gemm_splitk_reduce(p, 2, 1, 128, p, None, p, None) == fg.FG_ERR_INVALID_ARG
    assert L.fg_gemm_splitk_reduce(ctypes.c_void_p((1 << 20) + 4), 2, 1, 128, None, None, p,
                                   None) == fg.FG_ERR_ALIGN
    # M == 0 is a no-op that touches nothing
    assert L.fg_gemm_splitk_reduce(p, 2, 0, 128, None, None, p, None) == fg.FG_OK


def test_product_path_has_no_oracle_dependency():
    """The library sources and binding never reference the oracle."""
    pkg = os.path.join(ROOT, "mx_gemm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "orc_" not in text, f


def test_decode_config_override_is_validated(fg, monkeypatch):
    monkeypatch.setenv("FG_DECODE_CONFIG", "1,4")
    p = fg.gemm_plan("fp8_tensor", 1, 2048, 7168)
    assert (p["stage_slabs"], p["stages"]) == (1, 4)
    for bad in ("3,3", "1", "x,y", "1,4,5", "2,5z"):
        monkeypatch.setenv("FG_DECODE_CONFIG", bad)
        with pytest.raises(fg.FgError) as e:
            fg.gemm_plan("fp8_tensor", 1, 2048, 7168)
        assert e.value.status == fg.FG_ERR_INVALID_ARG


def test_binding_refuses_views_and_host_tensors(fg):
    """The binding hands raw pointers to the C ABI, so it refuses tensors the
    library would misread: a transposed or column-sliced view, a host
    tensor, a tensor of another element type (checks only, no arithmetic)."""
    import torch
    desc = fg.BShuf()
    desc.mode, desc.N, desc.K = fg.FG_FP8_TENSOR, 256, 128
    pb = fg.PreshuffledB(desc, torch.empty(0, dtype=torch.uint8), None)
    A = torch.zeros(128, 4, dtype=torch.uint8)
    with pytest.raises(ValueError, match="contiguous"):
        fg.gemm(A.t(), pb)                       # transposed [4][128] view
    with pytest.raises(ValueError, match="contiguous"):
        fg.gemm(torch.zeros(4, 256, dtype=torch.uint8)[:, :128], pb)
    with pytest.raises(ValueError, match="CUDA"):
        fg.gemm(torch.zeros(4, 128, dtype=torch.uint8), pb)
    with pytest.raises(ValueError, match="contiguous"):
        fg.preshuffle_b("fp8_tensor", torch.zeros(128, 256, dtype=torch.uint8).t())
    with pytest.raises(ValueError, match="CUDA"):
        fg.preshuffle_b("fp8_tensor", torch.zeros(256, 128, dtype=torch.uint8))
    with pytest.raises(ValueError, match="Y"):
        fg.gemm_noalloc(torch.zeros(4, 128, dtype=torch.uint8), pb, None)
    with pytest.raises(ValueError, match="contiguous"):
        fg.gemm_splitk_reduce(torch.zeros(8, 4).t(), 1, 4, 8)
