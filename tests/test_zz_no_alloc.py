"""fg_gemm_noalloc, called through the C ABI, against fg_gemm.

fg_gemm_noalloc serves callers that cannot allocate device memory while they
run (a serving loop with every buffer sized at start-up, or a plug-in whose
host framework owns all device memory): whatever fg_gemm would keep in a
caller workspace goes to the library's own 8 MiB device array instead.  These
cases make the kernels write and read that array -- the fp32 partials of
splits above 8, the A scale image of the large-M MX kernel -- plus a large-M
bf16 shape whose optional stream-K buffer does not fit (it must run with
whole tiles, not be refused).  Each output must match fg_gemm's with a caller
workspace (same kernels, same split: the same bits) and lie within the output
bound the other tests use, on consecutive calls with other inputs and shapes
(so stale scratch contents from an earlier call cannot leak in).  Calls that
need more than the array holds must be refused before anything is launched.

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import inputs
import mx_gemm_gb300 as fg
from tests import parity
from tests.gpu_util import Case, dev, y_to_f64

pytestmark = pytest.mark.gpu

SCRATCH = 8 << 20


def _noalloc(c, split_k, Y, A=None, a_s=None, M=None):
    """One fg_gemm_noalloc call through the C ABI (ctypes, no binding logic)."""
    L = fg.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    A = c.dA if A is None else A
    a_s = c.da_s if a_s is None else a_s
    return L.fg_gemm_noalloc(ctypes.c_void_p(A.data_ptr()), None if a_s is None else ctypes.c_void_p(a_s.data_ptr()),
                             c.M if M is None else M, ctypes.byref(c.pb.desc), fg.MODES[c.mode], split_k,
                             ctypes.c_void_p(Y.data_ptr()), 0, stream)


def _check_against_fg_gemm(c, S, what, workspace=None):
    Y = torch.full((c.M, c.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = _noalloc(c, S, Y)
    assert rc == fg.FG_OK, fg.last_error_message()
    torch.cuda.synchronize()
    y_ref = c.gemm(split_k=S, workspace=workspace)
    parity.assert_y_close(y_to_f64(Y), y_to_f64(y_ref), what)
    assert torch.equal(Y.view(torch.int16), y_ref.view(torch.int16)), what + ": not the same bits as fg_gemm"
    return Y


def test_noalloc_split_partials_in_scratch_on_consecutive_calls():
    """Splits of 12 and 16 keep their fp32 partials in the scratch (the
    two-pass path): three calls in a row, the third repeating the first
    shape with other inputs after a different shape overwrote part of the
    array."""
    calls = [("fp8_tensor", 16, 2048, 7168, 16, 500),    # 2 MiB of partials
             ("mxfp4", 1, 16384, 7168, 12, 510),         # 768 KiB
             ("fp8_tensor", 16, 2048, 7168, 16, 520)]    # same shape, other inputs
    for i, (mode, M, N, K, S, seed) in enumerate(calls):
        assert 8 < S and S * M * N * 4 <= SCRATCH
        assert fg.gemm_workspace_size(mode, M, N, K, S) == S * M * N * 4
        c = Case(mode, *inputs.operands(mode, M, N, K, seed, seed + 1, seed + 2))
        Y = _check_against_fg_gemm(c, S, f"no-alloc call {i + 1} ({mode} {M}x{N}x{K} S={S})")
        parity.assert_y_close(y_to_f64(Y), c.ref(), f"no-alloc call {i + 1} vs oracle")
    assert fg.get_error() == fg.FG_OK


def test_noalloc_large_mx_scale_image_in_scratch():
    """Large-M MX calls relay A's scales into the scratch every call: two
    calls of different modes and shapes, then the pages' mxfp4 shape."""
    for i, (mode, M, N, K) in enumerate([("mxfp4", 300, 512, 1024), ("mxfp8_b32", 129, 384, 2048),
                                        ("mxfp8", 1000, 1280, 1536)]):
        assert fg.gemm_plan(mode, M, N, K)["path"] == 1
        need = fg.gemm_workspace_size(mode, M, N, K)
        assert 0 < need <= SCRATCH
        c = Case(mode, *inputs.operands(mode, M, N, K, 530 + i, 540 + i, 550 + i))
        Y = _check_against_fg_gemm(c, 0, f"no-alloc large {mode} {M}x{N}x{K}")
        parity.assert_y_close(y_to_f64(Y), c.ref(), f"no-alloc large {mode} vs oracle")
    A, B, a_s, b_s = inputs.workload_operands("mx_mxfp8_mxfp4_n16384_k7168", 5)   # mxfp4 4096x16384x7168
    c = Case("mxfp4", A, B, a_s, b_s)
    Y = _check_against_fg_gemm(c, 0, "no-alloc large mxfp4 4096x16384x7168")
    rows = inputs.sample_rows(4096, n=32)
    parity.assert_y_close(y_to_f64(Y[torch.from_numpy(rows).cuda()]), c.ref(rows=rows), "mxfp4 4096 rows")
    assert fg.get_error() == fg.FG_OK


@pytest.mark.parametrize("mode", ["bf16", "fp8_tensor"])
def test_noalloc_large_partial_wave_runs_whole_tiles(mode):
    """160 tiles of 128 x 256 on the GPU's CTAs leave a partial last wave;
    the optional stream-K buffer (about 128 KiB per CTA) does not fit the
    scratch, so the call runs every tile whole -- the same bits as fg_gemm
    with too small a workspace -- and stays within the bound of fg_gemm's
    stream-K result."""
    M, N, K = 2560, 2048, 2048
    plan = fg.gemm_plan(mode, M, N, K)
    assert plan["path"] == 1 and plan["tile_m"] == 128
    assert fg.gemm_workspace_size(mode, M, N, K) > SCRATCH
    c = Case(mode, *inputs.operands(mode, M, N, K, 561, 562, 563))
    no_ws = torch.empty(4, dtype=torch.float32, device="cuda")
    Y = _check_against_fg_gemm(c, 0, f"no-alloc {mode} {M}x{N}x{K}", workspace=no_ws)
    parity.assert_y_close(y_to_f64(Y), y_to_f64(c.gemm()), f"no-alloc {mode} vs stream-K")
    rows = inputs.sample_rows(M, n=64)
    parity.assert_y_close(y_to_f64(Y[torch.from_numpy(rows).cuda()]), c.ref(rows=rows), f"{mode} vs oracle")
    assert fg.get_error() == fg.FG_OK


def test_noalloc_refuses_what_does_not_fit_and_launches_nothing():
    mode, M, N, K = "fp8_tensor", 16, 16384, 7168
    c = Case(mode, *inputs.operands(mode, M, N, K, 801, 802, 803))
    Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    rc = _noalloc(c, 16, Y)         # 16 * 16 * 16384 * 4 bytes = 16 MiB > 8 MiB
    assert rc == fg.FG_ERR_WORKSPACE
    assert "partials" in fg.last_error_message() and "scratch" in fg.last_error_message()
    # a large-M MX call whose A scale image is above the limit (224 bytes per
    # row of A for mxfp4 at K = 7168): refused before any launch, so the
    # operand contents do not matter
    Nb, Kb, Mbig = 128, 7168, 40000
    _, B, _, b_s = inputs.operands("mxfp4", 1, Nb, Kb, 804, 805, 806)
    big = Case.__new__(Case)
    big.mode, big.M, big.N, big.K = "mxfp4", Mbig, Nb, Kb
    big.pb = fg.preshuffle_b("mxfp4", dev(B), dev(b_s), K=Kb)
    assert fg.gemm_workspace_size("mxfp4", Mbig, Nb, Kb) > SCRATCH
    A_big = torch.zeros((Mbig, Kb // 2), dtype=torch.uint8, device="cuda")
    s_big = torch.zeros((Mbig, Kb // 32), dtype=torch.uint8, device="cuda")
    Y_big = torch.zeros((Mbig, Nb), dtype=torch.bfloat16, device="cuda")
    rc = _noalloc(big, 0, Y_big, A=A_big, a_s=s_big, M=Mbig)
    assert rc == fg.FG_ERR_WORKSPACE
    assert "scale image" in fg.last_error_message()
    # deferring the reduce would leave the partials in the private scratch
    L = fg.lib()
    rc = L.fg_gemm_noalloc(ctypes.c_void_p(c.dA.data_ptr()), ctypes.c_void_p(c.da_s.data_ptr()), M,
                           ctypes.byref(c.pb.desc), fg.MODES[mode], 2, ctypes.c_void_p(Y.data_ptr()),
                           fg.FG_FLAG_DEFER_REDUCE, None)
    assert rc == fg.FG_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert not Y.any() and not Y_big.any()       # nothing was launched
    rc = _noalloc(c, 2, Y)                       # split 2 reduces in a cluster: no scratch
    assert rc == fg.FG_OK
    parity.assert_y_close(y_to_f64(Y), c.ref(), "no-alloc within the limit")
    assert np.isfinite(y_to_f64(Y)).all()
    assert fg.get_error() == fg.FG_OK
