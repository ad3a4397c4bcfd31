"""Parity of the large-M GEMM (bf16, fp8 per-tensor, mxfp8, mxfp4) with the
oracle.

Small shapes compare every output (ragged M tiles, a half-empty last weight
tile); the pages' shapes (bf16 54560x8192x8192, fp8 4096x4096x8192, MX
4096x16384x7168) run in the dispatch configuration the bench times and
compare 256 seeded full rows.
"""
import numpy as np
import pytest
import torch

import inputs
import mx_gemm_gb300 as fg
import oracle
from tests import parity
from tests.gpu_util import Case, y_to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["bf16", "fp8_tensor", "fp8_block128", "mxfp8", "mxfp4", "mxfp8_b32", "mxfp4_fp8a"])
@pytest.mark.parametrize("M,N,K", [(33, 256, 512), (129, 384, 1024), (300, 512, 2048), (1000, 1280, 1536)])
def test_large_small_shapes(mode, M, N, K):
    c = Case(mode, *inputs.operands(mode, M, N, K, 10 + M, 20 + N, 30 + K))
    plan = fg.gemm_plan(mode, M, N, K)
    assert plan["path"] == 1
    parity.assert_y_close(y_to_f64(c.gemm()), c.ref(), f"{mode} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(300, 512, 640), (129, 384, 1152), (40, 256, 384)])
def test_large_blockscale_ragged_scale_blocks(M, N, K):
    """K/128 not a multiple of 4: the large-M blockscale epilogue reads its
    scale products one by one instead of four at a time."""
    mode = "fp8_block128"
    c = Case(mode, *inputs.operands(mode, M, N, K, 40 + M, 50 + N, 60 + K))
    assert fg.gemm_plan(mode, M, N, K)["path"] == 1
    parity.assert_y_close(y_to_f64(c.gemm()), c.ref(), f"{mode} {M}x{N}x{K}")


def test_large_blockscale_scales_not_16_byte_aligned():
    """A scales that are 4-byte but not 16-byte aligned (a view one float into
    a buffer) take the scalar scale reads; the result is the same."""
    mode, M, N, K = "fp8_block128", 300, 512, 1024
    c = Case(mode, *inputs.operands(mode, M, N, K, 70, 71, 72))
    buf = torch.zeros(M * (K // 128) + 1, dtype=torch.float32, device="cuda")
    a_s = buf[1:].view(M, K // 128)
    a_s.copy_(c.da_s)
    assert a_s.data_ptr() % 16 != 0
    Y = fg.gemm(c.dA, c.pb, a_s)
    assert np.array_equal(y_to_f64(Y), y_to_f64(c.gemm()))
    parity.assert_y_close(y_to_f64(Y), c.ref(), "misaligned A scales")


@pytest.mark.parametrize("mode", ["bf16", "fp8_tensor", "fp8_block128", "mxfp8", "mxfp4", "mxfp8_b32",
                                  "mxfp4_fp8a"])
def test_large_identity_is_bit_exact(mode):
    M, N, K = 300, 512, 1024
    _, B, _, b_s = inputs.operands(mode, 1, N, K, 3, 4, 5)
    A = np.zeros((M, K), np.uint16 if mode == "bf16" else np.uint8)
    one = {"bf16": 0x3F80, "mxfp4": 0x2}.get(mode, 0x38)
    for m in range(M):
        A[m, (3 * m + 1) % K] = one
    a_s = None
    if mode == "fp8_tensor":
        a_s, b_s = np.array([1.0], np.float32), np.array([1.0], np.float32)
    elif mode == "fp8_block128":
        a_s, b_s = np.ones((M, K // 128), np.float32), np.full_like(b_s, 0.5)
    elif mode == "mxfp8":
        a_s = np.full((M, K // 128), 127, np.uint8)
    elif mode == "mxfp4":
        A = inputs.pack_e2m1(A)
        a_s = np.full((M, K // 32), 127, np.uint8)
    elif mode in ("mxfp8_b32", "mxfp4_fp8a"):
        a_s = np.full((M, K // 32), 127, np.uint8)
    c = Case(mode, A, B, a_s, b_s)
    ref = c.ref()
    assert np.array_equal(y_to_f64(c.gemm()), parity.bf16_bits_to_f64(oracle.round_bf16(ref)))


@pytest.mark.parametrize("mode,M,N,K,name,idx", [
    ("fp8_tensor", 4096, 4096, 8192, "large_bf16_54560x8192x8192_fp8_4096x4096x8192", 1),
    ("bf16", 54560, 8192, 8192, "large_bf16_54560x8192x8192_fp8_4096x4096x8192", 0),
    ("mxfp8", 4096, 16384, 7168, "mx_mxfp8_mxfp4_n16384_k7168", 2),
    ("mxfp4", 4096, 16384, 7168, "mx_mxfp8_mxfp4_n16384_k7168", 5),
    ("mxfp4_fp8a", 4096, 16384, 7168, "mx_fp8a_fp4w_n16384_k7168", 2),
    ("mxfp8_b32", 4096, 16384, 7168, "mx_mxfp8_b32_n16384_k7168", 2),
    ("fp8_block128", 4096, 16384, 7168, "large_fp8_block128_4096x16384x7168", 0),
])
def test_large_workload_parity_sampled_rows(mode, M, N, K, name, idx):
    A, B, a_s, b_s = inputs.workload_operands(name, idx)
    c = Case(mode, A, B, a_s, b_s)
    Y = c.gemm()
    rows = inputs.sample_rows(M)
    y = y_to_f64(Y[torch.from_numpy(rows).cuda()])
    ref = c.ref(rows=rows)
    parity.assert_y_close(y, ref, f"{mode} {M}x{N}x{K} sampled rows")
    assert fg.get_error() == fg.FG_OK


@pytest.mark.parametrize("mode", ["bf16", "fp8_tensor"])
@pytest.mark.parametrize("tile,M,N,K", [("128", 2560, 2048, 2048), ("256", 6144, 6144, 1024)])
def test_streamk_tail_matches_whole_tiles(mode, tile, M, N, K, monkeypatch):
    """160 (128 x 256) or 576 (256 x 256) tiles on the GPU's CTAs leave a
    partial wave: with the workspace the tail runs stream-K (tiles split
    between CTAs, fp32 partials passed between them); without it every tile
    runs whole.  Both match the oracle."""
    monkeypatch.setenv("FG_LARGE_TILE", tile)
    assert fg.gemm_plan(mode, M, N, K)["tile_m"] == int(tile)
    c = Case(mode, *inputs.operands(mode, M, N, K, 91, 92, 93))
    need = fg.gemm_workspace_size(mode, M, N, K)
    assert need > 0
    rows = inputs.sample_rows(M)
    ref = c.ref(rows=rows)
    idx = torch.from_numpy(rows).cuda()
    ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
    y_sk = c.gemm(workspace=ws)
    y_whole = c.gemm(workspace=torch.empty(4, dtype=torch.float32, device="cuda"))
    parity.assert_y_close(y_to_f64(y_sk[idx]), ref, f"{mode} stream-K")
    parity.assert_y_close(y_to_f64(y_whole[idx]), ref, f"{mode} whole tiles")
    parity.assert_y_close(y_to_f64(y_sk), y_to_f64(y_whole), f"{mode} stream-K vs whole")
    # a second call with the same workspace (flags from the first call must not be mistaken)
    y_sk2 = c.gemm(workspace=ws)
    assert torch.equal(y_sk.view(torch.int16), y_sk2.view(torch.int16))
    assert fg.get_error() == fg.FG_OK


@pytest.mark.parametrize("mode,M,N,K,streamk", [
    ("fp8_tensor", 2560, 2048, 1024, True),    # stream-K tail: cooperative CTAs that wait on one another
    ("bf16", 300, 512, 1024, False),
    ("mxfp4", 300, 512, 1024, False),
    ("fp8_block128", 300, 512, 1024, False),
])
def test_large_bounded_wait_reports_timeout(mode, M, N, K, streamk):
    """The MMA issuer waits on a barrier nothing arrives at: every wait of the
    large-M kernels runs out after the limit, the kernel drains what it
    started and returns, the host reads FG_ERR_TIMEOUT, and a normal call
    afterwards is correct."""
    c = Case(mode, *inputs.operands(mode, M, N, K, 81, 82, 83))
    assert fg.get_error() == fg.FG_OK
    ws = torch.empty(max(4, fg.gemm_workspace_size(mode, M, N, K)) // 4, dtype=torch.float32, device="cuda")
    assert (fg.gemm_workspace_size(mode, M, N, K) > 0) == (streamk or mode == "mxfp4")
    assert fg.gemm_plan(mode, M, N, K)["path"] == 1
    fg.set_wait_timeout_ns(20_000_000)
    try:
        c.gemm(workspace=ws, flags=fg.FG_FLAG_DEBUG_STALL)
        assert fg.get_error() == fg.FG_ERR_TIMEOUT
    finally:
        fg.set_wait_timeout_ns(4_000_000_000)
    assert fg.get_error() == fg.FG_OK
    rows = inputs.sample_rows(M, n=64)
    y = c.gemm(workspace=ws)
    parity.assert_y_close(y_to_f64(y[torch.from_numpy(rows).cuda()]), c.ref(rows=rows), f"{mode} after timeout")


@pytest.mark.parametrize("mode", ["bf16", "fp8_tensor"])
@pytest.mark.parametrize("M,N,K", [(257, 256, 512), (300, 384, 1024), (1000, 1280, 1536)])
def test_wide_tile_small_shapes(mode, M, N, K, monkeypatch):
    """The 256 x 256 form forced on small shapes: a second 128-row half that
    is partly or wholly past M, a last weight tile with one slab; every
    output against the oracle."""
    monkeypatch.setenv("FG_LARGE_TILE", "256")
    c = Case(mode, *inputs.operands(mode, M, N, K, 40 + M, 50 + N, 60 + K))
    plan = fg.gemm_plan(mode, M, N, K)
    assert plan["path"] == 1 and plan["tile_m"] == 256
    assert fg.gemm_workspace_size(mode, M, N, K) == 0
    parity.assert_y_close(y_to_f64(c.gemm()), c.ref(), f"{mode} {M}x{N}x{K} 256x256")
    assert fg.get_error() == fg.FG_OK


@pytest.mark.parametrize("mode", ["bf16", "fp8_tensor"])
def test_wide_and_narrow_tiles_agree_bit_for_bit(mode, monkeypatch):
    """Both large-M forms accumulate every output over the same K order with
    the same MMA shape: without the stream-K tail their results are the same
    bits.  160 wide tiles on the GPU's CTAs: some CTAs run two tiles, so the
    accumulator hand-over between tiles is exercised."""
    M, N, K = 2560, 4096, 1024
    c = Case(mode, *inputs.operands(mode, M, N, K, 71, 72, 73))
    no_ws = torch.empty(4, dtype=torch.float32, device="cuda")   # too small: no stream-K
    monkeypatch.setenv("FG_LARGE_TILE", "256")
    y_wide = c.gemm(workspace=no_ws)
    monkeypatch.setenv("FG_LARGE_TILE", "128")
    y_narrow = c.gemm(workspace=no_ws)
    assert torch.equal(y_wide.view(torch.int16), y_narrow.view(torch.int16))
    rows = inputs.sample_rows(M, n=64)
    parity.assert_y_close(y_to_f64(y_wide[torch.from_numpy(rows).cuda()]), c.ref(rows=rows), f"{mode} wide")
    assert fg.get_error() == fg.FG_OK


@pytest.mark.parametrize("mode", ["bf16", "fp8_tensor"])
def test_wide_tile_bounded_wait_reports_timeout(mode, monkeypatch):
    monkeypatch.setenv("FG_LARGE_TILE", "256")
    M, N, K = 600, 512, 1024
    c = Case(mode, *inputs.operands(mode, M, N, K, 84, 85, 86))
    assert fg.get_error() == fg.FG_OK
    fg.set_wait_timeout_ns(20_000_000)
    try:
        c.gemm(flags=fg.FG_FLAG_DEBUG_STALL)
        assert fg.get_error() == fg.FG_ERR_TIMEOUT
    finally:
        fg.set_wait_timeout_ns(4_000_000_000)
    assert fg.get_error() == fg.FG_OK
    parity.assert_y_close(y_to_f64(c.gemm()), c.ref(), f"{mode} 256x256 after timeout")


# ------------------------------------------------------ MX on CTA pairs

MX = ["mxfp8", "mxfp4", "mxfp8_b32", "mxfp4_fp8a"]


@pytest.mark.parametrize("mode", MX)
@pytest.mark.parametrize("M,N,K", [(33, 256, 512), (129, 384, 2048), (300, 512, 1024), (1000, 1280, 1536)])
def test_pair_small_shapes(mode, M, N, K, monkeypatch):
    """The CTA-pair form (256 x 256 tiles on two SMs) forced on small shapes:
    an odd CTA whose rows of A lie past M, a weight tile whose second half
    lies past N, several tiles per pair; every output against the oracle."""
    monkeypatch.setenv("FG_LARGE_PAIR", "1")
    plan = fg.gemm_plan(mode, M, N, K)
    assert plan["path"] == 1 and plan["name"].endswith("pair256x256")
    c = Case(mode, *inputs.operands(mode, M, N, K, 110 + M, 120 + N, 130 + K))
    parity.assert_y_close(y_to_f64(c.gemm()), c.ref(), f"{mode} {M}x{N}x{K} pair")
    assert fg.get_error() == fg.FG_OK


@pytest.mark.parametrize("mode", MX)
def test_pair_identity_is_bit_exact(mode, monkeypatch):
    monkeypatch.setenv("FG_LARGE_PAIR", "1")
    M, N, K = 300, 512, 1024
    _, B, _, b_s = inputs.operands(mode, 1, N, K, 3, 4, 5)
    A = np.zeros((M, K), np.uint8)
    for m in range(M):
        A[m, (3 * m + 1) % K] = 0x2 if mode == "mxfp4" else 0x38
    if mode == "mxfp4":
        A = inputs.pack_e2m1(A)
    a_s = np.full((M, K // (128 if mode == "mxfp8" else 32)), 127, np.uint8)
    c = Case(mode, A, B, a_s, b_s)
    ref = c.ref()
    assert np.array_equal(y_to_f64(c.gemm()), parity.bf16_bits_to_f64(oracle.round_bf16(ref)))


@pytest.mark.parametrize("mode", MX)
def test_pair_and_single_cta_forms_agree(mode, monkeypatch):
    """Both large-M MX forms accumulate every output over the same K order
    with MMAs of the same K: the same results within the output bound, and a
    pair tile count that leaves some pairs a second tile."""
    M, N, K = 2304, 2560, 1024        # 9 x 10 pair tiles on 76 pairs
    c = Case(mode, *inputs.operands(mode, M, N, K, 141, 142, 143))
    monkeypatch.setenv("FG_LARGE_PAIR", "1")
    y_pair = c.gemm()
    monkeypatch.setenv("FG_LARGE_PAIR", "0")
    y_one = c.gemm()
    parity.assert_y_close(y_to_f64(y_pair), y_to_f64(y_one), f"{mode} pair vs one-CTA")
    rows = inputs.sample_rows(M, n=64)
    parity.assert_y_close(y_to_f64(y_pair[torch.from_numpy(rows).cuda()]), c.ref(rows=rows), f"{mode} pair")
    assert fg.get_error() == fg.FG_OK


@pytest.mark.parametrize("mode,name,idx", [("mxfp4", "mx_mxfp8_mxfp4_n16384_k7168", 5),
                                           ("mxfp8", "mx_mxfp8_mxfp4_n16384_k7168", 2)])
def test_pair_workload_parity_sampled_rows(mode, name, idx, monkeypatch):
    """The pair form at the pages' MX shape (4096 x 16384 x 7168): 256 seeded
    rows against the oracle."""
    monkeypatch.setenv("FG_LARGE_PAIR", "1")
    A, B, a_s, b_s = inputs.workload_operands(name, idx)
    c = Case(mode, A, B, a_s, b_s)
    assert fg.gemm_plan(mode, 4096, 16384, 7168)["name"].endswith("pair256x256")
    Y = c.gemm()
    rows = inputs.sample_rows(4096)
    parity.assert_y_close(y_to_f64(Y[torch.from_numpy(rows).cuda()]), c.ref(rows=rows), f"{mode} pair workload")
    assert fg.get_error() == fg.FG_OK


@pytest.mark.parametrize("mode", ["mxfp8", "mxfp4"])
def test_pair_bounded_wait_reports_timeout(mode, monkeypatch):
    """The even CTA's MMA issuer waits on a barrier nothing arrives at: both
    CTAs' waits run out, the even CTA completes every stage either producer
    started, the pair releases its memory and returns, the host reads
    FG_ERR_TIMEOUT, and a normal call afterwards is correct."""
    monkeypatch.setenv("FG_LARGE_PAIR", "1")
    M, N, K = 600, 512, 2048
    c = Case(mode, *inputs.operands(mode, M, N, K, 87, 88, 89))
    assert fg.get_error() == fg.FG_OK
    fg.set_wait_timeout_ns(20_000_000)
    try:
        c.gemm(flags=fg.FG_FLAG_DEBUG_STALL)
        assert fg.get_error() == fg.FG_ERR_TIMEOUT
    finally:
        fg.set_wait_timeout_ns(4_000_000_000)
    assert fg.get_error() == fg.FG_OK
    parity.assert_y_close(y_to_f64(c.gemm()), c.ref(), f"{mode} pair after timeout")


@pytest.mark.parametrize("tile", ["128", "256"])
def test_streamk_graph_replay_sees_new_inputs(tile, monkeypatch):
    """A stream-K call captured in a CUDA graph and replayed twice with A
    overwritten in between: the second replay must use its own partials, not
    those the first replay published under the same launch tag."""
    monkeypatch.setenv("FG_LARGE_TILE", tile)
    mode = "fp8_tensor"
    M, N, K = (2560, 2048, 1024) if tile == "128" else (6144, 6144, 1024)
    c = Case(mode, *inputs.operands(mode, M, N, K, 370, 371, 372))
    A2, _, _, _ = inputs.operands(mode, M, N, K, 373, 371, 372)
    need = fg.gemm_workspace_size(mode, M, N, K)
    assert need > 0
    ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    A = c.dA.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        fg.gemm(A, c.pb, c.da_s, Y=Y, workspace=ws)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    A.copy_(torch.from_numpy(A2).cuda())
    g.replay()
    torch.cuda.synchronize()
    rows = inputs.sample_rows(M, n=64)
    c2 = Case(mode, A2, c.B, c.a_s, c.b_s)
    parity.assert_y_close(y_to_f64(Y[torch.from_numpy(rows).cuda()]), c2.ref(rows=rows), f"stream-K {tile} replay")
    assert fg.get_error() == fg.FG_OK
