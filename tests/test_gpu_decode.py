"""Parity of the split-K decode GEMM (all scale modes) with the oracle.

Bounds: fp32 workspace |ws - ref| <= 1e-5 |ref| + 1e-6 rms(ref); bf16 Y
|y - ref| <= 2e-2 rms(ref) per element; closed forms bit-exact.
"""
import numpy as np
import pytest
import torch

import inputs
import mx_gemm_gb300 as fg
import oracle
from tests import parity
from tests.gpu_util import Case, dev, host, y_to_f64

pytestmark = pytest.mark.gpu

MODES = ["bf16", "fp8_tensor", "fp8_block128", "mxfp8", "mxfp4", "mxfp8_b32", "mxfp4_fp8a"]


def _slabs(mode, K):
    return {"bf16": K // 64, "mxfp4": K // 256}.get(mode, K // 128)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("M,N,K", [(1, 128, 1536), (3, 384, 1536), (16, 256, 3072), (17, 128, 1536),
                                   (24, 384, 1536), (32, 256, 2048), (40, 256, 1024)])
@pytest.mark.parametrize("S", [1, 2, 4, 8])
def test_decode_small_shapes(mode, M, N, K, S):
    if S > _slabs(mode, K):
        pytest.skip("more splits than K slabs")
    c = Case(mode, *inputs.operands(mode, M, N, K, 100 + M, 200 + N, 300 + K))
    ref = c.ref()
    if S > 1:
        ws = c.partials(S)
        parity.assert_ws_close(ws, c.ref_ws(S), f"{mode} ws S={S}")
    y = y_to_f64(c.gemm(split_k=S))
    parity.assert_y_close(y, ref, f"{mode} y S={S}")


@pytest.mark.parametrize("mode", MODES)
def test_split_outputs_agree(mode):
    M, N, K = 4, 256, 2048
    c = Case(mode, *inputs.operands(mode, M, N, K, 1, 2, 3))
    y1 = y_to_f64(c.gemm(split_k=1))
    for S in (2, 4, 8, 16):   # 2..8 reduce in a cluster, 16 through the workspace + reduce kernel
        if S > _slabs(mode, K):
            continue
        yS = y_to_f64(c.gemm(split_k=S))
        parity.assert_y_close(yS, y1, f"{mode} split {S} vs 1")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("S", [2, 3, 4, 5, 6, 7, 8])
def test_deferred_reduce_equals_fused_call(mode, S):
    """Two-pass (fp32 workspace + reduce kernel) and the in-cluster reduce sum
    the same partials in the same order: identical bits, for every cluster
    size (uneven ones give the CTAs of a tile unequal row counts)."""
    M, N, K = 16, 256, 2048
    if S > _slabs(mode, K):
        pytest.skip("more splits than K slabs")
    c = Case(mode, *inputs.operands(mode, M, N, K, 9, 10, 11))
    ws = torch.empty(S * M * N, dtype=torch.float32, device="cuda")
    c.gemm(split_k=S, flags=fg.FG_FLAG_DEFER_REDUCE, workspace=ws)
    y_two = c.reduce(ws, S)
    y_one = c.gemm(split_k=S)
    assert torch.equal(y_two.view(torch.int16), y_one.view(torch.int16))


@pytest.mark.parametrize("mode", ["fp8_tensor", "fp8_block128", "mxfp4", "bf16"])
@pytest.mark.parametrize("S", [3, 5, 6, 7])
@pytest.mark.parametrize("M", [1, 6, 21])
def test_fused_uneven_split_matches_oracle(mode, S, M):
    """Cluster sizes that do not divide the 128 rows of a tile, with ragged
    token tiles (M = 21: a full tile of 16 and one of 5): every output against
    the oracle."""
    N, K = 384, 2048
    if S > _slabs(mode, K):
        pytest.skip("more splits than K slabs")
    c = Case(mode, *inputs.operands(mode, M, N, K, 400 + S, 500 + M, 600))
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fg.gemm(c.dA, c.pb, c.da_s, split_k=S, Y=Y)
    parity.assert_y_close(y_to_f64(Y), c.ref(), f"{mode} M={M} fused split {S}")
    assert fg.get_error() == fg.FG_OK


PIPELINES = ["1,4", "1,5", "1,6", "1,8", "2,3", "2,5", "4,2"]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("cfg", PIPELINES)
def test_every_pipeline_config(mode, cfg, monkeypatch):
    """Each instantiated (slabs per stage, stages) pipeline, forced through the
    FG_DECODE_CONFIG hook: ragged token tile, splits 1 and 3 (three CTAs with
    unequal K shares and unequal row counts), stage buffers reused several
    times, every output against the oracle."""
    monkeypatch.setenv("FG_DECODE_CONFIG", cfg)
    M, N, K = 5, 256, 3072
    c = Case(mode, *inputs.operands(mode, M, N, K, 700, 701, 702))
    ref = c.ref()
    for S in (1, 3):
        plan = fg.gemm_plan(mode, M, N, K, split_k=S)
        assert f"{plan['stage_slabs']},{plan['stages']}" == cfg
        parity.assert_y_close(y_to_f64(c.gemm(split_k=S)), ref, f"{mode} {cfg} S={S}")
    assert fg.get_error() == fg.FG_OK


@pytest.mark.parametrize("mode", ["mxfp8", "mxfp4", "mxfp8_b32", "mxfp4_fp8a"])
def test_unaligned_mx_activation_scales(mode):
    """E8M0 activation scales passed at an odd address (a byte view one past
    an allocation's start) are read byte by byte: same result as aligned."""
    M, N, K = 5, 256, 2048
    c = Case(mode, *inputs.operands(mode, M, N, K, 801, 802, 803))
    buf = torch.zeros(c.a_s.size + 16, dtype=torch.uint8, device="cuda")
    odd = buf[1:1 + c.a_s.size]
    odd.copy_(dev(np.ascontiguousarray(c.a_s).reshape(-1)))
    assert odd.data_ptr() % 4 != 0
    for S in (1, 2):
        y = y_to_f64(fg.gemm(c.dA, c.pb, odd.view(c.a_s.shape), split_k=S))
        parity.assert_y_close(y, c.ref(), f"{mode} unaligned scales S={S}")
        assert np.array_equal(y, y_to_f64(c.gemm(split_k=S)))
    assert fg.get_error() == fg.FG_OK


ONE = {"bf16": 0x3F80, "fp8_tensor": 0x38, "fp8_block128": 0x38, "mxfp8": 0x38, "mxfp4": 0x2,
       "mxfp8_b32": 0x38, "mxfp4_fp8a": 0x38}   # the activation's code for 1.0


def _unit_a_scales(mode, M, K):
    return {"fp8_tensor": np.array([1.0], np.float32),
            "fp8_block128": np.ones((M, K // 128), np.float32),
            "mxfp8": np.full((M, K // 128), 127, np.uint8),
            "mxfp4": np.full((M, K // 32), 127, np.uint8),
            "mxfp8_b32": np.full((M, K // 32), 127, np.uint8),
            "mxfp4_fp8a": np.full((M, K // 32), 127, np.uint8)}.get(mode)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("S", [1, 4])
def test_identity_is_bit_exact(mode, S):
    """A = rows of the identity: Y[m, n] = Bd[n, m] exactly (bf16 holds every
    e4m3/e2m1 value times a power-of-two scale)."""
    M, N, K = 16, 256, 2048
    _, B, _, b_s = inputs.operands(mode, 1, N, K, 41, 42, 43)
    if mode == "fp8_block128":
        b_s = np.full_like(b_s, 0.5)
    if mode == "fp8_tensor":
        b_s = np.array([1.0], np.float32)
    A = np.zeros((M, K), np.uint16 if mode == "bf16" else np.uint8)
    for m in range(M):
        A[m, 37 * m + 5] = ONE[mode]
    if mode == "mxfp4":
        A = inputs.pack_e2m1(A)
    c = Case(mode, A, B, _unit_a_scales(mode, M, K), b_s)
    ref = c.ref()
    y = y_to_f64(c.gemm(split_k=S))
    assert np.array_equal(y, parity.bf16_bits_to_f64(oracle.round_bf16(ref)))
    assert np.array_equal(parity.bf16_bits_to_f64(oracle.round_bf16(ref)), ref)  # exact in bf16


@pytest.mark.parametrize("mode", MODES)
def test_all_ones_is_exact(mode):
    M, N, K = 3, 128, 7168 if mode != "bf16" else 4096
    A = np.full((M, K if mode != "mxfp4" else K // 2),
                ONE[mode] if mode != "mxfp4" else 0x22, np.uint16 if mode == "bf16" else np.uint8)
    B = np.full((N, A.shape[1]), A.flat[0], A.dtype)
    if mode == "mxfp4_fp8a":
        B = np.full((N, K // 2), 0x22, np.uint8)    # packed fp4 weights: two codes for 1.0
    b_s = {"fp8_tensor": np.array([1.0], np.float32), "fp8_block128": np.ones((1, K // 128), np.float32),
           "mxfp8": np.full((N, K // 128), 127, np.uint8), "mxfp4": np.full((N, K // 32), 127, np.uint8),
           "mxfp8_b32": np.full((N, K // 32), 127, np.uint8),
           "mxfp4_fp8a": np.full((N, K // 32), 127, np.uint8)}.get(mode)
    c = Case(mode, A, B, _unit_a_scales(mode, M, K), b_s)
    for S in (1, 4):
        y = y_to_f64(c.gemm(split_k=S))
        assert np.all(y == K)


# ----------------------------------------------------- full decode shapes

DECODE = [(m, n) for m, n in inputs.DECODE_SHAPES]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("M,N", DECODE)
def test_decode_workload_parity(mode, M, N):
    """The pages' decode shapes (K=7168) in the dispatch-chosen configuration,
    every output compared."""
    K = 7168
    c = Case(mode, *inputs.operands(mode, M, N, K, 1000 + M, 2000 + N, 3000))
    plan = fg.gemm_plan(mode, M, N, K)
    ref = c.ref()
    S = plan["split_k"]
    if S > 1:
        parity.assert_ws_close(c.partials(S), c.ref_ws(S), f"{mode} {M}x{N} ws")
    y = y_to_f64(c.gemm())
    parity.assert_y_close(y, ref, f"{mode} {M}x{N}")


@pytest.mark.parametrize("mode", ["fp8_tensor", "fp8_block128"])
@pytest.mark.parametrize("M", [1, 16])
def test_heuristic_two_per_sm_pipeline(mode, M):
    """A shape without a dispatch-table row whose grid needs one to two CTAs
    per SM with a long K range: the heuristic takes split 4 with 1 x 5
    stages; the fp32 partials at the workspace bound and every output."""
    N, K = 8192, 7168
    plan = fg.gemm_plan(mode, M, N, K)
    assert not plan["from_table"] and plan["split_k"] == 4 and (plan["stage_slabs"], plan["stages"]) == (1, 5)
    c = Case(mode, *inputs.operands(mode, M, N, K, 1100 + M, 2100, 3100))
    parity.assert_ws_close(c.partials(4), c.ref_ws(4), f"{mode} {M}x{N} ws")
    parity.assert_y_close(y_to_f64(c.gemm()), c.ref(), f"{mode} {M}x{N}")
    assert fg.get_error() == fg.FG_OK


def test_c1_split4_parity():
    """The first of the pages' decode configurations as stated: fp8
    per-tensor, M=1, N=2048, K=7168 with split_k fixed at 4 (not the
    dispatch's choice): the fp32 partials of the four splits at the
    workspace bound, and every output."""
    A, B, a_s, b_s = inputs.workload_operands("fp8_tensor_decode_m1_n2048_k7168_split4", 0)
    c = Case("fp8_tensor", A, B, a_s, b_s)
    assert fg.gemm_plan("fp8_tensor", 1, 2048, 7168, split_k=4)["split_k"] == 4
    parity.assert_ws_close(c.partials(4), c.ref_ws(4), "C1 ws S=4")
    parity.assert_y_close(y_to_f64(c.gemm(split_k=4)), c.ref(), "C1 y S=4")
    assert fg.get_error() == fg.FG_OK


@pytest.mark.parametrize("mode", MODES)
def test_two_pass_split16_matches_oracle(mode):
    """Splits above the cluster limit take the workspace + reduce-kernel
    path: 16 splits (ragged token tile, three weight tiles), the partials at
    the workspace bound and every output against the oracle."""
    M, N, K = 5, 384, 4096
    c = Case(mode, *inputs.operands(mode, M, N, K, 910, 911, 912))
    assert fg.gemm_workspace_size(mode, M, N, K, 16) == 16 * M * N * 4
    parity.assert_ws_close(c.partials(16), c.ref_ws(16), f"{mode} ws S=16")
    parity.assert_y_close(y_to_f64(c.gemm(split_k=16)), c.ref(), f"{mode} y S=16")
    assert fg.get_error() == fg.FG_OK


@pytest.mark.parametrize("mode", ["fp8_tensor", "fp8_block128", "mxfp4"])
def test_two_pass_split16_workload_shape(mode):
    """Split 16 at a decode shape of the pages (M=16, N=2048, K=7168):
    every output against the oracle."""
    M, N, K = 16, 2048, 7168
    c = Case(mode, *inputs.operands(mode, M, N, K, 920, 921, 922))
    parity.assert_y_close(y_to_f64(c.gemm(split_k=16)), c.ref(), f"{mode} {M}x{N}x{K} S=16")
    assert fg.get_error() == fg.FG_OK


# -------------------------------------------------------- negative controls

def test_negative_controls_diverge():
    """Planted mistakes must fail the bounds: a wrong scale, a weight that was
    not preshuffled, swapped fp4 nibbles."""
    M, N, K = 4, 256, 2048
    c = Case("fp8_tensor", *inputs.operands("fp8_tensor", M, N, K, 51, 52, 53))
    ref = c.ref()
    y = y_to_f64(fg.gemm(c.dA, c.pb, dev(c.a_s * 2)))
    assert parity.y_violations(y, ref)[0] > 0
    raw = Case("fp8_tensor", c.A, c.B, c.a_s, c.b_s)
    raw.pb.data.copy_(dev(np.ascontiguousarray(c.B).reshape(-1)))   # un-preshuffled bytes
    assert parity.y_violations(y_to_f64(raw.gemm()), ref)[0] > 0
    f = Case("mxfp4", *inputs.operands("mxfp4", M, N, K, 54, 55, 56))
    ref4 = f.ref()
    swapped = ((f.A & 15) << 4) | (f.A >> 4)
    y4 = y_to_f64(fg.gemm(dev(swapped.astype(np.uint8)), f.pb, f.da_s))
    assert parity.y_violations(y4, ref4)[0] > 0
    assert parity.y_violations(y_to_f64(f.gemm()), ref4)[0] == 0


# ------------------------------------------------------------ error paths

def test_error_paths_on_device():
    M, N, K = 2, 256, 1024
    c = Case("fp8_tensor", *inputs.operands("fp8_tensor", M, N, K, 61, 62, 63))
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fg.FgError) as e:
        fg.gemm(c.dA, c.pb, c.da_s, mode="mxfp8", Y=Y)
    assert e.value.status == fg.FG_ERR_LAYOUT
    with pytest.raises(fg.FgError) as e:     # deferred partials need split*M*N*4 bytes
        fg.gemm(c.dA, c.pb, c.da_s, split_k=4, Y=Y, workspace=torch.empty(8, device="cuda"),
                flags=fg.FG_FLAG_DEFER_REDUCE)
    assert e.value.status == fg.FG_ERR_WORKSPACE
    buf = torch.zeros(M * K + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fg.FgError) as e:
        fg.gemm(buf[1:1 + M * K].view(M, K), c.pb, c.da_s, Y=Y)
    assert e.value.status == fg.FG_ERR_ALIGN
    with pytest.raises(fg.FgError) as e:
        fg.gemm(c.dA, c.pb, None, Y=Y)
    assert e.value.status == fg.FG_ERR_INVALID_ARG
    fg.debug_override_cc(9, 0)
    try:
        with pytest.raises(fg.FgError) as e:
            fg.gemm(c.dA, c.pb, c.da_s, Y=Y)
        assert e.value.status == fg.FG_ERR_UNSUPPORTED_ARCH
    finally:
        fg.debug_override_cc(-1, 0)
    # M == 0: no-op
    fg.gemm(c.dA[:0], c.pb, c.da_s, Y=Y[:0])
    parity.assert_y_close(y_to_f64(c.gemm()), c.ref(), "after errors")


def test_binding_rejects_views_that_would_be_misread():
    """A transposed A, a column slice of a wider buffer, activations of the
    wrong element type, and a Y of the wrong shape are refused by the
    binding with ValueError before anything is launched."""
    M, N, K = 4, 256, 1024
    c = Case("fp8_tensor", *inputs.operands("fp8_tensor", M, N, K, 64, 65, 66))
    Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="contiguous"):
        fg.gemm(c.dA.t().contiguous().t(), c.pb, c.da_s, Y=Y)      # same shape, column-major
    with pytest.raises(ValueError, match="contiguous"):
        wide = torch.zeros((M, 2 * K), dtype=torch.uint8, device="cuda")
        fg.gemm(wide[:, :K], c.pb, c.da_s, Y=Y)
    with pytest.raises(ValueError, match="dtype"):
        fg.gemm(c.dA.float(), c.pb, c.da_s, Y=Y)
    with pytest.raises(ValueError, match="shape"):
        fg.gemm(c.dA, c.pb, c.da_s, Y=torch.zeros((M, N // 2), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError, match="dtype"):
        fg.gemm(c.dA, c.pb, c.da_s.double(), Y=Y)
    torch.cuda.synchronize()
    assert not Y.any()
    parity.assert_y_close(y_to_f64(fg.gemm(c.dA, c.pb, c.da_s, Y=Y)), c.ref(), "after refusals")


def test_bounded_wait_reports_timeout_and_context_survives():
    """The MMA issuer waits on a barrier nothing arrives at; every wait runs
    out after the limit, the kernel cleans up and returns, and the host reads
    FG_ERR_TIMEOUT.  A normal call afterwards is still correct."""
    M, N, K = 1, 256, 2048
    assert fg.get_error() == fg.FG_OK
    for mode in ("fp8_tensor", "fp8_block128", "mxfp4", "mxfp4_fp8a"):
        c = Case(mode, *inputs.operands(mode, M, N, K, 71, 72, 73))
        fg.set_wait_timeout_ns(20_000_000)
        try:
            c.gemm(split_k=2, flags=fg.FG_FLAG_DEBUG_STALL)
            assert fg.get_error() == fg.FG_ERR_TIMEOUT
        finally:
            fg.set_wait_timeout_ns(4_000_000_000)
        assert fg.get_error() == fg.FG_OK
        parity.assert_y_close(y_to_f64(c.gemm(split_k=2)), c.ref(), f"{mode} after timeout")


# -------------------------------------------------------- 32-token tiles

@pytest.mark.parametrize("M", [17, 32])
def test_up_to_32_tokens_take_one_token_tile(M):
    """17..32 tokens run as one 32-token tile (the MMA's N = 32), so the
    weights stream once; 33..64 take two."""
    p = fg.gemm_plan("fp8_tensor", M, 16384, 7168)
    assert p["path"] == 0 and p["tile_m"] == 32
    assert p["ctas"] == 128 * p["split_k"]
    p = fg.gemm_plan("fp8_tensor", 2 * M, 2048, 7168, split_k=2)  # an explicit split keeps decode: two tiles
    assert p["path"] == 0 and p["tile_m"] == 32 and p["ctas"] == 16 * 2 * 2


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("cfg", ["1,4", "1,5", "1,6", "1,8"])
def test_32_token_pipelines(mode, cfg, monkeypatch):
    """Every pipeline instantiated for 32-token tiles (one slab per stage),
    ragged (29 tokens), splits 1 and 3, every output against the oracle."""
    monkeypatch.setenv("FG_DECODE_CONFIG", cfg)
    M, N, K = 29, 256, 3072
    c = Case(mode, *inputs.operands(mode, M, N, K, 710, 711, 712))
    ref = c.ref()
    for S in (1, 3):
        plan = fg.gemm_plan(mode, M, N, K, split_k=S)
        assert plan["tile_m"] == 32 and f"{plan['stage_slabs']},{plan['stages']}" == cfg
        parity.assert_y_close(y_to_f64(c.gemm(split_k=S)), ref, f"{mode} {cfg} 32 tokens S={S}")
    assert fg.get_error() == fg.FG_OK


def test_32_token_tiles_refuse_multi_slab_stages(monkeypatch):
    monkeypatch.setenv("FG_DECODE_CONFIG", "2,3")
    with pytest.raises(fg.FgError) as e:
        fg.gemm_plan("fp8_tensor", 20, 2048, 7168)
    assert e.value.status == fg.FG_ERR_INVALID_ARG


@pytest.mark.parametrize("mode", MODES)
def test_identity_is_bit_exact_32_tokens(mode):
    M, N, K = 32, 256, 2048
    _, B, _, b_s = inputs.operands(mode, 1, N, K, 44, 45, 46)
    if mode == "fp8_block128":
        b_s = np.full_like(b_s, 0.5)
    if mode == "fp8_tensor":
        b_s = np.array([1.0], np.float32)
    A = np.zeros((M, K), np.uint16 if mode == "bf16" else np.uint8)
    for m in range(M):
        A[m, 29 * m + 3] = ONE[mode]
    if mode == "mxfp4":
        A = inputs.pack_e2m1(A)
    c = Case(mode, A, B, _unit_a_scales(mode, M, K), b_s)
    ref = c.ref()
    for S in (1, 4):
        assert np.array_equal(y_to_f64(c.gemm(split_k=S)), parity.bf16_bits_to_f64(oracle.round_bf16(ref)))


def test_32_token_bounded_wait_reports_timeout():
    M, N, K = 20, 256, 2048
    assert fg.get_error() == fg.FG_OK
    for mode in ("fp8_tensor", "fp8_block128", "mxfp4"):
        c = Case(mode, *inputs.operands(mode, M, N, K, 74, 75, 76))
        fg.set_wait_timeout_ns(20_000_000)
        try:
            c.gemm(split_k=2, flags=fg.FG_FLAG_DEBUG_STALL)
            assert fg.get_error() == fg.FG_ERR_TIMEOUT
        finally:
            fg.set_wait_timeout_ns(4_000_000_000)
        assert fg.get_error() == fg.FG_OK
        parity.assert_y_close(y_to_f64(c.gemm(split_k=2)), c.ref(), f"{mode} 32 tokens after timeout")


# ---------------------------------------- partial commits in groups of slabs

@pytest.mark.parametrize("mode", ["fp8_block128", "bf16"])
@pytest.mark.parametrize("group", ["1", "2", "4"])
@pytest.mark.parametrize("cfg", ["1,4", "1,5", "2,3", "2,5", "4,2"])
def test_partial_commit_groups(mode, group, cfg, monkeypatch):
    """bf16 and blockscale announce their per-slab TMEM partials with one
    commit per group of 1, 2 or 4 slabs (FG_DECODE_PGROUP); forced for each
    pipeline, including 2 x 5, whose stages are released by their own
    commits, and splits whose slab counts leave a short last group.  Every
    output against the oracle, the fp32 partials against the workspace
    bound, and the same bits as the default grouping (the sums do not depend
    on when a partial is announced)."""
    M, N, K = 5, 256, 3072
    c = Case(mode, *inputs.operands(mode, M, N, K, 730, 731, 732))
    ref = c.ref()
    monkeypatch.setenv("FG_DECODE_CONFIG", cfg)
    base = {S: c.gemm(split_k=S) for S in (1, 3, 7)}
    monkeypatch.setenv("FG_DECODE_PGROUP", group)
    for S in (1, 3, 7):
        y = c.gemm(split_k=S)
        parity.assert_y_close(y_to_f64(y), ref, f"{mode} {cfg} group {group} S={S}")
        assert torch.equal(y.view(torch.int16), base[S].view(torch.int16))
    parity.assert_ws_close(c.partials(3), c.ref_ws(3), f"{mode} {cfg} group {group} ws")
    if cfg.startswith("1,"):   # 32-token tiles: one slab per stage
        c32 = Case(mode, *inputs.operands(mode, 29, N, K, 733, 734, 735))
        parity.assert_y_close(y_to_f64(c32.gemm(split_k=3)), c32.ref(), f"{mode} {cfg} group {group} 32 tokens")
    assert fg.get_error() == fg.FG_OK
