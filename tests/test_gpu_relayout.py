"""GPU weight relayout and split-K reduce against the oracle (bit-exact /
within the output bound)."""
import numpy as np
import pytest
import torch

import inputs
import mx_gemm_gb300 as fg
import oracle
from tests import parity
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu


def _kb(mode, K):
    return K * 2 if mode == "bf16" else (K // 2 if mode in ("mxfp4", "mxfp4_fp8a") else K)


@pytest.mark.parametrize("mode", ["bf16", "fp8_tensor", "fp8_block128", "mxfp8", "mxfp4", "mxfp8_b32", "mxfp4_fp8a"])
@pytest.mark.parametrize("N,K", [(128, 256), (384, 1536), (256, 7168)])
def test_relayout_matches_spec_and_inverts(mode, N, K):
    A, B, a_s, b_s = inputs.operands(mode, 1, N, K, 5, 6, 7)
    pb = fg.preshuffle_b(mode, dev(B), dev(b_s), K=K)
    torch.cuda.synchronize()
    kb = _kb(mode, K)
    Bb = np.ascontiguousarray(B).view(np.uint8).reshape(N, kb)
    spec = oracle.block64_b(Bb, N, kb) if mode == "mxfp4_fp8a" else oracle.preshuffle_b(Bb, N, kb)
    assert np.array_equal(host(pb.data), spec)
    if mode in ("mxfp8", "mxfp4", "mxfp8_b32", "mxfp4_fp8a"):
        orc_mode = {"mxfp8": oracle.MXFP8, "mxfp4": oracle.MXFP4, "mxfp8_b32": oracle.MXFP8_B32,
                    "mxfp4_fp8a": oracle.MXFP4_FP8A}[mode]
        assert np.array_equal(host(pb.sf), oracle.sf_image(orc_mode, b_s, N, K))
    back, sc = fg.unshuffle_b(pb)
    torch.cuda.synchronize()
    assert np.array_equal(host(back), np.ascontiguousarray(B).view(np.uint8).reshape(N, kb))
    if b_s is not None:
        assert np.array_equal(host(sc).reshape(-1).view(np.uint8), np.ascontiguousarray(b_s).reshape(-1).view(np.uint8))


def test_relayout_is_a_bijection_on_unique_chunks():
    N, kb = 384, 2048
    idx = np.zeros((N * kb // 16, 2), np.uint64)
    idx[:, 0] = np.arange(N * kb // 16, dtype=np.uint64)
    B = idx.view(np.uint8).reshape(N, kb)
    pb = fg.preshuffle_b("fp8_tensor", dev(B), dev(np.array([1.0], np.float32)), K=kb)
    torch.cuda.synchronize()
    img = host(pb.data)
    assert np.array_equal(img, oracle.preshuffle_b(B, N, kb))
    moved = img.view(np.uint64).reshape(-1, 2)[:, 0]
    assert np.array_equal(np.sort(moved), idx[:, 0])


@pytest.mark.parametrize("S", [1, 2, 3, 8])
@pytest.mark.parametrize("scaled", [False, True])
def test_splitk_reduce(S, scaled):
    M, N = 5, 1024
    g = np.random.default_rng(S)
    ws = g.standard_normal((S, M, N)).astype(np.float32)
    a_s = np.array([0.37], np.float32) if scaled else None
    b_s = np.array([1.9], np.float32) if scaled else None
    Y = fg.gemm_splitk_reduce(dev(ws), S, M, N, dev(a_s), dev(b_s))
    y = parity.bf16_bits_to_f64(host(Y.view(torch.int16)))
    ref = ws.astype(np.float64).sum(axis=0) * (float(a_s[0]) * float(b_s[0]) if scaled else 1.0)
    parity.assert_y_close(y, ref, "reduce")
    # the sum runs in split order in fp32, then one scale and one bf16 rounding
    acc = ws[0].copy()
    for s in range(1, S):
        acc = acc + ws[s]
    if scaled:
        acc = acc * np.float32(a_s[0] * b_s[0])
    exp = torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(host(Y.view(torch.int16)), exp)
