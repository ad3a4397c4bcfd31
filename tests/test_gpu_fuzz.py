"""Seeded random shapes, modes and splits through the public API, every
output against the oracle.

Draws cover both kernels (M up to 300 so that the large-M forms run too),
ragged token tiles, weight widths that leave a half-empty 256-column tile,
K from one slab to many, and every split the dispatch allows (explicit 1-8
and 16, or the dispatch's own choice).  Each case is run twice: the bits
must repeat.
"""
import numpy as np
import pytest
import torch

import inputs
import mx_gemm_gb300 as fg
from tests import parity
from tests.gpu_util import Case, y_to_f64

pytestmark = pytest.mark.gpu

MODES = ["bf16", "fp8_tensor", "fp8_block128", "mxfp8", "mxfp4", "mxfp8_b32", "mxfp4_fp8a"]
K_UNIT = {"bf16": 64, "mxfp4": 256}  # elements per 128-byte slab; 128 otherwise


def _draw(i):
    g = np.random.default_rng(9000 + i)
    mode = MODES[i % len(MODES)]
    unit = K_UNIT.get(mode, 128)
    if mode in ("fp8_block128", "mxfp8"):
        unit = 128
    K = unit * int(g.integers(1, 25))
    N = 128 * int(g.integers(1, 13))
    M = int(g.choice([1, 2, 5, 16, 17, 31, 40, 64, 129, 300]))
    slabs = K // unit if mode != "bf16" else K // 64
    splits = [0] + [s for s in (1, 2, 3, 4, 5, 8, 16) if s <= slabs]
    split = int(g.choice(splits))
    if M > 32 and g.random() < 0.5:
        split = 0                      # the dispatch's choice: the large-M forms where they exist
    return mode, M, N, K, split


@pytest.mark.parametrize("i", range(48))
def test_random_case_matches_oracle(i):
    mode, M, N, K, split = _draw(i)
    c = Case(mode, *inputs.operands(mode, M, N, K, 100 + i, 200 + i, 300 + i))
    y1 = c.gemm(split_k=split)
    y2 = c.gemm(split_k=split)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), f"{mode} {M}x{N}x{K} S={split} not repeatable"
    parity.assert_y_close(y_to_f64(y1), c.ref(), f"{mode} {M}x{N}x{K} S={split}")
    assert fg.get_error() == fg.FG_OK
