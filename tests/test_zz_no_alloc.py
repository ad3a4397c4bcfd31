"""fg_gemm_noalloc, called through the C ABI, against fg_gemm.

fg_gemm_noalloc serves callers that cannot allocate device memory while they
run (a serving loop with every buffer sized at start-up, or a plug-in whose
host framework owns all device memory): it keeps the split-K partials in the
library's own 8 MiB device array instead of a caller workspace.  Its output
must match fg_gemm's (same kernels, same split) within the output bound the
other tests use, on two calls in a row (the second with other inputs and a
different shape, so stale partials from the first call cannot leak in), and a
split that needs more than the scratch holds must be refused.

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import inputs
import mx_gemm_gb300 as fg
from tests import parity
from tests.gpu_util import Case, y_to_f64

pytestmark = pytest.mark.gpu


def _noalloc(c, split_k, Y):
    """One fg_gemm_noalloc call through the C ABI (ctypes, no binding logic)."""
    L = fg.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    a_s = None if c.da_s is None else ctypes.c_void_p(c.da_s.data_ptr())
    return L.fg_gemm_noalloc(ctypes.c_void_p(c.dA.data_ptr()), a_s, c.M, ctypes.byref(c.pb.desc),
                             fg.MODES[c.mode], split_k, ctypes.c_void_p(Y.data_ptr()), 0, stream)


def _with_workspace(c, split_k):
    return c.gemm(split_k=split_k)


@pytest.mark.parametrize("first,second", [
    (("fp8_tensor", 16, 2048, 7168, 8), ("fp8_tensor", 1, 16384, 7168, 4)),
    (("fp8_block128", 16, 2048, 7168, 8), ("mxfp4", 16, 2048, 7168, 4)),
])
def test_noalloc_matches_fg_gemm_on_two_calls(first, second):
    for i, (mode, M, N, K, S) in enumerate((first, second)):
        c = Case(mode, *inputs.operands(mode, M, N, K, 500 + 7 * i, 600 + 7 * i, 700 + 7 * i))
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = _noalloc(c, S, Y)
        assert rc == fg.FG_OK, fg.last_error_message()
        torch.cuda.synchronize()
        y_ref = _with_workspace(c, S)
        parity.assert_y_close(y_to_f64(Y), y_to_f64(y_ref), f"no-alloc call {i + 1} ({mode} {M}x{N} S={S})")
        # same kernels and split: the results agree bit for bit
        assert torch.equal(Y.view(torch.int16), y_ref.view(torch.int16))
    assert fg.get_error() == fg.FG_OK


def test_noalloc_refuses_a_split_larger_than_its_scratch():
    mode, M, N, K = "fp8_tensor", 16, 16384, 7168
    c = Case(mode, *inputs.operands(mode, M, N, K, 801, 802, 803))
    Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    rc = _noalloc(c, 16, Y)         # 16 * 16 * 16384 * 4 bytes = 16 MiB > 8 MiB
    assert rc == fg.FG_ERR_WORKSPACE
    assert "scratch" in fg.last_error_message()
    torch.cuda.synchronize()
    assert not Y.any()                # nothing was launched
    rc = _noalloc(c, 2, Y)            # 2 MiB fits
    assert rc == fg.FG_OK
    parity.assert_y_close(y_to_f64(Y), c.ref(), "no-alloc within the limit")
    assert np.isfinite(y_to_f64(Y)).all()
