"""Helpers shared by the GPU tests: move seeded host operands to the device,
run the library through its Python binding, and compare with the oracle."""
import numpy as np
import torch

import mx_gemm_gb300 as fg
import oracle
from tests import parity

ORC = {"bf16": oracle.BF16, "fp8_tensor": oracle.FP8_TENSOR, "fp8_block128": oracle.FP8_BLOCK128,
       "mxfp8": oracle.MXFP8, "mxfp4": oracle.MXFP4, "mxfp8_b32": oracle.MXFP8_B32,
       "mxfp4_fp8a": oracle.MXFP4_FP8A}


def dev(x):
    if x is None:
        return None
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        x = x.view(np.int16)
    return torch.from_numpy(x).cuda()


def host(t):
    return t.cpu().numpy()


def y_to_f64(Y):
    return parity.bf16_bits_to_f64(Y.view(torch.int16).cpu().numpy())


class Case:
    """One GEMM's operands on host and device, with its preshuffled weight."""

    def __init__(self, mode, A, B, a_s, b_s):
        self.mode, self.A, self.B, self.a_s, self.b_s = mode, A, B, a_s, b_s
        self.M, self.N = A.shape[0], B.shape[0]
        self.K = A.shape[1] * (2 if mode == "mxfp4" else 1)
        self.dA, self.da_s = dev(A), dev(a_s)
        self.pb = fg.preshuffle_b(mode, dev(B), dev(b_s), K=self.K)

    def gemm(self, split_k=0, flags=0, workspace=None):
        return fg.gemm(self.dA, self.pb, self.da_s, split_k=split_k, flags=flags, workspace=workspace)

    def ref(self, tensor_scale=True, rows=None):
        return oracle.gemm(ORC[self.mode], self.A, self.B, self.a_s, self.b_s, M=self.M, N=self.N,
                           K=self.K, tensor_scale=tensor_scale, rows=rows)

    def ref_ws(self, S):
        return oracle.workspace(ORC[self.mode], self.A, self.B, self.a_s, self.b_s, S, M=self.M,
                                N=self.N, K=self.K)

    def partials(self, S):
        """Run with the reduce deferred; return the fp32 workspace [S][M][N]."""
        ws = torch.full((S * self.M * self.N,), float("nan"), dtype=torch.float32, device="cuda")
        self.gemm(split_k=S, flags=fg.FG_FLAG_DEFER_REDUCE, workspace=ws)
        torch.cuda.synchronize()
        return host(ws).reshape(S, self.M, self.N).astype(np.float64)

    def reduce(self, ws_dev, S):
        a_s = b_s = None
        if self.mode == "fp8_tensor":
            a_s, b_s = self.da_s, dev(self.b_s)
        return fg.gemm_splitk_reduce(ws_dev, S, self.M, self.N, a_s, b_s)
