"""Seeded synthetic inputs for the preshuffled-weight GEMM.

This module produces operands only: raw codes and scales, as numpy arrays on
the host.  It holds none of the GEMM's arithmetic (no dequantisation, no
products, no sums), so the CPU oracle and the CUDA path can both be fed from
it without sharing any of the method.

Recipe (the pages measure on bare GEMM shapes, not on a dataset):
  * values x ~ N(0, 1), fp32, numpy PCG64 seeded per operand;
  * bf16: round-to-nearest-even of x;
  * fp8 per-tensor: a_s = fp32(amax/448), code = e4m3(x / a_s) (amax maps to 448);
  * fp8 blockscale: each block (1x128 for A, 128x128 for B) is rescaled so its
    amax equals T, T log-uniform in [1e-2, 1e2]; scale = fp32(T/448),
    code = e4m3(x_block / scale);
  * MX: per 1 x blk block, E8M0 c = 127 + ceil(log2(amax / elem_max)), clamped
    to [0, 254] (an all-zero block gets 127); code = RNE(x / 2^(c-127)) in the
    element format (e4m3, elem_max 448, blk 128 -- or 32 for the OCP block;
    or e2m1, elem_max 6, blk 32, two codes per byte, low nibble = even k).
e4m3 and bf16 encodings use torch's dtype casts; e2m1 rounding is done here
(ties to the even code) and pinned against an independent dtype library in
the CPU tests.
"""
import math

import numpy as np

MODES = ("bf16", "fp8_tensor", "fp8_block128", "mxfp8", "mxfp4", "mxfp8_b32", "mxfp4_fp8a")
E4M3_MAX = 448.0
E2M1_MAX = 6.0
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float64)
_E2M1_MID = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float64)


def randn(rows, cols, seed):
    """fp32 N(0,1) of shape (rows, cols), generated in row chunks from one stream."""
    g = np.random.default_rng(seed)
    out = np.empty((rows, cols), np.float32)
    step = max(1, (1 << 24) // max(cols, 1))
    for r in range(0, rows, step):
        out[r:r + step] = g.standard_normal((min(step, rows - r), cols), dtype=np.float32)
    return out


def _torch():
    import torch
    return torch


def to_bf16_bits(x):
    torch = _torch()
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def to_e4m3_codes(x):
    """e4m3 'fn' codes (uint8) of fp32 values, RNE, saturating at +-448."""
    torch = _torch()
    t = torch.from_numpy(np.clip(np.ascontiguousarray(x, np.float32), -E4M3_MAX, E4M3_MAX))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def to_e2m1_codes(x):
    """e2m1 4-bit codes (uint8, one per element), RNE with ties to the even code.

    Inputs must already lie in [-6, 6].
    """
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    idx = np.searchsorted(_E2M1_MID, a, side="left")
    tie = np.zeros(a.shape, bool)
    inb = idx < _E2M1_MID.size
    tie[inb] = a[inb] == _E2M1_MID[idx[inb]]
    idx = idx + (tie & (idx % 2 == 1))
    code = idx.astype(np.uint8)
    return np.where(np.signbit(x) & (code != 0), code | 8, code).astype(np.uint8)


def pack_e2m1(codes):
    """Pack [rows][K] 4-bit codes into [rows][K/2] bytes, low nibble = even k."""
    codes = np.asarray(codes, np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def e8m0_for(amax, elem_max):
    """E8M0 code c = 127 + ceil(log2(amax/elem_max)), clamped to [0, 254]; 127 for 0."""
    amax = np.asarray(amax, np.float64)
    out = np.full(amax.shape, 127, np.int64)
    nz = amax > 0
    r = amax[nz] / elem_max
    f, e = np.frexp(r)              # r = f * 2^e, f in [0.5, 1)
    ceil_log2 = np.where(f == 0.5, e - 1, e)
    out[nz] = 127 + ceil_log2
    return np.clip(out, 0, 254).astype(np.uint8)


# ------------------------------------------------------------- operands

def bf16_operand(rows, K, seed):
    return to_bf16_bits(randn(rows, K, seed))


def fp8_tensor_operand(rows, K, seed):
    """(codes uint8 [rows][K], scale fp32 scalar)."""
    x = randn(rows, K, seed)
    amax = np.float32(np.max(np.abs(x)))
    s = np.float32(amax / np.float32(E4M3_MAX))
    return to_e4m3_codes(x / s), np.array([s], np.float32)


def fp8_block128_operand(rows, K, seed, scale_seed, block_rows):
    """(codes uint8 [rows][K], scales fp32 [rows/block_rows][K/128]).

    block_rows is 1 for the activation A and 128 for the weight B.
    """
    assert K % 128 == 0 and rows % block_rows == 0
    x = randn(rows, K, seed).reshape(rows // block_rows, block_rows, K // 128, 128)
    amax = np.max(np.abs(x), axis=(1, 3)).astype(np.float64)
    g = np.random.default_rng(scale_seed)
    target = np.exp(g.uniform(math.log(1e-2), math.log(1e2), size=amax.shape))
    scale = (target / E4M3_MAX).astype(np.float32)
    xs = x.astype(np.float64) * (target / amax)[:, None, :, None]
    q = xs / scale.astype(np.float64)[:, None, :, None]
    codes = to_e4m3_codes(q.astype(np.float32)).reshape(rows, K)
    return codes, scale


def mx_operand(rows, K, seed, fmt):
    """MX operand: fmt 'mxfp8' -> (e4m3 codes [rows][K], E8M0 [rows][K/128]);
    'mxfp8_b32' -> (e4m3 codes [rows][K], E8M0 [rows][K/32]);
    'mxfp4' -> (packed e2m1 [rows][K/2], E8M0 [rows][K/32])."""
    blk, emax = {"mxfp8": (128, E4M3_MAX), "mxfp8_b32": (32, E4M3_MAX), "mxfp4": (32, E2M1_MAX)}[fmt]
    assert K % blk == 0
    x = randn(rows, K, seed).reshape(rows, K // blk, blk)
    amax = np.max(np.abs(x), axis=2)
    c = e8m0_for(amax, emax)
    scale = np.ldexp(1.0, c.astype(np.int64) - 127)
    q = (x.astype(np.float64) / scale[:, :, None]).reshape(rows, K)
    if fmt in ("mxfp8", "mxfp8_b32"):
        return to_e4m3_codes(q.astype(np.float32)), c
    return pack_e2m1(to_e2m1_codes(q)), c


def operands(mode, M, N, K, seed_a, seed_b, seed_s):
    """(A, B, a_scale, b_scale) host arrays for one GEMM of the given mode."""
    if mode == "bf16":
        return bf16_operand(M, K, seed_a), bf16_operand(N, K, seed_b), None, None
    if mode == "fp8_tensor":
        A, a_s = fp8_tensor_operand(M, K, seed_a)
        B, b_s = fp8_tensor_operand(N, K, seed_b)
        return A, B, a_s, b_s
    if mode == "fp8_block128":
        A, a_s = fp8_block128_operand(M, K, seed_a, seed_s, 1)
        B, b_s = fp8_block128_operand(N, K, seed_b, seed_s + 500, 128)
        return A, B, a_s, b_s
    if mode in ("mxfp8", "mxfp4", "mxfp8_b32"):
        A, a_s = mx_operand(M, K, seed_a, mode)
        B, b_s = mx_operand(N, K, seed_b, mode)
        return A, B, a_s, b_s
    if mode == "mxfp4_fp8a":   # fp8 activations (32-K E8M0), fp4 weights (32-K E8M0)
        A, a_s = mx_operand(M, K, seed_a, "mxfp8_b32")
        B, b_s = mx_operand(N, K, seed_b, "mxfp4")
        return A, B, a_s, b_s
    raise ValueError(mode)


def sample_rows(M, n=256, seed=1234):
    """n distinct sorted rows of [0, M), always including 0 and M-1."""
    if M <= n:
        return np.arange(M, dtype=np.int64)
    g = np.random.default_rng(seed)
    rest = g.choice(np.arange(1, M - 1), size=n - 2, replace=False)
    return np.unique(np.concatenate([[0, M - 1], rest]).astype(np.int64))


# ----------------------------------------------------------- workloads
# The five workloads the pages measure on (shapes, splits, seeds).  Seeds:
# A = 1000+i, B = 2000+i, scales = 3000+i for workload i.

DECODE_SHAPES = ((1, 2048), (1, 16384), (16, 2048), (16, 16384))

WORKLOADS = {
    "fp8_tensor_decode_m1_n2048_k7168_split4": dict(
        idx=0, cases=[dict(mode="fp8_tensor", M=1, N=2048, K=7168, split_k=4)]),
    "fp8_tensor_decode_sweep_k7168": dict(
        idx=1, cases=[dict(mode="fp8_tensor", M=m, N=n, K=7168, split_k=0)
                      for m, n in DECODE_SHAPES]),
    "fp8_block128_decode_sweep_k7168": dict(
        idx=2, cases=[dict(mode="fp8_block128", M=m, N=n, K=7168, split_k=0)
                      for m, n in DECODE_SHAPES]),
    "large_bf16_54560x8192x8192_fp8_4096x4096x8192": dict(
        idx=3, cases=[dict(mode="bf16", M=54560, N=8192, K=8192, split_k=1),
                      dict(mode="fp8_tensor", M=4096, N=4096, K=8192, split_k=1)]),
    "mx_mxfp8_mxfp4_n16384_k7168": dict(
        idx=4, cases=[dict(mode=f, M=m, N=16384, K=7168, split_k=0)
                      for f in ("mxfp8", "mxfp4") for m in (1, 16, 4096)]),
    # next rows: the OCP 32-element mxfp8 block, the bf16 decode sweep, and
    # fp8 activations against fp4 weights (on the MX shapes above)
    "mx_mxfp8_b32_n16384_k7168": dict(
        idx=5, cases=[dict(mode="mxfp8_b32", M=m, N=16384, K=7168, split_k=0) for m in (1, 16, 4096)]),
    "bf16_decode_sweep_k7168": dict(
        idx=6, cases=[dict(mode="bf16", M=m, N=n, K=7168, split_k=0) for m, n in DECODE_SHAPES]),
    "mx_fp8a_fp4w_n16384_k7168": dict(
        idx=7, cases=[dict(mode="mxfp4_fp8a", M=m, N=16384, K=7168, split_k=0) for m in (1, 16, 4096)]),
    # FP8 blockscale at large M
    "large_fp8_block128_4096x16384x7168": dict(
        idx=9, cases=[dict(mode="fp8_block128", M=4096, N=16384, K=7168, split_k=1)]),
    # half of it (still larger than L2): the case a full kernel profile takes
    "large_fp8_block128_4096x8192x7168": dict(
        idx=10, cases=[dict(mode="fp8_block128", M=4096, N=8192, K=7168, split_k=1)]),
    # the same for mxfp4 (packed operands: 4096 x 16384 x 7168 is 201 MB of A, B and Y)
    "large_mxfp4_4096x8192x7168": dict(
        idx=11, cases=[dict(mode="mxfp4", M=4096, N=8192, K=7168, split_k=1)]),
    # 32 tokens: one 32-token tile per weight tile
    "fp8_tensor_decode_m32_k7168": dict(
        idx=8, cases=[dict(mode="fp8_tensor", M=32, N=n, K=7168, split_k=0) for n in (2048, 16384)]),
}


def workload_operands(name, case_index):
    w = WORKLOADS[name]
    c = w["cases"][case_index]
    i = w["idx"]
    # distinct streams per case inside one workload
    off = 10 * case_index
    return operands(c["mode"], c["M"], c["N"], c["K"], 1000 + i + off, 2000 + i + off,
                    3000 + i + off)
