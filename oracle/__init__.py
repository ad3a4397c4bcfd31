"""CPU oracle for the preshuffled-weight GEMM (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never calls it; it shares
no code with the CUDA path.

The arithmetic lives in ``fg_oracle.c`` (fp64, table decode of the bit
patterns, k-ascending sums); this module only marshals numpy arrays through
ctypes.  What it computes follows the aiter PR "FlyDSL split-K preshuffle
decode GEMM for small-M shapes (FP8 + MX, gfx950/gfx942)" (Summary, What's
included: per-tensor, blockscale and MX scale modes, fp32 split-K partials,
one downcast at the final store) and the FlyDSL PR "Enable the gmem->LDS
async copy for f16/bf16 preshuffle GEMM" (the bf16 large-M form).
"""
import ctypes
import os

import numpy as np

from . import build as _build

BF16, FP8_TENSOR, FP8_BLOCK128, MXFP8, MXFP4, MXFP8_B32, MXFP4_FP8A = 0, 1, 2, 3, 4, 5, 6
MODE_NAMES = {BF16: "bf16", FP8_TENSOR: "fp8_tensor", FP8_BLOCK128: "fp8_block128",
              MXFP8: "mxfp8", MXFP4: "mxfp4", MXFP8_B32: "mxfp8_b32", MXFP4_FP8A: "mxfp4_fp8a"}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.POINTER(ctypes.c_double)
        L.orc_gemm.argtypes = [ctypes.c_int, i64, i64, i64, vp, vp, vp, vp, i64, i64,
                               vp, i64, ctypes.c_int, vp, ctypes.c_int]
        L.orc_gemm.restype = ctypes.c_int
        L.orc_splitk_range.argtypes = [ctypes.c_int, i64, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.orc_splitk_range.restype = ctypes.c_int
        L.orc_preshuffle_b.argtypes = [vp, i64, i64, vp]
        L.orc_preshuffle_b.restype = ctypes.c_int
        L.orc_unshuffle_b.argtypes = [vp, i64, i64, vp]
        L.orc_unshuffle_b.restype = ctypes.c_int
        L.orc_block64_b.argtypes = [vp, i64, i64, vp]
        L.orc_block64_b.restype = ctypes.c_int
        L.orc_unblock64_b.argtypes = [vp, i64, i64, vp]
        L.orc_unblock64_b.restype = ctypes.c_int
        L.orc_sf_image.argtypes = [ctypes.c_int, vp, i64, i64, vp]
        L.orc_sf_image.restype = ctypes.c_int
        L.orc_round_bf16.argtypes = [vp, i64, vp]
        L.orc_decode_bf16.argtypes = [vp, i64, vp]
        for f in (L.orc_table_e4m3, L.orc_table_e2m1, L.orc_table_e8m0):
            f.argtypes = [dp]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def table_e4m3():
    out = np.empty(256, np.float64)
    lib().orc_table_e4m3(out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def table_e2m1():
    out = np.empty(16, np.float64)
    lib().orc_table_e2m1(out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def table_e8m0():
    out = np.empty(256, np.float64)
    lib().orc_table_e8m0(out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def decode_bf16(bits):
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    lib().orc_decode_bf16(_ptr(bits), bits.size, _ptr(out))
    return out


def default_threads():
    return max(1, os.cpu_count() or 1)


def gemm(mode, A, B, a_scale=None, b_scale=None, M=None, N=None, K=None,
         k_range=None, rows=None, tensor_scale=True, threads=None):
    """fp64 y[rows, :] = sum_{k in k_range} Ad[m, k] * Bd[n, k].

    A, B are the raw codes as numpy arrays: uint16 bf16 bits [M][K],
    uint8 e4m3 codes [M][K], or uint8 packed e2m1 pairs [M][K/2].  Scales:
    fp32 scalars (FP8_TENSOR), fp32 [M][K/128] and [N/128][K/128]
    (FP8_BLOCK128), uint8 E8M0 [M][K/128] (MXFP8) or [M][K/32] (MXFP4,
    MXFP8_B32, MXFP4_FP8A).  MXFP4_FP8A: A e4m3 [M][K], B packed e2m1 [N][K/2].
    ``tensor_scale`` False gives the unscaled per-tensor sum, which is what a
    split-K partial holds in that mode.
    """
    if M is None:
        M = A.shape[0]
    if N is None:
        N = B.shape[0]
    if K is None:
        K = A.shape[1] * (2 if mode == MXFP4 else 1)
    if mode == BF16:
        A, B = _c(A, np.uint16), _c(B, np.uint16)
    else:
        A, B = _c(A, np.uint8), _c(B, np.uint8)
    if mode in (FP8_TENSOR, FP8_BLOCK128):
        a_scale = _c(np.asarray(a_scale, np.float32).reshape(-1), np.float32)
        b_scale = _c(np.asarray(b_scale, np.float32).reshape(-1), np.float32)
    elif mode in (MXFP8, MXFP4, MXFP8_B32, MXFP4_FP8A):
        a_scale, b_scale = _c(a_scale, np.uint8), _c(b_scale, np.uint8)
    else:
        a_scale = b_scale = None
    k0, k1 = (0, K) if k_range is None else k_range
    if rows is not None:
        rows = np.ascontiguousarray(np.asarray(rows, np.int64))
        n_rows = rows.size
    else:
        n_rows = M
    out = np.empty((n_rows, N), np.float64)
    rc = lib().orc_gemm(mode, M, N, K, _ptr(A), _ptr(B), _ptr(a_scale), _ptr(b_scale),
                        k0, k1, _ptr(rows), n_rows, 1 if tensor_scale else 0, _ptr(out),
                        threads or default_threads())
    if rc != 0:
        raise ValueError("orc_gemm rejected its arguments")
    return out


def splitk_range(mode, K, S, s):
    b, e = ctypes.c_int64(), ctypes.c_int64()
    if lib().orc_splitk_range(mode, K, S, s, ctypes.byref(b), ctypes.byref(e)) != 0:
        raise ValueError("bad split arguments")
    return b.value, e.value


def workspace(mode, A, B, a_scale, b_scale, S, **kw):
    """Reference split-K partials ws[s][m][n]; per-tensor partials are unscaled."""
    K = kw.get("K") or A.shape[1] * (2 if mode == MXFP4 else 1)
    parts = [gemm(mode, A, B, a_scale, b_scale, k_range=splitk_range(mode, K, S, s),
                  tensor_scale=False, **kw) for s in range(S)]
    return np.stack(parts)


def preshuffle_b(B_bytes, N, Kb):
    B_bytes = _c(B_bytes, np.uint8)
    out = np.empty(N * Kb, np.uint8)
    if lib().orc_preshuffle_b(_ptr(B_bytes), N, Kb, _ptr(out)) != 0:
        raise ValueError("bad preshuffle shape")
    return out


def unshuffle_b(img, N, Kb):
    img = _c(img, np.uint8)
    out = np.empty((N, Kb), np.uint8)
    if lib().orc_unshuffle_b(_ptr(img), N, Kb, _ptr(out)) != 0:
        raise ValueError("bad preshuffle shape")
    return out


def block64_b(B_bytes, N, Kb):
    """MXFP4_FP8A weight image (layout spec): 128-row x 64-byte blocks of the
    packed fp4 bytes, unswizzled."""
    B_bytes = _c(B_bytes, np.uint8)
    out = np.empty(N * Kb, np.uint8)
    if lib().orc_block64_b(_ptr(B_bytes), N, Kb, _ptr(out)) != 0:
        raise ValueError("bad block shape")
    return out


def unblock64_b(img, N, Kb):
    img = _c(img, np.uint8)
    out = np.empty((N, Kb), np.uint8)
    if lib().orc_unblock64_b(_ptr(img), N, Kb, _ptr(out)) != 0:
        raise ValueError("bad block shape")
    return out


def sf_image(mode, sf, N, K):
    """MX weight-scale image (layout spec), uint8: N/128 * slabs * atoms * 512 bytes
    (MXFP8: N/128 * ceil(slabs / 4) * 512, four 128-K slabs per atom)."""
    sf = _c(sf, np.uint8)
    if mode == MXFP8:
        n_atoms = (N // 128) * (-(-(K // 128) // 4))
    else:
        atoms, slab_k = (2, 256) if mode == MXFP4 else (1, 128)
        n_atoms = (N // 128) * (K // slab_k) * atoms
    out = np.zeros(n_atoms * 512, np.uint8)
    if lib().orc_sf_image(mode, _ptr(sf), N, K, _ptr(out)) != 0:
        raise ValueError("bad scale image arguments")
    return out


def round_bf16(y):
    """fp64 -> fp32 -> bf16 (RNE) bit patterns, as uint16."""
    y = np.ascontiguousarray(y, np.float64)
    out = np.empty(y.shape, np.uint16)
    lib().orc_round_bf16(_ptr(y), y.size, _ptr(out))
    return out
