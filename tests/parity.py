"""Tolerance checks shared by the oracle pins and the GPU parity tests.

The bounds are the ones the method's statement fixes for this GEMM:
  * fp32 split-K workspace:  |ws - ref| <= 1e-5 |ref| + 1e-6 rms(ref)
  * bf16 output Y:           |y - ref|  <= 2e-2 rms(ref) + 2^-8 |ref|   (per element)
  * the weight relayout:     bit-exact
The 2^-8 |ref| term is at least half a bf16 ulp of ref: the rounding of the
output itself, which the 2e-2 rms(ref) bound alone cannot absorb once
|ref| > 10 rms(ref) (heavy-tailed outputs, e.g. block scales spanning four
decades).  Any computational mistake (a lost scale, a lost K block, a sign)
is still orders of magnitude outside the bound.
"""
import numpy as np

WS_REL, WS_ABS_RMS = 1e-5, 1e-6
Y_RMS = 2e-2
Y_ULP = 2.0 ** -8


def rms(x):
    x = np.asarray(x, np.float64)
    return float(np.sqrt(np.mean(x * x))) if x.size else 0.0


def bf16_bits_to_f64(bits):
    bits = np.asarray(bits).view(np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def ws_violations(ws, ref):
    ws = np.asarray(ws, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = WS_REL * np.abs(ref) + WS_ABS_RMS * rms(ref)
    err = np.abs(ws - ref)
    bad = ~(err <= bound)
    return int(np.count_nonzero(bad)), float(np.max(err / np.maximum(bound, 1e-300))) if ws.size else 0.0


def y_violations(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = Y_RMS * rms(ref) + Y_ULP * np.abs(ref)
    err = np.abs(y - ref)
    bad = ~(err <= bound)
    return int(np.count_nonzero(bad)), float(np.max(err / np.maximum(bound, 1e-300))) if y.size else 0.0


def assert_ws_close(ws, ref, what=""):
    n, worst = ws_violations(ws, ref)
    assert n == 0, f"{what}: {n} workspace elements out of tolerance (worst {worst:.3g}x bound)"


def assert_y_close(y, ref, what=""):
    n, worst = y_violations(y, ref)
    assert n == 0, f"{what}: {n} output elements out of tolerance (worst {worst:.3g}x bound)"
