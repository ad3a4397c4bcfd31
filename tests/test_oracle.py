"""Pins of the CPU oracle against things other than itself (no GPU).

Each pin is chosen so that a plausible mistake in the oracle (a dropped
term, a wrong sign, a transposed operand, a wrong scale index, a wrong
nibble order) fails at least one test here:
  * decode tables against an independent dtype library, exhaustively;
  * exact rational brute force (fractions.Fraction) on tiny shapes, with
    values decoded by that independent library;
  * identity and all-ones closed forms ("mxfp4 is bit-exact on the identity
    case", aiter PR "FlyDSL split-K preshuffle decode GEMM for small-M
    shapes", Correctness);
  * split sums that add up exactly to the unsplit result;
  * the weight layout spec: bijective, inverse exact, equal to an
    independent reshape/transpose construction.
"""
from fractions import Fraction

import numpy as np
import pytest

import inputs
import oracle
from tests import parity

ml = pytest.importorskip("ml_dtypes")

MODES = [oracle.BF16, oracle.FP8_TENSOR, oracle.FP8_BLOCK128, oracle.MXFP8, oracle.MXFP4, oracle.MXFP8_B32,
         oracle.MXFP4_FP8A]


def _enc(mode, is_b):
    """Encoding of one operand: MXFP4_FP8A has e4m3 activations (as MXFP8_B32)
    and packed e2m1 weights (as MXFP4); every other mode uses one for both."""
    if mode == oracle.MXFP4_FP8A:
        return oracle.MXFP4 if is_b else oracle.MXFP8_B32
    return mode


# ------------------------------------------------------------ decode tables

def test_e4m3_table_matches_ml_dtypes_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = codes.view(ml.float8_e4m3fn).astype(np.float64)
    got = oracle.table_e4m3()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_e4m3_table_matches_torch_all_codes():
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.table_e4m3()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_e2m1_table_matches_ml_dtypes_all_codes():
    codes = np.arange(16, dtype=np.uint8)
    ref = codes.view(ml.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(ref, oracle.table_e2m1())


def test_e8m0_table_matches_ml_dtypes_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = codes.view(ml.float8_e8m0fnu).astype(np.float64)
    got = oracle.table_e8m0()
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(ref[:255], got[:255])


def test_bf16_decode_matches_torch_all_patterns():
    import torch
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.decode_bf16(bits)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


# --------------------------------------------------------- output rounding

def _bf16_round_cases():
    """fp32 values that a wrong bf16 rounding (truncation, ties away from zero
    or to odd, a lost sign, a flushed subnormal, no overflow to inf, a NaN
    turned into inf) gets wrong: random values over every binade, the exact
    midpoint between every pair of neighbouring finite bf16 values (both
    signs), the values one fp32 ulp either side of those midpoints, +-0,
    fp32 subnormals, the overflow boundary, +-inf and NaNs."""
    g = np.random.default_rng(77)
    rand_bits = g.integers(0, 2 ** 32, 200_000, dtype=np.uint64).astype(np.uint32)
    # every finite non-negative bf16 pattern b and its successor b + 1:
    # their midpoint is b's fp32 pattern + 0x8000 (exact in fp32)
    b = np.arange(0x0000, 0x7F7F, dtype=np.uint32)
    mid = (b << 16) + 0x8000
    near = np.concatenate([mid - 1, mid, mid + 1])
    special = np.array([0x00000000, 0x80000000, 0x00000001, 0x807FFFFF, 0x00400000, 0x00008000,
                        0x7F7F7FFF, 0x7F7F8000, 0x7F7FFFFF, 0xFF7F8000, 0x7F800000, 0xFF800000,
                        0x7FC00000, 0x7F800001, 0xFFFFFFFF, 0x7FBFFFFF], np.uint32)
    bits = np.concatenate([rand_bits, near, near | 0x80000000, special]).astype(np.uint32)
    return bits.view(np.float32)


def test_round_bf16_matches_torch_and_ml_dtypes():
    """orc_round_bf16 (fp64 -> fp32 -> bf16, round to nearest even) against
    two independent casts on fp32-exact inputs, including every tie."""
    import torch
    x32 = _bf16_round_cases()
    got = oracle.round_bf16(x32.astype(np.float64))
    ref_t = torch.from_numpy(x32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    with np.errstate(invalid="ignore"):
        ref_m = x32.astype(ml.bfloat16).view(np.uint16)
    nan = np.isnan(x32)
    # NaN payloads may differ between implementations; a NaN must stay a NaN
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x007F) != 0)
    assert np.array_equal(got[~nan], ref_t[~nan])
    assert np.array_equal(got[~nan], ref_m[~nan])
    # ties go to the even bf16 code: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
    assert oracle.round_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert oracle.round_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82
    assert oracle.round_bf16(np.array([-(1.0 + 2.0 ** -8)]))[0] == 0xBF80


def test_round_bf16_rounds_fp64_through_fp32():
    """The oracle's fp64 results are rounded first to fp32 (the kernels'
    accumulator type) and then to bf16, each step to nearest even -- the
    same as an independent library taking the same two steps."""
    import torch
    g = np.random.default_rng(78)
    x = g.standard_normal(100_000) * np.exp2(g.integers(-30, 30, 100_000))
    got = oracle.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    # a value just above a bf16 midpoint in fp64 that lands exactly on the
    # midpoint in fp32 is decided by the fp32 tie rule (even), as on the GPU
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert oracle.round_bf16(np.array([v]))[0] == 0x3F80


# ------------------------------------------------- independent brute force

def _frac_values(mode, X, S, rows, K, is_b):
    """Exact Fraction dequantised operand, decoded with ml_dtypes."""
    mode = _enc(mode, is_b)
    if mode == oracle.BF16:
        v = X.view(np.uint16).view(ml.bfloat16).astype(np.float64)
    elif mode == oracle.MXFP4:
        lo, hi = X & 15, X >> 4
        nib = np.empty((rows, K), np.uint8)
        nib[:, 0::2], nib[:, 1::2] = lo, hi
        v = nib.view(ml.float4_e2m1fn).astype(np.float64)
    else:
        v = X.view(ml.float8_e4m3fn).astype(np.float64)
    out = [[Fraction(float(v[r, k])) for k in range(K)] for r in range(rows)]
    if mode == oracle.FP8_BLOCK128:
        kb = -(-K // 128)
        for r in range(rows):
            for k in range(K):
                sr = r // 128 if is_b else r
                out[r][k] *= Fraction(float(np.float32(S.reshape(-1)[sr * kb + k // 128])))
    elif mode in (oracle.MXFP8, oracle.MXFP4, oracle.MXFP8_B32):
        blk = 128 if mode == oracle.MXFP8 else 32
        kb = -(-K // blk)
        sv = S.reshape(-1).view(ml.float8_e8m0fnu).astype(np.float64)
        for r in range(rows):
            for k in range(K):
                out[r][k] *= Fraction(float(sv[r * kb + k // blk]))
    return out


def _rand_case(mode, M, N, K, seed):
    g = np.random.default_rng(seed)
    if mode == oracle.BF16:
        A = inputs.to_bf16_bits(g.standard_normal((M, K)).astype(np.float32))
        B = inputs.to_bf16_bits(g.standard_normal((N, K)).astype(np.float32))
        return A, B, None, None
    # all e4m3 codes except the two NaN patterns
    pool = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    A = g.integers(0, 256, (M, K // 2), dtype=np.uint8) if _enc(mode, False) == oracle.MXFP4 else g.choice(pool, (M, K))
    B = g.integers(0, 256, (N, K // 2), dtype=np.uint8) if _enc(mode, True) == oracle.MXFP4 else g.choice(pool, (N, K))
    if mode == oracle.FP8_TENSOR:
        return A, B, np.float32(g.uniform(0.01, 2)), np.float32(g.uniform(0.01, 2))
    if mode == oracle.FP8_BLOCK128:
        kb = -(-K // 128)
        return (A, B, g.uniform(0.01, 3, (M, kb)).astype(np.float32),
                g.uniform(0.01, 3, (-(-N // 128), kb)).astype(np.float32))
    blk = 128 if mode == oracle.MXFP8 else 32
    kb = -(-K // blk)
    # exponents within 2^+-2 keep every partial sum inside fp64's 53 bits at these
    # sizes (products on a 2^-22 grid, |sum| < 2^30), so the oracle must be exact
    return (A, B, g.integers(125, 130, (M, kb), dtype=np.uint8),
            g.integers(125, 130, (N, kb), dtype=np.uint8))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", [(4, 8, 64), (3, 256, 256)])
def test_bruteforce_fraction(mode, shape):
    M, N, K = shape
    if shape == (3, 256, 256) and mode == oracle.BF16:
        N = 16
    A, B, a_s, b_s = _rand_case(mode, M, N, K, seed=7 + mode)
    got = oracle.gemm(mode, A, B, a_s, b_s, M=M, N=N, K=K, threads=2)
    Af = _frac_values(mode, A, a_s, M, K, False)
    Bf = _frac_values(mode, B, b_s, N, K, True)
    ts = Fraction(1)
    if mode == oracle.FP8_TENSOR:
        ts = Fraction(float(a_s)) * Fraction(float(b_s))
    for m in range(M):
        for n in range(N):
            terms = [Af[m][k] * Bf[n][k] for k in range(K)]
            exact = sum(terms, Fraction(0)) * ts
            if mode == oracle.FP8_BLOCK128:
                # fp32 scales make products wider than 53 bits: each product and each
                # partial sum rounds once in fp64, so the error is below K * 2^-52 * sum|terms|
                mag = float(sum(abs(t) for t in terms))
                assert abs(got[m, n] - float(exact)) <= K * 2.0 ** -52 * mag
            elif mode == oracle.FP8_TENSOR:
                # the integer-grid sum is exact; one rounding for the scale product
                assert got[m, n] == pytest.approx(float(exact), rel=4e-16, abs=0)
            else:
                assert got[m, n] == float(exact), (m, n)


def test_bruteforce_catches_transposed_operand():
    """Negative control: reading B as [K][N] instead of [N][K] (square case)
    gives a different result, and the exact brute force picks the right one."""
    A, B, _, _ = _rand_case(oracle.FP8_TENSOR, 4, 64, 64, seed=11)
    y = oracle.gemm(oracle.FP8_TENSOR, A, B, 1.0, 1.0, threads=1)
    y_bad = oracle.gemm(oracle.FP8_TENSOR, A, np.ascontiguousarray(B.T), 1.0, 1.0, threads=1)
    Af = _frac_values(oracle.FP8_TENSOR, A, None, 4, 64, False)
    Bf = _frac_values(oracle.FP8_TENSOR, B, None, 64, 64, True)
    exact = np.array([[float(sum(Af[m][k] * Bf[n][k] for k in range(64))) for n in range(64)]
                      for m in range(4)])
    assert np.array_equal(y, exact)
    assert not np.array_equal(y_bad, exact)
    # and the roles of A and B are symmetric: (A B^T)^T = B A^T
    assert np.array_equal(y, oracle.gemm(oracle.FP8_TENSOR, B, A, 1.0, 1.0, threads=1).T)


# ----------------------------------------------------------- closed forms

ONE = {oracle.BF16: 0x3F80, oracle.FP8_TENSOR: 0x38, oracle.FP8_BLOCK128: 0x38,
       oracle.MXFP8: 0x38, oracle.MXFP4: 0x2, oracle.MXFP8_B32: 0x38}


def _unit_scales(mode, rows, K):
    if mode == oracle.MXFP4_FP8A:
        return np.full((rows, K // 32), 127, np.uint8)
    if mode == oracle.FP8_TENSOR:
        return np.float32(1.0)
    if mode == oracle.FP8_BLOCK128:
        return np.ones((rows, K // 128), np.float32)
    if mode == oracle.MXFP8:
        return np.full((rows, K // 128), 127, np.uint8)
    if mode in (oracle.MXFP4, oracle.MXFP8_B32):
        return np.full((rows, K // 32), 127, np.uint8)
    return None


def _const_operand(mode, rows, K, code):
    """Constant operand in encoding `mode` (an operand encoding, see _enc)."""
    if mode == oracle.BF16:
        return np.full((rows, K), code, np.uint16)
    if mode == oracle.MXFP4:
        return np.full((rows, K // 2), code | (code << 4), np.uint8)
    return np.full((rows, K), code, np.uint8)


def _identity_operand(mode, M, K):
    """Identity rows in the activation encoding of `mode`."""
    mode = _enc(mode, False)
    X = np.zeros((M, K), np.uint16 if mode == oracle.BF16 else np.uint8)
    for m in range(M):
        X[m, m % K] = ONE[mode]
    if mode == oracle.MXFP4:
        X = inputs.pack_e2m1(X)
    return X


@pytest.mark.parametrize("mode", MODES)
def test_identity_closed_form_is_exact(mode):
    M, N, K = 300, 256, 256
    A = _identity_operand(mode, M, K)
    _, B, _, b_s = _rand_case(mode, 1, N, K, seed=3)
    if mode == oracle.BF16:
        B = inputs.to_bf16_bits(np.random.default_rng(5).standard_normal((N, K)).astype(np.float32))
    a_s = _unit_scales(mode, M, K)
    if mode == oracle.FP8_BLOCK128:
        b_s = np.ones_like(b_s) * np.float32(0.5)  # powers of two keep the closed form exact
    y = oracle.gemm(mode, A, B, a_s, b_s, M=M, N=N, K=K, threads=4)
    # closed form: y[m, n] = Bd[n, m mod K]; Bd from the unit-A-scale gemm of B with itself
    Bd = oracle.gemm(mode, _identity_operand(mode, K, K), B, _unit_scales(mode, K, K), b_s,
                     M=K, N=N, K=K, threads=4)            # Bd^T, rows = k
    expect = Bd[np.arange(M) % K, :]
    assert np.array_equal(y, expect)
    # and the decoded weight agrees with the independent library on raw codes
    if _enc(mode, True) == oracle.MXFP4:
        nib = np.empty((N, K), np.uint8)
        nib[:, 0::2], nib[:, 1::2] = B & 15, B >> 4
        vals = nib.view(ml.float4_e2m1fn).astype(np.float64)
        sv = np.repeat(b_s.view(ml.float8_e8m0fnu).astype(np.float64), 32, axis=1)
        assert np.array_equal(Bd.T, vals * sv)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("K", [128, 7168])
def test_all_ones_closed_form(mode, K):
    if mode == oracle.MXFP4 and K % 256:
        pytest.skip("packed fp4 rows are cut in 128-byte (256-element) slabs")
    M, N = 3, 128
    A = _const_operand(_enc(mode, False), M, K, ONE[_enc(mode, False)])
    B = _const_operand(_enc(mode, True), N, K, ONE[_enc(mode, True)])
    a_s, b_s = _unit_scales(mode, M, K), _unit_scales(mode, N, K)
    if mode == oracle.FP8_BLOCK128:
        b_s = np.ones((1, K // 128), np.float32)
    y = oracle.gemm(mode, A, B, a_s, b_s, M=M, N=N, K=K, threads=2)
    assert np.all(y == K)
    # bf16 output of K is exact for K = 7 * 2^10
    assert np.all(parity.bf16_bits_to_f64(oracle.round_bf16(y)) == K)
    for S in (1, 2, 4, 8):
        ws = oracle.workspace(mode, A, B, a_s, b_s, S, M=M, N=N, K=K, threads=2)
        sizes = [e - b for b, e in (oracle.splitk_range(mode, K, S, s) for s in range(S))]
        for s in range(S):
            assert np.all(ws[s] == sizes[s])


def test_tensor_scale_applies_after_sum():
    A = _const_operand(oracle.FP8_TENSOR, 2, 256, ONE[oracle.FP8_TENSOR])
    y = oracle.gemm(oracle.FP8_TENSOR, A, A, np.float32(0.5), np.float32(0.25))
    y0 = oracle.gemm(oracle.FP8_TENSOR, A, A, np.float32(0.5), np.float32(0.25), tensor_scale=False)
    assert np.all(y0 == 256) and np.all(y == 256 * 0.125)


def test_mxfp4_nibble_order_low_is_even_k():
    K = 64
    A = np.zeros((1, K // 2), np.uint8)
    A[0, 3] = 0x20                      # code 2 (=1.0) in the HIGH nibble of byte 3 -> k = 7
    B = np.zeros((128, K), np.uint8)
    B[:, 7] = 0x6                       # 4.0 at k = 7
    B[:, 6] = 0x7                       # 6.0 at k = 6 (must not be picked up)
    Bp = inputs.pack_e2m1(B)
    sf = np.full((1, K // 32), 127, np.uint8)
    y = oracle.gemm(oracle.MXFP4, A, Bp, sf, np.full((128, K // 32), 127, np.uint8), K=K)
    assert np.all(y == 4.0)


# ----------------------------------------------------- split invariance

@pytest.mark.parametrize("mode", [oracle.FP8_TENSOR, oracle.MXFP8, oracle.MXFP4, oracle.MXFP8_B32,
                                  oracle.MXFP4_FP8A])
def test_split_sums_are_exact(mode):
    name = oracle.MODE_NAMES[mode]
    M, N, K = 5, 128, 2048
    A, B, a_s, b_s = inputs.operands(name, M, N, K, 11, 12, 13)
    y = oracle.gemm(mode, A, B, a_s, b_s, tensor_scale=False, threads=4)
    for S in (2, 4, 8):
        ws = oracle.workspace(mode, A, B, a_s, b_s, S, threads=4)
        assert np.array_equal(ws.sum(axis=0), y)
        acc = ws[0].copy()
        for s in range(1, S):
            acc = acc + ws[s]
        assert np.array_equal(acc, y)


@pytest.mark.parametrize("mode", [oracle.BF16, oracle.FP8_BLOCK128])
def test_split_sums_fp64_close(mode):
    name = {oracle.BF16: "bf16", oracle.FP8_BLOCK128: "fp8_block128"}[mode]
    M, N, K = 4, 128, 1024
    A, B, a_s, b_s = inputs.operands(name, M, N, K, 21, 22, 23)
    y = oracle.gemm(mode, A, B, a_s, b_s, threads=4)
    for S in (2, 8):
        ws = oracle.workspace(mode, A, B, a_s, b_s, S, threads=4)
        assert np.allclose(ws.sum(axis=0), y, rtol=1e-13, atol=1e-13 * parity.rms(y))


def test_splitk_partition():
    # fp8 K=7168 -> 56 slabs; fp4 -> 28 slabs
    assert [oracle.splitk_range(oracle.FP8_TENSOR, 7168, 4, s) for s in range(4)] == \
        [(0, 1792), (1792, 3584), (3584, 5376), (5376, 7168)]
    sizes = [(lambda b_e: (b_e[1] - b_e[0]) // 256)(oracle.splitk_range(oracle.MXFP4, 7168, 8, s))
             for s in range(8)]
    assert sizes == [4, 4, 4, 4, 3, 3, 3, 3]
    for mode, K in [(oracle.BF16, 8192), (oracle.FP8_BLOCK128, 7168), (oracle.MXFP4, 7168),
                    (oracle.MXFP8, 128), (oracle.MXFP8_B32, 7168), (oracle.MXFP4_FP8A, 7168),
                    (oracle.MXFP4_FP8A, 384)]:
        for S in (1, 2, 3, 4, 8):
            rs = [oracle.splitk_range(mode, K, S, s) for s in range(S)]
            assert rs[0][0] == 0 and rs[-1][1] == K
            assert all(rs[i][1] == rs[i + 1][0] for i in range(S - 1))
            lens = [e - b for b, e in rs]
            assert max(lens) - min(lens) <= (64 if mode == oracle.BF16 else
                                             256 if mode == oracle.MXFP4 else 128)
    with pytest.raises(ValueError):
        oracle.splitk_range(oracle.FP8_TENSOR, 7100, 2, 0)


# ----------------------------------------------------------- layout spec

def _layout_independent(Bb, N, Kb):
    """The same layout built with reshapes and a gather (no shared code)."""
    x = Bb.reshape(N // 128, 128, Kb // 128, 8, 16)        # nb, r, kb, c, byte
    x = x.transpose(0, 2, 1, 3, 4)                          # nb, kb, r, c, byte
    r = np.arange(128)[:, None]
    c = np.arange(8)[None, :]
    dst_chunk = c ^ (r % 8)                                  # chunk c lands at c ^ (r%8)
    out = np.empty_like(x)
    out[:, :, r, dst_chunk, :] = x[:, :, r, c, :]
    return out.reshape(-1)


@pytest.mark.parametrize("N,Kb", [(128, 128), (256, 384), (384, 1024)])
def test_layout_spec(N, Kb):
    g = np.random.default_rng(N + Kb)
    Bb = g.integers(0, 256, (N, Kb), dtype=np.uint8)
    img = oracle.preshuffle_b(Bb, N, Kb)
    assert np.array_equal(img, _layout_independent(Bb, N, Kb))
    assert np.array_equal(oracle.unshuffle_b(img, N, Kb), Bb)
    # bijection: a buffer of unique 16-byte-chunk indices maps to a permutation of them
    idx = np.arange(N * Kb // 16, dtype=np.uint64)
    chunks = np.zeros((N * Kb // 16, 2), np.uint64)
    chunks[:, 0] = idx
    img2 = oracle.preshuffle_b(chunks.view(np.uint8).reshape(N, Kb), N, Kb)
    moved = img2.view(np.uint64).reshape(-1, 2)[:, 0]
    assert np.array_equal(np.sort(moved), idx)
    # a single slab row keeps its 128 bytes together inside the slab
    KB = Kb // 128
    for n in (0, N - 1):
        for kb in range(KB):
            slab = img[((n // 128) * KB + kb) * 16384:][:16384].reshape(128, 128)
            assert sorted(slab[n % 128].tolist()) == sorted(Bb[n, kb * 128:(kb + 1) * 128].tolist())


@pytest.mark.parametrize("N,Kb", [(128, 64), (256, 192), (384, 3584)])
def test_block64_layout_spec(N, Kb):
    """The fp8-A x fp4-B weight image: 128-row x 64-byte blocks, unswizzled --
    checked against a reshape/transpose restatement, its inverse, and a
    bijection on unique 8-byte ids."""
    g = np.random.default_rng(N + Kb)
    Bb = g.integers(0, 256, (N, Kb), dtype=np.uint8)
    img = oracle.block64_b(Bb, N, Kb)
    indep = Bb.reshape(N // 128, 128, Kb // 64, 64).transpose(0, 2, 1, 3).reshape(-1)
    assert np.array_equal(img, indep)
    assert np.array_equal(oracle.unblock64_b(img, N, Kb), Bb)
    ids = np.arange(N * Kb // 8, dtype=np.uint64)
    moved = oracle.block64_b(ids.view(np.uint8).reshape(N, Kb), N, Kb).view(np.uint64)
    assert np.array_equal(np.sort(moved), ids)


def test_mixed_mode_equals_its_two_encodings():
    """fp8-A x fp4-B is the sum of products of an mxfp8_b32 activation and an
    mxfp4 weight: with the weight's fp4 values rewritten as the e4m3 codes of
    the same numbers (every e2m1 value is an e4m3 value), the mxfp8_b32 oracle
    gives the same bits; the weight's scale image equals mxfp8_b32's."""
    M, N, K = 5, 256, 1024
    A, B, a_s, b_s = inputs.operands("mxfp4_fp8a", M, N, K, 41, 42, 43)
    y = oracle.gemm(oracle.MXFP4_FP8A, A, B, a_s, b_s, threads=2)
    nib = np.empty((N, K), np.uint8)
    nib[:, 0::2], nib[:, 1::2] = B & 15, B >> 4
    B8 = nib.view(ml.float4_e2m1fn).astype(np.float32).astype(ml.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(oracle.table_e2m1()[nib], oracle.table_e4m3()[B8])
    assert np.array_equal(y, oracle.gemm(oracle.MXFP8_B32, A, B8, a_s, b_s, threads=2))
    assert np.array_equal(oracle.sf_image(oracle.MXFP4_FP8A, b_s, N, K), oracle.sf_image(oracle.MXFP8_B32, b_s, N, K))


# ------------------------------------------------------------- inputs

def test_e2m1_rounding_matches_ml_dtypes():
    x = np.concatenate([np.linspace(-6, 6, 4801), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0,
                                                   -0.25, -0.75, -5.0, -0.0]])
    ours = inputs.to_e2m1_codes(x)
    theirs = x.astype(ml.float4_e2m1fn).view(np.uint8) & 15
    vo = ours.view(ml.float4_e2m1fn).astype(np.float64)
    vt = theirs.view(ml.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(vo, vt)


def test_e8m0_choice_bounds_block():
    for fmt, emax in (("mxfp8", 448.0), ("mxfp4", 6.0), ("mxfp8_b32", 448.0)):
        A, sf = inputs.mx_operand(64, 1024, 5, fmt)
        blk = 128 if fmt == "mxfp8" else 32
        x = inputs.randn(64, 1024, 5).reshape(64, -1, blk)
        amax = np.abs(x).max(axis=2).astype(np.float64)
        scale = np.ldexp(1.0, sf.astype(np.int64) - 127)
        assert np.all(amax / scale <= emax) and np.all(amax / scale > emax / 2)


def test_per_tensor_amax_maps_to_448():
    A, s = inputs.fp8_tensor_operand(16, 7168, 1000)
    v = oracle.table_e4m3()[A]
    assert np.max(np.abs(v)) == 448.0


def test_tolerance_check_catches_planted_mistakes():
    """Planted oracle mistakes (dropped scale, transposed operand, sign flip,
    a dropped k term) all fail the output and workspace bounds."""
    M, N, K = 4, 256, 1024
    A, B, a_s, b_s = inputs.operands("fp8_block128", M, N, K, 31, 32, 33)
    ref = oracle.gemm(oracle.FP8_BLOCK128, A, B, a_s, b_s)
    wrong_scale = oracle.gemm(oracle.FP8_BLOCK128, A, B, a_s * 2, b_s)
    assert parity.y_violations(wrong_scale, ref)[0] > 0
    flipped = -ref
    assert parity.y_violations(flipped, ref)[0] > 0
    A2 = A.copy()
    A2[:, 5] = 0
    dropped = oracle.gemm(oracle.FP8_BLOCK128, A2, B, a_s, b_s)
    assert parity.ws_violations(dropped, ref)[0] > 0
    bs_swapped = oracle.gemm(oracle.FP8_BLOCK128, A, B, a_s, b_s[::-1].copy())
    assert parity.y_violations(bs_swapped, ref)[0] > 0


def test_sf_image_spec_is_a_bijection_onto_atoms():
    """Every scale lands in exactly one atom byte (one per 32-K block, or per
    128-K slab for mxfp8, four slabs to an atom); the bytes a short last
    mxfp8 group leaves over are zero."""
    for mode, cols_per_row, K in ((oracle.MXFP4, 7168 // 32, 7168), (oracle.MXFP8_B32, 1024 // 32, 1024),
                                  (oracle.MXFP8, 1024 // 128, 1024), (oracle.MXFP8, 640 // 128, 640)):
        N = 256
        ids = np.arange(N * cols_per_row, dtype=np.int64)
        for byte in range(2):   # unique 16-bit ids, one byte at a time
            sf = ((ids >> (8 * byte)) & 255).astype(np.uint8).reshape(N, cols_per_row)
            img = oracle.sf_image(mode, sf, N, K)
            if byte == 0:
                lo = img.astype(np.int64)
            else:
                hi = img.astype(np.int64)
        got = np.sort(lo | (hi << 8))
        pad = got.size - ids.size
        assert pad == ((N // 128) * 128 * (-cols_per_row % 4) if mode == oracle.MXFP8 else 0)
        assert np.array_equal(got[pad:], np.sort(ids)) and not got[:pad].any()
    # mxfp8: row r's scale for slab u sits at byte 16*(r%32) + 4*(r/32) + u%4 of atom (r/128, u/4)
    N, K = 256, 896
    sf = np.random.default_rng(9).integers(0, 255, (N, K // 128), dtype=np.uint8)
    img = oracle.sf_image(oracle.MXFP8, sf, N, K).reshape(N // 128, 2, 512)
    for r, u in ((0, 0), (37, 5), (200, 6), (255, 3)):
        assert img[r // 128, u // 4, 16 * (r % 128 % 32) + 4 * (r % 128 // 32) + u % 4] == sf[r, u]
