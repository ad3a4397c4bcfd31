"""Python binding of the sm_103a preshuffled-weight GEMM library (libfg.so).

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch supplies device memory and streams.  The functions carry the names
of the C ABI in ``include/fg.h`` without the ``fg_`` prefix.  There is no
fallback: if the library has not been built, loading it raises.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfg.so")

FG_BF16, FG_FP8_TENSOR, FG_FP8_BLOCK128, FG_MXFP8, FG_MXFP4, FG_MXFP8_B32, FG_MXFP4_FP8A = 0, 1, 2, 3, 4, 5, 6
MODES = {"bf16": FG_BF16, "fp8_tensor": FG_FP8_TENSOR, "fp8_block128": FG_FP8_BLOCK128,
         "mxfp8": FG_MXFP8, "mxfp4": FG_MXFP4, "mxfp8_b32": FG_MXFP8_B32, "mxfp4_fp8a": FG_MXFP4_FP8A}
STATUS = ["FG_OK", "FG_ERR_INVALID_ARG", "FG_ERR_SHAPE", "FG_ERR_ALIGN", "FG_ERR_LAYOUT",
          "FG_ERR_WORKSPACE", "FG_ERR_UNSUPPORTED_ARCH", "FG_ERR_CUDA", "FG_ERR_TIMEOUT"]
(FG_OK, FG_ERR_INVALID_ARG, FG_ERR_SHAPE, FG_ERR_ALIGN, FG_ERR_LAYOUT, FG_ERR_WORKSPACE,
 FG_ERR_UNSUPPORTED_ARCH, FG_ERR_CUDA, FG_ERR_TIMEOUT) = range(9)
FG_FLAG_DEFER_REDUCE = 0x1
FG_FLAG_DEBUG_STALL = 0x40000000


class FgError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (STATUS[status] if 0 <= status < len(STATUS) else status, message))
        self.status = status


class BShuf(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32), ("mode", ctypes.c_int32),
                ("tile_rows", ctypes.c_int32), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("data", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("data_bytes", ctypes.c_uint64),
                ("sf_bytes", ctypes.c_uint64), ("check", ctypes.c_uint64)]


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("split_k", ctypes.c_int32), ("tile_m", ctypes.c_int32),
                ("tile_n", ctypes.c_int32), ("stage_slabs", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("ctas", ctypes.c_int32), ("from_table", ctypes.c_int32), ("name", ctypes.c_char * 96)]


_lib = None


def lib():
    """Load libfg.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libfg.so is not built (%s); run mx_gemm_gb300.build.build()" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    i32, i64, u32, u64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_void_p
    sig = {
        "fg_version": ([], i32),
        "fg_status_str": ([i32], ctypes.c_char_p),
        "fg_last_error_message": ([], ctypes.c_char_p),
        "fg_preshuffle_b_size": ([i32, i64, i64, ctypes.POINTER(u64), ctypes.POINTER(u64)], i32),
        "fg_preshuffle_b": ([i32, vp, vp, i64, i64, vp, u64, vp, u64, ctypes.POINTER(BShuf), vp], i32),
        "fg_unshuffle_b": ([ctypes.POINTER(BShuf), vp, vp, vp], i32),
        "fg_gemm_plan": ([i32, i64, i64, i64, i32, ctypes.POINTER(Plan)], i32),
        "fg_gemm_workspace_size": ([i32, i64, i64, i64, i32, ctypes.POINTER(u64)], i32),
        "fg_gemm": ([vp, vp, i64, ctypes.POINTER(BShuf), i32, i32, vp, vp, u64, u32, vp], i32),
        "fg_gemm_splitk_reduce": ([vp, i32, i64, i64, vp, vp, vp, vp], i32),
        "fg_gemm_noalloc": ([vp, vp, i64, ctypes.POINTER(BShuf), i32, i32, vp, u32, vp], i32),
        "fg_get_error": ([], i32),
        "fg_set_wait_timeout_ns": ([u64], None),
        "fg_debug_override_cc": ([i32, i32], None),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def version():
    return lib().fg_version()


def status_str(status):
    return lib().fg_status_str(status).decode()


def last_error_message():
    return lib().fg_last_error_message().decode()


def _check(status):
    if status != FG_OK:
        raise FgError(status, last_error_message())


def _mode(mode):
    return MODES[mode] if isinstance(mode, str) else int(mode)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# ----------------------------------------------------------- argument checks
# The C ABI sees raw bytes: a transposed or sliced view, a tensor on another
# device or of another element type would be read as if it were the row-major
# operand.  These checks (no arithmetic) refuse such tensors with ValueError.

def _dtypes(*names):
    return tuple(getattr(torch, n) for n in names if hasattr(torch, n))


_BYTES = _dtypes("uint8", "int8")
_BF16 = _dtypes("bfloat16", "int16", "uint16")
_FP8 = _BYTES + _dtypes("float8_e4m3fn")
_FP4 = _BYTES + _dtypes("float4_e2m1fn_x2")
_E8M0 = _BYTES + _dtypes("float8_e8m0fnu")
_F32 = (torch.float32,)


def _a_dtypes(mode):
    return {FG_BF16: _BF16, FG_MXFP4: _FP4}.get(mode, _FP8)


def _b_dtypes(mode):
    return {FG_BF16: _BF16, FG_MXFP4: _FP4, FG_MXFP4_FP8A: _FP4}.get(mode, _FP8)


def _a_row_bytes(mode, K):
    return {FG_BF16: 2 * K, FG_MXFP4: K // 2}.get(mode, K)


def _b_row_bytes(mode, K):
    return K // 2 if mode == FG_MXFP4_FP8A else _a_row_bytes(mode, K)


def _scale_spec(mode, rows, K, is_b):
    """(dtypes, element count) of the scales of an operand with `rows` rows."""
    if mode == FG_FP8_TENSOR:
        return _F32, 1
    if mode == FG_FP8_BLOCK128:
        return _F32, ((rows // 128) if is_b else rows) * (K // 128)
    if mode == FG_MXFP8:
        return _E8M0, rows * (K // 128)
    if mode in (FG_MXFP4, FG_MXFP8_B32, FG_MXFP4_FP8A):
        return _E8M0, rows * (K // 32)
    return None, 0


def _require(t, name, dtypes=None, device=None, shape=None, numel=None, min_numel=None):
    if not isinstance(t, torch.Tensor):
        raise ValueError("%s must be a torch.Tensor, got %s" % (name, type(t).__name__))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous row-major memory (shape %s, strides %s): a transposed or "
                         "column-sliced view would be read as raw bytes" % (name, tuple(t.shape), t.stride()))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (it is on %s)" % (name, t.device))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, the other operands on %s" % (name, t.device, device))
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError("%s has dtype %s; expected one of %s" % (name, t.dtype, ", ".join(str(d) for d in dtypes)))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if numel is not None and t.numel() != numel:
        raise ValueError("%s has %d elements, expected %d" % (name, t.numel(), numel))
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError("%s has %d elements, needs at least %d" % (name, t.numel(), min_numel))


def _row_bytes_of(t):
    return t.shape[1] * t.element_size() if t.dim() == 2 else -1


def _check_gemm_args(mode, A, pb, a_scales, Y):
    dev = pb.data.device
    _require(A, "A", _a_dtypes(mode), dev)
    M = A.shape[0] if A.dim() == 2 else -1
    if A.dim() != 2 or _row_bytes_of(A) != _a_row_bytes(mode, pb.K):
        raise ValueError("A must be [M][K] codes of the mode (%d bytes per row for K=%d), got shape %s dtype %s"
                         % (_a_row_bytes(mode, pb.K), pb.K, tuple(A.shape), A.dtype))
    # a missing scale tensor or a mode that differs from the weight's is the
    # library's to report (FG_ERR_INVALID_ARG / FG_ERR_LAYOUT)
    if a_scales is not None and mode == pb.mode and mode != FG_BF16:
        dts, n = _scale_spec(mode, M, pb.K, False)
        _require(a_scales, "a_scales", dts, dev, numel=n)
    if Y is not None:
        _require(Y, "Y", _dtypes("bfloat16", "int16"), dev, shape=(M, pb.N))
    return M


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def set_wait_timeout_ns(ns):
    lib().fg_set_wait_timeout_ns(int(ns))


def debug_override_cc(major, minor=0):
    lib().fg_debug_override_cc(int(major), int(minor))


def get_error():
    """Synchronise and return (and clear) the kernels' error word as a status code."""
    return lib().fg_get_error()


def preshuffle_b_size(mode, N, K):
    b, s = ctypes.c_uint64(), ctypes.c_uint64()
    _check(lib().fg_preshuffle_b_size(_mode(mode), N, K, ctypes.byref(b), ctypes.byref(s)))
    return b.value, s.value


class PreshuffledB:
    """A preshuffled weight: the descriptor plus the device buffers it points at."""

    def __init__(self, desc, data, sf):
        self.desc, self.data, self.sf = desc, data, sf

    @property
    def mode(self):
        return self.desc.mode

    @property
    def N(self):
        return self.desc.N

    @property
    def K(self):
        return self.desc.K


def preshuffle_b(mode, B, b_scales=None, K=None, stream=None):
    """One-time relayout of weight B (device tensor [N][K] bf16 / uint8 codes /
    packed fp4 [N][K/2]) and its scales; returns a PreshuffledB."""
    mode = _mode(mode)
    _require(B, "B", _b_dtypes(mode))
    if B.dim() != 2:
        raise ValueError("B must be 2-D [N][K] codes, got shape %s" % (tuple(B.shape),))
    N = B.shape[0]
    rb = _row_bytes_of(B)
    if K is None:
        K = {FG_BF16: rb // 2, FG_MXFP4: 2 * rb, FG_MXFP4_FP8A: 2 * rb}.get(mode, rb)
    if rb != _b_row_bytes(mode, K):
        raise ValueError("B has %d bytes per row; K=%d needs %d" % (rb, K, _b_row_bytes(mode, K)))
    if b_scales is not None and mode != FG_BF16:
        dts, n = _scale_spec(mode, N, K, True)
        _require(b_scales, "b_scales", dts, B.device, numel=n)
    nb, ns = preshuffle_b_size(mode, N, K)
    data = torch.empty(nb, dtype=torch.uint8, device=B.device)
    sf = torch.empty(max(ns, 16), dtype=torch.uint8, device=B.device) if ns else None
    desc = BShuf()
    _check(lib().fg_preshuffle_b(mode, _ptr(B), _ptr(b_scales), N, K, _ptr(data), nb, _ptr(sf), ns,
                                 ctypes.byref(desc), _stream(stream)))
    return PreshuffledB(desc, data, sf)


def unshuffle_b(pb, stream=None):
    """Inverse relayout: (B bytes [N][Kb] uint8, scales in the caller layout or None)."""
    mode, N, K = pb.mode, pb.N, pb.K
    kb = K * (2 if mode == FG_BF16 else 1) // (2 if mode in (FG_MXFP4, FG_MXFP4_FP8A) else 1)
    B = torch.empty((N, kb), dtype=torch.uint8, device=pb.data.device)
    sc = None
    if mode == FG_FP8_TENSOR:
        sc = torch.empty(1, dtype=torch.float32, device=B.device)
    elif mode == FG_FP8_BLOCK128:
        sc = torch.empty((N // 128, K // 128), dtype=torch.float32, device=B.device)
    elif mode == FG_MXFP8:
        sc = torch.empty((N, K // 128), dtype=torch.uint8, device=B.device)
    elif mode in (FG_MXFP4, FG_MXFP8_B32, FG_MXFP4_FP8A):
        sc = torch.empty((N, K // 32), dtype=torch.uint8, device=B.device)
    _check(lib().fg_unshuffle_b(ctypes.byref(pb.desc), _ptr(B), _ptr(sc), _stream(stream)))
    return B, sc


def gemm_plan(mode, M, N, K, split_k=0):
    p = Plan()
    _check(lib().fg_gemm_plan(_mode(mode), M, N, K, split_k, ctypes.byref(p)))
    return {"path": p.path, "split_k": p.split_k, "tile_m": p.tile_m, "tile_n": p.tile_n,
            "stage_slabs": p.stage_slabs, "stages": p.stages, "ctas": p.ctas,
            "from_table": bool(p.from_table), "name": p.name.decode()}


def gemm_workspace_size(mode, M, N, K, split_k=0):
    b = ctypes.c_uint64()
    _check(lib().fg_gemm_workspace_size(_mode(mode), M, N, K, split_k, ctypes.byref(b)))
    return b.value


def gemm(A, pb, a_scales=None, mode=None, split_k=0, Y=None, workspace=None, flags=0, stream=None):
    """Y[M][N] (bf16) = dequant(A) . dequant(B)^T for the preshuffled weight pb.

    A is the device tensor of codes ([M][K] bf16 or uint8, or packed fp4
    [M][K/2]).  A workspace is allocated here when the resolved split needs
    one and none is given.  Returns Y.
    """
    mode = pb.mode if mode is None else _mode(mode)
    M = _check_gemm_args(mode, A, pb, a_scales, Y)
    if Y is None:
        Y = torch.empty((M, pb.N), dtype=torch.bfloat16, device=A.device)
    if workspace is not None:
        _require(workspace, "workspace", device=A.device)
    ws_bytes = 0
    if workspace is None:
        need = gemm_workspace_size(mode, M, pb.N, pb.K, split_k) if M > 0 else 0
        if need:
            workspace = torch.empty(need // 4, dtype=torch.float32, device=A.device)
    if workspace is not None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().fg_gemm(_ptr(A), _ptr(a_scales), M, ctypes.byref(pb.desc), mode, split_k, _ptr(Y),
                         _ptr(workspace), ws_bytes, flags, _stream(stream)))
    return Y


def gemm_noalloc(A, pb, Y, a_scales=None, mode=None, split_k=0, flags=0, stream=None):
    """gemm() for callers that cannot allocate device memory: whatever would
    need a workspace goes to the library's built-in 8 MiB scratch (see
    fg_gemm_noalloc in include/fg.h).  The caller passes Y (this wrapper
    allocates nothing either); returns Y."""
    mode = pb.mode if mode is None else _mode(mode)
    if Y is None:
        raise ValueError("gemm_noalloc needs the caller's output Y (it allocates nothing)")
    _check_gemm_args(mode, A, pb, a_scales, Y)
    _check(lib().fg_gemm_noalloc(_ptr(A), _ptr(a_scales), A.shape[0], ctypes.byref(pb.desc), mode, split_k,
                                 _ptr(Y), flags, _stream(stream)))
    return Y


def gemm_splitk_reduce(ws, split_k, M, N, a_s=None, b_s=None, Y=None, stream=None):
    _require(ws, "ws", _F32, min_numel=split_k * M * N)
    for name, t in (("a_s", a_s), ("b_s", b_s)):
        if t is not None:
            _require(t, name, _F32, ws.device, numel=1)
    if Y is not None:
        _require(Y, "Y", _dtypes("bfloat16", "int16"), ws.device, shape=(M, N))
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=ws.device)
    _check(lib().fg_gemm_splitk_reduce(_ptr(ws), split_k, M, N, _ptr(a_s), _ptr(b_s), _ptr(Y),
                                       _stream(stream)))
    return Y
