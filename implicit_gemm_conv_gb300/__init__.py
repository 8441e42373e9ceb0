"""Stream-K GEMM, implicit-GEMM conv wgrad and fp8 row/col GEMM on one GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/skgemm.h`` (``libskgemm.so``, built in-tree by
``implicit_gemm_conv_gb300/build.py``). The functions carry the C names; they only marshal
arguments: torch tensors supply device pointers and the current CUDA stream, and every step of the
computation runs in the library's kernels. There is no fallback: importing this package fails if the
library is missing, and every call raises ``SkError`` on a non-zero return code.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libskgemm.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python implicit_gemm_conv_gb300/build.py` "
                      "(or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)

F16, BF16, F32, E4M3 = 0, 1, 2, 3
OFF, DP_SK, PERSISTENT, SPLITK, AUTO, HYBRID = 0, 1, 2, 3, 4, 5
LINEAR, TREE, ATOMIC, WORKSPACE, REDUCTION_AUTO = 0, 1, 2, 3, 4
OP_GEMM, OP_FP8_ROWCOL, OP_WGRAD, OP_FPROP, OP_DGRAD, OP_FP8_BLOCK = 0, 1, 2, 3, 4, 5
SEG_FULL, SEG_OWNER, SEG_PEER = 0, 1, 2
TILE_AUTO, TILE_128, TILE_256_PAIR, TILE_256x256_PAIR = 0, 1, 2, 3

MODES = {"off": OFF, "dp_sk": DP_SK, "persistent": PERSISTENT, "splitk": SPLITK, "auto": AUTO,
         "hybrid": HYBRID}
REDUCTIONS = {"linear": LINEAR, "tree": TREE, "atomic": ATOMIC, "workspace": WORKSPACE,
              "auto": REDUCTION_AUTO}
DTYPES = {"f16": F16, "bf16": BF16, "f32": F32, "e4m3": E4M3}
TILES = {"auto": TILE_AUTO, "128": TILE_128, "256_pair": TILE_256_PAIR,
         "256x256_pair": TILE_256x256_PAIR}

_i64, _i32, _p, _sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t


class sk_problem(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("ab_dtype", ctypes.c_int32), ("c_dtype", ctypes.c_int32),
                ("groups", ctypes.c_int32), ("M", _i64), ("N", _i64), ("K", _i64),
                ("n", _i64), ("h", _i64), ("w", _i64), ("c", _i64), ("k", _i64), ("r", _i64),
                ("s", _i64), ("stride_h", ctypes.c_int32), ("stride_w", ctypes.c_int32),
                ("pad_h", ctypes.c_int32), ("pad_w", ctypes.c_int32)]


PLAN_FIELDS = ["op", "mode", "reduction", "tm", "tn", "tk", "gemm_m", "gemm_n", "kred", "groups",
               "tiles_m", "tiles_n", "tiles", "iters_per_tile", "pool", "sk_tiles", "dp_tiles",
               "sk_ctas", "sk_iters", "iters_per_sk_cta", "extra_iters", "splits", "grid",
               "publishers", "max_contributors", "tree_rounds", "shared_tiles", "flag_bytes",
               "control_offset", "partial_offset", "partial_bytes", "scratch_offset",
               "scratch_bytes", "ws_bytes", "partial_slots"]


class sk_plan_t(ctypes.Structure):
    _fields_ = [(f, _i64) for f in PLAN_FIELDS]

    def as_dict(self):
        return {f: getattr(self, f) for f in PLAN_FIELDS}


class sk_segment_t(ctypes.Structure):
    _fields_ = [(f, _i64) for f in ("tile", "k_begin", "k_end", "kind", "index", "n_contrib",
                                    "first_cta")]


_lib.sk_gemm_rcr.argtypes = [_i32, _i32, _i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64, _i32, _i32,
                             _i32, _p, _sz, _p]
_lib.sk_gemm_rowcol_fp8.argtypes = [_i64, _i64, _i64, _p, _p, _p, _p, _p, _i64, _i32, _i32, _i32,
                                    _p, _sz, _p]
_lib.sk_conv2d_wgrad_nhwc.argtypes = [_i32, _i32, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i32,
                                      _i32, _i32, _i32, _i32, _p, _p, _p, _i32, _i32, _i32, _p,
                                      _sz, _p]
_lib.sk_gemm_tensorquant_fp8.argtypes = [_i64, _i64, _i64, _p, _p, ctypes.c_float, ctypes.c_float,
                                         _p, _i64, _i32, _i32, _i32, _p, _sz, _p]
_lib.sk_gemm_blockscale_fp8.argtypes = [_i64, _i64, _i64, _p, _p, _p, _i64, _p, _i64, _i64, _p,
                                        _i64, _i32, _i32, _i32, _p, _sz, _p]
_lib.sk_conv2d_fprop_nhwc.argtypes = _lib.sk_conv2d_wgrad_nhwc.argtypes
_lib.sk_conv2d_dgrad_nhwc.argtypes = _lib.sk_conv2d_wgrad_nhwc.argtypes
_lib.sk_workspace_bytes.argtypes = [ctypes.POINTER(sk_problem), _i32, _i32, _i32,
                                    ctypes.POINTER(_sz)]
_lib.sk_plan.argtypes = [ctypes.POINTER(sk_problem), _i32, _i32, _i32, _i32,
                         ctypes.POINTER(sk_plan_t)]
_lib.sk_plan_cta_work.argtypes = [ctypes.POINTER(sk_plan_t), _i64, ctypes.POINTER(sk_segment_t),
                                  _i32, ctypes.POINTER(_i32)]
_lib.sk_default_pool.argtypes = [_i32, _i32, _i32, ctypes.POINTER(_i32)]
_lib.sk_device_status.argtypes = [_p]
_lib.sk_probe_flag_timeout.argtypes = [_i32, _p]
_lib.sk_last_error.restype = ctypes.c_char_p
_lib.sk_version.restype = _i32
_lib.sk_gemm_rcr_static_ws.argtypes = [_i32, _i32, _i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64,
                                       _i32, _i32, _i32, _p]
_lib.sk_timing_enable.argtypes = [_i32]
_lib.sk_set_tile.argtypes = [_i32]
_lib.sk_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_i64),
                                ctypes.POINTER(_i64)]

EXPORTS = ["sk_gemm_rcr", "sk_gemm_rowcol_fp8", "sk_conv2d_wgrad_nhwc", "sk_workspace_bytes",
           "sk_plan", "sk_plan_cta_work", "sk_default_pool", "sk_device_status", "sk_last_error",
           "sk_version", "sk_timing_enable", "sk_timing_read", "sk_gemm_rcr_static_ws",
           "sk_set_tile", "sk_conv2d_fprop_nhwc", "sk_conv2d_dgrad_nhwc",
           "sk_gemm_tensorquant_fp8", "sk_gemm_blockscale_fp8", "sk_probe_flag_timeout"]


class SkError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"skgemm error {code}: {msg}")
        self.code = code


def library() -> ctypes.CDLL:
    return _lib


def last_error() -> str:
    return _lib.sk_last_error().decode()


def _check(rc: int) -> int:
    if rc != 0:
        raise SkError(rc, last_error())
    return rc


def _code(table, v):
    return table[v] if isinstance(v, str) else int(v)


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _torch_dtype_code(t) -> int:
    import torch
    return {torch.float16: F16, torch.bfloat16: BF16, torch.float32: F32,
            torch.float8_e4m3fn: E4M3}[t.dtype]


def _ws(ws):
    if ws is None:
        return None, 0
    return ws.data_ptr(), ws.numel() * ws.element_size()


def sk_set_tile(tile) -> int:
    """Tile shape for later calls of this thread ("auto", "128", "256_pair", "256x256_pair" or the
    TILE_* code); returns the previous code."""
    rc = _lib.sk_set_tile(_code(TILES, tile))
    if rc < 0:
        raise SkError(rc, last_error())
    return rc


@contextlib.contextmanager
def tile(t):
    """``with tile("256x256_pair"): ...`` -- sk_set_tile for the block, restored afterwards."""
    prev = sk_set_tile(t)
    try:
        yield
    finally:
        sk_set_tile(prev)


# ---- compute calls -----------------------------------------------------------------------------

def sk_gemm_rcr(A, B, C, streamk="dp_sk", reduction="linear", ctas=-1, ws=None, stream=None):
    """C = A @ B.T for A [M, K], B [N, K] (i.e. B column-major K x N), C [M, N] (row-major, any
    leading dimension). fp32 accumulation."""
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K and C.shape == (M, N)
    assert A.stride(1) == 1 and B.stride(1) == 1 and C.stride(1) == 1
    wp, wb = _ws(ws)
    return _check(_lib.sk_gemm_rcr(_torch_dtype_code(A), _torch_dtype_code(C), M, N, K,
                                   A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                                   C.data_ptr(), C.stride(0), _code(MODES, streamk),
                                   _code(REDUCTIONS, reduction), ctas, wp, wb, _stream_ptr(stream)))


def sk_gemm_rcr_static_ws(A, B, C, streamk="dp_sk", reduction="linear", ctas=-1, stream=None):
    """sk_gemm_rcr using the library's fixed 16 MiB device scratch instead of a workspace: for
    callers that must not allocate device memory during the call. Calls sharing the scratch must
    be ordered on one stream."""
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K and C.shape == (M, N)
    assert A.stride(1) == 1 and B.stride(1) == 1 and C.stride(1) == 1
    return _check(_lib.sk_gemm_rcr_static_ws(_torch_dtype_code(A), _torch_dtype_code(C), M, N, K,
                                             A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                                             C.data_ptr(), C.stride(0), _code(MODES, streamk),
                                             _code(REDUCTIONS, reduction), ctas,
                                             _stream_ptr(stream)))


def sk_gemm_rowcol_fp8(A8, B8, sa, sb, C, streamk="dp_sk", reduction="linear", ctas=-1, ws=None,
                       stream=None):
    """C[m, n] = bf16((A8 @ B8.T)[m, n] * sa[m] * sb[n]); A8 [M, K], B8 [N, K] e4m3 (or uint8)."""
    import torch
    M, K = A8.shape
    N = B8.shape[0]
    if A8.element_size() != 1 or B8.element_size() != 1:
        raise TypeError("A8 and B8 must hold one byte per element (float8_e4m3fn or uint8)")
    if sa.dtype != torch.float32 or sb.dtype != torch.float32:
        raise TypeError("sa and sb must be float32")
    if C.dtype != torch.bfloat16:
        raise TypeError("C must be bfloat16")
    assert A8.is_contiguous() and B8.is_contiguous() and C.stride(1) == 1
    wp, wb = _ws(ws)
    return _check(_lib.sk_gemm_rowcol_fp8(M, N, K, A8.data_ptr(), B8.data_ptr(), sa.data_ptr(),
                                          sb.data_ptr(), C.data_ptr(), C.stride(0),
                                          _code(MODES, streamk), _code(REDUCTIONS, reduction),
                                          ctas, wp, wb, _stream_ptr(stream)))


def sk_gemm_tensorquant_fp8(A8, B8, scale_a, scale_b, C, streamk="dp_sk", reduction="linear",
                            ctas=-1, ws=None, stream=None):
    """C [M, N] bf16 = (A8 @ B8.T) * scale_a * scale_b for e4m3 A8 [M, K], B8 [N, K] and two
    scalar (per-tensor) scales."""
    M, K = A8.shape
    N = B8.shape[0]
    assert A8.is_contiguous() and B8.is_contiguous() and C.stride(1) == 1
    wp, wb = _ws(ws)
    return _check(_lib.sk_gemm_tensorquant_fp8(M, N, K, A8.data_ptr(), B8.data_ptr(),
                                               float(scale_a), float(scale_b), C.data_ptr(),
                                               C.stride(0), _code(MODES, streamk),
                                               _code(REDUCTIONS, reduction), ctas, wp, wb,
                                               _stream_ptr(stream)))


def sk_gemm_blockscale_fp8(A8, B8, sa, a_group_k, sb, b_group_n, b_group_k, C, streamk="dp_sk",
                           reduction="linear", ctas=-1, ws=None, stream=None):
    """C [M, N] bf16 = sum_k A8[m, k] * B8[n, k] * sa[m, k // a_group_k] *
    sb[n // b_group_n, k // b_group_k] for e4m3 A8 [M, K], B8 [N, K]; sa [M, ceil(K/a_group_k)]
    and sb [ceil(N/b_group_n), ceil(K/b_group_k)] float32, either may be None (scale 1)."""
    import torch
    M, K = A8.shape
    N = B8.shape[0]
    if A8.element_size() != 1 or B8.element_size() != 1:
        raise TypeError("A8 and B8 must hold one byte per element (float8_e4m3fn or uint8)")
    for name, t in (("sa", sa), ("sb", sb)):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise TypeError(f"{name} must be a contiguous float32 tensor")
    if C.dtype != torch.bfloat16:
        raise TypeError("C must be bfloat16")
    assert A8.is_contiguous() and B8.is_contiguous() and C.stride(1) == 1
    wp, wb = _ws(ws)
    return _check(_lib.sk_gemm_blockscale_fp8(
        M, N, K, A8.data_ptr(), B8.data_ptr(), None if sa is None else sa.data_ptr(), a_group_k,
        None if sb is None else sb.data_ptr(), b_group_n, b_group_k, C.data_ptr(), C.stride(0),
        _code(MODES, streamk), _code(REDUCTIONS, reduction), ctas, wp, wb, _stream_ptr(stream)))


def sk_conv2d_wgrad_nhwc(x, dy, dw, R, S, stride=(1, 1), pad=(0, 0), groups=1, streamk="dp_sk",
                         reduction="linear", ctas=-1, ws=None, stream=None):
    """dw [K, R, S, C/groups] = backward-weight of a 2-D convolution with NHWC x [N, H, W, C] and
    dy [N, Ho, Wo, K]."""
    N, H, W, C = x.shape
    K = dy.shape[3]
    assert x.is_contiguous() and dy.is_contiguous() and dw.is_contiguous()
    wp, wb = _ws(ws)
    return _check(_lib.sk_conv2d_wgrad_nhwc(_torch_dtype_code(x), _torch_dtype_code(dw), N, H, W, C,
                                            K, R, S, stride[0], stride[1], pad[0], pad[1], groups,
                                            x.data_ptr(), dy.data_ptr(), dw.data_ptr(),
                                            _code(MODES, streamk), _code(REDUCTIONS, reduction),
                                            ctas, wp, wb, _stream_ptr(stream)))


def sk_conv2d_fprop_nhwc(x, w, y, stride=(1, 1), pad=(0, 0), groups=1, streamk="dp_sk",
                         reduction="linear", ctas=-1, ws=None, stream=None):
    """y [N, Ho, Wo, K] = forward 2-D convolution of NHWC x [N, H, W, C] with the KRSC filter
    w [K, R, S, C/groups]."""
    N, H, W, C = x.shape
    K, R, S = w.shape[0], w.shape[1], w.shape[2]
    assert x.is_contiguous() and w.is_contiguous() and y.is_contiguous()
    wp, wb = _ws(ws)
    return _check(_lib.sk_conv2d_fprop_nhwc(_torch_dtype_code(x), _torch_dtype_code(y), N, H, W, C,
                                            K, R, S, stride[0], stride[1], pad[0], pad[1], groups,
                                            x.data_ptr(), w.data_ptr(), y.data_ptr(),
                                            _code(MODES, streamk), _code(REDUCTIONS, reduction),
                                            ctas, wp, wb, _stream_ptr(stream)))


def sk_conv2d_dgrad_nhwc(dy, w, dx, stride=(1, 1), pad=(0, 0), groups=1, streamk="dp_sk",
                         reduction="linear", ctas=-1, ws=None, stream=None):
    """dx [N, H, W, C] = data gradient of a 2-D convolution, from NHWC dy [N, Ho, Wo, K] and the
    KRSC filter w [K, R, S, C/groups]; dx's shape gives the input size. Strides 1..8 (a stride
    above 1 runs one launch per output phase)."""
    N, H, W, C = dx.shape
    K, R, S = w.shape[0], w.shape[1], w.shape[2]
    assert dy.is_contiguous() and w.is_contiguous() and dx.is_contiguous()
    wp, wb = _ws(ws)
    return _check(_lib.sk_conv2d_dgrad_nhwc(_torch_dtype_code(dy), _torch_dtype_code(dx), N, H, W,
                                            C, K, R, S, stride[0], stride[1], pad[0], pad[1], groups,
                                            dy.data_ptr(), w.data_ptr(), dx.data_ptr(),
                                            _code(MODES, streamk), _code(REDUCTIONS, reduction),
                                            ctas, wp, wb, _stream_ptr(stream)))


# ---- planning (host only) --------------------------------------------------------------------

def make_problem(op, **kw) -> sk_problem:
    p = sk_problem()
    p.op = _code({"gemm": OP_GEMM, "fp8": OP_FP8_ROWCOL, "wgrad": OP_WGRAD, "fprop": OP_FPROP,
                  "dgrad": OP_DGRAD, "fp8_block": OP_FP8_BLOCK}, op)
    p.groups = 1
    for k, v in kw.items():
        if k in ("ab_dtype", "c_dtype"):
            v = _code(DTYPES, v)
        setattr(p, k, v)
    return p


def sk_plan(problem: sk_problem, streamk, reduction, ctas=-1, num_sms=0) -> sk_plan_t:
    out = sk_plan_t()
    _check(_lib.sk_plan(ctypes.byref(problem), _code(MODES, streamk), _code(REDUCTIONS, reduction),
                        ctas, num_sms, ctypes.byref(out)))
    return out


def sk_plan_cta_work(plan: sk_plan_t, cta: int):
    n = _i32(0)
    _check(_lib.sk_plan_cta_work(ctypes.byref(plan), cta, None, 0, ctypes.byref(n)))
    buf = (sk_segment_t * max(1, n.value))()
    _check(_lib.sk_plan_cta_work(ctypes.byref(plan), cta, buf, n.value, ctypes.byref(n)))
    return [buf[i] for i in range(n.value)]


def sk_default_pool(reduction, num_sms: int, ctas_per_sm: int) -> int:
    out = _i32(0)
    _check(_lib.sk_default_pool(_code(REDUCTIONS, reduction), num_sms, ctas_per_sm,
                                ctypes.byref(out)))
    return out.value


def sk_workspace_bytes(problem: sk_problem, streamk, reduction, ctas=-1) -> int:
    out = _sz(0)
    _check(_lib.sk_workspace_bytes(ctypes.byref(problem), _code(MODES, streamk),
                                   _code(REDUCTIONS, reduction), ctas, ctypes.byref(out)))
    return out.value


def sk_device_status(stream=None) -> int:
    return _check(_lib.sk_device_status(_stream_ptr(stream)))


def sk_probe_flag_timeout(timeout_ms: int = 20, stream=None) -> int:
    """Failure-detection self-test: a bounded flag wait that runs out after timeout_ms; the next
    sk_device_status on the stream raises SkError(-1) with the hand-off timeout message."""
    return _check(_lib.sk_probe_flag_timeout(int(timeout_ms), _stream_ptr(stream)))


def sk_version() -> int:
    return _lib.sk_version()


def sk_last_error() -> str:
    return last_error()


def sk_timing_enable(on: bool = True) -> int:
    return _check(_lib.sk_timing_enable(1 if on else 0))


def sk_timing_read():
    """(summed main-kernel ms, main-kernel launches, all library kernel launches) since the last
    enable/read; clears the records."""
    ms, n_main, n_all = ctypes.c_double(0), _i64(0), _i64(0)
    _check(_lib.sk_timing_read(ctypes.byref(ms), ctypes.byref(n_main), ctypes.byref(n_all)))
    return ms.value, n_main.value, n_all.value

