"""ctypes front end of the fp64 C oracle (``oracle/ref.c``) plus the rounding step to the output
type.

TEST INFRASTRUCTURE. Part of the CPU oracle; see ``oracle/__init__.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

from . import codec

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref.c")
_LIB = os.path.join(_HERE, "_build", "liboracle_ref.so")

FMT = {"f16": 0, "bf16": 1, "e4m3": 3}

_lib = None


def build(force: bool = False) -> str:
    """Compile ``ref.c`` with the host gcc (OpenMP, -O2, no fast-math). Returns the library path."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC", "-std=c11",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, p, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.oracle_decode.argtypes = [i32, p, i64, p]
        lib.oracle_threads.argtypes = [i32]
        lib.oracle_threads.restype = i32
        lib.oracle_gemm_rcr_points.argtypes = [i32, i64, p, i64, p, i64, p, p, i64, p, i32]
        lib.oracle_gemm_rcr_rows.argtypes = [i32, i64, i64, i64, i64, p, i64, p, i64, p, i32]
        lib.oracle_fp8_rowcol_points.argtypes = [i64, p, i64, p, i64, p, p, p, p, i64, p, i32]
        lib.oracle_fp8_rowcol_rows.argtypes = [i64, i64, i64, i64, p, i64, p, i64, p, p, p, i32]
        lib.oracle_wgrad_nhwc.argtypes = [i32, i64, i64, i64, i64, i64, i64, i64, i32, i32, i32,
                                          i32, i32, p, p, i64, i64, p, i32]
        lib.oracle_fp8_blockscale_points.argtypes = [i64, i64, i64, p, p, p, i64, p, i64, i64, p,
                                                     p, i64, p, i32]
        lib.oracle_fprop_nhwc.argtypes = [i32, i64, i64, i64, i64, i64, i64, i64, i32, i32, i32,
                                          i32, i32, p, p, i64, i64, p, i32]
        lib.oracle_dgrad_nhwc.argtypes = [i32, i64, i64, i64, i64, i64, i64, i64, i32, i32, i32,
                                          i32, i32, p, p, i64, i64, p, i32]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def threads(n: int = 0) -> int:
    """Number of OpenMP threads the oracle uses (``n > 0`` sets it)."""
    return _load().oracle_threads(n)


def decode(bits: np.ndarray, fmt: str) -> np.ndarray:
    """The C decoder (the one the numerics use), for pinning."""
    bits = np.ascontiguousarray(bits)
    out = np.empty(bits.size, dtype=np.float64)
    _load().oracle_decode(FMT[fmt], _ptr(bits), bits.size, _ptr(out))
    return out.reshape(bits.shape)


def gemm_rcr_rows(fmt, A_bits, B_bits, m0=0, m1=None, nthreads=0):
    """fp64 C[m0:m1, :] of C = A * B^T for A [M][K], B [N][K] given as 16-bit patterns."""
    A = np.ascontiguousarray(A_bits, dtype=np.uint16)
    B = np.ascontiguousarray(B_bits, dtype=np.uint16)
    M, K = A.shape
    N = B.shape[0]
    m1 = M if m1 is None else m1
    out = np.empty((m1 - m0, N), dtype=np.float64)
    _load().oracle_gemm_rcr_rows(FMT[fmt], m0, m1, N, K, _ptr(A), K, _ptr(B), K, _ptr(out), nthreads)
    return out


def gemm_rcr_points(fmt, A_bits, B_bits, ms, ns, nthreads=0):
    A = np.ascontiguousarray(A_bits, dtype=np.uint16)
    B = np.ascontiguousarray(B_bits, dtype=np.uint16)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.size, dtype=np.float64)
    K = A.shape[1]
    _load().oracle_gemm_rcr_points(FMT[fmt], K, _ptr(A), K, _ptr(B), K, _ptr(ms), _ptr(ns),
                                   ms.size, _ptr(out), nthreads)
    return out


def fp8_rowcol_rows(A8, B8, sa, sb, m0=0, m1=None, nthreads=0):
    A = np.ascontiguousarray(A8, dtype=np.uint8)
    B = np.ascontiguousarray(B8, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    M, K = A.shape
    N = B.shape[0]
    m1 = M if m1 is None else m1
    out = np.empty((m1 - m0, N), dtype=np.float64)
    _load().oracle_fp8_rowcol_rows(m0, m1, N, K, _ptr(A), K, _ptr(B), K, _ptr(sa), _ptr(sb),
                                   _ptr(out), nthreads)
    return out


def fp8_rowcol_points(A8, B8, sa, sb, ms, ns, nthreads=0):
    A = np.ascontiguousarray(A8, dtype=np.uint8)
    B = np.ascontiguousarray(B8, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.size, dtype=np.float64)
    K = A.shape[1]
    _load().oracle_fp8_rowcol_points(K, _ptr(A), K, _ptr(B), K, _ptr(sa), _ptr(sb), _ptr(ms),
                                     _ptr(ns), ms.size, _ptr(out), nthreads)
    return out


def fp8_tensorquant_rows(A8, B8, scale_a, scale_b, m0=0, m1=None):
    """Per-tensor fp8 GEMM (PR #10439, Summary, "tensor_quant": one scalar scale for all of A,
    one for all of B): C[m][n] = (sum_k deq(A8[m][k]) * deq(B8[n][k])) * scale_a * scale_b, rows
    [m0, m1), in fp64 from the E4M3 definitions (the product of decoded operands is exact in
    fp64; numpy's matmul sums it). The scales are the fp32 values the kernel receives."""
    A = decode(np.ascontiguousarray(A8), "e4m3")
    B = decode(np.ascontiguousarray(B8), "e4m3")
    m1 = A.shape[0] if m1 is None else m1
    sa = float(np.float32(scale_a))
    sb = float(np.float32(scale_b))
    return (A[m0:m1] @ B.T) * sa * sb


def fp8_blockscale_points(A8, B8, sa, gka, sb, gnb, gkb, ms, ns, nthreads=0):
    """Block-scaled fp8 GEMM at the points (ms[i], ns[i]), fp64: sa [M][ceil(K/gka)] or None,
    sb [ceil(N/gnb)][ceil(K/gkb)] or None (a missing scale is 1)."""
    A = np.ascontiguousarray(A8, dtype=np.uint8)
    B = np.ascontiguousarray(B8, dtype=np.uint8)
    M, K = A.shape
    N = B.shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    sa_ = None if sa is None else np.ascontiguousarray(sa, dtype=np.float32)
    sb_ = None if sb is None else np.ascontiguousarray(sb, dtype=np.float32)
    out = np.empty(ms.size, dtype=np.float64)
    _load().oracle_fp8_blockscale_points(M, N, K, _ptr(A), _ptr(B),
                                         None if sa_ is None else _ptr(sa_), gka,
                                         None if sb_ is None else _ptr(sb_), gnb, gkb, _ptr(ms),
                                         _ptr(ns), ms.size, _ptr(out), nthreads)
    return out


def fp8_blockscale_rows(A8, B8, sa, gka, sb, gnb, gkb, m0=0, m1=None, nthreads=0):
    """Rows [m0, m1) of the block-scaled fp8 GEMM (see fp8_blockscale_points)."""
    M, N = A8.shape[0], B8.shape[0]
    m1 = M if m1 is None else m1
    mm, nn = np.meshgrid(np.arange(m0, m1), np.arange(N), indexing="ij")
    return fp8_blockscale_points(A8, B8, sa, gka, sb, gnb, gkb, mm.ravel(), nn.ravel(),
                                 nthreads).reshape(m1 - m0, N)


def wgrad_nhwc(fmt, x_bits, dy_bits, R, S, stride=(1, 1), pad=(0, 0), groups=1, k0=0, k1=None,
               nthreads=0):
    """fp64 dW[k0:k1] ([k][r][s][c], c per group) of the NHWC backward-weight convolution."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    dy = np.ascontiguousarray(dy_bits, dtype=np.uint16)
    N, H, W, C = x.shape
    K = dy.shape[3]
    k1 = K if k1 is None else k1
    Cg = C // groups
    out = np.empty((k1 - k0, R, S, Cg), dtype=np.float64)
    _load().oracle_wgrad_nhwc(FMT[fmt], N, H, W, C, K, R, S, stride[0], stride[1], pad[0], pad[1],
                              groups, _ptr(x), _ptr(dy), k0, k1, _ptr(out), nthreads)
    return out


def fprop_nhwc(fmt, x_bits, w_bits, stride=(1, 1), pad=(0, 0), groups=1, p0=0, p1=None,
               nthreads=0):
    """fp64 y[p0:p1] ([output pixel][K]) of the NHWC forward convolution, filter w [K][R][S][C/G]."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    N, H, W, C = x.shape
    K, R, S = w.shape[0], w.shape[1], w.shape[2]
    Ho, Wo = conv_out_size(H, R, stride[0], pad[0]), conv_out_size(W, S, stride[1], pad[1])
    p1 = N * Ho * Wo if p1 is None else p1
    out = np.empty((p1 - p0, K), dtype=np.float64)
    _load().oracle_fprop_nhwc(FMT[fmt], N, H, W, C, K, R, S, stride[0], stride[1], pad[0], pad[1],
                              groups, _ptr(x), _ptr(w), p0, p1, _ptr(out), nthreads)
    return out


def dgrad_nhwc(fmt, dy_bits, w_bits, H, W, stride=(1, 1), pad=(0, 0), groups=1, p0=0, p1=None,
               nthreads=0):
    """fp64 dx[p0:p1] ([input pixel][C]) of the NHWC convolution's data gradient; (H, W) is the
    input image size, dy [N][Ho][Wo][K], filter w [K][R][S][C/G]."""
    dy = np.ascontiguousarray(dy_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    N, Ho, Wo, K = dy.shape
    R, S, Cg = w.shape[1], w.shape[2], w.shape[3]
    C = Cg * groups
    assert (Ho, Wo) == (conv_out_size(H, R, stride[0], pad[0]), conv_out_size(W, S, stride[1], pad[1]))
    p1 = N * H * W if p1 is None else p1
    out = np.empty((p1 - p0, C), dtype=np.float64)
    _load().oracle_dgrad_nhwc(FMT[fmt], N, H, W, C, K, R, S, stride[0], stride[1], pad[0], pad[1],
                              groups, _ptr(dy), _ptr(w), p0, p1, _ptr(out), nthreads)
    return out


def conv_out_size(H, R, stride, pad):
    return (H + 2 * pad - R) // stride + 1


def round_output(ref: np.ndarray, out_dtype: str) -> np.ndarray:
    """Round the fp64 reference to the output type (round to nearest even), as float64 values."""
    if out_dtype == "f32":
        return ref.astype(np.float32).astype(np.float64)
    return codec.round_to(ref, out_dtype)


def tolerance(ref_rounded: np.ndarray, kred: int, kind: str = "16bit") -> float:
    """Parity bound: 2e-2*sqrt(K/4096)*max|ref| for 16-bit inputs (K = reduction length),
    2e-2*max|ref| for fp8."""
    amax = float(np.max(np.abs(ref_rounded))) if ref_rounded.size else 0.0
    if kind == "fp8":
        return 2e-2 * amax
    return 2e-2 * np.sqrt(kred / 4096.0) * amax
