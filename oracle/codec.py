"""Number formats used by the oracle: IEEE binary16, bfloat16 and OCP FP8 E4M3 ("e4m3fn").

TEST INFRASTRUCTURE. Part of the CPU oracle; see ``oracle/__init__.py``.

Written from the format definitions, not from any library routine:

* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits, subnormals, inf/NaN.
* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits (the top half of binary32).
* OCP FP8 E4M3 (the "fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits,
  subnormals, no infinities, NaN only at S.1111.111, largest finite value 448 (S.1111.110).

The format comes from the RowColQuant GEMM bridge page (rocm-libraries PR #9979, "Round-3" and
"GPU validation" comments): the reference must push its inputs through the same fp8
quantise -> dequantise as the kernel, with OCP E4M3 on the newer parts. Encoding rounds to nearest,
ties to even, from float64 in one step (no double rounding). ``encode_e4m3`` saturates finite
overflow to +-448 ("satfinite"); binary16 and bfloat16 overflow to +-inf.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "FORMATS", "decode", "encode", "round_to",
    "decode_f16", "decode_bf16", "decode_e4m3",
    "encode_f16", "encode_bf16", "encode_e4m3",
]


class _Fmt:
    def __init__(self, name, ebits, mbits, bias, has_inf, nan_bits, max_finite, storage):
        self.name = name
        self.ebits = ebits
        self.mbits = mbits
        self.bias = bias
        self.has_inf = has_inf
        self.nan_bits = nan_bits
        self.max_finite = max_finite
        self.storage = storage
        self.emin = 1 - bias                      # exponent of the smallest normal
        self.sign_shift = ebits + mbits


FORMATS = {
    # largest finite: (2 - 2^-10) * 2^15
    "f16": _Fmt("f16", 5, 10, 15, True, 0x7E00, (2.0 - 2.0 ** -10) * 2.0 ** 15, np.uint16),
    # largest finite: (2 - 2^-7) * 2^127
    "bf16": _Fmt("bf16", 8, 7, 127, True, 0x7FC0, (2.0 - 2.0 ** -7) * 2.0 ** 127, np.uint16),
    # largest finite: exponent field 15, fraction 110b -> 1.75 * 2^8 = 448
    "e4m3": _Fmt("e4m3", 4, 3, 7, False, 0x7F, 448.0, np.uint8),
}


def decode(bits, fmt: str) -> np.ndarray:
    """Bit patterns -> float64 values (exact)."""
    f = FORMATS[fmt]
    b = np.asarray(bits).astype(np.int64)
    sign = np.where((b >> f.sign_shift) & 1, -1.0, 1.0)
    efield = (b >> f.mbits) & ((1 << f.ebits) - 1)
    frac = (b & ((1 << f.mbits) - 1)).astype(np.float64)
    emax_field = (1 << f.ebits) - 1
    normal = sign * (1.0 + frac / 2.0 ** f.mbits) * np.exp2((efield - f.bias).astype(np.float64))
    sub = sign * (frac / 2.0 ** f.mbits) * 2.0 ** f.emin
    out = np.where(efield == 0, sub, normal)
    if f.has_inf:
        special = efield == emax_field
        out = np.where(special & (frac == 0), sign * np.inf, out)
        out = np.where(special & (frac != 0), np.nan, out)
    else:
        # E4M3 "fn": only S.1111.111 is NaN; S.1111.xxx otherwise stays a normal number
        out = np.where((efield == emax_field) & (frac == (1 << f.mbits) - 1), np.nan, out)
    return out


def round_to(x, fmt: str) -> np.ndarray:
    """Round float64 values to the nearest value of ``fmt`` (ties to even), returned as float64."""
    f = FORMATS[fmt]
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    finite = np.isfinite(ax) & (ax > 0)
    safe = np.where(finite, ax, 1.0)
    # frexp: safe = m * 2^E with m in [0.5, 1), so floor(log2(safe)) = E - 1
    _, E = np.frexp(safe)
    e = np.maximum(E.astype(np.int64) - 1, f.emin)          # subnormals share emin's quantum
    quantum = np.exp2((e - f.mbits).astype(np.float64))
    r = np.rint(safe / quantum) * quantum                    # np.rint: round half to even
    if f.has_inf:
        r = np.where(r > f.max_finite, np.inf, r)
    else:
        r = np.minimum(r, f.max_finite)                      # satfinite
    r = np.where(finite, r, ax)                              # 0, inf, nan pass through
    if not f.has_inf:
        r = np.where(np.isinf(ax), f.max_finite, r)          # satfinite: +-inf -> +-max
    return np.copysign(r, x)


def encode(x, fmt: str) -> np.ndarray:
    """float64 -> bit patterns of ``fmt`` (round to nearest even)."""
    f = FORMATS[fmt]
    x = np.asarray(x, dtype=np.float64)
    r = round_to(x, fmt)
    neg = np.signbit(r)
    a = np.abs(r)
    is_nan = np.isnan(a)
    is_inf = np.isinf(a)
    ok = ~(is_nan | is_inf) & (a > 0)
    safe = np.where(ok, a, 1.0)
    _, E = np.frexp(safe)
    e = E.astype(np.int64) - 1
    normal = e >= f.emin
    efield = np.where(normal, e + f.bias, 0)
    mant = np.where(normal,
                    safe / np.exp2((e - f.mbits).astype(np.float64)) - 2.0 ** f.mbits,
                    safe / 2.0 ** (f.emin - f.mbits))
    bits = (efield << f.mbits) | mant.astype(np.int64)
    bits = np.where(ok, bits, 0)
    if f.has_inf:
        bits = np.where(is_inf, ((1 << f.ebits) - 1) << f.mbits, bits)
    bits = bits | (neg.astype(np.int64) << f.sign_shift)
    bits = np.where(is_nan, f.nan_bits, bits)
    return bits.astype(f.storage)


def decode_f16(bits):
    return decode(bits, "f16")


def decode_bf16(bits):
    return decode(bits, "bf16")


def decode_e4m3(bits):
    return decode(bits, "e4m3")


def encode_f16(x):
    return encode(x, "f16")


def encode_bf16(x):
    return encode(x, "bf16")


def encode_e4m3(x):
    return encode(x, "e4m3")
