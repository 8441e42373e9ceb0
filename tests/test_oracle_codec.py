"""Pins for the oracle's number formats: exhaustive decode tables and round-to-nearest-even
encoding, checked against torch's own casts (a library routine) and against closed-form values of
the format definitions (IEEE 754 binary16, bfloat16, OCP FP8 E4M3)."""
import numpy as np
import pytest
import torch

from oracle import codec, numerics


def _torch_decode(bits, dtype):
    t = torch.from_numpy(bits.astype(np.int64))
    if dtype == torch.float8_e4m3fn:
        return t.to(torch.uint8).view(dtype).double().numpy()
    return t.to(torch.int16).view(dtype).double().numpy()


@pytest.mark.parametrize("fmt,dtype,n", [("f16", torch.float16, 65536),
                                         ("bf16", torch.bfloat16, 65536),
                                         ("e4m3", torch.float8_e4m3fn, 256)])
def test_decode_exhaustive(fmt, dtype, n):
    bits = np.arange(n, dtype=np.int64)
    ref = _torch_decode(bits, dtype)
    py = codec.decode(bits, fmt)
    c = numerics.decode(bits.astype(np.uint8 if n == 256 else np.uint16), fmt)
    np.testing.assert_array_equal(py, ref)
    np.testing.assert_array_equal(c, ref)


def test_format_closed_forms():
    # binary16: 1.0 = 0x3C00, largest finite 65504 = 0x7BFF, smallest subnormal 2^-24 = 0x0001
    assert codec.decode(np.array([0x3C00, 0x7BFF, 0x0001, 0xC000]), "f16").tolist() == \
        [1.0, 65504.0, 2.0 ** -24, -2.0]
    # bfloat16: 1.0 = 0x3F80, -0.5 = 0xBF00, smallest subnormal 2^-133 = 0x0001
    assert codec.decode(np.array([0x3F80, 0xBF00, 0x0001]), "bf16").tolist() == \
        [1.0, -0.5, 2.0 ** -133]
    # E4M3: 1.0 = 0x38, largest finite 448 = 0x7E, smallest subnormal 2^-9 = 0x01,
    # smallest normal 2^-6 = 0x08, 0x7F is NaN, 0xFE = -448
    d = codec.decode(np.array([0x38, 0x7E, 0x01, 0x08, 0xFE]), "e4m3").tolist()
    assert d == [1.0, 448.0, 2.0 ** -9, 2.0 ** -6, -448.0]
    assert np.isnan(codec.decode(np.array([0x7F]), "e4m3"))[0]
    assert codec.encode(np.array([500.0, np.inf, -1e9]), "e4m3").tolist() == [0x7E, 0x7E, 0xFE]


def _edge_values():
    rng = np.random.default_rng(7)
    v = [rng.standard_normal(20000).astype(np.float32),
         (rng.standard_normal(5000) * 1e-5).astype(np.float32),      # f16 subnormal range
         (rng.standard_normal(5000) * 1e4).astype(np.float32),
         np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e-8, 2.0 ** -25,
                   3 * 2.0 ** -26, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -8,
                   1.0 + 3 * 2.0 ** -9], dtype=np.float32)]
    return np.concatenate(v).astype(np.float64)


@pytest.mark.parametrize("fmt,dtype", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_encode_matches_torch_rne(fmt, dtype):
    x = _edge_values()
    ref = torch.from_numpy(x.astype(np.float32)).to(dtype).view(torch.int16).numpy()
    ours = codec.encode(x, fmt).view(np.int16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(codec.round_to(x, fmt), codec.decode(ours.view(np.uint16), fmt))


def test_encode_e4m3_matches_torch_in_range():
    x = _edge_values()
    x = x[np.abs(x) <= 448.0]
    ties = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 440.0, 447.9], dtype=np.float64)
    x = np.concatenate([x, ties, -ties])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codec.encode(x, "e4m3"), ref)


def test_round_is_single_step_from_fp64():
    # 1 + 2^-11 + 2^-40 lies just above the binary16 tie between 1 and 1 + 2^-10, so one rounding
    # step from fp64 goes up. A detour through fp32 (23 fraction bits) would land on the tie itself
    # and then round to even, down to 1.0.
    x = np.array([1.0 + 2.0 ** -11 + 2.0 ** -40])
    assert codec.round_to(x, "f16")[0] == 1.0 + 2.0 ** -10
