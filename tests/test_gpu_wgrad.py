"""GPU parity of the implicit-GEMM conv wgrad (sk_conv2d_wgrad_nhwc through the C ABI) against the
fp64 direct-loop oracle: both launch modes x four reductions on dense, strided and grouped shapes
with a partial last M tile and a ragged pixel tail, and the two named wgrad workloads in full."""
import numpy as np
import pytest
import torch

from oracle import numerics
from workloads import conv_out, wgrad_operands

pytestmark = pytest.mark.gpu

import implicit_gemm_conv_gb300 as sk  # noqa: E402  (no skip: a missing library must fail)
from gpu_helpers import DEV, bits, check_parity, poisoned  # noqa: E402

TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
_REF = {}


def case(dt, N, H, W, C, K, R, S, stride, pad, groups, dist="u11", off=0):
    key = (dt, N, H, W, C, K, R, S, stride, pad, groups, dist, off)
    if key not in _REF:
        x, dy = wgrad_operands(N, H, W, C, K, R, S, stride, pad, dt, dist, seed_offset=off)
        ref = numerics.wgrad_nhwc(dt, bits(x), bits(dy), R, S, stride, pad, groups)
        _REF[key] = (x, dy, ref)
    return _REF[key]


def run(x, dy, K, R, S, stride, pad, groups, out, mode, red, ctas):
    C = x.shape[3]
    dw = poisoned((K, R, S, C // groups), TD[out])
    sk.sk_conv2d_wgrad_nhwc(x.to(DEV), dy.to(DEV), dw, R, S, stride, pad, groups, streamk=mode,
                            reduction=red, ctas=ctas)
    sk.sk_device_status()
    return dw


SHAPES = {
    # ragged pixel tail: 3*7*9 = 189 pixels = 2 full steps + 61
    "dense_3x3": dict(dt="f16", N=3, H=7, W=9, C=64, K=64, R=3, S=3, stride=(1, 1), pad=(1, 1),
                      groups=1),
    # stride 2, two groups, Kg = 64 < 128: a partial last M tile in every group
    "grouped_s2": dict(dt="bf16", N=2, H=12, W=10, C=128, K=128, R=3, S=3, stride=(2, 2),
                       pad=(1, 1), groups=2),
    # 1x1, no padding, Kg = 192 (one full and one partial M tile), two 64-channel slabs per tap
    "pointwise": dict(dt="f16", N=2, H=9, W=9, C=128, K=192, R=1, S=1, stride=(1, 1), pad=(0, 0),
                      groups=1),
    # asymmetric filter and stride, one padding side
    "asym": dict(dt="bf16", N=2, H=11, W=8, C=64, K=32, R=3, S=2, stride=(2, 1), pad=(1, 0),
                 groups=1),
}


@pytest.mark.parametrize("red", ["linear", "tree", "atomic", "workspace"])
@pytest.mark.parametrize("mode", ["dp_sk", "persistent", "off", "splitk", "hybrid"])
@pytest.mark.parametrize("name", list(SHAPES))
def test_wgrad_shapes(name, mode, red):
    s = SHAPES[name]
    x, dy, ref = case(s["dt"], s["N"], s["H"], s["W"], s["C"], s["K"], s["R"], s["S"], s["stride"],
                      s["pad"], s["groups"])
    Ho, Wo = conv_out(s["H"], s["R"], s["stride"][0], s["pad"][0]), \
        conv_out(s["W"], s["S"], s["stride"][1], s["pad"][1])
    dw = run(x, dy, s["K"], s["R"], s["S"], s["stride"], s["pad"], s["groups"], "f32", mode, red, 7)
    check_parity(dw, ref, "f32", s["N"] * Ho * Wo, what=f"{name} {mode}/{red}")


def test_wgrad_16bit_output():
    s = SHAPES["dense_3x3"]
    x, dy, ref = case(s["dt"], s["N"], s["H"], s["W"], s["C"], s["K"], s["R"], s["S"], s["stride"],
                      s["pad"], s["groups"])
    dw = run(x, dy, s["K"], s["R"], s["S"], s["stride"], s["pad"], s["groups"], "f16", "dp_sk",
             "linear", -1)
    check_parity(dw, ref, "f16", 189, what="f16 dW")


@pytest.mark.parametrize("mode", ["dp_sk", "persistent"])
@pytest.mark.parametrize("red", ["linear", "tree", "atomic", "workspace"])
def test_wgrad_n32_56x56_c64_k64(mode, red):
    x, dy, ref = case("f16", 32, 56, 56, 64, 64, 3, 3, (1, 1), (1, 1), 1, "u11")
    dw = run(x, dy, 64, 3, 3, (1, 1), (1, 1), 1, "f32", mode, red, -1)
    check_parity(dw, ref, "f32", 32 * 56 * 56, what=f"cfg n32 {mode}/{red}")


@pytest.mark.parametrize("mode", ["dp_sk", "persistent"])
@pytest.mark.parametrize("red", ["atomic", "workspace", "linear", "tree"])
def test_wgrad_n64_28x28_g4_s2(mode, red):
    x, dy, ref = case("bf16", 64, 28, 28, 256, 256, 3, 3, (2, 2), (1, 1), 4, "n0.5")
    dw = run(x, dy, 256, 3, 3, (2, 2), (1, 1), 4, "f32", mode, red, -1)
    check_parity(dw, ref, "f32", 64 * 14 * 14, what=f"cfg g4 {mode}/{red}")


def test_wgrad_auto_selection():
    x, dy, ref = case("f16", 32, 56, 56, 64, 64, 3, 3, (1, 1), (1, 1), 1, "u11")
    dw = run(x, dy, 64, 3, 3, (1, 1), (1, 1), 1, "f32", "auto", "auto", -1)
    check_parity(dw, ref, "f32", 32 * 56 * 56, what="wgrad auto")
