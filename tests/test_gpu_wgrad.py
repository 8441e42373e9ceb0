"""GPU parity of the implicit-GEMM conv wgrad (sk_conv2d_wgrad_nhwc through the C ABI) against the
fp64 direct-loop oracle: every launch mode x four reductions on dense, strided and grouped shapes
with a partial last M tile and a ragged pixel tail, under both wgrad kernels (the automatic tile,
which takes the shifted-row kernel for 64-channel, 64-filter groups, its CTA-pair form with several
K steps per ring stage on request, and the 128 x 128 tile of the pages' GEMM view), shapes that reach the shifted-row
kernel's edges (one to five tap rows; one to three column taps; column stride 2; rows packed several to a K step with a ragged
last step; the widest rows it takes), and the two named wgrad workloads in full."""
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


def run(x, dy, K, R, S, stride, pad, groups, out, mode, red, ctas, tile="auto"):
    C = x.shape[3]
    dw = poisoned((K, R, S, C // groups), TD[out])
    with sk.tile(tile):
        sk.sk_conv2d_wgrad_nhwc(x.to(DEV), dy.to(DEV), dw, R, S, stride, pad, groups, streamk=mode,
                                reduction=red, ctas=ctas)
    sk.sk_device_status()
    return dw


def row_plan(s, tile="auto"):
    """The plan of this shape under a tile setting."""
    N, H, W, C, K, R, S = s["N"], s["H"], s["W"], s["C"], s["K"], s["R"], s["S"]
    prob = sk.make_problem("wgrad", ab_dtype=s["dt"], c_dtype="f32", n=N, h=H, w=W, c=C, k=K,
                           r=R, s=S, stride_h=s["stride"][0], stride_w=s["stride"][1],
                           pad_h=s["pad"][0], pad_w=s["pad"][1], groups=s["groups"])
    with sk.tile(tile):
        return sk.sk_plan(prob, "dp_sk", "atomic", 7, 148)


def row_kernel(s) -> bool:
    """Whether the automatic tile runs this shape on the shifted-row kernel (its 192-wide tile)."""
    return row_plan(s).tn == 192


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


# Shapes for the shifted-row kernel (64 channels and 64 filters per group), each at an edge of it.
ROW_SHAPES = {
    # one tap row (the tile's lower half unused), one column tap, no padding
    "row_r1s1": dict(dt="f16", N=2, H=5, W=7, C=64, K=64, R=1, S=1, stride=(1, 1), pad=(0, 0),
                     groups=1),
    # two tap rows (one full tile), two column taps
    "row_r2s2": dict(dt="bf16", N=3, H=6, W=9, C=64, K=64, R=2, S=2, stride=(1, 1), pad=(1, 1),
                     groups=1),
    # five tap rows: three tiles, the last with its lower half unused; asymmetric padding
    "row_r5s3": dict(dt="f16", N=2, H=9, W=13, C=64, K=64, R=5, S=3, stride=(1, 1), pad=(2, 1),
                     groups=1),
    # column stride 2: even and odd x columns; 8 output columns + 1 shift -> 16-position segments,
    # four output rows per K step, 7 rows per image (ragged last step of each image)
    "row_sw2": dict(dt="bf16", N=2, H=7, W=16, C=64, K=64, R=3, S=3, stride=(1, 2), pad=(1, 1),
                    groups=1),
    # row stride 2 only: two 32-position rows per K step
    "row_sh2": dict(dt="f16", N=3, H=11, W=20, C=64, K=64, R=3, S=3, stride=(2, 1), pad=(1, 1),
                    groups=1),
    # stride 2 both ways with 2x2 taps: one tap per column phase, no shift, 16 rows per K step
    "row_s2_2x2": dict(dt="bf16", N=2, H=9, W=9, C=64, K=64, R=2, S=2, stride=(2, 2),
                       pad=(0, 0), groups=1),
    # four tap rows (the CTA pair's 256 rows all used), two groups, row padding only
    "row_r4s2_g2": dict(dt="bf16", N=2, H=8, W=10, C=128, K=128, R=4, S=2, stride=(1, 1),
                        pad=(1, 0), groups=2),
    # the widest rows the kernel takes: 62 output columns + 2 shifts = 64 positions
    "row_wide": dict(dt="f16", N=1, H=3, W=62, C=64, K=64, R=3, S=3, stride=(1, 1), pad=(1, 1),
                     groups=1),
    # three groups of 64 channels and 64 filters
    "row_g3": dict(dt="bf16", N=2, H=6, W=6, C=192, K=192, R=3, S=3, stride=(1, 1), pad=(1, 1),
                   groups=3),
    # padding 2 on a 3x3 filter: output larger than the input
    "row_pad2": dict(dt="f16", N=2, H=5, W=6, C=64, K=64, R=3, S=3, stride=(1, 1), pad=(2, 2),
                     groups=1),
}
ALL_SHAPES = {**SHAPES, **ROW_SHAPES}


def test_row_kernel_takes_its_shapes():
    """The shifted-row shapes reach the shifted-row kernel; of the others, the 64-channel,
    64-filter dense and grouped ones do, the rest stay on the 128 x 128 tile. Rows one position
    too wide for a K step fall back too."""
    for name, s in ROW_SHAPES.items():
        assert row_kernel(s), name
        # at these sizes the one-CTA 128 x 192 tile; the pair tile on request
        assert row_plan(s).tm == 128, name
        assert row_plan(s, "256_pair").tm == 256, name
    assert row_kernel(SHAPES["dense_3x3"]) and row_kernel(SHAPES["grouped_s2"])
    assert not row_kernel(SHAPES["pointwise"]) and not row_kernel(SHAPES["asym"])
    too_wide = dict(ROW_SHAPES["row_wide"], W=63)
    assert not row_kernel(too_wide)


@pytest.mark.parametrize("red", ["linear", "tree", "atomic", "workspace"])
@pytest.mark.parametrize("mode", ["dp_sk", "persistent", "off", "splitk", "hybrid"])
@pytest.mark.parametrize("tile", ["auto", "128", "256_pair"])
@pytest.mark.parametrize("name", list(ALL_SHAPES))
def test_wgrad_shapes(name, tile, mode, red):
    """auto: the one-CTA shifted-row kernel on these sizes; 256_pair: its CTA-pair form (several
    K steps per ring stage); 128: the pages' view."""
    s = ALL_SHAPES[name]
    if tile == "128" and name in ROW_SHAPES and mode not in ("dp_sk", "off"):
        pytest.skip("the 128 x 128 tile's modes are covered on the first four shapes")
    if tile == "256_pair" and not row_kernel(s):
        pytest.skip("the pair tile serves the shifted-row view only")
    x, dy, ref = case(s["dt"], s["N"], s["H"], s["W"], s["C"], s["K"], s["R"], s["S"], s["stride"],
                      s["pad"], s["groups"])
    Ho, Wo = conv_out(s["H"], s["R"], s["stride"][0], s["pad"][0]), \
        conv_out(s["W"], s["S"], s["stride"][1], s["pad"][1])
    dw = run(x, dy, s["K"], s["R"], s["S"], s["stride"], s["pad"], s["groups"], "f32", mode, red, 7,
             tile)
    check_parity(dw, ref, "f32", s["N"] * Ho * Wo, what=f"{name} {tile} {mode}/{red}")


@pytest.mark.parametrize("out", ["f16", "bf16"])
def test_wgrad_row_16bit_output(out):
    s = ROW_SHAPES["row_r5s3"] if out == "f16" else ROW_SHAPES["row_sw2"]
    x, dy, ref = case(s["dt"], s["N"], s["H"], s["W"], s["C"], s["K"], s["R"], s["S"], s["stride"],
                      s["pad"], s["groups"])
    Ho, Wo = conv_out(s["H"], s["R"], s["stride"][0], s["pad"][0]), \
        conv_out(s["W"], s["S"], s["stride"][1], s["pad"][1])
    for mode, red in (("dp_sk", "linear"), ("dp_sk", "workspace"), ("off", "linear")):
        dw = run(x, dy, s["K"], s["R"], s["S"], s["stride"], s["pad"], s["groups"], s["dt"], mode,
                 red, 5)
        check_parity(dw, ref, s["dt"], s["N"] * Ho * Wo, what=f"{s['dt']} dW {mode}/{red}")


def test_wgrad_16bit_output():
    s = SHAPES["dense_3x3"]
    x, dy, ref = case(s["dt"], s["N"], s["H"], s["W"], s["C"], s["K"], s["R"], s["S"], s["stride"],
                      s["pad"], s["groups"])
    dw = run(x, dy, s["K"], s["R"], s["S"], s["stride"], s["pad"], s["groups"], "f16", "dp_sk",
             "linear", -1)
    check_parity(dw, ref, "f16", 189, what="f16 dW")


@pytest.mark.parametrize("tile", ["auto", "128"])
@pytest.mark.parametrize("mode", ["dp_sk", "persistent", "splitk"])
@pytest.mark.parametrize("red", ["linear", "tree", "atomic", "workspace"])
def test_wgrad_n32_56x56_c64_k64(tile, mode, red):
    x, dy, ref = case("f16", 32, 56, 56, 64, 64, 3, 3, (1, 1), (1, 1), 1, "u11")
    dw = run(x, dy, 64, 3, 3, (1, 1), (1, 1), 1, "f32", mode, red, -1, tile)
    check_parity(dw, ref, "f32", 32 * 56 * 56, what=f"cfg n32 {tile} {mode}/{red}")


@pytest.mark.parametrize("tile", ["auto", "128"])
@pytest.mark.parametrize("mode", ["dp_sk", "persistent", "splitk"])
@pytest.mark.parametrize("red", ["atomic", "workspace", "linear", "tree"])
def test_wgrad_n64_28x28_g4_s2(tile, mode, red):
    x, dy, ref = case("bf16", 64, 28, 28, 256, 256, 3, 3, (2, 2), (1, 1), 4, "n0.5")
    dw = run(x, dy, 256, 3, 3, (2, 2), (1, 1), 4, "f32", mode, red, -1, tile)
    check_parity(dw, ref, "f32", 64 * 14 * 14, what=f"cfg g4 {tile} {mode}/{red}")


def test_wgrad_auto_selection():
    x, dy, ref = case("f16", 32, 56, 56, 64, 64, 3, 3, (1, 1), (1, 1), 1, "u11")
    dw = run(x, dy, 64, 3, 3, (1, 1), (1, 1), 1, "f32", "auto", "auto", -1)
    check_parity(dw, ref, "f32", 32 * 56 * 56, what="wgrad auto")
