"""GPU parity of the forward convolution and the data gradient (sk_conv2d_fprop_nhwc and
sk_conv2d_dgrad_nhwc through the C ABI) against the fp64 oracle: every mode x reduction on ragged
shapes (pixel counts that leave partial tiles, partial channel tiles), groups, strides and padding
(the strided data gradient runs one launch per output phase), a 1x1 convolution, sampled tile-edge
pixels of a 32x56x56 workload, and bit-identical linear/tree hand-offs."""
import numpy as np
import pytest
import torch

from oracle import numerics
from workloads import dgrad_operands, fprop_operands

pytestmark = pytest.mark.gpu

import implicit_gemm_conv_gb300 as sk  # noqa: E402  (no skip: a missing library must fail)
from gpu_helpers import DEV, bits, check_parity, poisoned  # noqa: E402

MODES = ["off", "dp_sk", "persistent", "splitk"]
REDS = ["linear", "tree", "atomic", "workspace"]
TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def out_size(H, R, s, p):
    return (H + 2 * p - R) // s + 1


def run_fprop(x, w, out, stride, pad, groups, mode, red, ctas, ws=None):
    N, H, W, _ = x.shape
    K, R, S = w.shape[0], w.shape[1], w.shape[2]
    y = poisoned((N, out_size(H, R, stride[0], pad[0]), out_size(W, S, stride[1], pad[1]), K), TD[out])
    sk.sk_conv2d_fprop_nhwc(x.to(DEV), w.to(DEV), y, stride, pad, groups, mode, red, ctas, ws=ws)
    sk.sk_device_status()
    return y


def run_dgrad(dy, w, H, W, C, out, pad, groups, mode, red, ctas, ws=None, stride=(1, 1)):
    N = dy.shape[0]
    dx = poisoned((N, H, W, C), TD[out])
    sk.sk_conv2d_dgrad_nhwc(dy.to(DEV), w.to(DEV), dx, stride, pad, groups, mode, red, ctas, ws=ws)
    sk.sk_device_status()
    return dx


_REF = {}


def fprop_case(N, H, W, C, K, R, S, stride, pad, groups, dt, off):
    key = ("f", N, H, W, C, K, R, S, stride, pad, groups, dt, off)
    if key not in _REF:
        x, w = fprop_operands(N, H, W, C, K, R, S, groups, dt, "u11", seed_offset=off)
        _REF[key] = (x, w, numerics.fprop_nhwc(dt, bits(x), bits(w), stride, pad, groups))
    return _REF[key]


def dgrad_case(N, H, W, C, K, R, S, pad, groups, dt, off, stride=(1, 1)):
    key = ("d", N, H, W, C, K, R, S, pad, groups, dt, off, stride)
    if key not in _REF:
        dy, w = dgrad_operands(N, H, W, C, K, R, S, stride, pad, groups, dt, "u11", seed_offset=off)
        _REF[key] = (dy, w, numerics.dgrad_nhwc(dt, bits(dy), bits(w), H, W, stride, pad, groups))
    return _REF[key]


@pytest.mark.parametrize("red", REDS)
@pytest.mark.parametrize("mode", MODES)
def test_fprop_ragged(mode, red):
    # 198 output pixels (a partial second tile), 72 filters (a partial tile), 9 reduction steps
    x, w, ref = fprop_case(2, 9, 11, 64, 72, 3, 3, (1, 1), (1, 1), 1, "f16", 1)
    out = "f32" if red == "atomic" else "f16"
    y = run_fprop(x, w, out, (1, 1), (1, 1), 1, mode, red, 5)
    check_parity(y.reshape(-1, 72), ref, out, 9 * 64, what=f"fprop {mode}/{red}")


@pytest.mark.parametrize("red", REDS)
@pytest.mark.parametrize("mode", MODES)
def test_dgrad_ragged(mode, red):
    # 198 input pixels, 72 channels, 9 reduction steps over (r, s, k)
    dy, w, ref = dgrad_case(2, 9, 11, 72, 64, 3, 3, (1, 1), 1, "f16", 2)
    out = "f32" if red == "atomic" else "f16"
    dx = run_dgrad(dy, w, 9, 11, 72, out, (1, 1), 1, mode, red, 5)
    check_parity(dx.reshape(-1, 72), ref, out, 9 * 64, what=f"dgrad {mode}/{red}")


@pytest.mark.parametrize("mode,red", [("dp_sk", "linear"), ("persistent", "tree"), ("off", "linear"),
                                      ("splitk", "workspace"), ("dp_sk", "atomic")])
def test_fprop_grouped_strided(mode, red):
    # 2 groups of 64 channels and 48 filters, stride (2, 1), padding (1, 0), R != S, bf16
    x, w, ref = fprop_case(3, 10, 13, 128, 96, 3, 2, (2, 1), (1, 0), 2, "bf16", 3)
    out = "f32" if red == "atomic" else "bf16"
    y = run_fprop(x, w, out, (2, 1), (1, 0), 2, mode, red, 7)
    check_parity(y.reshape(-1, 96), ref, out, 6 * 64, what=f"fprop grouped {mode}/{red}")


@pytest.mark.parametrize("mode,red", [("dp_sk", "linear"), ("persistent", "tree"), ("off", "linear"),
                                      ("splitk", "workspace"), ("dp_sk", "atomic")])
def test_dgrad_grouped(mode, red):
    # 2 groups of 48 channels and 64 filters, padding (1, 0), R != S, bf16
    dy, w, ref = dgrad_case(3, 8, 10, 96, 128, 3, 2, (1, 0), 2, "bf16", 4)
    out = "f32" if red == "atomic" else "bf16"
    dx = run_dgrad(dy, w, 8, 10, 96, out, (1, 0), 2, mode, red, 7)
    check_parity(dx.reshape(-1, 96), ref, out, 6 * 64, what=f"dgrad grouped {mode}/{red}")


def test_fprop_1x1_and_padding_free():
    x, w, ref = fprop_case(4, 7, 7, 192, 256, 1, 1, (1, 1), (0, 0), 1, "bf16", 5)
    for mode, red in [("dp_sk", "linear"), ("off", "linear"), ("splitk", "tree")]:
        y = run_fprop(x, w, "bf16", (1, 1), (0, 0), 1, mode, red, 11)
        check_parity(y.reshape(-1, 256), ref, "bf16", 192, what=f"fprop 1x1 {mode}/{red}")


def test_dgrad_5x5_no_padding():
    dy, w, ref = dgrad_case(2, 12, 9, 64, 64, 5, 5, (0, 0), 1, "f16", 6)
    for mode, red in [("dp_sk", "linear"), ("persistent", "workspace")]:
        dx = run_dgrad(dy, w, 12, 9, 64, "f16", (0, 0), 1, mode, red, 9)
        check_parity(dx.reshape(-1, 64), ref, "f16", 25 * 64, what=f"dgrad 5x5 {mode}/{red}")


def _pixel_ranges(P):
    """Tile-edge pixel ranges of a P-pixel output: the first tiles, a middle stretch and the end."""
    return [(0, 300), (P // 2 - 130, P // 2 + 130), (P - 300, P)]


@pytest.mark.parametrize("tile", ["auto", "128"])   # auto: the shifted-row kernel
@pytest.mark.parametrize("red", ["linear", "atomic"])
def test_fprop_32x56x56_sampled(red, tile):
    N, H, W, C, K = 32, 56, 56, 64, 64
    x, w = fprop_operands(N, H, W, C, K, 3, 3, 1, "f16", "u11")
    out = "f32" if red == "atomic" else "f16"
    with sk.tile(tile):
        y = run_fprop(x, w, out, (1, 1), (1, 1), 1, "dp_sk", red, -1).reshape(-1, K)
    assert torch.isfinite(y.float()).all(), "unwritten outputs"
    for p0, p1 in _pixel_ranges(N * H * W):
        ref = numerics.fprop_nhwc("f16", bits(x), bits(w), (1, 1), (1, 1), 1, p0=p0, p1=p1)
        check_parity(y[p0:p1], ref, out, 9 * C, what=f"fprop 32x56x56 {red} pixels {p0}..{p1}")


@pytest.mark.parametrize("tile", ["auto", "128"])   # auto: the shifted-row kernel
@pytest.mark.parametrize("red", ["linear", "workspace"])
def test_dgrad_32x56x56_sampled(red, tile):
    N, H, W, C, K = 32, 56, 56, 64, 64
    dy, w = dgrad_operands(N, H, W, C, K, 3, 3, (1, 1), (1, 1), 1, "f16", "u11")
    with sk.tile(tile):
        dx = run_dgrad(dy, w, H, W, C, "f16", (1, 1), 1, "dp_sk", red, -1).reshape(-1, C)
    assert torch.isfinite(dx.float()).all(), "unwritten outputs"
    for p0, p1 in _pixel_ranges(N * H * W):
        ref = numerics.dgrad_nhwc("f16", bits(dy), bits(w), H, W, (1, 1), (1, 1), 1, p0=p0, p1=p1)
        check_parity(dx[p0:p1], ref, "f16", 9 * K, what=f"dgrad 32x56x56 {red} pixels {p0}..{p1}")


@pytest.mark.parametrize("op", ["fprop", "dgrad"])
@pytest.mark.parametrize("red", ["linear", "tree"])
def test_conv_bit_identical(op, red):
    # 20 launches with the workspace and the output poisoned before each one; a small pool so
    # that tiles are shared by several CTAs
    if op == "fprop":
        x, w, _ = fprop_case(2, 9, 11, 64, 72, 3, 3, (1, 1), (1, 1), 1, "f16", 1)
        launch = lambda o, ws: sk.sk_conv2d_fprop_nhwc(xd, wd, o, (1, 1), (1, 1), 1, "dp_sk", red,
                                                       5, ws=ws)
        shape = (2, 9, 11, 72)
        xd, wd = x.to(DEV), w.to(DEV)
        prob = sk.make_problem("fprop", ab_dtype="f16", c_dtype="f16", n=2, h=9, w=11, c=64, k=72,
                               r=3, s=3, stride_h=1, stride_w=1, pad_h=1, pad_w=1, groups=1)
    else:
        dy, w, _ = dgrad_case(2, 9, 11, 72, 64, 3, 3, (1, 1), 1, "f16", 2)
        launch = lambda o, ws: sk.sk_conv2d_dgrad_nhwc(xd, wd, o, (1, 1), (1, 1), 1, "dp_sk", red,
                                                       5, ws=ws)
        shape = (2, 9, 11, 72)
        xd, wd = dy.to(DEV), w.to(DEV)
        prob = sk.make_problem("dgrad", ab_dtype="f16", c_dtype="f16", n=2, h=9, w=11, c=72, k=64,
                               r=3, s=3, stride_h=1, stride_w=1, pad_h=1, pad_w=1, groups=1)
    ws = torch.empty(sk.sk_workspace_bytes(prob, "dp_sk", red, 5), dtype=torch.uint8, device=DEV)
    o = poisoned(shape, torch.float16)
    first = None
    for _ in range(20):
        ws.fill_(0xFF)
        o.view(torch.uint8).fill_(0xFF)
        launch(o, ws)
        sk.sk_device_status()
        b = o.view(torch.uint8).clone()
        assert torch.isfinite(o.float()).all()
        if first is None:
            first = b
        else:
            assert torch.equal(first, b), "result changed between launches"


STRIDED = {
    # N, H, W, C, K, R, S, stride, pad, groups, dtype
    "s2_3x3_ragged": (2, 9, 11, 72, 64, 3, 3, (2, 2), (1, 1), 1, "f16"),
    "s2x3_3x2_g2": (2, 10, 7, 64, 128, 3, 2, (2, 3), (1, 0), 2, "bf16"),
    "s2_1x1": (3, 8, 8, 64, 64, 1, 1, (2, 2), (0, 0), 1, "f16"),       # 3 of 4 phases get no taps
    "s3_3x3_pad2x1": (1, 13, 12, 64, 64, 3, 3, (3, 3), (2, 1), 1, "bf16"),   # negative padding
}


@pytest.mark.parametrize("mode,red", [("dp_sk", "linear"), ("persistent", "tree"), ("off", "linear"),
                                      ("splitk", "workspace"), ("dp_sk", "atomic"),
                                      ("hybrid", "linear")])
@pytest.mark.parametrize("name", list(STRIDED))
def test_dgrad_strided(name, mode, red):
    N, H, W, C, K, R, S, stride, pad, groups, dt = STRIDED[name]
    dy, w, ref = dgrad_case(N, H, W, C, K, R, S, pad, groups, dt, 7, stride)
    out = "f32" if red == "atomic" else dt
    dx = run_dgrad(dy, w, H, W, C, out, pad, groups, mode, red, 5, stride=stride)
    check_parity(dx.reshape(-1, C), ref, out, R * S * K // groups,
                 what=f"dgrad {name} {mode}/{red}")


def test_dgrad_strided_caller_workspace_and_bit_identical():
    # the caller's workspace, sized by sk_workspace_bytes for all phases; 10 launches, poisoned
    N, H, W, C, K, R, S, stride, pad, groups, dt = STRIDED["s2_3x3_ragged"]
    dy, w, ref = dgrad_case(N, H, W, C, K, R, S, pad, groups, dt, 7, stride)
    prob = sk.make_problem("dgrad", ab_dtype=dt, c_dtype=dt, n=N, h=H, w=W, c=C, k=K, r=R, s=S,
                           stride_h=stride[0], stride_w=stride[1], pad_h=pad[0], pad_w=pad[1],
                           groups=groups)
    ws = torch.empty(sk.sk_workspace_bytes(prob, "dp_sk", "linear", 5), dtype=torch.uint8,
                     device=DEV)
    dyd, wd = dy.to(DEV), w.to(DEV)
    dx = poisoned((N, H, W, C), TD[dt])
    first = None
    for _ in range(10):
        ws.fill_(0xFF)
        dx.view(torch.uint8).fill_(0xFF)
        sk.sk_conv2d_dgrad_nhwc(dyd, wd, dx, stride, pad, groups, "dp_sk", "linear", 5, ws=ws)
        sk.sk_device_status()
        b = dx.view(torch.uint8).clone()
        if first is None:
            first = b
            check_parity(dx.reshape(-1, C), ref, dt, R * S * K, what="strided dgrad, caller ws")
        else:
            assert torch.equal(first, b), "result changed between launches"


# ---- the shifted-row forward convolution (stride 1, 64 channels -> 64 filters, <= 3x3 taps)

ROW_FPROP = {   # (N, H, W, R, S, pad, dtype)
    # odd Ho (the last tile's second row is padding), 11 of 64 positions per row
    "ragged_3x3": (2, 9, 11, 3, 3, (1, 1), "f16"),
    # the widest rows it takes: 62 output columns + 2 column taps = 64 positions
    "wide_3x3": (1, 5, 62, 3, 3, (1, 1), "bf16"),
    # 2x2 taps, padding on one side only
    "2x2_pad01": (3, 7, 7, 2, 2, (0, 1), "f16"),
    # 1x1
    "1x1": (2, 6, 20, 1, 1, (0, 0), "bf16"),
    # three tap rows, one column tap, row padding 2
    "3x1_pad2": (1, 4, 30, 3, 1, (2, 0), "f16"),
}


def row_fprop_plan(N, H, W, R, S, pad, dt, tile="auto"):
    prob = sk.make_problem("fprop", ab_dtype=dt, c_dtype=dt, n=N, h=H, w=W, c=64, k=64, r=R, s=S,
                           stride_h=1, stride_w=1, pad_h=pad[0], pad_w=pad[1], groups=1)
    with sk.tile(tile):
        return sk.sk_plan(prob, "dp_sk", "linear", 5, 148)


def test_fprop_row_kernel_takes_its_shapes():
    """The automatic tile runs these shapes on the shifted-row kernel (a 128 x 64 tile, a K step
    per tap); the 128 x 128 tile keeps the pages' im2col view; other shapes keep the im2col view."""
    for name, (N, H, W, R, S, pad, dt) in ROW_FPROP.items():
        p = row_fprop_plan(N, H, W, R, S, pad, dt)
        ho = H + 2 * pad[0] - R + 1
        assert (p.tn, p.iters_per_tile, p.gemm_m) == (64, R * S, N * (ho + ho % 2) * 64), name
        assert row_fprop_plan(N, H, W, R, S, pad, dt, tile="128").tn == 128, name
    # 72 filters, or rows too wide for a 64-position segment: the im2col view
    prob = sk.make_problem("fprop", ab_dtype="f16", c_dtype="f16", n=2, h=9, w=11, c=64, k=72, r=3,
                           s=3, stride_h=1, stride_w=1, pad_h=1, pad_w=1, groups=1)
    assert sk.sk_plan(prob, "dp_sk", "linear", 5, 148).tn == 128
    assert row_fprop_plan(1, 5, 63, 3, 3, (1, 1), "f16").tn == 128


@pytest.mark.parametrize("red", REDS)
@pytest.mark.parametrize("mode", MODES + ["hybrid"])
@pytest.mark.parametrize("name", list(ROW_FPROP))
def test_fprop_row_shapes(name, mode, red):
    N, H, W, R, S, pad, dt = ROW_FPROP[name]
    x, w, ref = fprop_case(N, H, W, 64, 64, R, S, (1, 1), pad, 1, dt, 31)
    out = "f32" if red == "atomic" else dt
    y = run_fprop(x, w, out, (1, 1), pad, 1, mode, red, 5)
    check_parity(y.reshape(-1, 64), ref, out, R * S * 64, what=f"fprop row {name} {mode}/{red}")


@pytest.mark.parametrize("red", ["linear", "tree"])
def test_fprop_row_bit_identical(red):
    """20 launches, workspace and output poisoned before each; pool 5 so that tiles are shared."""
    N, H, W, R, S, pad, dt = ROW_FPROP["ragged_3x3"]
    x, w, _ = fprop_case(N, H, W, 64, 64, R, S, (1, 1), pad, 1, dt, 31)
    xd, wd = x.to(DEV), w.to(DEV)
    prob = sk.make_problem("fprop", ab_dtype=dt, c_dtype=dt, n=N, h=H, w=W, c=64, k=64, r=R, s=S,
                           stride_h=1, stride_w=1, pad_h=pad[0], pad_w=pad[1], groups=1)
    ws = torch.empty(sk.sk_workspace_bytes(prob, "dp_sk", red, 5), dtype=torch.uint8, device=DEV)
    y = poisoned((N, 9, 11, 64), TD[dt])
    first = None
    for _ in range(20):
        ws.fill_(0xFF)
        y.view(torch.uint8).fill_(0xFF)
        sk.sk_conv2d_fprop_nhwc(xd, wd, y, (1, 1), pad, 1, "dp_sk", red, 5, ws=ws)
        sk.sk_device_status()
        b = y.view(torch.uint8).clone()
        assert torch.isfinite(y.float()).all()
        if first is None:
            first = b
        else:
            assert torch.equal(first, b), "result changed between launches"


# ---- the shifted-row data gradient (stride 1, 64 filters -> 64 channels, <= 3x3 taps): the
# stride-1 convolution of dy with the flipped filter on the same kernel

ROW_DGRAD = {   # (N, H, W, R, S, pad, dtype): dx is N x H x W x 64
    "ragged_3x3": (2, 9, 11, 3, 3, (1, 1), "f16"),
    "wide_3x3": (1, 5, 62, 3, 3, (1, 1), "bf16"),
    "2x2_pad01": (3, 7, 7, 2, 2, (0, 1), "f16"),
    "1x1": (2, 6, 20, 1, 1, (0, 0), "bf16"),
    "3x1_pad2": (1, 4, 30, 3, 1, (2, 0), "f16"),
    "3x3_unpadded": (2, 8, 10, 3, 3, (0, 0), "f16"),   # the traversal pads by 2 on every side
}


def row_dgrad_plan(N, H, W, R, S, pad, dt, tile="auto"):
    prob = sk.make_problem("dgrad", ab_dtype=dt, c_dtype=dt, n=N, h=H, w=W, c=64, k=64, r=R, s=S,
                           stride_h=1, stride_w=1, pad_h=pad[0], pad_w=pad[1], groups=1)
    with sk.tile(tile):
        return sk.sk_plan(prob, "dp_sk", "linear", 5, 148)


def test_dgrad_row_kernel_takes_its_shapes():
    for name, (N, H, W, R, S, pad, dt) in ROW_DGRAD.items():
        p = row_dgrad_plan(N, H, W, R, S, pad, dt)
        assert (p.tn, p.iters_per_tile, p.gemm_m) == (64, R * S, N * (H + H % 2) * 64), name
        assert row_dgrad_plan(N, H, W, R, S, pad, dt, tile="128").tn == 128, name
    # 72 channels, or rows too wide: the im2col view
    prob = sk.make_problem("dgrad", ab_dtype="f16", c_dtype="f16", n=2, h=9, w=11, c=72, k=64,
                           r=3, s=3, stride_h=1, stride_w=1, pad_h=1, pad_w=1, groups=1)
    assert sk.sk_plan(prob, "dp_sk", "linear", 5, 148).tn == 128
    assert row_dgrad_plan(1, 5, 63, 3, 3, (1, 1), "f16").tn == 128


@pytest.mark.parametrize("red", REDS)
@pytest.mark.parametrize("mode", MODES + ["hybrid"])
@pytest.mark.parametrize("name", list(ROW_DGRAD))
def test_dgrad_row_shapes(name, mode, red):
    N, H, W, R, S, pad, dt = ROW_DGRAD[name]
    dy, w, ref = dgrad_case(N, H, W, 64, 64, R, S, pad, 1, dt, 33)
    out = "f32" if red == "atomic" else dt
    dx = run_dgrad(dy, w, H, W, 64, out, pad, 1, mode, red, 5)
    check_parity(dx.reshape(-1, 64), ref, out, R * S * 64, what=f"dgrad row {name} {mode}/{red}")


@pytest.mark.parametrize("red", ["linear", "tree"])
def test_dgrad_row_bit_identical(red):
    """20 launches, workspace and output poisoned before each; pool 5 so that tiles are shared."""
    N, H, W, R, S, pad, dt = ROW_DGRAD["ragged_3x3"]
    dy, w, _ = dgrad_case(N, H, W, 64, 64, R, S, pad, 1, dt, 33)
    dyd, wd = dy.to(DEV), w.to(DEV)
    prob = sk.make_problem("dgrad", ab_dtype=dt, c_dtype=dt, n=N, h=H, w=W, c=64, k=64, r=R, s=S,
                           stride_h=1, stride_w=1, pad_h=pad[0], pad_w=pad[1], groups=1)
    ws = torch.empty(sk.sk_workspace_bytes(prob, "dp_sk", red, 5), dtype=torch.uint8, device=DEV)
    dx = poisoned((N, H, W, 64), TD[dt])
    first = None
    for _ in range(20):
        ws.fill_(0xFF)
        dx.view(torch.uint8).fill_(0xFF)
        sk.sk_conv2d_dgrad_nhwc(dyd, wd, dx, (1, 1), pad, 1, "dp_sk", red, 5, ws=ws)
        sk.sk_device_status()
        b = dx.view(torch.uint8).clone()
        assert torch.isfinite(dx.float()).all()
        if first is None:
            first = b
        else:
            assert torch.equal(first, b), "result changed between launches"


def test_dgrad_strided_phases_keep_the_im2col_view():
    """A stride-2 dgrad of 64 -> 64 channels: its phase problems fit the shifted-row shape, but the
    phases run the im2col kernel; the workspace query sizes them the same way."""
    N, H, W, C, K, R, S, stride, pad, groups, dt = STRIDED["s2_1x1"]
    prob = sk.make_problem("dgrad", ab_dtype=dt, c_dtype=dt, n=N, h=H, w=W, c=C, k=K, r=R, s=S,
                           stride_h=2, stride_w=2, pad_h=0, pad_w=0, groups=1)
    ws = torch.empty(sk.sk_workspace_bytes(prob, "dp_sk", "linear", 5), dtype=torch.uint8,
                     device=DEV)
    dy, w, ref = dgrad_case(N, H, W, C, K, R, S, pad, groups, dt, 7, stride)
    dx = poisoned((N, H, W, C), TD[dt])
    sk.sk_conv2d_dgrad_nhwc(dy.to(DEV), w.to(DEV), dx, stride, pad, groups, "dp_sk", "linear", 5,
                            ws=ws)
    sk.sk_device_status()
    check_parity(dx.reshape(-1, C), ref, dt, R * S * K, what="strided dgrad phases, auto tile")


@pytest.mark.parametrize("mode", ["off", "dp_sk"])
def test_dgrad_strided_phases_finish_before_the_next_work(mode):
    """The phases of a strided data gradient may overlap one another (programmatic dependent
    launches where a phase shares no tile); work queued after the call on the same stream still
    sees every phase's pixels: a copy of dx enqueued right after the call, with no host
    synchronisation, equals dx read after synchronising, 20 times over, and matches the oracle."""
    N, H, W, C, K, R, S, stride, pad, groups, dt = STRIDED["s3_3x3_pad2x1"]
    dy, w, ref = dgrad_case(N, H, W, C, K, R, S, pad, groups, dt, 7, stride)
    dyd, wd = dy.to(DEV), w.to(DEV)
    dx = poisoned((N, H, W, C), TD[dt])
    first = None
    for _ in range(20):
        dx.view(torch.uint8).fill_(0xFF)
        sk.sk_conv2d_dgrad_nhwc(dyd, wd, dx, stride, pad, groups, mode, "linear", 5)
        early = dx.clone()   # same stream, no synchronisation in between
        sk.sk_device_status()
        assert torch.equal(early.view(torch.uint8), dx.view(torch.uint8)), "a phase was still running"
        if first is None:
            first = early
        assert torch.equal(first.view(torch.uint8), early.view(torch.uint8)), "result changed"
    check_parity(dx.reshape(-1, C), ref, dt, R * S * K, what=f"strided dgrad {mode}, chained phases")


def test_dgrad_strided_workspace_of_the_largest_phase_only():
    """A caller's workspace that holds only the largest phase's plan (smaller than
    sk_workspace_bytes, which gives all phases side by side): the phases with shared tiles then run
    one after another in it; the result matches the oracle and is bit-identical over 10 launches."""
    from oracle import partition as P
    N, H, W, C, K, R, S, stride, pad, groups, dt = STRIDED["s2_3x3_ragged"]
    dy, w, ref = dgrad_case(N, H, W, C, K, R, S, pad, groups, dt, 7, stride)
    prob = sk.make_problem("dgrad", ab_dtype=dt, c_dtype=dt, n=N, h=H, w=W, c=C, k=K, r=R, s=S,
                           stride_h=stride[0], stride_w=stride[1], pad_h=pad[0], pad_w=pad[1],
                           groups=groups)
    most = 0
    for a in range(stride[0]):
        for b in range(stride[1]):
            hp = len(range(a, H, stride[0]))
            wp = len(range(b, W, stride[1]))
            rt = len([r for r in range(R) if (a + pad[0] - r) % stride[0] == 0])
            st = len([s for s in range(S) if (b + pad[1] - s) % stride[1] == 0])
            if not (hp and wp and rt and st):
                continue
            plan = P.make_plan(tiles_m=-(-N * hp * wp // 128), tiles_n=-(-C // 128), groups=1,
                               kred=rt * st * K, tm=128, tn=128, tk=64, pool=5, mode=P.DP_SK,
                               reduction=P.LINEAR)
            most = max(most, plan.ws_bytes)
    full = sk.sk_workspace_bytes(prob, "dp_sk", "linear", 5)
    assert most < full
    ws = torch.empty(-(-most // 256) * 256, dtype=torch.uint8, device=DEV)
    dyd, wd = dy.to(DEV), w.to(DEV)
    dx = poisoned((N, H, W, C), TD[dt])
    first = None
    for _ in range(10):
        ws.fill_(0xFF)
        dx.view(torch.uint8).fill_(0xFF)
        sk.sk_conv2d_dgrad_nhwc(dyd, wd, dx, stride, pad, groups, "dp_sk", "linear", 5, ws=ws)
        sk.sk_device_status()
        b = dx.view(torch.uint8).clone()
        if first is None:
            first = b
            check_parity(dx.reshape(-1, C), ref, dt, R * S * K, what="strided dgrad, one phase's ws")
        else:
            assert torch.equal(first, b), "result changed between launches"
