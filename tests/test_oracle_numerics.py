"""Pins for the fp64 oracle numerics (oracle/ref.c) against library routines evaluated in fp64 on
the CPU (torch.matmul, torch.nn.grad.conv2d_weight) and against closed forms. Shapes are
non-square and asymmetric so that a transposed operand, a swapped index or a dropped term fails."""
import numpy as np
import pytest
import torch

from oracle import codec, numerics
from workloads import (blockscale_scales, dgrad_operands, fp8_operands, fprop_operands,
                       gemm_operands, wgrad_operands)


def _bits(t):
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.uint8).numpy()


@pytest.mark.parametrize("dtype,M,N,K", [("f16", 37, 53, 72), ("bf16", 64, 17, 136),
                                         ("f16", 1, 129, 8)])
def test_gemm_rcr_vs_torch_fp64(oracle_lib, dtype, M, N, K):
    A, B = gemm_operands(M, N, K, dtype, "u11", seed_offset=11)
    ref = A.double() @ B.double().T
    out = numerics.gemm_rcr_rows(dtype, _bits(A), _bits(B))
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    ms = np.array([0, M - 1, M // 2]); ns = np.array([N - 1, 0, N // 3])
    pts = numerics.gemm_rcr_points(dtype, _bits(A), _bits(B), ms, ns)
    np.testing.assert_allclose(pts, ref.numpy()[ms, ns], rtol=1e-12, atol=1e-12)
    part = numerics.gemm_rcr_rows(dtype, _bits(A), _bits(B), m0=M // 2, m1=M)
    np.testing.assert_array_equal(part, out[M // 2:])


def test_fp8_rowcol_vs_torch_fp64(oracle_lib):
    M, N, K = 40, 24, 96
    A, B, sa, sb = fp8_operands(M, N, K, seed_offset=3)
    ref = (A.double() @ B.double().T) * sa.double()[:, None] * sb.double()[None, :]
    out = numerics.fp8_rowcol_rows(_bits(A), _bits(B), sa.numpy(), sb.numpy())
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    ms = np.array([3, 39]); ns = np.array([23, 0])
    pts = numerics.fp8_rowcol_points(_bits(A), _bits(B), sa.numpy(), sb.numpy(), ms, ns)
    np.testing.assert_allclose(pts, ref.numpy()[ms, ns], rtol=1e-12, atol=1e-12)


def _torch_wgrad(x, dy, R, S, stride, pad, groups):
    xn = x.double().permute(0, 3, 1, 2)
    dyn = dy.double().permute(0, 3, 1, 2)
    K = dy.shape[3]
    w = torch.nn.grad.conv2d_weight(xn, (K, x.shape[3] // groups, R, S), dyn, stride=stride,
                                    padding=pad, groups=groups)
    return w.permute(0, 2, 3, 1).numpy()          # KCRS -> KRSC


@pytest.mark.parametrize("shape", [
    dict(N=2, H=7, W=9, C=8, K=6, R=3, S=3, stride=(1, 1), pad=(1, 1), groups=1, dt="f16"),
    dict(N=3, H=10, W=8, C=16, K=8, R=3, S=2, stride=(2, 2), pad=(1, 0), groups=2, dt="bf16"),
    dict(N=1, H=9, W=11, C=12, K=12, R=1, S=3, stride=(2, 1), pad=(0, 2), groups=4, dt="f16"),
    dict(N=2, H=5, W=5, C=4, K=4, R=5, S=5, stride=(3, 3), pad=(2, 2), groups=1, dt="bf16"),
])
def test_wgrad_vs_torch_conv2d_weight(oracle_lib, shape):
    s = shape
    x, dy = wgrad_operands(s["N"], s["H"], s["W"], s["C"], s["K"], s["R"], s["S"], s["stride"],
                           s["pad"], s["dt"], "u11", seed_offset=5)
    ref = _torch_wgrad(x, dy, s["R"], s["S"], s["stride"], s["pad"], s["groups"])
    out = numerics.wgrad_nhwc(s["dt"], _bits(x), _bits(dy), s["R"], s["S"], s["stride"], s["pad"],
                              s["groups"])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    k0 = s["K"] // 2
    part = numerics.wgrad_nhwc(s["dt"], _bits(x), _bits(dy), s["R"], s["S"], s["stride"], s["pad"],
                               s["groups"], k0=k0)
    np.testing.assert_array_equal(part, out[k0:])


def test_wgrad_all_ones_closed_form(oracle_lib):
    # x = dy = 1: dW[k,r,s,c] counts the (n, ho, wo) whose input tap (ho*sh-ph+r, wo*sw-pw+s)
    # lies inside the image, which factors into N * rows(r) * cols(s).
    N, H, W, C, K, R, S, sh, sw, ph, pw, G = 2, 6, 7, 4, 4, 3, 3, 2, 1, 1, 1, 2
    Ho, Wo = (H + 2 * ph - R) // sh + 1, (W + 2 * pw - S) // sw + 1
    one = 0x3C00
    x = np.full((N, H, W, C), one, np.uint16)
    dy = np.full((N, Ho, Wo, K), one, np.uint16)
    out = numerics.wgrad_nhwc("f16", x, dy, R, S, (sh, sw), (ph, pw), G)
    for r in range(R):
        rows = sum(0 <= ho * sh - ph + r < H for ho in range(Ho))
        for s_ in range(S):
            cols = sum(0 <= wo * sw - pw + s_ < W for wo in range(Wo))
            assert np.all(out[:, r, s_, :] == N * rows * cols)


CONV_SHAPES = [
    dict(N=2, H=7, W=9, C=8, K=6, R=3, S=3, stride=(1, 1), pad=(1, 1), groups=1, dt="f16"),
    dict(N=3, H=10, W=8, C=16, K=8, R=3, S=2, stride=(2, 2), pad=(1, 0), groups=2, dt="bf16"),
    dict(N=1, H=9, W=11, C=12, K=12, R=1, S=3, stride=(2, 1), pad=(0, 2), groups=4, dt="f16"),
    dict(N=2, H=5, W=5, C=4, K=4, R=5, S=5, stride=(3, 3), pad=(2, 2), groups=1, dt="bf16"),
    dict(N=2, H=6, W=5, C=6, K=9, R=2, S=3, stride=(1, 1), pad=(0, 1), groups=3, dt="f16"),
]


def _nhwc(t):          # NCHW fp64 -> NHWC numpy
    return t.permute(0, 2, 3, 1).numpy()


@pytest.mark.parametrize("shape", CONV_SHAPES)
def test_fprop_vs_torch_conv2d(oracle_lib, shape):
    s = shape
    x, w = fprop_operands(s["N"], s["H"], s["W"], s["C"], s["K"], s["R"], s["S"], s["groups"],
                          s["dt"], "u11", seed_offset=6)
    ref = torch.nn.functional.conv2d(x.double().permute(0, 3, 1, 2), w.double().permute(0, 3, 1, 2),
                                     stride=s["stride"], padding=s["pad"], groups=s["groups"])
    ref = _nhwc(ref).reshape(-1, s["K"])                  # [output pixel][K]
    out = numerics.fprop_nhwc(s["dt"], _bits(x), _bits(w), s["stride"], s["pad"], s["groups"])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    p0 = ref.shape[0] // 3
    part = numerics.fprop_nhwc(s["dt"], _bits(x), _bits(w), s["stride"], s["pad"], s["groups"],
                               p0=p0, p1=p0 + 5)
    np.testing.assert_array_equal(part, out[p0:p0 + 5])


@pytest.mark.parametrize("shape", CONV_SHAPES)
def test_dgrad_vs_torch_conv2d_input(oracle_lib, shape):
    s = shape
    dy, w = dgrad_operands(s["N"], s["H"], s["W"], s["C"], s["K"], s["R"], s["S"], s["stride"],
                           s["pad"], s["groups"], s["dt"], "u11", seed_offset=7)
    ref = torch.nn.grad.conv2d_input((s["N"], s["C"], s["H"], s["W"]),
                                     w.double().permute(0, 3, 1, 2),
                                     dy.double().permute(0, 3, 1, 2), stride=s["stride"],
                                     padding=s["pad"], groups=s["groups"])
    ref = _nhwc(ref).reshape(-1, s["C"])                  # [input pixel][C]
    out = numerics.dgrad_nhwc(s["dt"], _bits(dy), _bits(w), s["H"], s["W"], s["stride"], s["pad"],
                              s["groups"])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    part = numerics.dgrad_nhwc(s["dt"], _bits(dy), _bits(w), s["H"], s["W"], s["stride"], s["pad"],
                               s["groups"], p0=3, p1=11)
    np.testing.assert_array_equal(part, out[3:11])


def test_fprop_and_dgrad_all_ones_closed_form(oracle_lib):
    # x = w = 1: y counts the in-image taps of each output pixel, times C/G. dy = w = 1: dx counts
    # the (r, s) whose output position (h+ph-r)/sh, (w+pw-s)/sw is whole and inside, times K/G.
    N, H, W, C, K, R, S, sh, sw, ph, pw, G = 2, 6, 7, 4, 6, 3, 2, 2, 1, 1, 1, 2
    Ho, Wo = (H + 2 * ph - R) // sh + 1, (W + 2 * pw - S) // sw + 1
    one = 0x3C00
    y = numerics.fprop_nhwc("f16", np.full((N, H, W, C), one, np.uint16),
                            np.full((K, R, S, C // G), one, np.uint16), (sh, sw), (ph, pw), G)
    for n in range(N):
        for ho in range(Ho):
            rows = sum(0 <= ho * sh - ph + r < H for r in range(R))
            for wo in range(Wo):
                cols = sum(0 <= wo * sw - pw + s_ < W for s_ in range(S))
                assert np.all(y[(n * Ho + ho) * Wo + wo] == rows * cols * (C // G))
    dx = numerics.dgrad_nhwc("f16", np.full((N, Ho, Wo, K), one, np.uint16),
                             np.full((K, R, S, C // G), one, np.uint16), H, W, (sh, sw), (ph, pw), G)
    for h in range(H):
        rows = sum((h + ph - r) % sh == 0 and 0 <= (h + ph - r) // sh < Ho and h + ph - r >= 0
                   for r in range(R))
        for w_ in range(W):
            cols = sum((w_ + pw - s_) % sw == 0 and 0 <= (w_ + pw - s_) // sw < Wo and w_ + pw - s_ >= 0
                       for s_ in range(S))
            for n in range(N):
                assert np.all(dx[(n * H + h) * W + w_] == rows * cols * (K // G))


def test_fp8_tensorquant_vs_torch(oracle_lib):
    # per-tensor scales: torch's own e4m3 decode and fp64 matmul, times the two scalars
    A, B, _, _ = fp8_operands(37, 29, 96, seed_offset=9)
    sa, sb = 0.75, 1.625
    ref = (A.double() @ B.double().T) * sa * sb
    out = numerics.fp8_tensorquant_rows(_bits(A), _bits(B), sa, sb)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    # the same as row/col scales with constant vectors
    rc = numerics.fp8_rowcol_rows(_bits(A), _bits(B), np.full(37, sa, np.float32),
                                  np.full(29, sb, np.float32))
    np.testing.assert_allclose(out, rc, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(numerics.fp8_tensorquant_rows(_bits(A), _bits(B), sa, sb, 5, 9),
                                  out[5:9])


@pytest.mark.parametrize("case", [
    dict(M=37, N=29, K=300, gka=128, gnb=8, gkb=64, a=True, b=False),    # aquant, ragged K block
    dict(M=20, N=50, K=256, gka=64, gnb=16, gkb=128, a=False, b=True),   # bquant
    dict(M=33, N=40, K=384, gka=128, gnb=32, gkb=128, a=True, b=True),   # abquant
    dict(M=9, N=7, K=96, gka=32, gnb=3, gkb=48, a=True, b=True),
])
def test_fp8_blockscale_vs_torch_scaled_operands(oracle_lib, case):
    # Independent formulation: scale every element of A and B by its block's scale in fp64, then
    # one matmul in torch (fp64).
    c = case
    A, B, _, _ = fp8_operands(c["M"], c["N"], c["K"], seed_offset=14)
    sa, sb = blockscale_scales(c["M"], c["N"], c["K"], c["gka"], c["gnb"], c["gkb"], seed_offset=14)
    k = torch.arange(c["K"])
    As = A.double() * (sa.double()[:, k // c["gka"]] if c["a"] else 1.0)
    Bs = B.double() * (sb.double()[torch.arange(c["N"]) // c["gnb"]][:, k // c["gkb"]] if c["b"] else 1.0)
    ref = (As @ Bs.T).numpy()
    out = numerics.fp8_blockscale_rows(_bits(A), _bits(B), sa.numpy() if c["a"] else None, c["gka"],
                                       sb.numpy() if c["b"] else None, c["gnb"], c["gkb"])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    if not c["a"] and not c["b"]:
        return
    # with every scale 1 it is the plain fp8 product
    one = numerics.fp8_blockscale_rows(_bits(A), _bits(B), np.ones_like(sa.numpy()), c["gka"],
                                       np.ones_like(sb.numpy()), c["gnb"], c["gkb"])
    np.testing.assert_allclose(one, (A.double() @ B.double().T).numpy(), rtol=1e-12, atol=1e-12)


def test_round_output_and_tolerance():
    ref = np.array([1.0 + 2.0 ** -12, -3.0, 0.1])
    np.testing.assert_array_equal(numerics.round_output(ref, "f16"), codec.round_to(ref, "f16"))
    assert numerics.round_output(ref, "f32")[2] == np.float64(np.float32(0.1))
    # 2e-2*sqrt(K/4096)*max|ref|: K = 4096 -> 2e-2 * 3
    assert numerics.tolerance(numerics.round_output(ref, "f32"), 4096) == pytest.approx(0.06)
    assert numerics.tolerance(np.array([2.0]), 16384) == pytest.approx(0.08)
    assert numerics.tolerance(np.array([2.0]), 10 ** 6, "fp8") == pytest.approx(0.04)
