"""linear and tree are bit-identical across 20 launches with the workspace (flags, control block,
partial tiles) and the output poisoned with 0xFF bytes before every launch: a missing release or
acquire on the partial hand-off would let an owner read poison (NaN) or a stale partial."""
import pytest
import torch

from workloads import fp8_operands, gemm_operands, wgrad_operands

pytestmark = pytest.mark.gpu

import implicit_gemm_conv_gb300 as sk  # noqa: E402  (no skip: a missing library must fail)
from gpu_helpers import DEV, poisoned  # noqa: E402


@pytest.fixture(autouse=True)
def tile_128():
    """The configurations these tests follow fix 128 x 128 tiles; the pair tiles have their own
    tests."""
    with sk.tile("128"):
        yield


def _repeat(launch, out, ws, n=20):
    first = None
    for _ in range(n):
        ws.fill_(0xFF)
        out.view(torch.uint8).fill_(0xFF)
        launch()
        sk.sk_device_status()
        b = out.view(torch.uint8).clone()
        assert torch.isfinite(out.float()).all()
        if first is None:
            first = b
        else:
            assert torch.equal(first, b), "result changed between launches"


@pytest.mark.parametrize("red", ["linear", "tree"])
@pytest.mark.parametrize("mode,shape,ctas", [("persistent", (256, 256, 4096), 3),
                                             ("dp_sk", (3840, 4096, 4096), 148),
                                             ("dp_sk", (512, 512, 65536), 148),
                                             ("hybrid", (3840, 4096, 4096), 148),
                                             ("hybrid", (1280, 1152, 2048), 13)])
def test_gemm_bit_identical(mode, shape, ctas, red):
    M, N, K = shape
    A, B = gemm_operands(M, N, K, "bf16", "n01")
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = poisoned((M, N), torch.bfloat16)
    prob = sk.make_problem("gemm", ab_dtype="bf16", c_dtype="bf16", M=M, N=N, K=K)
    ws = torch.empty(sk.sk_workspace_bytes(prob, mode, red, ctas), dtype=torch.uint8, device=DEV)
    _repeat(lambda: sk.sk_gemm_rcr(Ad, Bd, C, streamk=mode, reduction=red, ctas=ctas, ws=ws), C, ws)


WGRAD = {   # (N, H, W, C, K, R, S, stride, pad, groups)
    "32x56x56x64": (32, 56, 56, 64, 64, 3, 3, (1, 1), (1, 1), 1),
    "64x28x28x256 g4 s2": (64, 28, 28, 256, 256, 3, 3, (2, 2), (1, 1), 4),
}


@pytest.mark.parametrize("red", ["linear", "tree"])
@pytest.mark.parametrize("tile", ["128", "auto", "256_pair"])   # auto / 256_pair: shifted rows
@pytest.mark.parametrize("name", list(WGRAD))
def test_wgrad_bit_identical(name, tile, red):
    N, H, W, C, K, R, S, st, pd, g = WGRAD[name]
    x, dy = wgrad_operands(N, H, W, C, K, R, S, st, pd, "f16" if g == 1 else "bf16", "u11")
    xd, dyd = x.to(DEV), dy.to(DEV)
    dw = poisoned((K, R, S, C // g), torch.float32)
    prob = sk.make_problem("wgrad", ab_dtype="f16" if g == 1 else "bf16", c_dtype="f32", n=N,
                           h=H, w=W, c=C, k=K, r=R, s=S, stride_h=st[0], stride_w=st[1],
                           pad_h=pd[0], pad_w=pd[1], groups=g)
    with sk.tile(tile):
        ws = torch.empty(sk.sk_workspace_bytes(prob, "dp_sk", red, -1), dtype=torch.uint8,
                         device=DEV)
        _repeat(lambda: sk.sk_conv2d_wgrad_nhwc(xd, dyd, dw, R, S, st, pd, g, streamk="dp_sk",
                                                reduction=red, ctas=-1, ws=ws), dw, ws)


@pytest.mark.parametrize("red", ["linear", "tree"])
@pytest.mark.parametrize("tile", ["128", "256x256_pair"])
def test_fp8_rowcol_bit_identical(tile, red):
    """The fp8 row/col-scaled GEMM at 8192^3 (bf16 output), both tiles, default pool."""
    M = N = K = 8192
    A, B, sa, sb = fp8_operands(M, N, K)
    Ad, Bd, sad, sbd = A.to(DEV), B.to(DEV), sa.to(DEV), sb.to(DEV)
    C = poisoned((M, N), torch.bfloat16)
    prob = sk.make_problem("fp8", ab_dtype="e4m3", c_dtype="bf16", M=M, N=N, K=K)
    with sk.tile(tile):
        ws = torch.empty(sk.sk_workspace_bytes(prob, "dp_sk", red, -1), dtype=torch.uint8,
                         device=DEV)
        _repeat(lambda: sk.sk_gemm_rowcol_fp8(Ad, Bd, sad, sbd, C, streamk="dp_sk",
                                              reduction=red, ctas=-1, ws=ws), C, ws)
