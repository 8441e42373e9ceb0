"""GPU parity of the block-scaled fp8 GEMM (sk_gemm_blockscale_fp8 through the C ABI) against the
fp64 oracle, on the 128 x 128 one-CTA tile and the 256 x 128 CTA-pair tile: the three scale layouts
(A blocks along K, B blocks along N and K, both), group sizes of one and several K steps, a ragged
last K step, every mode x deterministic/workspace reduction, sampled outputs of a 4096^3 problem,
bit-identical linear/tree hand-offs and the smallest shapes."""
import pytest
import torch

from oracle import numerics
from workloads import blockscale_scales, fp8_operands

pytestmark = pytest.mark.gpu

import implicit_gemm_conv_gb300 as sk  # noqa: E402  (no skip: a missing library must fail)
from gpu_helpers import DEV, bits, check_parity, poisoned, sample_points  # noqa: E402

MODES = ["off", "dp_sk", "persistent", "splitk", "hybrid"]


@pytest.fixture(autouse=True, params=["128", "256_pair"])
def block_tile(request):
    with sk.tile(request.param):
        yield request.param

REDS = ["linear", "tree", "workspace"]
LAYOUTS = ["aquant", "bquant", "abquant"]


def operands(M, N, K, layout, gka, gnb, gkb, off):
    A, B, _, _ = fp8_operands(M, N, K, seed_offset=off)
    sa, sb = blockscale_scales(M, N, K, gka, gnb, gkb, seed_offset=off)
    if layout == "bquant":
        sa = None
    if layout == "aquant":
        sb = None
    return A, B, sa, sb


def run(A, B, sa, sb, gka, gnb, gkb, mode, red, ctas, ws=None):
    M, N = A.shape[0], B.shape[0]
    C = poisoned((M, N), torch.bfloat16)
    dev = lambda t: None if t is None else t.to(DEV)
    sk.sk_gemm_blockscale_fp8(A.to(DEV), B.to(DEV), dev(sa), gka, dev(sb), gnb, gkb, C,
                              streamk=mode, reduction=red, ctas=ctas, ws=ws)
    sk.sk_device_status()
    return C


def np_or_none(t):
    return None if t is None else t.numpy()


_REF = {}


def case(M, N, K, layout, gka, gnb, gkb, off):
    key = (M, N, K, layout, gka, gnb, gkb, off)
    if key not in _REF:
        A, B, sa, sb = operands(M, N, K, layout, gka, gnb, gkb, off)
        ref = numerics.fp8_blockscale_rows(bits(A), bits(B), np_or_none(sa), gka, np_or_none(sb),
                                           gnb, gkb)
        _REF[key] = (A, B, sa, sb, ref)
    return _REF[key]


@pytest.mark.parametrize("red", REDS)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_blockscale_ragged(layout, mode, red):
    # 300 x 392: partial last row and column tiles; K = 1040: 9 steps, the last 16 wide;
    # A blocks of one step, B blocks of 128 columns x 2 steps
    A, B, sa, sb, ref = case(300, 392, 1040, layout, 128, 128, 256, 1)
    C = run(A, B, sa, sb, 128, 128, 256, mode, red, 5)
    check_parity(C, ref, "bf16", 1040, kind="fp8", what=f"block {layout} {mode}/{red}")


@pytest.mark.parametrize("gka,gnb,gkb", [(256, 128, 128), (512, 256, 384), (1024, 384, 1024)])
@pytest.mark.parametrize("mode,red", [("dp_sk", "linear"), ("persistent", "tree"),
                                      ("splitk", "workspace")])
def test_blockscale_group_sizes(gka, gnb, gkb, mode, red):
    # groups spanning several K steps and B blocks of 2 and 3 column tiles; 24 K steps over 7
    # CTAs so that stream-K ranges start inside a block
    A, B, sa, sb, ref = case(384, 448, 3072, "abquant", gka, gnb, gkb, 2)
    C = run(A, B, sa, sb, gka, gnb, gkb, mode, red, 7)
    check_parity(C, ref, "bf16", 3072, kind="fp8", what=f"block groups {gka}/{gnb}/{gkb}")


@pytest.mark.parametrize("shape", [(1, 8, 16), (129, 136, 144), (128, 128, 128)])
def test_blockscale_small_shapes(shape):
    M, N, K = shape
    A, B, sa, sb, ref = case(M, N, K, "abquant", 128, 128, 128, 3)
    for mode, red, ctas in [("dp_sk", "linear", -1), ("off", "linear", 1),
                            ("persistent", "workspace", 3)]:
        C = run(A, B, sa, sb, 128, 128, 128, mode, red, ctas)
        check_parity(C, ref, "bf16", K, kind="fp8", what=f"block {shape} {mode}/{red}")


def test_blockscale_scales_matter():
    # The same operands with one A block scale doubled: exactly the outputs of that row and
    # block change, so the block index arithmetic cannot be off by one step.
    M, N, K = 256, 256, 1024
    A, B, sa, sb, ref = case(M, N, K, "abquant", 128, 128, 128, 4)
    sa2 = sa.clone()
    sa2[5, 3] *= 2.0
    ref2 = numerics.fp8_blockscale_rows(bits(A), bits(B), sa2.numpy(), 128, sb.numpy(), 128, 128)
    C = run(A, B, sa2, sb, 128, 128, 128, "dp_sk", "linear", -1)
    check_parity(C, ref2, "bf16", K, kind="fp8", what="block one scale doubled")
    C0 = run(A, B, sa, sb, 128, 128, 128, "dp_sk", "linear", -1)
    changed = (C.float() != C0.float()).any(dim=1).nonzero().flatten().tolist()
    assert changed == [5]


@pytest.mark.parametrize("red", ["linear", "workspace"])
def test_blockscale_4096_sampled(red):
    M = N = K = 4096
    A, B, sa, sb = operands(M, N, K, "abquant", 128, 128, 128, 0)
    C = run(A, B, sa, sb, 128, 128, 128, "dp_sk", red, -1)
    assert torch.isfinite(C.float()).all(), "unwritten outputs"
    ms, ns = sample_points(M, N, n_random=4096, tile=128)
    ref = numerics.fp8_blockscale_points(bits(A), bits(B), sa.numpy(), 128, sb.numpy(), 128, 128,
                                         ms, ns)
    out = C[torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)]
    check_parity(out, ref, "bf16", K, kind="fp8", what=f"block 4096^3 {red} sampled")


@pytest.mark.parametrize("red", ["linear", "tree"])
def test_blockscale_bit_identical(red):
    # 20 launches with the workspace and the output poisoned before each one
    M, N, K = 300, 392, 1040
    A, B, sa, sb, _ = case(M, N, K, "abquant", 128, 128, 256, 1)
    Ad, Bd, sad, sbd = A.to(DEV), B.to(DEV), sa.to(DEV), sb.to(DEV)
    prob = sk.make_problem("fp8_block", ab_dtype="e4m3", c_dtype="bf16", M=M, N=N, K=K)
    ws = torch.empty(sk.sk_workspace_bytes(prob, "dp_sk", red, 5), dtype=torch.uint8, device=DEV)
    C = poisoned((M, N), torch.bfloat16)
    first = None
    for _ in range(20):
        ws.fill_(0xFF)
        C.view(torch.uint8).fill_(0xFF)
        sk.sk_gemm_blockscale_fp8(Ad, Bd, sad, 128, sbd, 128, 256, C, streamk="dp_sk",
                                  reduction=red, ctas=5, ws=ws)
        sk.sk_device_status()
        b = C.view(torch.uint8).clone()
        assert torch.isfinite(C.float()).all()
        if first is None:
            first = b
        else:
            assert torch.equal(first, b), "result changed between launches"
