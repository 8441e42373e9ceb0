"""GPU parity of the CTA-pair tiles, 256 x 128 and 256 x 256 (two CTAs of a cluster share each tile
through the two-SM tensor-core instruction), against the fp64 oracle, through the same C ABI calls
as the 128 x 128 tile: every mode x reduction on ragged shapes, the fp8 GEMM, sampled outputs of the
large workloads, bit-identical linear/tree hand-offs, and the wgrad rejection."""
import pytest
import torch

from oracle import numerics
from workloads import fp8_operands, gemm_operands

pytestmark = pytest.mark.gpu

import implicit_gemm_conv_gb300 as sk  # noqa: E402  (no skip: a missing library must fail)
from gpu_helpers import DEV, bits, check_parity, poisoned, sample_points  # noqa: E402

MODES = ["off", "dp_sk", "persistent", "splitk", "hybrid"]
REDS = ["linear", "tree", "atomic", "workspace"]
TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(autouse=True, params=["256_pair", "256x256_pair"])
def pair_tile(request):
    with sk.tile(request.param):
        yield request.param


def run_gemm(A, B, out_dtype, mode, red, ctas, ws=None):
    M, N = A.shape[0], B.shape[0]
    C = poisoned((M, N), TD[out_dtype])
    sk.sk_gemm_rcr(A.to(DEV), B.to(DEV), C, streamk=mode, reduction=red, ctas=ctas, ws=ws)
    sk.sk_device_status()
    return C


_REF = {}


def ref_full(ab, M, N, K, dist, off):
    key = (ab, M, N, K, dist, off)
    if key not in _REF:
        A, B = gemm_operands(M, N, K, ab, dist, seed_offset=off)
        _REF[key] = (A, B, numerics.gemm_rcr_rows(ab, bits(A), bits(B)))
    return _REF[key]


def test_pair_single_tile(pair_tile):
    # one pair tile, one K step: the smallest use of both CTAs' operands
    n = 256 if pair_tile == "256x256_pair" else 128
    A, B, ref = ref_full("bf16", 256, n, 64, "n01", 21)
    C = run_gemm(A, B, "bf16", "off", "linear", 1)
    check_parity(C, ref, "bf16", 64, what=f"pair 256x{n}x64")


@pytest.mark.parametrize("red", REDS)
@pytest.mark.parametrize("mode", MODES)
def test_pair_ragged_bf16(mode, red):
    # 300 x 392: a partial second M half and a partial last N tile of either pair tile;
    # K = 520: a ragged last K step (8 of 64)
    A, B, ref = ref_full("bf16", 300, 392, 520, "n01", 7)
    out = "f32" if red == "atomic" else "bf16"
    C = run_gemm(A, B, out, mode, red, 5)
    check_parity(C, ref, out, 520, what=f"pair {mode}/{red}")


@pytest.mark.parametrize("red", REDS)
@pytest.mark.parametrize("mode", MODES)
def test_pair_512x384x4096_pool3(mode, red):
    A, B, ref = ref_full("f16", 512, 384, 4096, "u11", 0)
    out = "f32" if red == "atomic" else "f16"
    C = run_gemm(A, B, out, mode, red, 3)
    check_parity(C, ref, out, 4096, what=f"pair pool 3 {mode}/{red}")


@pytest.mark.parametrize("shape", [(1, 8, 8), (129, 8, 64), (257, 1024, 8192), (640, 640, 1088)])
@pytest.mark.parametrize("red", ["linear", "tree", "workspace"])
def test_pair_edges(shape, red):
    M, N, K = shape
    A, B, ref = ref_full("f16", M, N, K, "u11", 3)
    for mode, ctas in [("dp_sk", -1), ("persistent", 7), ("dp_sk", 13)]:
        C = run_gemm(A, B, "f16", mode, red, ctas)
        check_parity(C, ref, "f16", K, what=f"pair {shape} {mode}/{red}/{ctas}")


def _sampled(ab, M, N, K, dist, mode, red, ctas):
    A, B = gemm_operands(M, N, K, ab, dist)
    C = run_gemm(A, B, ab, mode, red, ctas)
    ms, ns = sample_points(M, N, tile=256)
    ref = numerics.gemm_rcr_points(ab, bits(A), bits(B), ms, ns)
    out = C[torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)]
    check_parity(out, ref, ab, K, what=f"pair {M}x{N}x{K} {mode}/{red}/{ctas} sampled")
    assert torch.isfinite(C.float()).all(), "unwritten outputs"


@pytest.mark.parametrize("red,ctas", [("linear", 148), ("tree", 148), ("linear", 74),
                                      ("workspace", -1)])
def test_pair_3840x4096x4096_sampled(red, ctas):
    _sampled("bf16", 3840, 4096, 4096, "n01", "dp_sk", red, ctas)


@pytest.mark.parametrize("mode,red", [("dp_sk", "linear"), ("dp_sk", "tree"),
                                      ("dp_sk", "workspace"), ("splitk", "workspace")])
def test_pair_512x512x65536_sampled(mode, red):
    _sampled("bf16", 512, 512, 65536, "n01", mode, red, 148)


def run_fp8(A, B, sa, sb, mode, red, ctas):
    M, N = A.shape[0], B.shape[0]
    C = poisoned((M, N), torch.bfloat16)
    sk.sk_gemm_rowcol_fp8(A.to(DEV), B.to(DEV), sa.to(DEV), sb.to(DEV), C, streamk=mode,
                          reduction=red, ctas=ctas)
    sk.sk_device_status()
    return C


@pytest.mark.parametrize("red", ["linear", "tree", "workspace"])
@pytest.mark.parametrize("mode", MODES)
def test_pair_fp8_small(mode, red):
    M, N, K = 300, 392, 1040
    A, B, sa, sb = fp8_operands(M, N, K, seed_offset=2)
    ref = numerics.fp8_rowcol_rows(bits(A), bits(B), sa.numpy(), sb.numpy())
    C = run_fp8(A, B, sa, sb, mode, red, 5)
    check_parity(C, ref, "bf16", K, kind="fp8", what=f"pair fp8 {mode}/{red}")


def test_pair_fp8_8192_sampled():
    M = N = K = 8192
    A, B, sa, sb = fp8_operands(M, N, K)
    C = run_fp8(A, B, sa, sb, "dp_sk", "linear", -1)
    ms, ns = sample_points(M, N, n_random=4096, tile=256)
    ref = numerics.fp8_rowcol_points(bits(A), bits(B), sa.numpy(), sb.numpy(), ms, ns)
    out = C[torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)]
    check_parity(out, ref, "bf16", K, kind="fp8", what="pair fp8 8192^3")
    assert torch.isfinite(C.float()).all()


@pytest.mark.parametrize("red", ["linear", "tree"])
@pytest.mark.parametrize("shape,ctas", [((3840, 4096, 4096), 74), ((512, 512, 65536), 148),
                                        ((512, 384, 4096), 3)])
def test_pair_bit_identical(shape, ctas, red):
    # 20 launches with the workspace and the output poisoned (0xFF bytes) before each one
    M, N, K = shape
    A, B = gemm_operands(M, N, K, "bf16", "n01")
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = poisoned((M, N), torch.bfloat16)
    mode = "persistent" if ctas == 3 else "dp_sk"
    prob = sk.make_problem("gemm", ab_dtype="bf16", c_dtype="bf16", M=M, N=N, K=K)
    ws = torch.empty(sk.sk_workspace_bytes(prob, mode, red, ctas), dtype=torch.uint8, device=DEV)
    first = None
    for _ in range(20):
        ws.fill_(0xFF)
        C.view(torch.uint8).fill_(0xFF)
        sk.sk_gemm_rcr(Ad, Bd, C, streamk=mode, reduction=red, ctas=ctas, ws=ws)
        sk.sk_device_status()
        b = C.view(torch.uint8).clone()
        assert torch.isfinite(C.float()).all()
        if first is None:
            first = b
        else:
            assert torch.equal(first, b), "result changed between launches"


def test_pair_agrees_with_single_tile():
    # The pair tile changes which CTA adds which partial, so the two results are compared within
    # a few fp32 roundings; each also meets the oracle bound (checked above).
    A, B, ref = ref_full("bf16", 300, 392, 520, "n01", 7)
    C2 = run_gemm(A, B, "f32", "dp_sk", "linear", 5)
    with sk.tile("128"):
        C1 = run_gemm(A, B, "f32", "dp_sk", "linear", 5)
    assert (C2 - C1).abs().max().item() <= 1e-3 * max(1.0, C1.abs().max().item())


def test_pair_rejects_wgrad_outside_the_row_view():
    """Under the pair tiles a wgrad of 128-channel groups (the pages' view) is refused; the
    shifted-row shapes run on the row kernel's pair tile (tests/test_gpu_wgrad.py)."""
    x = torch.zeros((1, 8, 8, 128), dtype=torch.float16, device=DEV)
    dy = torch.zeros((1, 8, 8, 64), dtype=torch.float16, device=DEV)
    dw = torch.zeros((64, 1, 1, 128), dtype=torch.float32, device=DEV)
    with pytest.raises(sk.SkError) as e:
        sk.sk_conv2d_wgrad_nhwc(x, dy, dw, 1, 1, (1, 1), (0, 0), 1, streamk="dp_sk",
                                reduction="linear", ctas=-1)
    assert e.value.code == -2 and "GEMMs and the shifted-row wgrad only" in str(e.value)


@pytest.mark.parametrize("mode,red", [("dp_sk", "linear"), ("off", "linear"), ("dp_sk", "tree"),
                                      ("persistent", "workspace")])
def test_pair_strided_16bit_output(mode, red):
    # A 16-bit C with a row stride larger than N: complete tiles leave through TMA tile stores
    # whose tensor map carries ldc; nothing outside the [M, N] window may be written.
    M, N, K = 520, 392, 1032
    A, B, ref = ref_full("bf16", M, N, K, "n01", 31)
    Cbig = poisoned((M, 512), torch.bfloat16)
    C = Cbig[:, :N]
    sk.sk_gemm_rcr(A.to(DEV), B.to(DEV), C, streamk=mode, reduction=red, ctas=5)
    sk.sk_device_status()
    check_parity(C, ref, "bf16", K, what=f"strided 16-bit C {mode}/{red}")
    assert torch.isnan(Cbig[:, N:].float()).all(), "wrote outside the [M, N] window"


def test_pair_auto_mode_and_reduction(pair_tile):
    # streamk = auto / reduction = auto over pair tiles: 2 tiles, a long reduction, 74 pairs ->
    # stream-K with the workspace reduction; 24 tiles on a pool of 3 pairs -> split-K (one slice)
    n = 256 if pair_tile == "256x256_pair" else 128
    prob = sk.make_problem("gemm", ab_dtype="bf16", c_dtype="bf16", M=512, N=n, K=32768)
    plan = sk.sk_plan(prob, "auto", "auto", 74)
    assert plan.mode == sk.DP_SK and plan.reduction == sk.WORKSPACE and plan.sk_ctas == 74
    A, B, ref = ref_full("bf16", 512, n, 32768, "n01", 13)
    C = run_gemm(A, B, "bf16", "auto", "auto", 74)
    check_parity(C, ref, "bf16", 32768, what="pair auto -> dp_sk/workspace")
    prob = sk.make_problem("gemm", ab_dtype="f16", c_dtype="f16", M=1536, N=1024, K=1024)
    assert sk.sk_plan(prob, "auto", "linear", 3).mode == sk.SPLITK
    A, B, ref = ref_full("f16", 1536, 1024, 1024, "u11", 14)
    C = run_gemm(A, B, "f16", "auto", "linear", 3)
    check_parity(C, ref, "f16", 1024, what="pair auto -> split-K")
