"""GPU parity of the stream-K rcr GEMM (sk_gemm_rcr through the C ABI) against the fp64 oracle:
every mode x reduction on the 256x256x4096 pool-3 workload and on a ragged shape, sampled outputs of
the 3840x4096x4096 pool-148 and 512x512x65536 workloads, and edge cases."""
import numpy as np
import pytest
import torch

from oracle import numerics
from workloads import gemm_operands

pytestmark = pytest.mark.gpu

import implicit_gemm_conv_gb300 as sk  # noqa: E402  (no skip: a missing library must fail)
from gpu_helpers import DEV, bits, check_parity, poisoned, sample_points  # noqa: E402


@pytest.fixture(autouse=True)
def tile_128():
    """The configurations these tests follow fix 128 x 128 tiles; the pair tiles have their own
    tests."""
    with sk.tile("128"):
        yield

MODES = ["off", "dp_sk", "persistent", "splitk", "hybrid"]
REDS = ["linear", "tree", "atomic", "workspace"]
TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


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


@pytest.mark.parametrize("red", REDS)
@pytest.mark.parametrize("mode", MODES)
def test_gemm_256x256x4096_pool3(mode, red):
    A, B, ref = ref_full("f16", 256, 256, 4096, "u11", 0)
    out = "f32" if red == "atomic" else "f16"
    C = run_gemm(A, B, out, mode, red, 3)
    check_parity(C, ref, out, 4096, what=f"{mode}/{red}")


@pytest.mark.parametrize("red", REDS)
@pytest.mark.parametrize("mode", MODES)
def test_gemm_ragged_bf16(mode, red):
    # 200 x 136: partial last M and N tiles; K = 520: a ragged last K step (8 of 64)
    A, B, ref = ref_full("bf16", 200, 136, 520, "n01", 7)
    out = "f32" if red == "atomic" else "bf16"
    C = run_gemm(A, B, out, mode, red, 5)
    check_parity(C, ref, out, 520, what=f"{mode}/{red}")


@pytest.mark.parametrize("shape", [(1, 8, 8), (129, 8, 64), (64, 1024, 8192), (384, 640, 1088)])
@pytest.mark.parametrize("red", ["linear", "tree", "workspace"])
def test_gemm_edges(shape, red):
    M, N, K = shape
    A, B, ref = ref_full("f16", M, N, K, "u11", 3)
    for mode, ctas in [("dp_sk", -1), ("persistent", 7), ("dp_sk", 13)]:
        C = run_gemm(A, B, "f16", mode, red, ctas)
        check_parity(C, ref, "f16", K, what=f"{shape} {mode}/{red}/{ctas}")


def test_gemm_f32_output_and_leading_dims():
    M, N, K = 192, 200, 256
    A, B, ref = ref_full("bf16", M, N, K, "u11", 9)
    Ad = torch.zeros((M, K + 64), dtype=torch.bfloat16, device=DEV)[:, :K]
    Ad.copy_(A.to(DEV))
    Bd = torch.zeros((N, K + 8), dtype=torch.bfloat16, device=DEV)[:, :K]
    Bd.copy_(B.to(DEV))
    Cbig = poisoned((M, 256), torch.float32)
    C = Cbig[:, :N]
    sk.sk_gemm_rcr(Ad, Bd, C, streamk="persistent", reduction="tree", ctas=4)
    sk.sk_device_status()
    check_parity(C, ref, "f32", K, what="strided")
    tail = Cbig[:, N:].cpu()
    assert torch.isnan(tail).all(), "wrote outside the [M, N] window"


def test_gemm_k_zero_gives_zeros():
    A = torch.zeros((64, 0), dtype=torch.float16, device=DEV)
    B = torch.zeros((32, 0), dtype=torch.float16, device=DEV)
    C = poisoned((64, 32), torch.float16)
    sk.sk_gemm_rcr(A, B, C, streamk="dp_sk", reduction="linear", ctas=-1)
    torch.cuda.synchronize()
    assert (C == 0).all()


def test_caller_workspace_and_size_check():
    A, B, ref = ref_full("f16", 256, 256, 4096, "u11", 0)
    prob = sk.make_problem("gemm", ab_dtype="f16", c_dtype="f16", M=256, N=256, K=4096)
    need = sk.sk_workspace_bytes(prob, "persistent", "linear", 3)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    ws.fill_(0xFF)
    C = run_gemm(A, B, "f16", "persistent", "linear", 3, ws=ws)
    check_parity(C, ref, "f16", 4096, what="caller ws")
    small = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(sk.SkError) as e:
        run_gemm(A, B, "f16", "persistent", "linear", 3, ws=small)
    assert e.value.code == -2 and "workspace too small" in str(e.value)


def _sampled(ab, M, N, K, dist, mode, red, ctas):
    A, B = gemm_operands(M, N, K, ab, dist)
    C = run_gemm(A, B, ab, mode, red, ctas)
    ms, ns = sample_points(M, N)
    ref = numerics.gemm_rcr_points(ab, bits(A), bits(B), ms, ns)
    out = C[torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)]
    check_parity(out, ref, ab, K, what=f"{M}x{N}x{K} {mode}/{red} sampled")
    assert torch.isfinite(C.float()).all(), "unwritten outputs"


@pytest.mark.parametrize("red", ["linear", "tree"])
def test_gemm_3840x4096x4096_pool148_sampled(red):
    _sampled("bf16", 3840, 4096, 4096, "n01", "dp_sk", red, 148)



@pytest.mark.parametrize("mode,red", [("dp_sk", "linear"), ("dp_sk", "tree"),
                                      ("persistent", "workspace"), ("splitk", "workspace"),
                                      ("off", "linear")])
def test_gemm_512x512x65536_pool148_sampled(mode, red):
    _sampled("bf16", 512, 512, 65536, "n01", mode, red, 148)


def test_gemm_auto_selection():
    # few tiles over a long reduction -> stream-K; reduction auto -> workspace
    prob = sk.make_problem("gemm", ab_dtype="bf16", c_dtype="bf16", M=512, N=512, K=65536)
    plan = sk.sk_plan(prob, "auto", "auto", 148)
    assert plan.mode == sk.DP_SK and plan.reduction == sk.WORKSPACE
    _sampled("bf16", 512, 512, 65536, "n01", "auto", "auto", 148)
    # the tiles fill the pool -> split-K with one slice, i.e. data-parallel
    A, B, ref = ref_full("f16", 256, 256, 4096, "u11", 0)
    assert sk.sk_plan(sk.make_problem("gemm", ab_dtype="f16", c_dtype="f16", M=256, N=256,
                                      K=4096), "auto", "linear", 3).mode == sk.SPLITK
    C = run_gemm(A, B, "f16", "auto", "linear", 3)
    check_parity(C, ref, "f16", 4096, what="auto pool 3")


@pytest.mark.parametrize("mode,red", [("dp_sk", "linear"), ("off", "linear"), ("persistent", "tree")])
def test_gemm_strided_16bit_output(mode, red):
    # 16-bit C with a row stride larger than N (TMA-store epilogue, 128x128 tile)
    M, N, K = 200, 136, 520
    A, B, ref = ref_full("bf16", M, N, K, "n01", 7)
    Cbig = poisoned((M, 256), torch.bfloat16)
    C = Cbig[:, :N]
    sk.sk_gemm_rcr(A.to(DEV), B.to(DEV), C, streamk=mode, reduction=red, ctas=5)
    sk.sk_device_status()
    check_parity(C, ref, "bf16", 520, what=f"strided 16-bit C {mode}/{red}")
    assert torch.isnan(Cbig[:, N:].float()).all(), "wrote outside the [M, N] window"


# ---- the automatic tile's deep-ring 256x256 CTA pair for few tiles over a long 16-bit reduction

@pytest.mark.parametrize("mode,red", [("dp_sk", "linear"), ("dp_sk", "tree"), ("dp_sk", "workspace"),
                                      ("splitk", "workspace"), ("persistent", "linear")])
def test_gemm_512x512x65536_auto_pair_sampled(mode, red):
    with sk.tile("auto"):
        prob = sk.make_problem("gemm", ab_dtype="bf16", c_dtype="bf16", M=512, N=512, K=65536)
        assert (sk.sk_plan(prob, mode, red, 74).tm, sk.sk_plan(prob, mode, red, 74).tn) == (256, 256)
        _sampled("bf16", 512, 512, 65536, "n01", mode, red, 74)


@pytest.mark.parametrize("red", ["linear", "atomic", "workspace"])
def test_gemm_ragged_long_k_auto_pair(red):
    """Partial M and N pair tiles and a ragged K tail (K = 33000) on the deep-ring pair."""
    M, N, K = 300, 392, 33000
    with sk.tile("auto"):
        prob = sk.make_problem("gemm", ab_dtype="bf16", c_dtype="bf16", M=M, N=N, K=K)
        assert sk.sk_plan(prob, "dp_sk", red, 5).tm == 256
        A, B, ref = ref_full("bf16", M, N, K, "u11", 21)
        out = "f32" if red == "atomic" else "bf16"
        C = run_gemm(A, B, out, "dp_sk", red, 5)
    check_parity(C, ref, out, K, what=f"ragged long-K pair {red}")
