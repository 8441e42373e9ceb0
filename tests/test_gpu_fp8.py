"""GPU parity of the fp8 e4m3 row/col-scaled GEMM (sk_gemm_rowcol_fp8 through the C ABI) against
the oracle, which decodes the same e4m3 bytes (quantise -> dequantise) and applies the scales."""
import numpy as np
import pytest
import torch

from oracle import numerics
from workloads import fp8_operands

pytestmark = pytest.mark.gpu

import implicit_gemm_conv_gb300 as sk  # noqa: E402  (no skip: a missing library must fail)
from gpu_helpers import DEV, bits, check_parity, poisoned, sample_points  # noqa: E402


@pytest.fixture(autouse=True)
def tile_128():
    """The configurations these tests follow fix 128 x 128 tiles; the pair tiles have their own
    tests."""
    with sk.tile("128"):
        yield


def run(A, B, sa, sb, mode, red, ctas):
    M, N = A.shape[0], B.shape[0]
    C = poisoned((M, N), torch.bfloat16)
    sk.sk_gemm_rowcol_fp8(A.to(DEV), B.to(DEV), sa.to(DEV), sb.to(DEV), C, streamk=mode,
                          reduction=red, ctas=ctas)
    sk.sk_device_status()
    return C


@pytest.mark.parametrize("red", ["linear", "tree", "workspace"])
@pytest.mark.parametrize("mode", ["off", "dp_sk", "persistent", "splitk"])
def test_fp8_small(mode, red):
    M, N, K = 200, 136, 1040
    A, B, sa, sb = fp8_operands(M, N, K, seed_offset=2)
    ref = numerics.fp8_rowcol_rows(bits(A), bits(B), sa.numpy(), sb.numpy())
    C = run(A, B, sa, sb, mode, red, 5)
    check_parity(C, ref, "bf16", K, kind="fp8", what=f"{mode}/{red}")


def test_fp8_atomic_rejected():
    A, B, sa, sb = fp8_operands(128, 128, 128)
    with pytest.raises(sk.SkError) as e:
        run(A, B, sa, sb, "dp_sk", "atomic", -1)
    assert e.value.code == -2


@pytest.mark.parametrize("red", ["linear", "workspace"])
def test_fp8_8192_sampled(red):
    M = N = K = 8192
    A, B, sa, sb = fp8_operands(M, N, K)
    C = run(A, B, sa, sb, "dp_sk", red, -1)
    ms, ns = sample_points(M, N, n_random=4096)
    ref = numerics.fp8_rowcol_points(bits(A), bits(B), sa.numpy(), sb.numpy(), ms, ns)
    out = C[torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)]
    check_parity(out, ref, "bf16", K, kind="fp8", what=f"8192^3 {red}")
    assert torch.isfinite(C.float()).all()


def run_tq(A, B, scale_a, scale_b, mode, red, ctas):
    M, N = A.shape[0], B.shape[0]
    C = poisoned((M, N), torch.bfloat16)
    sk.sk_gemm_tensorquant_fp8(A.to(DEV), B.to(DEV), scale_a, scale_b, C, streamk=mode,
                               reduction=red, ctas=ctas)
    sk.sk_device_status()
    return C


@pytest.mark.parametrize("red", ["linear", "tree", "workspace"])
@pytest.mark.parametrize("mode", ["off", "dp_sk", "persistent", "splitk"])
def test_fp8_tensorquant_small(mode, red):
    # per-tensor scales (PR #10439 "tensor_quant"): one scalar for A, one for B
    M, N, K = 200, 136, 1040
    A, B, _, _ = fp8_operands(M, N, K, seed_offset=12)
    ref = numerics.fp8_tensorquant_rows(bits(A), bits(B), 0.8125, 1.375)
    C = run_tq(A, B, 0.8125, 1.375, mode, red, 5)
    check_parity(C, ref, "bf16", K, kind="fp8", what=f"tensorquant {mode}/{red}")


@pytest.mark.parametrize("tile", ["128", "256x256_pair"])
def test_fp8_tensorquant_pair_and_large(tile):
    M, N, K = 2048, 2048, 4096
    A, B, _, _ = fp8_operands(M, N, K, seed_offset=13)
    with sk.tile(tile):
        C = run_tq(A, B, 0.5, 1.5, "dp_sk", "linear", -1)
    rows = np.r_[0:130, 1000:1030, M - 130:M]
    ref = np.concatenate([numerics.fp8_tensorquant_rows(bits(A), bits(B), 0.5, 1.5, a, b)
                          for a, b in [(0, 130), (1000, 1030), (M - 130, M)]])
    check_parity(C[torch.from_numpy(rows).to(DEV)], ref, "bf16", K, kind="fp8",
                 what=f"tensorquant 2048^2x4096 {tile}")
