"""Seeded synthetic inputs and the named workloads.

This module is shared by the CUDA-path tests, the benchmark and the CPU oracle's callers. It holds
shapes, seeds and random-number draws only -- none of the method's arithmetic. Values are drawn on
the CPU with ``torch.Generator().manual_seed(seed)`` and cast to the storage type once; every
consumer reads the same bytes.

Seeds: A=1, B=2, x=3, dy=4, sa=5, sb=6, conv filter w=7 (a shape-specific offset is added for the small
test cases).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Tuple

import torch

SEED_A, SEED_B, SEED_X, SEED_DY, SEED_SA, SEED_SB, SEED_W = 1, 2, 3, 4, 5, 6, 7

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def draw(shape, dist: str, seed: int) -> torch.Tensor:
    """fp32 samples: ``"u11"`` = uniform[-1, 1], ``"n01"`` = N(0, 1), ``"n0.5"`` = N(0, 0.5^2)
    (0.5 read as the standard deviation), ``"u0.5_2"`` = uniform[0.5, 2]."""
    g = _gen(seed)
    if dist == "u11":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    if dist == "n01":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    if dist == "n0.5":
        return torch.randn(shape, generator=g, dtype=torch.float32) * 0.5
    if dist == "u0.5_2":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 1.5 + 0.5
    raise ValueError(dist)


def gemm_operands(M: int, N: int, K: int, dtype: str, dist: str, seed_offset: int = 0):
    """rcr operands: A [M][K] row-major, B [N][K] (= B col-major K x N)."""
    A = draw((M, K), dist, SEED_A + seed_offset).to(TORCH_DTYPE[dtype])
    B = draw((N, K), dist, SEED_B + seed_offset).to(TORCH_DTYPE[dtype])
    return A, B


def fp8_operands(M: int, N: int, K: int, seed_offset: int = 0):
    """e4m3 A [M][K], B [N][K] from N(0,1) samples (torch's cast, values clipped to the finite
    range first), fp32 scales sa [M], sb [N] from uniform[0.5, 2]."""
    A = draw((M, K), "n01", SEED_A + seed_offset).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    B = draw((N, K), "n01", SEED_B + seed_offset).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    sa = draw((M,), "u0.5_2", SEED_SA + seed_offset)
    sb = draw((N,), "u0.5_2", SEED_SB + seed_offset)
    return A, B, sa, sb


def blockscale_scales(M: int, N: int, K: int, gka: int, gnb: int, gkb: int, seed_offset: int = 0):
    """Block scales from uniform[0.5, 2]: sa [M][ceil(K/gka)] (A blocks along K) and
    sb [ceil(N/gnb)][ceil(K/gkb)] (B blocks along N and K)."""
    sa = draw((M, -(-K // gka)), "u0.5_2", SEED_SA + seed_offset)
    sb = draw((-(-N // gnb), -(-K // gkb)), "u0.5_2", SEED_SB + seed_offset)
    return sa, sb


def conv_out(H: int, R: int, stride: int, pad: int) -> int:
    return (H + 2 * pad - R) // stride + 1


def wgrad_operands(N, H, W, C, K, R, S, stride, pad, dtype, dist, seed_offset: int = 0):
    """NHWC x [N][H][W][C] and dy [N][Ho][Wo][K]."""
    Ho, Wo = conv_out(H, R, stride[0], pad[0]), conv_out(W, S, stride[1], pad[1])
    x = draw((N, H, W, C), dist, SEED_X + seed_offset).to(TORCH_DTYPE[dtype])
    dy = draw((N, Ho, Wo, K), dist, SEED_DY + seed_offset).to(TORCH_DTYPE[dtype])
    return x, dy


def fprop_operands(N, H, W, C, K, R, S, groups, dtype, dist, seed_offset: int = 0):
    """NHWC x [N][H][W][C] and the filter w [K][R][S][C/groups]."""
    x = draw((N, H, W, C), dist, SEED_X + seed_offset).to(TORCH_DTYPE[dtype])
    w = draw((K, R, S, C // groups), dist, SEED_W + seed_offset).to(TORCH_DTYPE[dtype])
    return x, w


def dgrad_operands(N, H, W, C, K, R, S, stride, pad, groups, dtype, dist, seed_offset: int = 0):
    """NHWC dy [N][Ho][Wo][K] and the filter w [K][R][S][C/groups]."""
    Ho, Wo = conv_out(H, R, stride[0], pad[0]), conv_out(W, S, stride[1], pad[1])
    dy = draw((N, Ho, Wo, K), dist, SEED_DY + seed_offset).to(TORCH_DTYPE[dtype])
    w = draw((K, R, S, C // groups), dist, SEED_W + seed_offset).to(TORCH_DTYPE[dtype])
    return dy, w


@dataclass
class Workload:
    name: str
    op: str                      # "gemm" | "wgrad" | "fp8" | "fp8_block" | "fprop" | "dgrad"
    ab: str                      # input storage type
    out: str                     # output type
    dist: str
    M: int = 0
    N: int = 0
    K: int = 0
    conv: Optional[dict] = None  # N,H,W,C,K,R,S,stride,pad,groups
    pool: int = -1
    modes: Tuple[str, ...] = ("dp_sk",)
    reductions: Tuple[str, ...] = ("linear",)
    blocks: Optional[Tuple[int, int, int]] = None   # fp8_block: (a_group_k, b_group_n, b_group_k)

    def _conv_dims(self):
        c = self.conv
        Ho = conv_out(c["H"], c["R"], c["stride"][0], c["pad"][0])
        Wo = conv_out(c["W"], c["S"], c["stride"][1], c["pad"][1])
        return c, Ho, Wo

    def flops(self) -> float:
        if self.op in ("fprop", "dgrad"):
            c, Ho, Wo = self._conv_dims()
            if self.op == "fprop":   # output pixels x filters x (r, s, c per group)
                return 2.0 * c["N"] * Ho * Wo * c["K"] * c["R"] * c["S"] * (c["C"] // c["groups"])
            return 2.0 * c["N"] * c["H"] * c["W"] * c["C"] * c["R"] * c["S"] * (c["K"] // c["groups"])
        if self.op == "wgrad":
            c = self.conv
            Ho = conv_out(c["H"], c["R"], c["stride"][0], c["pad"][0])
            Wo = conv_out(c["W"], c["S"], c["stride"][1], c["pad"][1])
            kred = c["N"] * Ho * Wo
            return 2.0 * c["K"] * c["R"] * c["S"] * (c["C"] // c["groups"]) * kred
        return 2.0 * self.M * self.N * self.K

    def kred(self) -> int:
        if self.op in ("fprop", "dgrad"):
            c = self.conv
            per = (c["C"] if self.op == "fprop" else c["K"]) // c["groups"]
            return c["R"] * c["S"] * per
        if self.op == "wgrad":
            c = self.conv
            return c["N"] * conv_out(c["H"], c["R"], c["stride"][0], c["pad"][0]) * \
                conv_out(c["W"], c["S"], c["stride"][1], c["pad"][1])
        return self.K

    def min_bytes(self) -> float:
        """Each operand read once, the output written once."""
        sz = {"f16": 2, "bf16": 2, "f32": 4, "e4m3": 1}
        if self.op in ("fprop", "dgrad"):
            c, Ho, Wo = self._conv_dims()
            x = c["N"] * c["H"] * c["W"] * c["C"]
            dy = c["N"] * Ho * Wo * c["K"]
            w = c["K"] * c["R"] * c["S"] * (c["C"] // c["groups"])
            inp, out = (x, dy) if self.op == "fprop" else (dy, x)
            return (inp + w) * sz[self.ab] + out * sz[self.out]
        if self.op == "wgrad":
            c = self.conv
            Ho = conv_out(c["H"], c["R"], c["stride"][0], c["pad"][0])
            Wo = conv_out(c["W"], c["S"], c["stride"][1], c["pad"][1])
            x = c["N"] * c["H"] * c["W"] * c["C"]
            dy = c["N"] * Ho * Wo * c["K"]
            dw = c["K"] * c["R"] * c["S"] * (c["C"] // c["groups"])
            return (x + dy) * sz[self.ab] + dw * sz[self.out]
        extra = 4 * (self.M + self.N) if self.op == "fp8" else 0
        if self.op == "fp8_block":
            gka, gnb, gkb = self.blocks
            extra = 4 * (self.M * -(-self.K // gka) + -(-self.N // gnb) * -(-self.K // gkb))
        return (self.M + self.N) * self.K * sz[self.ab] + self.M * self.N * sz[self.out] + extra


WORKLOADS = {
    w.name: w for w in [
        Workload("gemm_f16_256x256x4096_pool3", "gemm", "f16", "f16", "u11", 256, 256, 4096,
                 pool=3, modes=("persistent",), reductions=("linear", "tree", "atomic", "workspace")),
        Workload("gemm_bf16_3840x4096x4096_pool148", "gemm", "bf16", "bf16", "n01", 3840, 4096, 4096,
                 pool=148, modes=("dp_sk",), reductions=("linear", "tree")),
        Workload("wgrad_f16_n32_56x56_c64_k64_3x3", "wgrad", "f16", "f32", "u11",
                 conv=dict(N=32, H=56, W=56, C=64, K=64, R=3, S=3, stride=(1, 1), pad=(1, 1),
                           groups=1),
                 pool=-1, modes=("dp_sk", "persistent"),
                 reductions=("linear", "tree", "atomic", "workspace")),
        Workload("wgrad_bf16_n64_28x28_c256_k256_g4_s2", "wgrad", "bf16", "f32", "n0.5",
                 conv=dict(N=64, H=28, W=28, C=256, K=256, R=3, S=3, stride=(2, 2), pad=(1, 1),
                           groups=4),
                 pool=-1, modes=("dp_sk", "persistent"), reductions=("atomic", "workspace")),
        Workload("fp8_rowcol_8192x8192x8192", "fp8", "e4m3", "bf16", "n01", 8192, 8192, 8192,
                 pool=-1, modes=("dp_sk",), reductions=("linear", "tree", "workspace")),
        # A scaled per row in blocks of 128 along K, B in 128 x 128 blocks.
        Workload("fp8_blockscale_8192x8192x8192_a1x128_b128x128", "fp8_block", "e4m3", "bf16",
                 "n01", 8192, 8192, 8192, pool=-1, modes=("dp_sk",),
                 reductions=("linear", "workspace"), blocks=(128, 128, 128)),
        Workload("gemm_bf16_512x512x65536_pool148", "gemm", "bf16", "bf16", "n01", 512, 512, 65536,
                 pool=148, modes=("dp_sk", "persistent"),
                 reductions=("linear", "tree", "workspace")),
        # The same 3x3 layer as the wgrad workload, forward and data gradient.
        # The automatic mode runs the shifted-row kernel persistently (all tiles data-parallel).
        Workload("fprop_f16_n32_56x56_c64_k64_3x3", "fprop", "f16", "f16", "u11",
                 conv=dict(N=32, H=56, W=56, C=64, K=64, R=3, S=3, stride=(1, 1), pad=(1, 1),
                           groups=1),
                 pool=-1, modes=("dp_sk", "persistent", "auto"), reductions=("linear", "tree")),
        Workload("dgrad_f16_n32_56x56_c64_k64_3x3", "dgrad", "f16", "f16", "u11",
                 conv=dict(N=32, H=56, W=56, C=64, K=64, R=3, S=3, stride=(1, 1), pad=(1, 1),
                           groups=1),
                 pool=-1, modes=("dp_sk", "persistent", "auto"), reductions=("linear", "tree")),
        # A downsampling layer's data gradient: stride 2, four output phases.
        Workload("dgrad_f16_n32_56x56_c64_k128_3x3_s2", "dgrad", "f16", "f16", "u11",
                 conv=dict(N=32, H=56, W=56, C=64, K=128, R=3, S=3, stride=(2, 2), pad=(1, 1),
                           groups=1),
                 pool=-1, modes=("dp_sk", "auto"), reductions=("linear", "tree")),
    ]
}
