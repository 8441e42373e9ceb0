"""The GEMM entry point that allocates nothing (sk_gemm_rcr_static_ws), for callers that cannot
allocate device memory during the call (their GPU memory belongs to another allocator, or they
cannot take the synchronisation an allocation may bring). Each case calls it twice in a row: both
outputs must match the regular entry point's (the second call finds the first call's leftovers in
the shared scratch), bit for bit under linear/tree. Around those calls the high-water mark of the
device's default memory pool, which the library's own workspace allocation (cudaMallocAsync)
draws from, must not move; a positive control shows the same mark moving when the regular entry
point is left to allocate its workspace. A problem whose workspace does not fit the fixed scratch
is refused with -2.

Collected last on purpose (file name), so that a run stopping at the first failure has already
run every other test; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import numerics
from workloads import gemm_operands

pytestmark = pytest.mark.gpu

import implicit_gemm_conv_gb300 as sk  # noqa: E402  (no skip: a missing library must fail)
from gpu_helpers import DEV, poisoned  # noqa: E402

LIB = sk.library()
STATIC_BYTES = 16 << 20

# CUDA driver: the device's default memory pool and its "used memory" high-water mark.
_CU_MEMPOOL_ATTR_USED_MEM_HIGH = 8


def _driver():
    cuda = ctypes.CDLL("libcuda.so.1")   # loaded here: collection on a machine without a GPU
    torch.cuda.init()
    assert cuda.cuInit(0) == 0
    cuda.cuDeviceGetDefaultMemPool.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
    cuda.cuMemPoolSetAttribute.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    cuda.cuMemPoolGetAttribute.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    return cuda


def _default_pool(cuda):
    pool = ctypes.c_void_p()
    assert cuda.cuDeviceGetDefaultMemPool(ctypes.byref(pool), DEV.index or 0) == 0
    return pool


def _reset_high(cuda, pool):
    torch.cuda.synchronize()
    zero = ctypes.c_uint64(0)
    assert cuda.cuMemPoolSetAttribute(pool, _CU_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(zero)) == 0


def _read_high(cuda, pool) -> int:
    torch.cuda.synchronize()
    v = ctypes.c_uint64(0)
    assert cuda.cuMemPoolGetAttribute(pool, _CU_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(v)) == 0
    return v.value


def _abi_static(A, B, C, mode, red, ctas):
    """Call the C ABI directly (ctypes), on torch's current stream."""
    M, K = A.shape
    N = B.shape[0]
    code = {torch.float16: sk.F16, torch.bfloat16: sk.BF16, torch.float32: sk.F32}
    return LIB.sk_gemm_rcr_static_ws(code[A.dtype], code[C.dtype], M, N, K, A.data_ptr(),
                                     A.stride(0), B.data_ptr(), B.stride(0), C.data_ptr(),
                                     C.stride(0), sk.MODES[mode], sk.REDUCTIONS[red], ctas,
                                     torch.cuda.current_stream().cuda_stream)


CASES = [  # (tile, dtype, out, M, N, K, mode, reduction, pool)
    ("128", "f16", "f16", 256, 256, 4096, "persistent", "linear", 3),
    ("128", "bf16", "f32", 200, 136, 520, "dp_sk", "workspace", 5),
    ("128", "bf16", "bf16", 512, 512, 8192, "dp_sk", "tree", 148),
    # 256x256 CTA-pair tiles: 40 pairs x 256 KiB partial slots fit the fixed scratch
    ("256x256_pair", "bf16", "bf16", 768, 512, 8192, "dp_sk", "linear", 40),
]
TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def test_static_scratch_matches_regular_entry_point_twice_in_a_row():
    cuda = _driver()
    pool = _default_pool(cuda)
    for i, (tile, ab, out, M, N, K, mode, red, ctas) in enumerate(CASES):
        A, B = gemm_operands(M, N, K, ab, "u11", seed_offset=40 + i)
        Ad, Bd = A.to(DEV), B.to(DEV)
        ref = poisoned((M, N), TD[out])
        got = [poisoned((M, N), TD[out]) for _ in range(2)]
        with sk.tile(tile):   # every call plans with the same tile
            # positive control: the regular entry point, left to allocate its own workspace,
            # moves the pool's high-water mark
            _reset_high(cuda, pool)
            sk.sk_gemm_rcr(Ad, Bd, ref, streamk=mode, reduction=red, ctas=ctas)
            assert _read_high(cuda, pool) > 0, f"case {i}: the allocation probe did not see the workspace"
            _reset_high(cuda, pool)
            for g in got:
                rc = _abi_static(Ad, Bd, g, mode, red, ctas)
                assert rc == 0, sk.last_error()
            assert _read_high(cuda, pool) == 0, f"case {i}: the fixed-scratch entry point allocated"
        sk.sk_device_status()
        r = ref.double().cpu().numpy()
        tol = numerics.tolerance(r, K)
        for j, g in enumerate(got):
            gv = g.double().cpu().numpy()
            assert np.isfinite(gv).all(), f"case {i} call {j}: unwritten outputs"
            err = float(np.max(np.abs(gv - r)))
            assert err <= tol, f"case {i} call {j}: max|err| {err:.3e} > {tol:.3e}"
            if red in ("linear", "tree"):   # same plan, deterministic fixup: identical bits
                assert torch.equal(ref.view(torch.uint8), g.view(torch.uint8)), f"case {i} call {j}"


def test_static_scratch_refuses_oversized_plans():
    M, N, K = 512, 512, 65536
    A = torch.zeros((M, K), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((N, K), dtype=torch.bfloat16, device=DEV)
    C = torch.zeros((M, N), dtype=torch.bfloat16, device=DEV)
    with sk.tile("128"):
        # 300 stream-K CTAs x 64 KiB partial slots = 19.7 MB > 16 MiB
        rc = _abi_static(A, B, C, "dp_sk", "linear", 300)
        assert rc == -2
        assert "fixed scratch holds" in sk.last_error()
        # in off mode the plan needs only the 512-byte flag/control header, which fits
        rc = _abi_static(A, B, C, "off", "linear", 300)
        assert rc == 0, sk.last_error()
    torch.cuda.synchronize()
