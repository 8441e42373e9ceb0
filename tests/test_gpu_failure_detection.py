"""Failure detection on the GPU without a fault: a bounded hand-off wait that nothing satisfies
runs out, the kernel records the timeout, the host reads it through sk_device_status, and the
context stays usable for the next launch."""
import time

import pytest
import torch

from oracle import numerics
from workloads import gemm_operands

pytestmark = pytest.mark.gpu

import implicit_gemm_conv_gb300 as sk  # noqa: E402  (no skip: a missing library must fail)
from gpu_helpers import DEV, bits, check_parity, poisoned  # noqa: E402


def test_flag_timeout_is_reported_and_the_context_survives():
    sk.sk_device_status()                    # nothing pending
    t0 = time.monotonic()
    sk.sk_probe_flag_timeout(20)
    with pytest.raises(sk.SkError) as e:
        sk.sk_device_status()                # synchronises, reads and clears the record
    assert e.value.code == -1 and "timed out" in str(e.value)
    assert time.monotonic() - t0 < 10.0      # bounded: the wait gave up
    sk.sk_device_status()                    # cleared
    # the context still computes: a stream-K GEMM with hand-offs matches the oracle
    A, B = gemm_operands(300, 392, 520, "bf16", "n01", seed_offset=41)
    ref = numerics.gemm_rcr_rows("bf16", bits(A), bits(B))
    C = poisoned((300, 392), torch.bfloat16)
    with sk.tile("128"):
        sk.sk_gemm_rcr(A.to(DEV), B.to(DEV), C, streamk="dp_sk", reduction="linear", ctas=5)
    sk.sk_device_status()
    check_parity(C, ref, "bf16", 520, what="GEMM after a reported timeout")


def test_first_error_wins_and_is_read_once():
    sk.sk_probe_flag_timeout(5)
    sk.sk_probe_flag_timeout(5)
    with pytest.raises(sk.SkError):
        sk.sk_device_status()
    sk.sk_device_status()                    # one record, read once
