"""The C ABI library: it loads without a GPU, exports every call include/skgemm.h declares, and its
argument gates return -2 (with a reason) before touching any device."""
import ctypes
import os
import re

import pytest

import implicit_gemm_conv_gb300 as sk

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "skgemm.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:int|const char\*)\s+(sk_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 10
    lib = sk.library()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(sk.EXPORTS)


def test_version_and_error_string():
    assert sk.sk_version() >= 100
    assert isinstance(sk.last_error(), str)


FAKE = 0x10000   # 16-byte aligned, never dereferenced: every call below stops at a gate


def _gemm(**kw):
    a = dict(ab=sk.F16, c=sk.F16, M=256, N=256, K=4096, A=FAKE, lda=4096, B=FAKE, ldb=4096,
             C=FAKE, ldc=256, mode=sk.PERSISTENT, red=sk.LINEAR, ctas=3)
    a.update(kw)
    lib = sk.library()
    rc = lib.sk_gemm_rcr(a["ab"], a["c"], a["M"], a["N"], a["K"], a["A"], a["lda"], a["B"],
                         a["ldb"], a["C"], a["ldc"], a["mode"], a["red"], a["ctas"], None, 0, None)
    return rc, sk.last_error()


@pytest.mark.parametrize("kw,reason", [
    (dict(red=sk.ATOMIC), "atomic"),                         # atomic needs an fp32 output
    (dict(ctas=0), "streamk_ctas"),
    (dict(ctas=-2), "streamk_ctas"),
    (dict(mode=7), "mode"),
    (dict(red=9), "reduction"),
    (dict(ab=sk.F32), "f16 or bf16"),
    (dict(c=sk.BF16), "output"),
    (dict(K=4100, lda=4100, ldb=4100), "multiple of 8"),
    (dict(lda=4099), "16 bytes"),
    (dict(ldc=100), "leading dimension"),
    (dict(A=FAKE + 2), "aligned"),
    (dict(C=0), "NULL"),
    (dict(M=-1), "negative"),
])
def test_gemm_rejections(kw, reason):
    rc, msg = _gemm(**kw)
    assert rc == -2
    assert reason in msg, msg


def test_empty_problem_is_a_noop():
    rc, _ = _gemm(M=0)
    assert rc == 0
    rc, _ = _gemm(N=0, C=0)
    assert rc == 0


def test_valid_call_without_a_gpu_is_refused_not_computed():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, msg = _gemm()
    assert rc == -2 and msg   # no device: nothing computed on the CPU


def _wgrad(**kw):
    a = dict(i=sk.F16, o=sk.F32, N=32, H=56, W=56, C=64, K=64, R=3, S=3, sh=1, sw=1, ph=1, pw=1,
             g=1, mode=sk.DP_SK, red=sk.LINEAR, ctas=-1)
    a.update(kw)
    lib = sk.library()
    rc = lib.sk_conv2d_wgrad_nhwc(a["i"], a["o"], a["N"], a["H"], a["W"], a["C"], a["K"], a["R"],
                                  a["S"], a["sh"], a["sw"], a["ph"], a["pw"], a["g"], FAKE, FAKE,
                                  FAKE, a["mode"], a["red"], a["ctas"], None, 0, None)
    return rc, sk.last_error()


@pytest.mark.parametrize("kw,reason", [
    (dict(g=3), "groups"),
    (dict(C=96, K=96), "multiple of 64"),
    (dict(K=60), "multiple of 8"),
    (dict(ph=3), "padding"),
    (dict(sh=0), "stride"),
    (dict(R=17, S=3), "16"),
    (dict(o=sk.F16, red=sk.ATOMIC), "atomic"),
    (dict(o=sk.BF16), "dW"),
    (dict(H=1, W=1, ph=0, pw=0), "larger than"),
])
def test_wgrad_rejections(kw, reason):
    rc, msg = _wgrad(**kw)
    assert rc == -2
    assert reason in msg, msg


def _conv(fn, **kw):
    a = dict(i=sk.BF16, o=sk.BF16, N=8, H=28, W=28, C=128, K=128, R=3, S=3, sh=1, sw=1, ph=1, pw=1,
             g=1, mode=sk.DP_SK, red=sk.LINEAR, ctas=-1)
    a.update(kw)
    rc = getattr(sk.library(), fn)(a["i"], a["o"], a["N"], a["H"], a["W"], a["C"], a["K"], a["R"],
                                   a["S"], a["sh"], a["sw"], a["ph"], a["pw"], a["g"], FAKE, FAKE,
                                   FAKE, a["mode"], a["red"], a["ctas"], None, 0, None)
    return rc, sk.last_error()


@pytest.mark.parametrize("fn", ["sk_conv2d_fprop_nhwc", "sk_conv2d_dgrad_nhwc"])
@pytest.mark.parametrize("kw,reason", [
    (dict(g=3), "groups"),
    (dict(C=96, K=96), "multiple of 64"),
    (dict(ph=3), "padding"),
    (dict(sh=0), "stride"),
    (dict(R=17, S=3), "16"),
    (dict(red=sk.ATOMIC), "atomic"),
    (dict(i=sk.F16, o=sk.BF16), "output"),
    (dict(H=1, W=1, ph=0, pw=0), "larger than"),
])
def test_conv_rejections(fn, kw, reason):
    rc, msg = _conv(fn, **kw)
    assert rc == -2
    assert reason in msg, msg


def _phase_1d(X, R, sigma, pad, a):
    """One dimension of an output phase of a strided data gradient, from its definition: the taps
    r with (a + pad - r) divisible by sigma, and the pixels a, a + sigma, ... below X."""
    taps = [r for r in range(R) if (a + pad - r) % sigma == 0]
    return len(range(a, X, sigma)), len(taps)


def test_strided_dgrad_gates_and_workspace():
    rc, msg = _conv("sk_conv2d_dgrad_nhwc", sh=2, sw=2)
    assert rc == -2 and "stride" not in msg          # past every argument gate (no device here)
    rc, msg = _conv("sk_conv2d_dgrad_nhwc", sh=9, sw=1)
    assert rc == -2 and "stride" in msg
    # the workspace holds every phase's plan side by side (each rounded up to 256 bytes), each plan
    # recomputed by the oracle partitioner
    N, H, W, C, K, R, S, sh, sw, ph, pw = 4, 17, 13, 64, 128, 3, 2, 2, 3, 1, 1
    prob = sk.make_problem("dgrad", ab_dtype="bf16", c_dtype="bf16", n=N, h=H, w=W, c=C, k=K,
                           r=R, s=S, stride_h=sh, stride_w=sw, pad_h=ph, pad_w=pw, groups=1)
    with pytest.raises(sk.SkError, match="one plan per output phase"):
        sk.sk_plan(prob, "dp_sk", "linear", 7, 148)
    from oracle import partition as P
    for mode, red, pm, pr in [("dp_sk", "linear", P.DP_SK, P.LINEAR),
                              ("splitk", "workspace", P.SPLITK, P.WORKSPACE)]:
        total = 0
        for a in range(sh):
            for b in range(sw):
                hp, rt = _phase_1d(H, R, sh, ph, a)
                wp, st = _phase_1d(W, S, sw, pw, b)
                if not (hp and wp and rt and st):
                    continue
                plan = P.make_plan(tiles_m=-(-N * hp * wp // 128), tiles_n=1, groups=1,
                                   kred=rt * st * K, tm=128, tn=128, tk=64, pool=7, mode=pm,
                                   reduction=pr)
                total += -(-plan.ws_bytes // 256) * 256
        assert sk.sk_workspace_bytes(prob, mode, red, 7) == total
    with sk.tile("256x256_pair"):
        rc, msg = _conv("sk_conv2d_fprop_nhwc", N=0)   # checked before any device work
    assert rc in (0, -2)
    prob = sk.make_problem("fprop", ab_dtype="bf16", c_dtype="bf16", n=8, h=28, w=28, c=128,
                           k=128, r=3, s=3, stride_h=1, stride_w=1, pad_h=1, pad_w=1, groups=1)
    with sk.tile("256x256_pair"):
        with pytest.raises(sk.SkError, match="GEMMs and the shifted-row wgrad only"):
            sk.sk_plan(prob, "dp_sk", "linear", 148, 148)
    plan = sk.sk_plan(prob, "dp_sk", "linear", 148, 148)   # auto: the 128x128 tile
    assert (plan.tm, plan.gemm_m, plan.gemm_n, plan.kred) == (128, 8 * 28 * 28, 128, 9 * 128)


def test_fp8_rejections():
    lib = sk.library()
    rc = lib.sk_gemm_rowcol_fp8(64, 64, 100, FAKE, FAKE, FAKE, FAKE, FAKE, 64, sk.DP_SK, sk.ATOMIC,
                                -1, None, 0, None)
    assert rc == -2 and "atomic" in sk.last_error()
    rc = lib.sk_gemm_rowcol_fp8(64, 64, 100, FAKE, FAKE, FAKE, FAKE, FAKE, 64, sk.DP_SK, sk.LINEAR,
                                -1, None, 0, None)
    assert rc == -2 and "multiple of 16" in sk.last_error()


@pytest.mark.parametrize("kw,reason", [
    (dict(gka=64), "a_group_k"),
    (dict(gka=200), "a_group_k"),
    (dict(gkb=0), "b_group_k"),
    (dict(gnb=64), "b_group_n"),
    (dict(gnb=192), "b_group_n"),
    (dict(red=sk.ATOMIC), "atomic"),
    (dict(K=100), "multiple of 16"),
    (dict(ldc=32), "ldc"),
])
def test_blockscale_rejections(kw, reason):
    a = dict(M=256, N=256, K=1024, sa=FAKE, gka=128, sb=FAKE, gnb=128, gkb=256, ldc=256,
             red=sk.LINEAR)
    a.update(kw)
    lib = sk.library()
    rc = lib.sk_gemm_blockscale_fp8(a["M"], a["N"], a["K"], FAKE, FAKE, a["sa"], a["gka"], a["sb"],
                                    a["gnb"], a["gkb"], FAKE, a["ldc"], sk.DP_SK, a["red"], -1, None,
                                    0, None)
    assert rc == -2 and reason in sk.last_error(), (rc, sk.last_error())


def test_blockscale_group_sizes_of_a_missing_scale_are_ignored():
    # sb == NULL: b_group_n / b_group_k are not checked; the call then stops at the device gate
    lib = sk.library()
    rc = lib.sk_gemm_blockscale_fp8(256, 256, 1024, FAKE, FAKE, FAKE, 128, None, 0, 0, FAKE, 256,
                                    sk.DP_SK, sk.LINEAR, -1, None, 0, None)
    assert rc == -2 and "group" not in sk.last_error()


def test_flag_timeout_probe_gates():
    lib = sk.library()
    for bad in (0, -5, 1001):
        assert lib.sk_probe_flag_timeout(bad, None) == -2 and "timeout_ms" in sk.last_error()


def test_default_pool():
    assert sk.sk_default_pool("linear", 148, 1) == 148
    assert sk.sk_default_pool("tree", 148, 2) == 148
    assert sk.sk_default_pool("workspace", 148, 1) == 148
    assert sk.sk_default_pool("atomic", 148, 2) == 296
    assert sk.sk_default_pool("atomic", 304, 8) == 1216
    with pytest.raises(sk.SkError):
        sk.sk_default_pool("linear", 0, 1)
