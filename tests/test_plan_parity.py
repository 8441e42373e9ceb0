"""The CUDA path's host planner (sk_plan / sk_plan_cta_work in libskgemm) against the oracle's
partition replica: every scalar field and every CTA's segment list must match bit for bit."""
import itertools
import random

import pytest

import implicit_gemm_conv_gb300 as sk
from oracle import partition as P


@pytest.fixture(autouse=True)
def tile_128():
    """The configurations these tests follow fix 128 x 128 tiles; the pair tiles have their own
    tests."""
    with sk.tile("128"):
        yield

MODES = [("off", P.OFF), ("dp_sk", P.DP_SK), ("persistent", P.PERSISTENT), ("splitk", P.SPLITK),
         ("hybrid", P.HYBRID)]
REDS = [("linear", P.LINEAR), ("tree", P.TREE), ("atomic", P.ATOMIC), ("workspace", P.WORKSPACE)]

FIELD_MAP = {  # C name -> oracle name
    "tiles": "T", "iters_per_tile": "I", "pool": "P", "sk_tiles": "sk_tiles",
    "dp_tiles": "dp_tiles", "sk_ctas": "sk_ctas", "sk_iters": "sk_iters",
    "iters_per_sk_cta": "iters_per_sk_cta", "extra_iters": "extra", "grid": "grid",
    "publishers": "publishers", "max_contributors": "max_contrib", "tree_rounds": "rounds",
    "shared_tiles": "shared_tiles", "flag_bytes": "flag_bytes", "partial_bytes": "partial_bytes",
    "partial_slots": "slots",
    "scratch_bytes": "scratch_bytes", "ws_bytes": "ws_bytes", "tiles_m": "tiles_m",
    "tiles_n": "tiles_n", "groups": "groups",
}


def compare(prob, oracle_kw, mode, red, ctas, num_sms=148, check_ctas=None, cluster=1):
    oracle_kw = dict(oracle_kw)
    cluster = oracle_kw.pop("cluster", cluster)
    cp = sk.sk_plan(prob, mode[0], red[0], ctas, num_sms)
    # a pair kernel's default pool is resolved over SM pairs
    pool = ctas if ctas > 0 else P.default_pool(red[1], num_sms // cluster, 1)
    op = P.make_plan(pool=pool, mode=mode[1], reduction=red[1], cluster=cluster, **oracle_kw)
    for c, o in FIELD_MAP.items():
        assert getattr(cp, c) == getattr(op, o), (c, getattr(cp, c), getattr(op, o))
    if mode[1] == P.SPLITK:
        assert cp.splits == op.splits
    ctas_to_check = range(cp.grid) if check_ctas is None else check_ctas(cp.grid)
    for c in ctas_to_check:
        got = [(s.tile, s.k_begin, s.k_end, s.kind, s.index, s.n_contrib, s.first_cta)
               for s in sk.sk_plan_cta_work(cp, c)]
        exp = [(s.tile, s.k_begin, s.k_end, s.kind, s.index, s.n_contrib, s.first_cta)
               for s in P.cta_segments(op, c)]
        assert got == exp, (c, got, exp)
    return cp


def gemm(M, N, K, ab="f16", tm=128, tn=128):
    tk = 128 if ab == "e4m3" else 64
    prob = sk.make_problem("fp8" if ab == "e4m3" else "gemm", ab_dtype=ab,
                           c_dtype="bf16" if ab == "e4m3" else ab, M=M, N=N, K=K)
    kw = dict(tiles_m=-(-M // tm), tiles_n=-(-N // tn), groups=1, kred=K, tm=tm, tn=tn, tk=tk)
    return prob, kw


def wgrad(N, H, W, C, K, R, S, stride, pad, groups):
    prob = sk.make_problem("wgrad", ab_dtype="bf16", c_dtype="f32", n=N, h=H, w=W, c=C, k=K, r=R,
                           s=S, stride_h=stride, stride_w=stride, pad_h=pad, pad_w=pad,
                           groups=groups)
    Ho = (H + 2 * pad - R) // stride + 1
    Wo = (W + 2 * pad - S) // stride + 1
    Kg, Cg = K // groups, C // groups
    kw = dict(tiles_m=-(-Kg // 128), tiles_n=-(-(R * S * Cg) // 128), groups=groups,
              kred=N * Ho * Wo, tm=128, tn=128, tk=64)
    return prob, kw


def conv(op, N, H, W, C, K, R, S, stride, pad, groups):
    prob = sk.make_problem(op, ab_dtype="bf16", c_dtype="bf16", n=N, h=H, w=W, c=C, k=K, r=R, s=S,
                           stride_h=stride, stride_w=stride, pad_h=pad, pad_w=pad, groups=groups)
    Ho = (H + 2 * pad - R) // stride + 1
    Wo = (W + 2 * pad - S) // stride + 1
    Kg, Cg = K // groups, C // groups
    if op == "fprop":   # output pixels x filters per group, reduction (r, s, c)
        m, n, kred = N * Ho * Wo, Kg, R * S * Cg
    else:               # input pixels x channels per group, reduction (r, s, k)
        m, n, kred = N * H * W, Cg, R * S * Kg
    kw = dict(tiles_m=-(-m // 128), tiles_n=-(-n // 128), groups=groups, kred=kred, tm=128, tn=128,
              tk=64)
    return prob, kw


NAMED = [
    ("gemm 256x256x4096", gemm(256, 256, 4096), 3),
    ("gemm 3840x4096x4096", gemm(3840, 4096, 4096, "bf16"), 148),
    ("wgrad 32x56x56x64", wgrad(32, 56, 56, 64, 64, 3, 3, 1, 1, 1), -1),
    ("wgrad 64x28x28x256 g4 s2", wgrad(64, 28, 28, 256, 256, 3, 3, 2, 1, 4), -1),
    ("fp8 8192^3", gemm(8192, 8192, 8192, "e4m3"), -1),
    ("gemm 512x512x65536", gemm(512, 512, 65536, "bf16"), 148),
    ("fprop 32x56x56x64 3x3", conv("fprop", 32, 56, 56, 64, 64, 3, 3, 1, 1, 1), -1),
    ("fprop 8x28x28x256 g2 s2", conv("fprop", 8, 28, 28, 256, 256, 3, 3, 2, 1, 2), 148),
    ("dgrad 32x56x56x64 3x3", conv("dgrad", 32, 56, 56, 64, 64, 3, 3, 1, 1, 1), -1),
    ("dgrad 4x14x14x128 g2", conv("dgrad", 4, 14, 14, 128, 256, 3, 3, 1, 1, 2), 148),
]


@pytest.mark.parametrize("name,pk,ctas", NAMED, ids=[n[0] for n in NAMED])
@pytest.mark.parametrize("mode", MODES, ids=[m[0] for m in MODES])
@pytest.mark.parametrize("red", REDS, ids=[r[0] for r in REDS])
def test_named_workloads(name, pk, ctas, mode, red):
    prob, kw = pk
    big = lambda g: sorted(set(list(range(min(g, 200))) + list(range(max(0, g - 50), g))))
    compare(prob, kw, mode, red, ctas, check_ctas=big)


def test_worked_vector_values_through_c():
    cp = sk.sk_plan(*gemm(3840, 4096, 4096, "bf16")[:1], "dp_sk", "linear", 148, 148)
    assert (cp.tiles, cp.dp_tiles, cp.sk_tiles, cp.sk_iters, cp.iters_per_sk_cta,
            cp.extra_iters, cp.grid) == (960, 888, 72, 4608, 31, 20, 1036)
    cp = sk.sk_plan(wgrad(64, 28, 28, 256, 256, 3, 3, 2, 1, 4)[0], "dp_sk", "workspace", -1, 148)
    assert (cp.tiles, cp.iters_per_tile, cp.sk_ctas, cp.iters_per_sk_cta, cp.extra_iters) == \
        (20, 196, 148, 26, 72)


def test_random_sweep():
    rng = random.Random(11)
    for _ in range(300):
        M, N = rng.randint(1, 1200), rng.randint(1, 1200)
        K = 8 * rng.randint(1, 400)
        mode = rng.choice(MODES)
        red = rng.choice(REDS)
        ctas = rng.choice([-1, 1, 2, 3, 5, 7, 31, 148, 300])
        prob, kw = gemm(M, N, K)
        compare(prob, kw, mode, red, ctas, num_sms=rng.choice([148, 152, 8]))


def test_grouped_wgrad_sweep():
    for N, H, C, K, R, s, p, g in itertools.product([1, 3], [5, 9], [64, 256], [64, 128],
                                                    [1, 3], [1, 2], [0, 1], [1, 2]):
        if C % g or K % g or (C // g) % 64 or p >= R:
            continue
        prob, kw = wgrad(N, H, H + 2, C, K, R, R, s, p, g)
        for mode in MODES:
            compare(prob, kw, mode, REDS[1], 7)


def test_auto_mode_matches_oracle():
    rng = random.Random(17)
    cases = [gemm(512, 512, 65536, "bf16"), gemm(3840, 4096, 4096, "bf16"), gemm(256, 256, 4096),
             gemm(128, 128, 64 * 1216), gemm(128, 128, 64 * 1215)]
    cases += [gemm(rng.randint(1, 900), rng.randint(1, 900), 8 * rng.randint(1, 4000))
              for _ in range(200)]
    for prob, kw in cases:
        for red, ored in [("linear", P.LINEAR), ("auto", P.REDUCTION_AUTO)]:
            for ctas in (-1, 148, 1216):
                cp = sk.sk_plan(prob, "auto", red, ctas, 152)
                pool = ctas if ctas > 0 else P.default_pool(
                    P.WORKSPACE if ored == P.REDUCTION_AUTO else ored, 152, 1)
                op = P.make_auto_plan(pool=pool, reduction=ored, **kw)
                assert cp.mode == op.mode and cp.reduction == op.reduction
                for c, o in FIELD_MAP.items():
                    assert getattr(cp, c) == getattr(op, o), (c, kw, ctas)


def test_plan_rejections():
    prob, _ = gemm(256, 256, 4096)
    for ctas in (0, -5):
        with pytest.raises(sk.SkError, match="streamk_ctas"):
            sk.sk_plan(prob, "dp_sk", "linear", ctas, 148)
    with pytest.raises(sk.SkError, match="mode"):
        sk.sk_plan(prob, 9, "linear", 3, 148)
    empty, _ = gemm(0, 256, 4096)
    with pytest.raises(sk.SkError, match="empty"):
        sk.sk_plan(empty, "dp_sk", "linear", 3, 148)


# ---- CTA-pair tiles: the same partition over pair tiles, pool in pairs, a flag per CTA

PAIR_TILES = [("256_pair", 128), ("256x256_pair", 256)]
PAIR_NAMED = [
    ("gemm 3840x4096x4096", (3840, 4096, 4096, "bf16"), 148),
    ("gemm 3840x4096x4096 pool 74", (3840, 4096, 4096, "bf16"), 74),
    ("gemm 512x512x65536", (512, 512, 65536, "bf16"), 148),
    ("fp8 8192^3", (8192, 8192, 8192, "e4m3"), -1),
    ("gemm 300x392x520", (300, 392, 520, "bf16"), 5),
]


@pytest.mark.parametrize("tile,tn", PAIR_TILES, ids=[t[0] for t in PAIR_TILES])
@pytest.mark.parametrize("name,shape,ctas", PAIR_NAMED, ids=[n[0] for n in PAIR_NAMED])
@pytest.mark.parametrize("mode", MODES, ids=[m[0] for m in MODES])
@pytest.mark.parametrize("red", REDS, ids=[r[0] for r in REDS])
def test_pair_tile_plans(tile, tn, name, shape, ctas, mode, red):
    prob, kw = gemm(*shape, tm=256, tn=tn)
    big = lambda g: sorted(set(list(range(min(g, 200))) + list(range(max(0, g - 50), g))))
    with sk.tile(tile):
        cp = compare(prob, kw, mode, red, ctas, num_sms=152, check_ctas=big, cluster=2)
    assert (cp.tm, cp.tn) == (256, tn)
    assert cp.flag_bytes >= 8 * cp.publishers


@pytest.mark.parametrize("tile,tn", PAIR_TILES, ids=[t[0] for t in PAIR_TILES])
def test_pair_tile_random_sweep(tile, tn):
    rng = random.Random(23)
    with sk.tile(tile):
        for _ in range(200):
            M, N = rng.randint(1, 1500), rng.randint(1, 1200)
            K = 8 * rng.randint(1, 400)
            prob, kw = gemm(M, N, K, tm=256, tn=tn)
            compare(prob, kw, rng.choice(MODES), rng.choice(REDS),
                    rng.choice([-1, 1, 2, 3, 5, 74, 148]), num_sms=rng.choice([148, 152, 8]),
                    cluster=2)


def test_pair_tile_setting():
    prob, _ = gemm(3840, 4096, 4096, "bf16")
    with sk.tile("auto"):   # 240 pair tiles: the pair; few pair tiles or 128 rows: one CTA per tile
        assert (sk.sk_plan(prob, "dp_sk", "linear", 74, 148).tm,
                sk.sk_plan(prob, "dp_sk", "linear", 74, 148).tn) == (256, 256)
        # 4 pair tiles over 1024 K steps: the deep-ring pair (one CTA per SM, 7 stages)
        assert sk.sk_plan(gemm(512, 512, 65536, "bf16")[0], "dp_sk", "linear", 74, 148).tm == 256
        assert sk.sk_plan(gemm(512, 512, 4096, "bf16")[0], "dp_sk", "linear", 148, 148).tm == 128
        assert sk.sk_plan(gemm(128, 8192, 4096, "bf16")[0], "dp_sk", "linear", 148, 148).tm == 128
        assert sk.sk_plan(gemm(2048, 2048, 4096, "bf16")[0], "dp_sk", "linear", 74, 148).tm == 256
        assert sk.sk_plan(gemm(2048, 1792, 4096, "bf16")[0], "dp_sk", "linear", 74, 148).tm == 128
    with sk.tile("128"):
        assert sk.sk_plan(prob, "dp_sk", "linear", 148, 148).tm == 128
    with sk.tile("256_pair"):
        assert (sk.sk_plan(prob, "dp_sk", "linear", 148, 148).tm,
                sk.sk_plan(prob, "dp_sk", "linear", 148, 148).tn) == (256, 128)
        # a shifted-row wgrad shape: its 256 x 192 pair tile; another wgrad shape: refused
        w, _ = wgrad(32, 56, 56, 64, 64, 3, 3, 1, 1, 1)
        assert (sk.sk_plan(w, "dp_sk", "linear", -1, 148).tm,
                sk.sk_plan(w, "dp_sk", "linear", -1, 148).tn) == (256, 192)
        w2, _ = wgrad(2, 9, 9, 128, 192, 1, 1, 1, 0, 1)
        with pytest.raises(sk.SkError, match="GEMMs and the shifted-row wgrad only"):
            sk.sk_plan(w2, "dp_sk", "linear", -1, 148)
    with sk.tile("256x256_pair"):
        assert sk.sk_plan(prob, "dp_sk", "linear", 148, 148).tn == 256
    with pytest.raises(sk.SkError, match="tile setting"):
        sk.sk_set_tile(7)


# ---- the block-scaled fp8 GEMM: 128 x 128 tiles, a 128-wide reduction step

BLOCK_NAMED = [
    ("fp8 block 4096x4096x4096", (4096, 4096, 4096), -1),
    ("fp8 block 300x392x1040", (300, 392, 1040), 5),
    ("fp8 block 512x512x32768", (512, 512, 32768), 148),
]


def block_gemm(M, N, K, tm=128):
    prob = sk.make_problem("fp8_block", ab_dtype="e4m3", c_dtype="bf16", M=M, N=N, K=K)
    kw = dict(tiles_m=-(-M // tm), tiles_n=-(-N // 128), groups=1, kred=K, tm=tm, tn=128, tk=128)
    return prob, kw


@pytest.mark.parametrize("tile,tm", [("128", 128), ("256_pair", 256)])
@pytest.mark.parametrize("name,shape,ctas", BLOCK_NAMED, ids=[n[0] for n in BLOCK_NAMED])
@pytest.mark.parametrize("mode", MODES, ids=[m[0] for m in MODES])
@pytest.mark.parametrize("red", REDS, ids=[r[0] for r in REDS])
def test_block_scale_plans(tile, tm, name, shape, ctas, mode, red):
    prob, kw = block_gemm(*shape, tm=tm)
    big = lambda g: sorted(set(list(range(min(g, 200))) + list(range(max(0, g - 50), g))))
    with sk.tile(tile):
        cp = compare(prob, kw, mode, red, ctas, num_sms=152, check_ctas=big, cluster=tm // 128)
    assert (cp.tm, cp.tn, cp.iters_per_tile) == (tm, 128, -(-shape[2] // 128))


def test_block_scale_tile_setting():
    prob, _ = block_gemm(4096, 4096, 4096)
    small, _ = block_gemm(128, 4096, 4096)
    with sk.tile("auto"):   # the one-CTA tile (the pair only on request)
        assert (sk.sk_plan(prob, "dp_sk", "linear", 148, 148).tm,
                sk.sk_plan(prob, "dp_sk", "linear", 148, 148).tn) == (128, 128)
        assert sk.sk_plan(small, "dp_sk", "linear", 148, 148).tm == 128
    with sk.tile("128"):
        assert sk.sk_plan(prob, "dp_sk", "linear", 148, 148).tm == 128
    with sk.tile("256_pair"):
        assert sk.sk_plan(prob, "dp_sk", "linear", 74, 148).tm == 256
    with sk.tile("256x256_pair"):
        with pytest.raises(sk.SkError, match="no 256 x 256 tile"):
            sk.sk_plan(prob, "dp_sk", "linear", 148, 148)


# ---- shifted-row wgrad (automatic tile, 64-channel and 64-filter groups): GEMM view
# M = (tap row, channel) in 128-row tiles of two tap rows (on request, 256-row tiles of four on a
# CTA pair), N = (column tap, filter) in one 192-wide tile, reduction over the padded positions: 64
# per K step, `64 / wseg` output rows of `wseg` positions (the power of two >= Wo + shifts), rows
# counted per image over Ho rounded up.

def wgrad_row(N, H, W, C, K, R, S, stride, pad, groups, dt="bf16", pair=False):
    sh, sw = stride
    ph, pw = pad
    prob = sk.make_problem("wgrad", ab_dtype=dt, c_dtype="f32", n=N, h=H, w=W, c=C, k=K, r=R,
                           s=S, stride_h=sh, stride_w=sw, pad_h=ph, pad_w=pw, groups=groups)
    Ho = (H + 2 * ph - R) // sh + 1
    Wo = (W + 2 * pw - S) // sw + 1
    shifts = -(-S // sw) - 1
    wseg = 1
    while wseg < Wo + shifts:
        wseg *= 2
    rows = 64 // wseg
    if rows == 0:   # rows too wide for one K step: not this view
        return prob, None
    ho_pad = -(-Ho // rows) * rows
    tm = 256 if pair else 128
    kw = dict(tiles_m=-(-(R * 64) // tm), tiles_n=1, groups=groups, kred=N * ho_pad * wseg,
              tm=tm, tn=192, tk=64, cluster=tm // 128)
    return prob, kw


ROW_NAMED = [
    ("wgrad 32x56x56x64", wgrad_row(32, 56, 56, 64, 64, 3, 3, (1, 1), (1, 1), 1), -1),
    ("wgrad 64x28x28x256 g4 s2", wgrad_row(64, 28, 28, 256, 256, 3, 3, (2, 2), (1, 1), 4), -1),
    ("wgrad 2x9x13 r5 s3", wgrad_row(2, 9, 13, 64, 64, 5, 3, (1, 1), (2, 1), 1), 7),
    ("wgrad 2x7x16 sw2", wgrad_row(2, 7, 16, 64, 64, 3, 3, (1, 2), (1, 1), 1), 7),
]


@pytest.mark.parametrize("name,pk,ctas", ROW_NAMED, ids=[n[0] for n in ROW_NAMED])
@pytest.mark.parametrize("mode", MODES, ids=[m[0] for m in MODES])
@pytest.mark.parametrize("red", REDS, ids=[r[0] for r in REDS])
def test_row_wgrad_plans(name, pk, ctas, mode, red):
    prob, kw = pk
    big = lambda g: sorted(set(list(range(min(g, 200))) + list(range(max(0, g - 50), g))))
    with sk.tile("auto"):
        cp = compare(prob, kw, mode, red, ctas, check_ctas=big)
    assert (cp.tm, cp.tn, cp.tk) == (kw["tm"], 192, 64)


ROW_PAIR_NAMED = [
    ("wgrad 32x56x56x64 pair", wgrad_row(32, 56, 56, 64, 64, 3, 3, (1, 1), (1, 1), 1, pair=True), -1),
    ("wgrad 64x28x28x256 g4 s2 pair",
     wgrad_row(64, 28, 28, 256, 256, 3, 3, (2, 2), (1, 1), 4, pair=True), -1),
    ("wgrad 2x9x13 r5 s3 pair", wgrad_row(2, 9, 13, 64, 64, 5, 3, (1, 1), (2, 1), 1, pair=True), 7),
]


@pytest.mark.parametrize("name,pk,ctas", ROW_PAIR_NAMED, ids=[n[0] for n in ROW_PAIR_NAMED])
@pytest.mark.parametrize("mode", MODES, ids=[m[0] for m in MODES])
@pytest.mark.parametrize("red", REDS, ids=[r[0] for r in REDS])
def test_row_wgrad_pair_plans(name, pk, ctas, mode, red):
    prob, kw = pk
    big = lambda g: sorted(set(list(range(min(g, 200))) + list(range(max(0, g - 50), g))))
    with sk.tile("256_pair"):
        cp = compare(prob, kw, mode, red, ctas, num_sms=152, check_ctas=big)
    assert (cp.tm, cp.tn, cp.tk) == (256, 192, 64)


def test_row_wgrad_worked_vectors():
    """32x56x56, 64 -> 64, 3x3: two tiles (tap rows {0,1} and {2}), 32*56 K steps of one
    56-column row each (64 positions); 148 CTAs: 3584 steps, 24 each and one more for the first
    32. Grouped stride 2 (4 groups of 64): 8 tiles, 14 output columns + 1 shift -> 16-position
    rows, 4 rows per step, 14 rows per image padded to 16: 64*16/4 = 256 steps per tile. On the
    CTA pair (on request): one 256 x 192 tile (tap rows 0-2) of 1792 steps on 74 pairs, 24 each
    and one more for the first 16; grouped: 4 tiles, 1024 steps, 13 each and one more for the
    first 62."""
    with sk.tile("auto"):
        cp = sk.sk_plan(ROW_NAMED[0][1][0], "dp_sk", "atomic", 148, 148)
        assert (cp.tm, cp.tiles, cp.iters_per_tile, cp.sk_tiles, cp.sk_iters, cp.iters_per_sk_cta,
                cp.extra_iters, cp.grid) == (128, 2, 1792, 2, 3584, 24, 32, 148)
        cp = sk.sk_plan(ROW_NAMED[1][1][0], "dp_sk", "atomic", 148, 148)
        assert (cp.tiles, cp.iters_per_tile, cp.sk_ctas, cp.iters_per_sk_cta, cp.extra_iters) == \
            (8, 256, 148, 13, 124)
    with sk.tile("256_pair"):
        cp = sk.sk_plan(ROW_NAMED[0][1][0], "dp_sk", "atomic", 74, 148)
        assert (cp.tm, cp.tiles, cp.iters_per_tile, cp.sk_tiles, cp.sk_iters, cp.iters_per_sk_cta,
                cp.extra_iters, cp.grid) == (256, 1, 1792, 1, 1792, 24, 16, 74)
        cp = sk.sk_plan(ROW_NAMED[1][1][0], "dp_sk", "atomic", 74, 148)
        assert (cp.tiles, cp.iters_per_tile, cp.sk_ctas, cp.iters_per_sk_cta, cp.extra_iters) == \
            (4, 256, 74, 13, 62)


def test_row_wgrad_pair_only_for_long_reductions():
    """The automatic tile takes the CTA pair for three tap rows once the reduction is long
    (about 128 K steps per SM): 32x56x56 stays on one CTA, 192x56x56 goes to the pair."""
    with sk.tile("auto"):
        assert sk.sk_plan(ROW_NAMED[0][1][0], "dp_sk", "atomic", -1, 148).tm == 128
        big = wgrad_row(192, 56, 56, 64, 64, 3, 3, (1, 1), (1, 1), 1)[0]
        assert sk.sk_plan(big, "dp_sk", "atomic", -1, 148).tm == 256


def test_row_wgrad_sweep():
    """Random shapes of the shifted-row kernel's domain (and some just outside it, which must keep
    the 128 x 128 view) against the oracle's partition."""
    rng = random.Random(29)
    seen_row = seen_generic = 0
    for _ in range(150):
        R, S = rng.randint(1, 5), rng.randint(1, 3)
        sh, sw = rng.randint(1, 3), rng.randint(1, 2)
        ph, pw = rng.randint(0, R - 1), rng.randint(0, S - 1)
        N, H, W = rng.randint(1, 4), rng.randint(R, 30), rng.randint(S, 80)
        g = rng.randint(1, 3)
        prob, kw = wgrad_row(N, H, W, 64 * g, 64 * g, R, S, (sh, sw), (ph, pw), g)
        with sk.tile("auto"):
            tn = sk.sk_plan(prob, "dp_sk", "atomic", 7, 148).tn
        Wo = (W + 2 * pw - S) // sw + 1
        fits = Wo + (-(-S // sw) - 1) <= 64
        assert (tn == 192) == fits, (R, S, sh, sw, W, Wo)
        if not fits:
            seen_generic += 1
            continue
        seen_row += 1
        with sk.tile("auto"):
            compare(prob, kw, rng.choice(MODES), rng.choice(REDS), rng.choice([-1, 1, 3, 7, 148]),
                    num_sms=rng.choice([148, 152, 8]))
    assert seen_row > 50 and seen_generic > 5



# ---- shifted-row forward convolution (automatic tile; stride 1, 64 channels, 64 filters, <= 3x3):
# M = positions, 64 per output row, rows counted per image over Ho rounded up to even, in 128-row
# tiles (two output rows); N = 64 filters; one K step per tap.

def fprop_row(N, H, W, R, S, pad):
    prob = sk.make_problem("fprop", ab_dtype="f16", c_dtype="f16", n=N, h=H, w=W, c=64, k=64, r=R,
                           s=S, stride_h=1, stride_w=1, pad_h=pad[0], pad_w=pad[1], groups=1)
    ho = H + 2 * pad[0] - R + 1
    ho_pad = ho + ho % 2
    kw = dict(tiles_m=N * ho_pad * 64 // 128, tiles_n=1, groups=1, kred=R * S * 64, tm=128, tn=64,
              tk=64)
    return prob, kw


FPROP_ROW_NAMED = [
    ("fprop 32x56x56 3x3", fprop_row(32, 56, 56, 3, 3, (1, 1)), -1),
    ("fprop 2x9x11 3x3", fprop_row(2, 9, 11, 3, 3, (1, 1)), 5),
    ("fprop 3x7x7 2x2", fprop_row(3, 7, 7, 2, 2, (0, 1)), 7),
]


@pytest.mark.parametrize("name,pk,ctas", FPROP_ROW_NAMED, ids=[n[0] for n in FPROP_ROW_NAMED])
@pytest.mark.parametrize("mode", MODES, ids=[m[0] for m in MODES])
@pytest.mark.parametrize("red", REDS, ids=[r[0] for r in REDS])
def test_fprop_row_plans(name, pk, ctas, mode, red):
    prob, kw = pk
    big = lambda g: sorted(set(list(range(min(g, 200))) + list(range(max(0, g - 50), g))))
    with sk.tile("auto"):
        cp = compare(prob, kw, mode, red, ctas, check_ctas=big)
    assert (cp.tm, cp.tn, cp.tk, cp.iters_per_tile) == (128, 64, 64, kw["kred"] // 64)


def test_fprop_row_worked_vector():
    """32x56x56, 64 -> 64, 3x3: 32 images x 56 rows / 2 = 896 tiles of 9 taps; 148 CTAs: 888
    tiles in six data-parallel waves, 8 left over (72 iterations, fewer than the pool: all
    data-parallel)."""
    with sk.tile("auto"):
        cp = sk.sk_plan(FPROP_ROW_NAMED[0][1][0], "dp_sk", "linear", 148, 148)
    assert (cp.tiles, cp.iters_per_tile, cp.sk_ctas, cp.dp_tiles, cp.grid) == (896, 9, 0, 896, 896)


def test_fprop_row_auto_mode_is_persistent():
    """The automatic mode runs the shifted-row fprop persistently when its tiles outnumber the CTAs
    (every CTA keeps the filter resident over its tiles), all tiles data-parallel (a stream-K wave's
    fixups cost more than one short tile): CTA c runs tiles c, c + pool, ... With fewer tiles than
    CTAs it keeps the pages' rule."""
    prob, kw = FPROP_ROW_NAMED[0][1]
    with sk.tile("auto"):
        for ctas, sms in ((-1, 152), (-1, 148), (300, 152)):
            cp = sk.sk_plan(prob, "auto", "linear", ctas, sms)
            pool = ctas if ctas > 0 else sms
            assert (cp.mode, cp.pool, cp.grid, cp.sk_tiles, cp.sk_ctas, cp.dp_tiles) == (
                P.PERSISTENT, pool, pool, 0, 0, 896)
            assert cp.ws_bytes <= 256 * 1024   # no partials: flags and the control block at most
            seen = []
            for c in range(pool):
                segs = sk.sk_plan_cta_work(cp, c)
                assert [s.tile for s in segs] == list(range(c, 896, pool))
                assert all((s.k_begin, s.k_end) == (0, 9) for s in segs)
                seen += [s.tile for s in segs]
            assert sorted(seen) == list(range(896))
        small, skw = fprop_row(1, 4, 8, 3, 3, (1, 1))   # 2 tiles, fewer than the pool
        cp = sk.sk_plan(small, "auto", "linear", -1, 152)
        op = P.make_auto_plan(pool=P.default_pool(P.LINEAR, 152, 1), reduction=P.LINEAR, **skw)
        assert cp.mode == op.mode != P.PERSISTENT


# ---- shifted-row data gradient (automatic tile; stride 1, 64 filters -> 64 channels, <= 3x3): the
# stride-1 convolution of dy with the flipped filter over the dx grid, in the same view.

def dgrad_row(N, H, W, R, S, pad):
    prob = sk.make_problem("dgrad", ab_dtype="f16", c_dtype="f16", n=N, h=H, w=W, c=64, k=64, r=R,
                           s=S, stride_h=1, stride_w=1, pad_h=pad[0], pad_w=pad[1], groups=1)
    kw = dict(tiles_m=N * (H + H % 2) * 64 // 128, tiles_n=1, groups=1, kred=R * S * 64, tm=128,
              tn=64, tk=64)
    return prob, kw


DGRAD_ROW_NAMED = [
    ("dgrad 32x56x56 3x3", dgrad_row(32, 56, 56, 3, 3, (1, 1)), -1),
    ("dgrad 2x9x11 3x3", dgrad_row(2, 9, 11, 3, 3, (1, 1)), 5),
    ("dgrad 2x8x10 3x3 unpadded", dgrad_row(2, 8, 10, 3, 3, (0, 0)), 7),
]


@pytest.mark.parametrize("name,pk,ctas", DGRAD_ROW_NAMED, ids=[n[0] for n in DGRAD_ROW_NAMED])
@pytest.mark.parametrize("mode", MODES, ids=[m[0] for m in MODES])
@pytest.mark.parametrize("red", REDS, ids=[r[0] for r in REDS])
def test_dgrad_row_plans(name, pk, ctas, mode, red):
    prob, kw = pk
    big = lambda g: sorted(set(list(range(min(g, 200))) + list(range(max(0, g - 50), g))))
    with sk.tile("auto"):
        cp = compare(prob, kw, mode, red, ctas, check_ctas=big)
    assert (cp.tm, cp.tn, cp.tk, cp.iters_per_tile) == (128, 64, 64, kw["kred"] // 64)


def test_row_views_need_their_shape():
    """The shifted-row view only for one group of 64 -> 64 channels, stride 1, at most 3 x 3 taps
    and rows of at most 64 positions with the column taps; the pages' im2col view otherwise, and
    always under the 128 x 128 tile."""
    def tn(op, tile="auto", **kw):
        a = dict(n=2, h=9, w=11, c=64, k=64, r=3, s=3, stride_h=1, stride_w=1, pad_h=1, pad_w=1,
                 groups=1)
        a.update(kw)
        with sk.tile(tile):
            return sk.sk_plan(sk.make_problem(op, ab_dtype="f16", c_dtype="f16", **a), "dp_sk",
                              "linear", 5, 148).tn
    for op in ("fprop", "dgrad"):
        assert tn(op) == 64
        assert tn(op, tile="128") == 128
        assert tn(op, c=128, k=128) == 128
        assert tn(op, r=5, s=5, pad_h=2, pad_w=2) == 128
        assert tn(op, groups=2, c=128, k=128) == 128
    assert tn("fprop", stride_h=2) == 128
    assert tn("fprop", w=63) == 128 and tn("fprop", w=62) == 64    # Wo + S - 1 = 64 fits
    assert tn("dgrad", w=63) == 128 and tn("dgrad", w=62) == 64    # W + S - 1 = 64 fits
