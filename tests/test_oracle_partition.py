"""Pins for the partition replica: values printed on the pages (tests/golden), closed-form
vectors worked by hand from the partition rule, a brute-force iteration assignment, the
invariants the pages fix, and a forward-progress simulation of the linear/tree hand-off."""
import itertools
import os
import random

import pytest

from oracle import partition as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "partition_page_points.txt")
RED = {"linear": P.LINEAR, "tree": P.TREE, "atomic": P.ATOMIC, "workspace": P.WORKSPACE}
MODE = {"off": P.OFF, "dp_sk": P.DP_SK, "persistent": P.PERSISTENT, "splitk": P.SPLITK,
        "hybrid": P.HYBRID}


def plan(T, I, Pool, mode=P.DP_SK, red=P.LINEAR, tm=128, tn=128, tk=64):
    # a 1 x T tile grid with kred = I*tk
    return P.make_plan(tiles_m=1, tiles_n=T, groups=1, kred=I * tk, tm=tm, tn=tn, tk=tk,
                       pool=Pool, mode=mode, reduction=red)


def _kv(s):
    return dict(x.split("=") for x in s.split())


def test_golden_page_points():
    n = 0
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, inp, exp = [x.strip() for x in line.split("|")]
        i = _kv(inp)
        if name.startswith("default_pool"):
            got = P.default_pool(RED[i["reduction"]], int(i["num_sms"]), int(i["ctas_per_sm"]))
            assert got == int(exp), name
        else:
            p = plan(int(i["T"]), int(i["I"]), int(i["P"]), MODE[i["mode"]])
            for k, v in _kv(exp).items():
                assert getattr(p, k) == int(v), (name, k)
        n += 1
    assert n == 8


# Hand-worked vectors for 128x128 tiles (TK = 64 for 16-bit, 128 for fp8):
#  T = tiles, I = ceil(Kred/TK), sk_tiles = T mod P, dp = T - sk_tiles, sk_iters = sk_tiles*I,
#  ipc = sk_iters // P, extra = sk_iters mod P.
VECTORS = [
    # name, T, I, P, dp, sk_tiles, sk_iters, ipc, extra
    ("gemm 256x256x4096 pool 3", 4, 64, 3, 3, 1, 64, 21, 1),
    ("gemm 3840x4096x4096 pool 148", 960, 64, 148, 888, 72, 4608, 31, 20),
    ("wgrad 32x56x56 c64 k64", 5, 1568, 148, 0, 5, 7840, 52, 144),
    ("wgrad 64x28x28 g4 s2", 20, 196, 148, 0, 20, 3920, 26, 72),
    ("fp8 8192^3 (TK=128)", 4096, 64, 148, 3996, 100, 6400, 43, 36),
    ("gemm 512x512x65536 pool 148", 16, 1024, 148, 0, 16, 16384, 110, 104),
]


@pytest.mark.parametrize("v", VECTORS, ids=[v[0] for v in VECTORS])
def test_worked_vectors(v):
    _, T, I, Pool, dp, skt, ski, ipc, extra = v
    p = plan(T, I, Pool)
    assert (p.dp_tiles, p.sk_tiles, p.sk_iters, p.iters_per_sk_cta, p.extra) == \
        (dp, skt, ski, ipc, extra)
    assert p.sk_ctas == Pool and p.grid == Pool + dp
    P.check_invariants(p)


def test_gemm_pool3_ranges_and_tree_rounds():
    p = plan(4, 64, 3, P.PERSISTENT)
    assert [P.sk_range(p, c) for c in range(3)] == [(0, 22), (22, 43), (43, 64)]
    assert P.contributors(p, 0) == [0, 1, 2]
    assert p.max_contrib == 3 and p.rounds == 2
    # tree of 3: index 0 takes 1 (round 0) then 2 (round 1); 1 and 2 only hand on
    assert P.tree_senders(0, 3, 2) == [1, 2]
    assert P.tree_senders(1, 3, 2) == [] and P.tree_senders(2, 3, 2) == []
    # persistent: CTA c runs DP tile 1 + c, then its SK range over tile 0
    segs = [P.cta_segments(p, c) for c in range(3)]
    assert [s[0].tile for s in segs] == [1, 2, 3]
    assert [(s[1].kind, s[1].k_begin, s[1].k_end) for s in segs] == \
        [(P.SEG_OWNER, 0, 22), (P.SEG_PEER, 22, 43), (P.SEG_PEER, 43, 64)]


def test_tree_senders_closed_form():
    # n = 8: a binary tree; index 0 takes 1, 2, 4; 4 takes 5, 6; 6 takes 7; odd indices take none
    assert P.tree_senders(0, 8, 3) == [1, 2, 4]
    assert P.tree_senders(4, 8, 3) == [5, 6]
    assert P.tree_senders(6, 8, 3) == [7]
    assert all(P.tree_senders(j, 8, 3) == [] for j in (1, 3, 5, 7))
    # every index but 0 hands on exactly once: sum of receives = n - 1
    for n in range(1, 40):
        r = max(0, (n - 1).bit_length())
        assert sum(len(P.tree_senders(j, n, r)) for j in range(n)) == n - 1


def test_brute_force_assignment_matches_closed_form():
    rng = random.Random(3)
    for _ in range(400):
        T, I, Pool = rng.randint(1, 300), rng.randint(1, 200), rng.randint(1, 300)
        p = plan(T, I, Pool)
        if not p.sk_ctas:
            continue
        owner = P.brute_force_assignment(p)
        assert all(P.cta_of_iter(p, i) == owner[i] for i in range(0, p.sk_iters, 7))


SWEEP = [(T, I, Pool) for T, I, Pool in itertools.product(
    [1, 2, 3, 4, 5, 7, 12, 13, 148, 149, 300], [1, 2, 3, 7, 64, 65], [1, 2, 3, 4, 5, 12, 148])]


@pytest.mark.parametrize("mode", [P.OFF, P.DP_SK, P.PERSISTENT, P.SPLITK, P.HYBRID])
def test_invariants_sweep(mode):
    for T, I, Pool in SWEEP:
        P.check_invariants(plan(T, I, Pool, mode))


def test_hybrid_worked_vector():
    # 10 tiles of 8 iterations on a pool of 4, worked by hand: the remainder (2 tiles) plus one
    # full wave (4) is stream-K, 48 iterations, 12 per CTA; tiles 6..9 run data-parallel
    p = plan(10, 8, 4, P.HYBRID)
    assert (p.sk_tiles, p.dp_tiles, p.sk_iters, p.sk_ctas) == (6, 4, 48, 4)
    assert (p.iters_per_sk_cta, p.extra, p.grid) == (12, 0, 8)
    seg = lambda c: [(s.tile, s.k_begin, s.k_end, s.kind) for s in P.cta_segments(p, c)]
    # CTA 0: iterations 0..11 = all of tile 0, then the first half of tile 1, which it owns
    assert seg(0) == [(0, 0, 8, P.SEG_FULL), (1, 0, 4, P.SEG_OWNER)]
    # CTA 1: iterations 12..23 = the second half of tile 1 (handed to CTA 0), all of tile 2
    assert seg(1) == [(1, 4, 8, P.SEG_PEER), (2, 0, 8, P.SEG_FULL)]
    assert seg(4) == [(6, 0, 8, P.SEG_FULL)] and seg(7) == [(9, 0, 8, P.SEG_FULL)]
    # dp_sk on the same problem balances only the remainder: half a tile per SK CTA
    d = plan(10, 8, 4, P.DP_SK)
    assert (d.sk_tiles, d.iters_per_sk_cta, d.grid) == (2, 4, 12)


def test_hybrid_reduces_to_dp_sk():
    # fewer tiles than the pool, or tiles that fill whole waves: the same plan as dp_sk
    for T, I, Pool in [(3, 64, 4), (1, 1216, 148), (12, 33, 4), (296, 64, 148)]:
        h, d = plan(T, I, Pool, P.HYBRID), plan(T, I, Pool, P.DP_SK)
        assert (h.sk_tiles, h.dp_tiles, h.sk_ctas, h.iters_per_sk_cta, h.extra, h.grid) == \
            (d.sk_tiles, d.dp_tiles, d.sk_ctas, d.iters_per_sk_cta, d.extra, d.grid)


def test_planted_hybrid_with_two_extra_waves_is_caught():
    # a stream-K region of two full waves plus the remainder gives every SK CTA 2.5 tiles
    import dataclasses
    p = plan(14, 8, 4, P.HYBRID)
    P.check_invariants(p)
    bad = dataclasses.replace(p, sk_tiles=10, dp_tiles=4, sk_iters=80, iters_per_sk_cta=20,
                              grid=8)
    with pytest.raises(AssertionError):
        P.check_invariants(bad)


def test_all_dp_when_tiles_divide_pool():
    for T, Pool in [(148, 148), (296, 148), (12, 3), (12, 4)]:
        p = plan(T, 33, Pool)
        assert p.sk_ctas == 0 and p.dp_tiles == T and p.iters_per_sk_cta == 1


def test_splitk_comparator():
    p = plan(16, 1024, 148, P.SPLITK)
    assert p.splits == 9 and p.grid == 144
    segs = P.cta_segments(p, 10)
    assert segs[0].tile == 1 and (segs[0].k_begin, segs[0].k_end) == (113, 227)
    assert plan(1, 3, 148, P.SPLITK).splits == 3          # never more slices than iterations
    assert plan(300, 8, 148, P.SPLITK).splits == 1         # tiles fill the pool: no split


def test_workspace_layout():
    # 4 tiles on 3 CTAs: one shared tile with 3 contributors; 3 + 1 partial slots of 64 KB
    p = plan(4, 64, 3, P.PERSISTENT, P.LINEAR)
    assert (p.publishers, p.slots) == (3, 4)
    assert p.flag_bytes == 256 and p.partial_bytes == 4 * 128 * 128 * 4
    assert p.ws_bytes == 256 + P.CONTROL_BYTES + 4 * 65536
    assert [P.slot(p, 0, j) for j in range(3)] == [0, 1, 2]
    w = plan(4, 64, 3, P.PERSISTENT, P.WORKSPACE)
    assert w.partial_bytes == 0 and w.scratch_bytes == 1 * 65536
    a = plan(4, 64, 3, P.PERSISTENT, P.ATOMIC)
    assert a.ws_bytes == 256 + P.CONTROL_BYTES


def test_flag_table_gives_every_cta_of_a_cluster_its_own_flag():
    # A logical CTA made of `cluster` CTAs that each hand on their own rows publishes one flag per
    # CTA: the flag of CTA r of publisher p sits at byte 4*(p*cluster + r), inside the table, and
    # no two (p, r) share one; the table still starts the 256-byte aligned control block.
    for T, I, Pool in [(240, 64, 74), (18, 64, 74), (5, 1568, 152), (1, 4096, 1216)]:
        for cluster in (1, 2):
            p = plan(T, I, Pool, tm=128 * cluster)
            p2 = P.make_plan(tiles_m=1, tiles_n=T, groups=1, kred=I * 64, tm=128 * cluster, tn=128,
                             tk=64, pool=Pool, mode=P.DP_SK, reduction=P.LINEAR, cluster=cluster)
            offs = {4 * (pub * cluster + r) for pub in range(p2.publishers) for r in range(cluster)}
            assert len(offs) == p2.publishers * cluster
            assert all(o + 4 <= p2.flag_bytes for o in offs)
            assert p2.flag_bytes % 256 == 0 and p2.flag_bytes - 256 < 4 * p2.publishers * cluster
            # the partition itself does not depend on how many CTAs make a logical CTA
            assert (p2.sk_tiles, p2.sk_ctas, p2.iters_per_sk_cta, p2.extra, p2.grid) == \
                (p.sk_tiles, p.sk_ctas, p.iters_per_sk_cta, p.extra, p.grid)
            # one fp32 partial slot per contributor of a shared tile, tm x tn x 4 bytes each
            assert p2.partial_bytes == p2.slots * (128 * cluster) * 128 * 4


def test_forward_progress_simulation():
    rng = random.Random(5)
    cases = [(4, 64, 3), (5, 1568 // 16, 148 // 4), (7, 5, 6), (3, 40, 12)]
    cases += [(rng.randint(1, 30), rng.randint(1, 40), rng.randint(2, 24)) for _ in range(60)]
    for T, I, Pool in cases:
        for mode in (P.DP_SK, P.PERSISTENT, P.SPLITK, P.HYBRID):
            for red in (P.LINEAR, P.TREE):
                p = plan(T, I, Pool, mode, red)
                # a blocked linear owner needs one more resident CTA to make progress; a tree
                # blocks at most `rounds` CTAs at a time
                need = 2 if red == P.LINEAR else p.rounds + 1
                for slots in sorted({need, need + 1, max(need, p.grid // 2), max(need, p.grid)}):
                    assert P.simulate_progress(p, slots, red), (T, I, Pool, mode, red, slots)


# --- planted mistakes: each must be caught by the checks above -------------------------------

def test_auto_selection_page_example():
    # review thread: pool 1216, one tile with 1024..1215 iterations passes the long-reduction
    # predicate but has no stream-K CTAs, so auto must keep split-K; from 1216 it is stream-K.
    kw = dict(tiles_m=1, tiles_n=1, groups=1, tm=128, tn=128, tk=64, pool=1216,
              reduction=P.WORKSPACE)
    for I in (1024, 1100, 1215):
        assert P.make_auto_plan(kred=I * 64, **kw).mode == P.SPLITK
    assert P.make_auto_plan(kred=1216 * 64, **kw).mode == P.DP_SK
    # many tiles: split-K, which degenerates to one slice per tile
    many = P.make_auto_plan(tiles_m=30, tiles_n=32, groups=1, kred=4096, tm=128, tn=128, tk=64,
                            pool=148, reduction=P.LINEAR)
    assert many.mode == P.SPLITK and many.splits == 1
    # few tiles, short reduction (T*I < 1024): split-K
    short = P.make_auto_plan(tiles_m=2, tiles_n=2, groups=1, kred=64 * 100, tm=128, tn=128, tk=64,
                             pool=148, reduction=P.LINEAR)
    assert short.mode == P.SPLITK
    # reduction auto -> workspace
    assert P.make_auto_plan(tiles_m=4, tiles_n=4, groups=1, kred=65536, tm=128, tn=128, tk=64,
                            pool=148, reduction=P.REDUCTION_AUTO).reduction == P.WORKSPACE


def test_single_slot_linear_owner_blocks():
    # with one resident CTA the owner of a shared tile waits for a CTA that never starts
    assert not P.simulate_progress(plan(4, 64, 3, P.DP_SK, P.LINEAR), 1, P.LINEAR)


def test_planted_extra_on_last_ctas_is_caught(monkeypatch):
    orig = P.sk_range

    def wrong(p, c):      # give the extra iteration to the LAST ctas instead of the first
        b, e = orig(p, c)
        if p.extra == 0:
            return b, e
        k = p.sk_ctas - p.extra
        size = p.iters_per_sk_cta + (1 if c >= k else 0)
        begin = c * p.iters_per_sk_cta + max(0, c - k)
        return begin, begin + size
    monkeypatch.setattr(P, "sk_range", wrong)
    with pytest.raises(AssertionError):
        P.check_invariants(plan(4, 64, 3))


def test_planted_missing_all_dp_rule_is_caught():
    p = plan(1, 1024, 1216)
    assert p.sk_ctas == 0
    q = plan(1, 1216, 1216)
    assert q.sk_ctas == 1216


def test_planted_wrong_tree_direction_is_caught(monkeypatch):
    monkeypatch.setattr(P, "tree_senders",
                        lambda j, n, r: [j - 1] if j % 2 == 1 else [])   # waits on a lower id
    with pytest.raises(AssertionError):
        P.check_invariants(plan(4, 64, 3, P.PERSISTENT, P.TREE))


def test_slot_worked_vector():
    # 2 tiles of 3 iterations on 4 CTAs: ranges [0,2) [2,4) [4,5) [5,6); tile 0 is shared by CTAs
    # 0 and 1, tile 1 by CTAs 1, 2 and 3; CTA 1 contributes to both and has a slot in each.
    p = plan(2, 3, 4, P.DP_SK, P.LINEAR)
    assert (p.sk_ctas, p.iters_per_sk_cta, p.extra, p.publishers, p.slots) == (4, 1, 2, 4, 6)
    assert P.contributors(p, 0) == [0, 1] and P.contributors(p, 1) == [1, 2, 3]
    assert [P.slot(p, 0, j) for j in range(2)] == [0, 1]
    assert [P.slot(p, 1, j) for j in range(3)] == [2, 3, 4]
    # CTA 1's flag reads 1 once its partial of tile 0 is out, 2 once that of tile 1 is too
    assert (P.publication(p, 1, 0), P.publication(p, 1, 1), P.publication(p, 2, 1)) == (1, 2, 1)
    assert p.partial_bytes == 6 * 128 * 128 * 4 and p.flag_bytes == 256
    s = plan(2, 64, 8, P.SPLITK, P.LINEAR)     # 4 slices per tile
    assert s.slots == 8 and [P.slot(s, 1, j) for j in range(4)] == [4, 5, 6, 7]


def test_slots_distinct_over_sweep():
    rng = random.Random(31)
    for _ in range(300):
        T, I, Pool = rng.randint(1, 40), rng.randint(1, 60), rng.randint(1, 160)
        for mode in (P.DP_SK, P.PERSISTENT, P.SPLITK, P.HYBRID):
            p = plan(T, I, Pool, mode, P.LINEAR)
            seen = set()
            for t in P._shared_tile_ids(p):
                for j in range(len(P.contributors(p, t))):
                    k = P.slot(p, t, j)
                    assert 0 <= k < p.slots and k not in seen, (T, I, Pool, mode, t, j)
                    seen.add(k)


def test_spread_fold_progress():
    """With every publishing CTA resident at once, the spread fold (all contributors publish, then
    each waits for every contributor of its tiles) always finishes; with fewer resident slots a
    one-tile plan deadlocks, which the owner fold of the pages avoids."""
    rng = random.Random(37)
    cases = [(4, 64, 3), (2, 1792, 148), (8, 256, 148), (5, 1568 // 16, 148 // 4), (1, 400, 148)]
    cases += [(rng.randint(1, 30), rng.randint(1, 40), rng.randint(2, 24)) for _ in range(60)]
    for T, I, Pool in cases:
        for mode in (P.DP_SK, P.PERSISTENT, P.SPLITK, P.HYBRID):
            for red in (P.LINEAR, P.TREE):
                p = plan(T, I, Pool, mode, red)
                publishing = p.grid if mode == P.SPLITK else p.sk_ctas
                for extra in (0, 1, p.grid):
                    assert P.simulate_progress(p, max(1, publishing) + extra, red, fold="spread"), \
                        (T, I, Pool, mode, red)
    one = plan(1, 400, 148, P.DP_SK, P.LINEAR)
    assert one.sk_ctas == 148
    assert not P.simulate_progress(one, 147, P.LINEAR, fold="spread")
    assert P.simulate_progress(one, 2, P.LINEAR, fold="owner")


# --- forward progress at the scale the pages checked it ---------------------------------------

FULL_PLANS = [   # (name, make_plan keywords) of the named workloads' whole partitions
    ("gemm 3840x4096x4096 128x128 P=148",
     dict(tiles_m=30, tiles_n=32, groups=1, kred=4096, tm=128, tn=128, tk=64, pool=148)),
    ("gemm 3840x4096x4096 256x256 pairs P=74",
     dict(tiles_m=15, tiles_n=16, groups=1, kred=4096, tm=256, tn=256, tk=64, pool=74, cluster=2)),
    ("gemm 3840x4096x4096 128x128 P=152",
     dict(tiles_m=30, tiles_n=32, groups=1, kred=4096, tm=128, tn=128, tk=64, pool=152)),
    ("gemm 512x512x65536 P=148",
     dict(tiles_m=4, tiles_n=4, groups=1, kred=65536, tm=128, tn=128, tk=64, pool=148)),
    ("gemm 512x512x65536 P=152",
     dict(tiles_m=4, tiles_n=4, groups=1, kred=65536, tm=128, tn=128, tk=64, pool=152)),
    ("fp8 8192^3 256x256 pairs P=76",
     dict(tiles_m=32, tiles_n=32, groups=1, kred=8192, tm=256, tn=256, tk=128, pool=76, cluster=2)),
    ("wgrad 32x56x56x64 rows P=148",
     dict(tiles_m=2, tiles_n=1, groups=1, kred=32 * 56 * 64, tm=128, tn=192, tk=64, pool=148)),
    ("wgrad 32x56x56x64 rows P=152",
     dict(tiles_m=2, tiles_n=1, groups=1, kred=32 * 56 * 64, tm=128, tn=192, tk=64, pool=152)),
    ("wgrad 64x28x28x256 g4 s2 rows P=148",
     dict(tiles_m=2, tiles_n=1, groups=4, kred=64 * 16 * 16, tm=128, tn=192, tk=64, pool=148)),
    ("wgrad 32x56x56x64 128x128 P=152",
     dict(tiles_m=1, tiles_n=5, groups=1, kred=32 * 56 * 56, tm=128, tn=128, tk=64, pool=152)),
]


def _need(p, red):
    # resident slots the owner fold needs: a blocked linear owner waits on one later CTA; a tree
    # blocks at most `rounds` CTAs at a time
    return 2 if red == P.LINEAR else p.rounds + 1


def test_forward_progress_5280_partitions():
    """The review thread on forward progress simulated the hand-off on 5280 partitions: here
    24 tile counts x 11 reduction lengths x 20 pool sizes = 5280 stream-K partitions, each run
    under both deterministic reductions with only the resident slots the owner fold needs, and
    under the spread fold with exactly its publishers resident."""
    Ts = list(range(1, 25))
    Is = [1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 144]
    Pools = [2, 3, 4, 5, 6, 7, 8, 12, 16, 24, 32, 37, 48, 64, 74, 96, 128, 148, 152, 304]
    n = 0
    for T in Ts:
        for I in Is:
            for Pool in Pools:
                n += 1
                for red in (P.LINEAR, P.TREE):
                    p = plan(T, I, Pool, P.DP_SK, red)
                    assert P.simulate_progress(p, _need(p, red), red), (T, I, Pool, red)
                    if red == P.LINEAR:
                        assert P.simulate_progress(p, max(1, p.sk_ctas), red, fold="spread"), \
                            (T, I, Pool)
    assert n == 5280


@pytest.mark.parametrize("name,kw", FULL_PLANS, ids=[f[0] for f in FULL_PLANS])
def test_forward_progress_named_full_plans(name, kw):
    """The named workloads' whole partitions, every mode, with the fewest resident slots each
    fold needs (owner: one or `rounds` more than the blocked CTAs; spread: every publisher)."""
    for mode in (P.DP_SK, P.PERSISTENT, P.SPLITK, P.HYBRID):
        for red in (P.LINEAR, P.TREE):
            p = P.make_plan(mode=mode, reduction=red, **kw)
            P.check_invariants(p)
            assert P.simulate_progress(p, _need(p, red), red), (name, mode, red)
            publishing = p.grid if mode == P.SPLITK else p.sk_ctas
            assert P.simulate_progress(p, max(1, publishing), red, fold="spread"), (name, mode, red)
