"""CPU replica of the stream-K iteration partitioner, plus a brute-force checker and a
forward-progress simulator.

TEST INFRASTRUCTURE. Part of the CPU oracle; see ``oracle/__init__.py``. Shares no code with the
C++ planner of the CUDA path: it is written step by step from the pages.

What the pages fix (rocm-libraries PR #13151, "feat(rocke): stream-K for implicit-GEMM conv wgrad"):

* PR body, Technical Details, "Partitioner": output tiles that fill whole waves of the CTA pool run
  data-parallel (DP); only the remainder is spread over the stream-K (SK) CTAs; ``iters_per_sk_cta``
  is clamped to at least 1 so an all-DP partition is safe; the flag table is sized from the CTA count.
* Commit "Add StreamKIterPartition": each SK CTA owns a contiguous, balanced range of MAC
  iterations that may straddle output tiles; the plan exposes the DP/SK split, the grid, the linear
  partner and tree round bounds and the flag-table size, and is resolved once, returned by value.
* Review thread (auto-selection finding): a one-tile shape whose ``tiles * iters`` is below the pool
  yields ``sk_ctas == 0``, i.e. an all-DP partition.
* Commit "Resolve streamk_ctas=-1 from the reduction": linear/tree use one CTA per compute unit;
  atomic/workspace size the pool for throughput (four CTAs per compute unit in the final rule,
  bounded here by how many CTAs of the kernel fit on one SM).

Readings where the pages are silent (each is listed in the design notes):

* ``sk_ctas == 0`` when the remainder has fewer iterations than the pool (``sk_tiles*I < P``).
* CTA ``c`` gets ``iters_per_sk_cta + (c < extra)`` iterations; the first ``extra`` CTAs take one more.
* SK tiles are tile ids ``[0, sk_tiles)``, DP tiles ``[sk_tiles, T)``; a tile id maps to
  ``(group, m-tile, n-tile)`` with the n-tile fastest.
* ``dp_sk``: logical ids ``[0, sk_ctas)`` are SK CTAs, the rest run one DP tile each.
  ``persistent``: grid = P; CTA ``c`` runs DP tiles ``sk_tiles + c + k*P`` and then its SK range.
  ``off``: one CTA per tile over the whole reduction.
* ``hybrid`` (a variant of the pages' rule, which balances only the remainder): when the pool
  does not divide the tiles and there is at least one full wave (``T >= P``, ``T mod P != 0``),
  the stream-K region takes one full wave more, ``P + T mod P`` tiles, so that every SK CTA runs
  between one and two tiles' worth of iterations; otherwise it is ``dp_sk``. Grid and CTA walk
  as in ``dp_sk``.
* Split-K comparator: ``s = clamp(P // T, 1, I)`` slices per tile, slice ``j`` covering
  iterations ``[j*I//s, (j+1)*I//s)``.
* Flag table: one 32-bit flag per CTA that can publish, rounded up to 256 bytes. When a logical CTA
  is a cluster of ``cluster`` CTAs that each hand on their own rows of the tile, each of those CTAs
  has its flag: ``4 * publishers * cluster`` bytes. A flag counts the partials its CTA has
  published (a stream-K CTA shares at most two tiles: the tail of one and the head of the next).
* Partial slots: one fp32 tile per contributor of every shared tile, so that every contributor can
  hand its partial on: slot ``first(t) + t + j`` for contributor ``j`` of stream-K tile ``t`` (the
  boundary CTA of two tiles contributes to both and has one slot in each), slot ``t*s + j`` for
  slice ``j`` of split-K tile ``t``: ``sk_ctas + sk_tiles`` (stream-K) or ``T*s`` (split-K) slots.
* Who adds the partials. The pages fix the order of the additions (linear: the owner's partial,
  then the others in increasing contributor order; tree: the index-based rounds), not which CTA
  performs them. Two ways reach the same sums: the owner (and in a tree each receiver) folds its
  senders' partials, waiting only on higher ids; or every contributor publishes and then adds, in
  that order, a share of the tile's elements from all the partials ("spread"), which waits on every
  contributor of the tile and therefore needs all of the plan's publishing CTAs resident at once.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List

OFF, DP_SK, PERSISTENT, SPLITK, AUTO, HYBRID = 0, 1, 2, 3, 4, 5
LINEAR, TREE, ATOMIC, WORKSPACE, REDUCTION_AUTO = 0, 1, 2, 3, 4

# Auto selection: "long reduction" once the tiles hold this many MAC iterations in total (the
# PR #13151 review thread shows the predicate passing for a one-tile shape from 1024 iterations).
AUTO_MIN_ITERATIONS = 1024

# segment kinds: a CTA's work on one tile
SEG_FULL = 0    # the CTA computes the whole reduction of the tile and writes it
SEG_OWNER = 1   # first contributor of a shared tile: it finishes the tile
SEG_PEER = 2    # later contributor of a shared tile: it hands its partial on

CONTROL_BYTES = 256   # ticket counter + spare words, after the flag table


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def round_up(a: int, b: int) -> int:
    return ceil_div(a, b) * b


@dataclass
class Plan:
    tiles_m: int
    tiles_n: int
    groups: int
    T: int
    I: int
    P: int
    mode: int
    reduction: int
    tm: int
    tn: int
    tk: int
    sk_tiles: int = 0
    dp_tiles: int = 0
    sk_ctas: int = 0
    sk_iters: int = 0
    iters_per_sk_cta: int = 1
    extra: int = 0
    splits: int = 0
    grid: int = 0
    publishers: int = 0          # CTAs that may publish a partial (one flag each)
    slots: int = 0               # fp32 partial slots, one per contributor of a shared tile
    max_contrib: int = 1
    rounds: int = 0
    flag_bytes: int = 0
    partial_bytes: int = 0
    scratch_bytes: int = 0
    ws_bytes: int = 0
    shared_tiles: int = 0        # tiles with more than one contributor


def default_pool(reduction: int, num_sms: int, ctas_per_sm: int) -> int:
    """``ctas = -1``: one CTA per SM for linear/tree (every CTA may wait on a later one), and
    ``num_sms * min(4, ctas_per_sm)`` for atomic/workspace, whose CTAs never wait."""
    if reduction in (LINEAR, TREE):
        return num_sms
    return num_sms * min(4, max(1, ctas_per_sm))


def make_plan(*, tiles_m: int, tiles_n: int, groups: int, kred: int, tm: int, tn: int, tk: int,
              pool: int, mode: int, reduction: int, cluster: int = 1) -> Plan:
    """Steps 1-8 of the partition, in order."""
    # 1. tile and iteration counts
    T = groups * tiles_m * tiles_n
    I = ceil_div(kred, tk)
    P = pool
    p = Plan(tiles_m=tiles_m, tiles_n=tiles_n, groups=groups, T=T, I=I, P=P, mode=mode,
             reduction=reduction, tm=tm, tn=tn, tk=tk)
    if mode == OFF:
        p.dp_tiles, p.grid = T, T
    elif mode == SPLITK:
        s = min(max(P // T, 1), I) if T > 0 else 1
        p.splits = s
        p.dp_tiles = T if s == 1 else 0
        p.grid = T * s
        p.publishers = T * s if s > 1 else 0
        p.slots = p.publishers
    else:
        # 2. the remainder of whole waves is the stream-K part (hybrid: plus one full wave)
        p.sk_tiles = T % P
        if mode == HYBRID and T >= P and p.sk_tiles:
            p.sk_tiles += P
        p.dp_tiles = T - p.sk_tiles
        # 3. its iterations; too few to give every pool CTA one -> all data-parallel
        p.sk_iters = p.sk_tiles * I
        if p.sk_tiles == 0 or p.sk_iters < P:
            p.sk_tiles, p.dp_tiles, p.sk_iters, p.sk_ctas = 0, T, 0, 0
        else:
            p.sk_ctas = P
        # 4. balanced contiguous ranges, never a zero divisor
        if p.sk_ctas > 0:
            p.iters_per_sk_cta = max(1, p.sk_iters // p.sk_ctas)
            p.extra = p.sk_iters % p.sk_ctas
        else:
            p.iters_per_sk_cta, p.extra = 1, 0
        # 6. grid
        p.grid = p.sk_ctas + p.dp_tiles if mode in (DP_SK, HYBRID) else P
        p.publishers = p.sk_ctas
        p.slots = p.sk_ctas + p.sk_tiles if p.sk_ctas else 0
    # 7. contributors of the shared tiles
    mc = 1
    shared = 0
    for t in _shared_tile_ids(p):
        n = len(contributors(p, t))
        mc = max(mc, n)
        shared += n > 1
    p.max_contrib = mc
    p.shared_tiles = shared
    p.rounds = 0
    while (1 << p.rounds) < mc:
        p.rounds += 1
    # 8. workspace: [flags][control][partials | scratch]
    p.flag_bytes = round_up(4 * p.publishers * cluster, 256)
    tile_bytes = tm * tn * 4
    if reduction in (LINEAR, TREE):
        p.partial_bytes = p.slots * tile_bytes
    if reduction == WORKSPACE:
        p.scratch_bytes = _n_sk_tiles(p) * tile_bytes
    p.ws_bytes = p.flag_bytes + CONTROL_BYTES + p.partial_bytes + p.scratch_bytes
    return p


def make_auto_plan(**kw) -> Plan:
    """streamk = auto (PR #13151, commit making "auto" the default, and the review fix that has it
    build the launch's partition): stream-K when the tiles are few (T < P) over a long reduction
    (T*I >= AUTO_MIN_ITERATIONS) and the partition really has stream-K CTAs; otherwise split-K.
    reduction = auto resolves to workspace (same commit)."""
    if kw.get("reduction") == REDUCTION_AUTO:
        kw["reduction"] = WORKSPACE
    kw.pop("mode", None)
    p = make_plan(mode=DP_SK, **kw)
    if p.T < p.P and p.T * p.I >= AUTO_MIN_ITERATIONS and p.sk_ctas > 0:
        return p
    return make_plan(mode=SPLITK, **kw)


def _n_sk_tiles(p: Plan) -> int:
    if p.mode == SPLITK:
        return p.T if p.splits > 1 else 0
    return p.sk_tiles


def _shared_tile_ids(p: Plan):
    return range(_n_sk_tiles(p))


def sk_range(p: Plan, c: int):
    """Iteration range ``[begin, end)`` of SK CTA ``c`` in the SK iteration space."""
    ipc, extra = p.iters_per_sk_cta, p.extra
    begin = c * ipc + min(c, extra)
    end = begin + ipc + (1 if c < extra else 0)
    return begin, end


def cta_of_iter(p: Plan, it: int) -> int:
    """SK CTA that holds SK iteration ``it`` (inverse of ``sk_range``)."""
    big = p.iters_per_sk_cta + 1
    boundary = p.extra * big
    if it < boundary:
        return it // big
    return p.extra + (it - boundary) // p.iters_per_sk_cta


def contributors(p: Plan, t: int) -> List[int]:
    """Logical ids of the CTAs that contribute to shared tile ``t``, the owner first."""
    if p.mode == SPLITK:
        if p.splits <= 1:
            return []
        return [t * p.splits + j for j in range(p.splits)]
    if t >= p.sk_tiles:
        return []
    first = cta_of_iter(p, t * p.I)
    last = cta_of_iter(p, (t + 1) * p.I - 1)
    return list(range(first, last + 1))


def tile_coords(p: Plan, t: int):
    """Tile id -> (group, m-tile, n-tile), n-tile fastest."""
    nt = t % p.tiles_n
    mt = (t // p.tiles_n) % p.tiles_m
    g = t // (p.tiles_n * p.tiles_m)
    return g, mt, nt


@dataclass
class Segment:
    tile: int
    k_begin: int
    k_end: int
    kind: int
    index: int = 0        # contributor index in the tile (0 = owner)
    n_contrib: int = 1
    first_cta: int = -1


def _sk_segments(p: Plan, c: int) -> List[Segment]:
    out = []
    begin, end = sk_range(p, c)
    it = begin
    while it < end:
        t = it // p.I
        tile_end = (t + 1) * p.I
        stop = min(end, tile_end)
        cs = contributors(p, t)
        if len(cs) == 1:
            kind = SEG_FULL
        elif cs[0] == c:
            kind = SEG_OWNER
        else:
            kind = SEG_PEER
        if kind == SEG_FULL:   # sole contributor: no hand-off partners
            out.append(Segment(t, it - t * p.I, stop - t * p.I, kind, 0, 1, -1))
        else:
            out.append(Segment(t, it - t * p.I, stop - t * p.I, kind, c - cs[0], len(cs), cs[0]))
        it = stop
    return out


def cta_segments(p: Plan, c: int) -> List[Segment]:
    """Work of logical CTA ``c``, in the order it runs it."""
    full = lambda t: Segment(t, 0, p.I, SEG_FULL, 0, 1, -1)
    if p.mode == OFF:
        return [full(c)] if c < p.T else []
    if p.mode == SPLITK:
        s = p.splits
        t, j = divmod(c, s)
        if t >= p.T:
            return []
        if s == 1:
            return [full(t)]
        lo, hi = j * p.I // s, (j + 1) * p.I // s
        return [Segment(t, lo, hi, SEG_OWNER if j == 0 else SEG_PEER, j, s, t * s)]
    if p.mode in (DP_SK, HYBRID):
        if c < p.sk_ctas:
            return _sk_segments(p, c)
        t = p.sk_tiles + (c - p.sk_ctas)
        return [full(t)] if t < p.T else []
    # persistent: DP tiles first, then the SK range
    out = []
    t = p.sk_tiles + c
    while t < p.T:
        out.append(full(t))
        t += p.P
    if c < p.sk_ctas:
        out.extend(_sk_segments(p, c))
    return out


def tree_senders(index: int, n: int, rounds: int) -> List[int]:
    """Tree fixup, contributor ``index`` of ``n``: in round r (stride s = 2^r) an index with
    ``index mod 2s == s`` hands its sum to ``index - s`` and drops out; one with
    ``index mod 2s == 0`` and ``index + s < n`` takes the sum of ``index + s``. Returns the
    contributor indices this one receives from, in round order."""
    out = []
    for r in range(rounds):
        s = 1 << r
        if index % (2 * s) == s:
            break
        if index % (2 * s) == 0 and index + s < n:
            out.append(index + s)
    return out


def slot(p: Plan, t: int, j: int) -> int:
    """Partial slot of contributor ``j`` of shared tile ``t``."""
    if p.mode == SPLITK:
        return t * p.splits + j
    return contributors(p, t)[0] + t + j


def publication(p: Plan, c: int, t: int) -> int:
    """How many partials CTA ``c`` has published once it has handed on its partial of shared tile
    ``t`` (its flag's value then): 2 for the second of its shared tiles, else 1."""
    shared = [s.tile for s in cta_segments(p, c) if s.kind in (SEG_OWNER, SEG_PEER)]
    return shared.index(t) + 1


def linear_senders(index: int, n: int) -> List[int]:
    """Linear fixup: the owner takes every later contributor's partial, in increasing order."""
    return list(range(1, n)) if index == 0 else []


# ----------------------------------------------------------------------------------------------
# brute force and invariants
# ----------------------------------------------------------------------------------------------

def brute_force_assignment(p: Plan):
    """Give SK iterations to CTAs one at a time, CTA by CTA, with the balanced sizes; return the
    iteration -> CTA map (a list) built without any closed form."""
    owner = []
    for c in range(p.sk_ctas):
        size = p.iters_per_sk_cta + (1 if c < p.extra else 0)
        owner.extend([c] * size)
    return owner


def check_invariants(p: Plan) -> None:
    """Raise AssertionError on any violated invariant of the partition."""
    assert p.iters_per_sk_cta >= 1
    if p.mode in (DP_SK, PERSISTENT, HYBRID):
        assert p.dp_tiles + p.sk_tiles == p.T
        if p.T % p.P == 0:
            assert p.sk_ctas == 0 and p.dp_tiles == p.T          # all-DP when tiles divide the pool
        if p.sk_ctas:
            owner = brute_force_assignment(p)
            assert len(owner) == p.sk_iters                      # complete coverage
            sizes = [sk_range(p, c)[1] - sk_range(p, c)[0] for c in range(p.sk_ctas)]
            assert max(sizes) - min(sizes) <= 1                  # balanced
            if p.mode == HYBRID and p.T >= p.P:                  # one to two tiles per SK CTA
                assert p.I <= min(sizes) and max(sizes) <= 2 * p.I
            for c in range(p.sk_ctas):
                b, e = sk_range(p, c)
                assert all(owner[i] == c for i in range(b, e))   # contiguous and disjoint
                assert all(cta_of_iter(p, i) == c for i in range(b, e))
                segs = _sk_segments(p, c)
                peers = [i for i, s in enumerate(segs) if s.kind == SEG_PEER]
                assert len(peers) <= 1 and (not peers or peers[0] == 0)   # <=1 non-owner, first
    # every tile is computed exactly once over all iterations
    cover = {}
    for c in range(p.grid):
        for s in cta_segments(p, c):
            cover.setdefault(s.tile, []).append((s.k_begin, s.k_end))
    assert sorted(cover) == list(range(p.T))
    for t, rs in cover.items():
        rs.sort()
        assert rs[0][0] == 0 and rs[-1][1] == p.I
        assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
    # every contributor of every shared tile has its own partial slot inside the table
    taken = set()
    for t in _shared_tile_ids(p):
        for j in range(len(contributors(p, t))):
            k = slot(p, t, j)
            assert 0 <= k < p.slots and k not in taken
            taken.add(k)
    # waits only target higher logical ids
    for t in _shared_tile_ids(p):
        cs = contributors(p, t)
        assert cs == list(range(cs[0], cs[0] + len(cs)))
        for j in range(len(cs)):
            for snd in linear_senders(j, len(cs)) + tree_senders(j, len(cs), p.rounds):
                assert cs[snd] > cs[j]


def simulate_progress(p: Plan, slots: int, reduction: int, fold: str = "owner") -> bool:
    """Discrete-event check that a pool of ``slots`` resident CTAs, started in logical-id order
    (a ticket counter), always finishes.

    ``fold="owner"``: each segment is one step; a receiving segment blocks until every sender has
    published; a peer publishes when its own receives are done.
    ``fold="spread"``: a CTA first runs all its segments, publishing every shared one without
    waiting; then it blocks until every contributor of each of its shared tiles has published."""
    if reduction not in (LINEAR, TREE):
        return True
    if fold == "spread":
        return _simulate_spread(p, slots)
    work = {c: list(cta_segments(p, c)) for c in range(p.grid)}
    published = set()
    nxt = 0
    running = []
    done = 0
    while done < p.grid:
        while len(running) < slots and nxt < p.grid:
            running.append(nxt)
            nxt += 1
        progressed = False
        for c in list(running):
            segs = work[c]
            while segs:
                s = segs[0]
                if s.kind in (SEG_OWNER, SEG_PEER):
                    snd = (linear_senders(s.index, s.n_contrib) if reduction == LINEAR
                           else tree_senders(s.index, s.n_contrib, p.rounds))
                    if not all(s.first_cta + j in published for j in snd):
                        break
                    if s.kind == SEG_PEER:
                        published.add(c)
                segs.pop(0)
                progressed = True
            if not segs:
                running.remove(c)
                done += 1
                progressed = True
        if not progressed:
            return False
    return True


def _simulate_spread(p: Plan, slots: int) -> bool:
    tiles_of = {c: [s.tile for s in cta_segments(p, c) if s.kind in (SEG_OWNER, SEG_PEER)]
                for c in range(p.grid)}
    published = set()   # (tile, cta)
    nxt, running, done = 0, [], 0
    while done < p.grid:
        while len(running) < slots and nxt < p.grid:
            for t in tiles_of[nxt]:   # a started CTA publishes all its shared segments
                published.add((t, nxt))
            running.append(nxt)
            nxt += 1
        finished = [c for c in running
                    if all((t, d) in published for t in tiles_of[c] for d in contributors(p, t))]
        if not finished:
            return False
        for c in finished:
            running.remove(c)
            done += 1
    return True
