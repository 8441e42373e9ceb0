// Stream-K partition: the host planner and the CTA -> work walk shared by the host and the
// kernels of the CUDA path.
//
// rocm-libraries PR #13151 "feat(rocke): stream-K for implicit-GEMM conv wgrad":
//  - PR body, Technical Details / Partitioner: tiles that fill whole waves of the CTA pool run
//    data-parallel; the remainder's MAC iterations are spread over the stream-K CTAs;
//    iters_per_sk_cta is clamped to at least 1; the flag table is sized from the CTA count.
//  - Commit "Add StreamKIterPartition": contiguous balanced ranges that may straddle tiles; the
//    plan carries the DP/SK split, grid, partner and round bounds, flag bytes; resolved once.
//  - Review thread on auto-selection: tiles*iters below the pool gives sk_ctas == 0.
//  - Commit "Address review feedback": CTAs wait only on later CTAs and publish before waiting.
// Where the pages are silent this follows one fixed reading: the first `extra` SK CTAs take one
// more iteration; SK tiles are ids [0, sk_tiles); tile ids are (group, m-tile, n-tile) with the
// n-tile fastest; persistent CTAs run their DP tiles before their SK range.
#pragma once

#include <stdint.h>

#include "skgemm.h"

#if defined(__CUDACC__)
#define SK_HD __host__ __device__ __forceinline__
#else
#define SK_HD inline
#endif

namespace sk {

constexpr int64_t kControlBytes = 256;   // ticket counter + spare words after the flag table

SK_HD int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
// Quotient of two non-negative values below 2^31 (every iteration, tile and CTA index of a plan is,
// which the host planner checks): a 32-bit division, several times cheaper on the GPU than a
// 64-bit one.
SK_HD int64_t udiv31(int64_t a, int64_t b) {
    return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
}
SK_HD int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
SK_HD int64_t imin(int64_t a, int64_t b) { return a < b ? a : b; }
SK_HD int64_t imax(int64_t a, int64_t b) { return a > b ? a : b; }

// --- SK iteration space ----------------------------------------------------------------------

SK_HD int64_t sk_begin(const sk_plan_t& p, int64_t c) {
    return c * p.iters_per_sk_cta + imin(c, p.extra_iters);
}
SK_HD int64_t sk_end(const sk_plan_t& p, int64_t c) {
    return sk_begin(p, c) + p.iters_per_sk_cta + (c < p.extra_iters ? 1 : 0);
}
// Inverse of sk_begin/sk_end: the SK CTA holding SK iteration `it`. The divisor is never 0
// because iters_per_sk_cta >= 1 in every plan.
SK_HD int64_t sk_cta_of_iter(const sk_plan_t& p, int64_t it) {
    const int64_t big = p.iters_per_sk_cta + 1;
    const int64_t boundary = p.extra_iters * big;
    if (it < boundary) return udiv31(it, big);
    return p.extra_iters + udiv31(it - boundary, p.iters_per_sk_cta);
}

// Tiles that may have several contributors: SK tiles, or every tile of a split-K plan.
SK_HD int64_t n_shared_candidates(const sk_plan_t& p) {
    if (p.mode == SK_SPLITK) return p.splits > 1 ? p.tiles : 0;
    return p.sk_tiles;
}

// Contributors of tile t (a candidate): consecutive logical ids [first, first + n).
SK_HD void tile_contributors(const sk_plan_t& p, int64_t t, int64_t& first, int64_t& n) {
    if (p.mode == SK_SPLITK) {
        first = t * p.splits;
        n = p.splits;
        return;
    }
    first = sk_cta_of_iter(p, t * p.iters_per_tile);
    const int64_t last = sk_cta_of_iter(p, (t + 1) * p.iters_per_tile - 1);
    n = last - first + 1;
}

// Partial slot of contributor `index` of the shared tile of segment `s`: first + t + index for a
// stream-K tile (the CTA at the boundary of two tiles has a slot in each), t*splits + index for
// split-K (first = t*splits).
SK_HD int64_t partial_slot(const sk_plan_t& p, int64_t tile, int64_t first, int64_t index) {
    return first + index + (p.mode == SK_SPLITK ? 0 : tile);
}

// The value of CTA c's flag once it has handed on its partial of shared tile t: the number of
// partials it has published by then. A stream-K CTA shares at most two tiles, the one its range
// starts in (if it is shared) and the one its range ends in; the first is published first.
SK_HD uint32_t publication(const sk_plan_t& p, int64_t c, int64_t t) {
    if (p.mode == SK_SPLITK) return 1u;
    const int64_t t0 = udiv31(sk_begin(p, c), p.iters_per_tile);
    if (t == t0) return 1u;
    int64_t first, n;
    tile_contributors(p, t0, first, n);
    return n > 1 ? 2u : 1u;
}

// Tree fixup, contributor `index` of `n`: in round r (stride s = 2^r) an index with
// index mod 2s == s hands its sum to index - s and stops; one with index mod 2s == 0 and
// index + s < n receives the sum of index + s. Calls f(sender_index) in round order.
template <typename F>
SK_HD void for_each_tree_sender(int64_t index, int64_t n, int64_t rounds, F&& f) {
    for (int64_t r = 0; r < rounds; ++r) {
        const int64_t s = int64_t(1) << r;
        if (index % (2 * s) == s) break;
        if (index % (2 * s) == 0 && index + s < n) f(index + s);
    }
}

// --- CTA -> segments walk ----------------------------------------------------------------------

struct SegCursor {
    int64_t dp_next;   // next DP tile of this CTA, -1 when none is left
    int64_t it;        // next SK (or split-K) iteration, in the plan's global iteration space
    int64_t it_end;
};

SK_HD void seg_init(const sk_plan_t& p, int64_t cta, SegCursor& c) {
    c.dp_next = -1;
    c.it = c.it_end = 0;
    if (p.mode == SK_OFF) {
        if (cta < p.tiles) c.dp_next = cta;
    } else if (p.mode == SK_SPLITK) {
        const int64_t t = udiv31(cta, p.splits), j = cta - t * p.splits;
        if (t < p.tiles) {
            if (p.splits == 1) {
                c.dp_next = t;
            } else {
                c.it = t * p.iters_per_tile + j * p.iters_per_tile / p.splits;
                c.it_end = t * p.iters_per_tile + (j + 1) * p.iters_per_tile / p.splits;
            }
        }
    } else if (p.mode == SK_DP_SK || p.mode == SK_HYBRID) {
        if (cta < p.sk_ctas) {
            c.it = sk_begin(p, cta);
            c.it_end = sk_end(p, cta);
        } else {
            const int64_t t = p.sk_tiles + (cta - p.sk_ctas);
            if (t < p.tiles) c.dp_next = t;
        }
    } else {  // SK_PERSISTENT: DP tiles sk_tiles + cta + k*pool, then the SK range
        const int64_t t = p.sk_tiles + cta;
        if (t < p.tiles) c.dp_next = t;
        if (cta < p.sk_ctas) {
            c.it = sk_begin(p, cta);
            c.it_end = sk_end(p, cta);
        }
    }
}

SK_HD bool seg_next(const sk_plan_t& p, int64_t cta, SegCursor& c, sk_segment_t& s) {
    if (c.dp_next >= 0) {
        s.tile = c.dp_next;
        s.k_begin = 0;
        s.k_end = p.iters_per_tile;
        s.kind = SK_SEG_FULL;
        s.index = 0;
        s.n_contrib = 1;
        s.first_cta = -1;
        if (p.mode == SK_PERSISTENT) {
            c.dp_next += p.pool;
            if (c.dp_next >= p.tiles) c.dp_next = -1;
        } else {
            c.dp_next = -1;
        }
        return true;
    }
    if (c.it >= c.it_end) return false;
    const int64_t I = p.iters_per_tile;
    const int64_t t = udiv31(c.it, I);
    const int64_t stop = imin(c.it_end, (t + 1) * I);
    int64_t first, n;
    tile_contributors(p, t, first, n);
    s.tile = t;
    s.k_begin = c.it - t * I;
    s.k_end = stop - t * I;
    s.n_contrib = n;
    s.index = cta - first;
    s.first_cta = n > 1 ? first : -1;
    s.kind = n == 1 ? SK_SEG_FULL : (first == cta ? SK_SEG_OWNER : SK_SEG_PEER);
    if (n == 1) s.index = 0;
    c.it = stop;
    return true;
}

// Order of the iterations inside one stream-K segment (an execution detail, not part of the
// plan). A CTA that has already run `tau` stream-K iterations starts its next segment at the
// iteration k whose k mod iters_per_sk_cta is closest above tau, and wraps around. Then every SK
// CTA reads reduction block k at a time close to k mod iters_per_sk_cta, whatever tile it works on,
// so tiles that share an A or B panel read each block of it at nearly the same moment and L2
// serves the repeats. Returns the offset of the first iteration processed, in [0, len).
SK_HD int64_t sk_segment_rotation(int64_t iters_per_sk_cta, int64_t k_begin, int64_t len,
                                  int64_t tau) {
    const int64_t q = iters_per_sk_cta;
    const int64_t d = k_begin - tau;   // |d| < 2^31
    int64_t r = d >= 0 ? d - udiv31(d, q) * q : q - 1 - ((-d - 1) - udiv31(-d - 1, q) * q);
    if (r == 0) return 0;
    const int64_t i = q - r;
    return i < len ? i : 0;
}

// Tile id -> (group, m-tile, n-tile), n-tile fastest.
SK_HD void tile_coords(const sk_plan_t& p, int64_t t, int64_t& g, int64_t& mt, int64_t& nt) {
    const int64_t q = udiv31(t, p.tiles_n);
    nt = t - q * p.tiles_n;
    g = udiv31(q, p.tiles_m);
    mt = q - g * p.tiles_m;
}

}  // namespace sk
