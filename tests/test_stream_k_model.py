"""The stream-K partition of the tensor-core attention kernel, on a model.

attn_tc_kernel cuts the flattened order of all units' tiles into ranges of
equal cost: a unit costs its tiles plus `c` tiles for the segment boundary it
causes.  In cost positions unit u (the u-th unit with tiles) starts at
U_u = P_u + c * u (P_u its first tile) and its tile o sits at U_u + c + o;
tile t belongs to range floor(cost(t) / T), the last range taking the rest.
Each CTA finds its range's first tile and the next range's first tile
(`find`), walks its range as segments (one per unit), and the CTA holding a
unit's first tile records (first range, ranges spanned or 0 when whole, slot
of the first piece) for the merge launch, which reads piece q from the CTA of
range first + q, slot `first_slot` for q = 0 and 0 after.

This model replays that arithmetic (in the kernel's order of operations) on
random batches and checks it against a direct assignment of every tile:
ranges tile the order exactly, no range but trailing ones is empty, each
unit's entry names exactly the ranges holding its tiles and the slots their
segments wrote, and no unit has more than 64 pieces.  (The kernel's code is
kept with this model: a change to one is a change to the other.)
"""
import random

import pytest

MAX_PIECES = 64


def partition(tiles_per_request, upr, ranges, seg_cost):
    """(T, c, range starts) as locate_range computes them."""
    tiles = sum(tiles_per_request) * upr
    units = sum(1 for v in tiles_per_request if v > 0) * upr
    nmax = max(tiles_per_request) if tiles_per_request else 0
    c = seg_cost if tiles >= ranges else 0
    cost = tiles + c * units
    T = max(-(-cost // ranges), (nmax + MAX_PIECES - 3) // (MAX_PIECES - 2), c + 1)

    def find(X):
        cum_cost = cum_tiles = 0
        for v in tiles_per_request:
            vc = upr * (v + c) if v > 0 else 0
            if cum_cost + vc > X:
                rem = X - cum_cost
                per = v + c
                j = rem // per
                r2 = rem - j * per
                o = 0 if r2 <= c else r2 - c
                return cum_tiles + j * v + o, cum_cost + j * per
            cum_cost += vc
            cum_tiles += upr * v
        return tiles, None

    starts = []
    for r in range(ranges):
        X0 = r * T
        s = find(X0) if X0 < cost else (tiles, None)
        if r + 1 < ranges and (r + 1) * T < cost:
            e = (r + 1) * T if c == 0 else find((r + 1) * T)[0]
        else:
            e = tiles
        if X0 >= cost:
            s = (tiles, None)
        starts.append((s[0], e, s[1]))
    return T, c, starts, tiles, cost


def unit_list(tiles_per_request, upr):
    """(unit id, first tile, tiles, cost position) of every unit with tiles."""
    out, pos, u = [], 0, 0
    for b, v in enumerate(tiles_per_request):
        for j in range(upr):
            if v > 0:
                out.append(((b, j), pos, v, u))
                pos += v
                u += 1
    return out


@pytest.mark.parametrize("seed", range(300))
def test_partition_matches_direct_assignment(seed):
    rng = random.Random(seed)
    batch = rng.randint(1, 64)
    upr = rng.choice([1, 2, 4, 8, 16])
    long_tail = rng.random() < 0.3
    tiles_per_request = [0 if rng.random() < 0.1 else
                         (rng.randint(1, 300) if long_tail else rng.randint(1, 20))
                         for _ in range(batch)]
    ranges = rng.choice([1, 2, 7, 64, 76, 152, 304])
    seg_cost = rng.choice([1, 2])
    T, c, rs, tiles, cost = partition(tiles_per_request, upr, ranges, seg_cost)
    units = unit_list(tiles_per_request, upr)

    # ranges tile [0, tiles) in order; only trailing ranges are empty
    prev_end = 0
    seen_empty = False
    for s, e, _ in rs:
        if s >= e:
            seen_empty = True
            continue
        assert not seen_empty, "an empty range before a non-empty one"
        assert s == prev_end
        prev_end = e
    assert prev_end == tiles

    # direct assignment of every tile to a range by its cost position
    owner = {}
    for (uid, p0, v, u) in units:
        for o in range(v):
            owner[p0 + o] = min((p0 + c * u + c + o) // T, ranges - 1)
    for r, (s, e, _) in enumerate(rs):
        for t in range(s, e):
            assert owner[t] == r, (t, owner[t], r)

    # segments as the CTAs walk them; entries as the CTA with x0 == 0 writes them
    entries, written = {}, {}
    for r, (s, e, ucost0) in enumerate(rs):
        if s >= e:
            continue
        for (uid, p0, v, u) in units:
            a, bnd = max(s, p0), min(e, p0 + v)
            if a >= bnd:
                continue
            ucost = p0 + c * u
            if a == p0 and a == s:
                assert ucost == ucost0          # the cost position find() returned
            slot = 0 if a == s else 1
            written.setdefault(uid, []).append((r, slot))
            if a == p0:
                whole = bnd == p0 + v
                r_last = min((ucost + c + v - 1) // T, ranges - 1)
                entries[uid] = (r, 0 if whole else r_last - r + 1, slot)
    for (uid, p0, v, u) in units:
        r0, np_, first_slot = entries[uid]
        pieces = written[uid]
        if np_ == 0:
            assert pieces == [(r0, pieces[0][1])] and len(pieces) == 1
            continue
        assert 2 <= np_ <= MAX_PIECES
        expect = [(r0 + q, first_slot if q == 0 else 0) for q in range(np_)]
        assert pieces == expect, (uid, pieces, expect)
    # a range writes at most two partials (its first and its last segment)
    per_range = {}
    for uid, pieces in written.items():
        if entries[uid][1] == 0:
            continue
        for (r, slot) in pieces:
            per_range.setdefault(r, []).append(slot)
    for r, slots in per_range.items():
        assert len(slots) == len(set(slots)) <= 2
