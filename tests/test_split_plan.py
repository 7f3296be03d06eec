"""The split-KV plan the decode kernels derive on the device, restated on the
host and checked for the properties the kernels rely on (CPU only).

Every (source, row group) pair contributes `pen` work-free items and then its
key tiles to one list of W items; CTA c of G takes items [c W / G, (c + 1) W /
G).  A pair cut by range boundaries becomes chunks on consecutive CTAs; chunk
k of a pair whose first chunk CTA c0 holds writes its partial rows at
chunk_slot(c0, k); CTA c0 publishes the pair in its split-table entry.  With
gangs of S CTAs a source's items are counted once (not once per row group):
gang j = c // S takes items [j W / G, (j + 1) W / G) of G gangs and its CTA
c % S runs that row group of every source over them, so a pair's chunks are
on CTAs S apart (chunk k of the pair starting on CTA c0 on CTA c0 + k S).  The
kernels compute quotients with a float estimate corrected by exact integer
products; that estimate is emulated here in float32.
"""
import numpy as np
import pytest


def quot_floor(t, W):
    q = int(np.float32(t) * (np.float32(1.0) / np.float32(W)))
    while q > 0 and q * W > t:
        q -= 1
    while (q + 1) * W <= t:
        q += 1
    return q


def range_owner(i, W, G):
    return quot_floor((i + 1) * G - 1, W)


def chunk_slot(c0, k, stride=1):
    return 2 * c0 + 1 if k == 0 else 2 * (c0 + k * stride)


def plan(pairs_per_source, tiles_per_source, pen, grid, S=1):
    """Units of every CTA: (source, group, first tile, tiles, cta0, split, nsplit)."""
    if S > 1:
        items = [nt + pen if nt > 0 and g > 0 else 0 for g, nt in zip(pairs_per_source, tiles_per_source)]
    else:
        items = [g * (nt + pen) if nt > 0 else 0 for g, nt in zip(pairs_per_source, tiles_per_source)]
    W = sum(items)
    nplan = grid // S
    G = min(nplan, W) if W > 0 else 1
    base = np.concatenate([[0], np.cumsum(items)]).astype(np.int64)
    units = [[] for _ in range(grid)]
    for c in range(grid):
        me, gg = c // S, c % S
        if W == 0 or me >= G:
            continue
        lo, hi = quot_floor(me * W, G), quot_floor((me + 1) * W, G)
        i = lo
        b = int(np.searchsorted(base, lo, side="right") - 1)
        while i < hi and b < len(items):
            rend = base[b] + items[b]
            if i >= rend:
                b += 1
                continue
            nt = tiles_per_source[b]
            vlen = nt + pen
            g = gg if S > 1 else quot_floor(i - base[b], vlen)
            item0 = base[b] + (0 if S > 1 else g * vlen) + pen
            if i < item0:
                i = item0
            if i >= hi:
                break
            end = min(hi, item0 + nt)
            if g >= pairs_per_source[b]:
                i = end
                continue
            own0 = range_owner(item0, W, G)
            cta0 = own0 * S + gg
            nsplit = range_owner(item0 + nt - 1, W, G) - own0 + 1
            units[c].append((b, g, i - item0, end - i, cta0, me - own0, nsplit))
            i = end
    return units, W, G


def check_plan(pairs, tiles, pen, grid, S=1):
    units, W, G = plan(pairs, tiles, pen, grid, S)
    covered = {}
    for c, us in enumerate(units):
        for k, (b, g, t0, n, cta0, split, nsplit) in enumerate(us):
            assert n > 0
            assert 0 <= split < nsplit and cta0 + split * S == c
            assert S == 1 or g == c % S
            for t in range(t0, t0 + n):
                assert (b, g, t) not in covered, "a tile in two units"
                covered[(b, g, t)] = c
            if nsplit > 1 and split == 0:
                assert k == len(us) - 1, "a pair's first chunk is its CTA's last unit"
            if split > 0:
                assert k == 0, "a continued pair is its CTA's first unit"
    # every tile of every pair exactly once
    expect = {(b, g, t) for b, (gs, nt) in enumerate(zip(pairs, tiles)) for g in range(gs) for t in range(nt)}
    assert set(covered) == expect
    # a pair's chunks: nsplit CTAs S apart in tile order; partial slots unique and in range
    slots = set()
    for b, (gs, nt) in enumerate(zip(pairs, tiles)):
        for g in range(gs):
            if nt == 0:
                continue
            ctas = [covered[(b, g, t)] for t in range(nt)]
            assert ctas == sorted(ctas) and set(ctas) == set(range(ctas[0], ctas[-1] + 1, S))
            nsplit = (ctas[-1] - ctas[0]) // S + 1
            if nsplit > 1:
                for k in range(nsplit):
                    s = chunk_slot(ctas[0], k, S)
                    assert s not in slots and 0 <= s < 2 * grid
                    slots.add(s)
    # quotient estimate = exact quotient
    for i in range(0, W, max(1, W // 50)):
        assert range_owner(i, W, G) == -(-((i + 1) * G) // W) - 1
    return units


def test_headline_plan():
    # 64 requests x 1 group x 64 tiles over 152 CTAs: every pair split
    units = check_plan([1] * 64, [64] * 64, 4, 152)
    per_cta = [sum(u[3] for u in us) for us in units]
    assert max(per_cta) - min(per_cta) <= 5
    assert all(1 <= len(us) <= 2 for us in units)


@pytest.mark.parametrize("seed", range(40))
def test_random_plans(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 400))
    pairs = rng.integers(1, 9, size=B).tolist()
    tiles = rng.integers(0, 200, size=B).tolist()
    if seed % 5 == 0:
        tiles = [int(x) if rng.random() < 0.5 else 0 for x in tiles]  # sources without keys
    grid = int(rng.choice([1, 3, 17, 148, 152, 300]))
    pen = int(rng.choice([0, 1, 4, 6]))
    check_plan(pairs, tiles, pen, grid)


def test_more_ctas_than_items():
    check_plan([1, 1], [1, 2], 0, 152)
    check_plan([2], [3], 4, 152)


def test_quotient_estimate_on_large_lists():
    # item counts far beyond float32's 24-bit mantissa still give exact owners
    for W, G in [(2 ** 31 - 1, 152), (10 ** 12 + 7, 148), (123456789, 151)]:
        for i in (0, 1, W // 3, W // 2 + 17, W - 2, W - 1):
            assert range_owner(i, W, G) == -(-((i + 1) * G) // W) - 1
            assert quot_floor(i, W) == 0 or quot_floor(i * G, W) == (i * G) // W


@pytest.mark.parametrize("seed", range(40))
def test_random_gang_plans(seed):
    # gangs of S CTAs (S = the largest request's row groups, 2..8), requests
    # with fewer groups (mixed query lengths) and without keys included
    rng = np.random.default_rng(1000 + seed)
    S = int(rng.integers(2, 9))
    B = int(rng.integers(1, 120))
    pairs = rng.integers(1, S + 1, size=B).tolist()
    pairs[int(rng.integers(0, B))] = S
    tiles = rng.integers(0, 400, size=B).tolist()
    if seed % 4 == 0:
        tiles = [int(x) if rng.random() < 0.6 else 0 for x in tiles]
    grid = (int(rng.choice([2 * S, 37, 148, 152])) // S) * S
    pen = int(rng.choice([0, 4]))
    check_plan(pairs, tiles, pen, grid, S)


def test_long_context_gang_plan():
    # 32 requests x 4 row groups of 64 rows (2 tokens x 128 heads), ~384
    # tiles each over all 8 shards, 38 gangs of 4 on 152 CTAs: every CTA
    # streams the same tiles as the 3 other members of its gang
    rng = np.random.default_rng(3)
    tiles = rng.integers(256, 513, size=32).tolist()
    units = check_plan([4] * 32, tiles, 4, 152, 4)
    for j in range(38):
        ranges = [[(b, t0, n) for (b, g, t0, n, *_rest) in units[4 * j + gg]] for gg in range(4)]
        assert all(r == ranges[0] for r in ranges)
    per_cta = [sum(u[3] for u in us) for us in units]
    assert max(per_cta) - min(per_cta) <= 12
