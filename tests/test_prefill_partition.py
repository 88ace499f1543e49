"""The chunked-prefill kernel's persistent work split, restated on the CPU.

The kernel cuts all key-tile steps of all units (128 queries of one row and
one head), in (row, head, query tile, key tile) order, into one equal range
per block, finds its first unit by closed forms and a binary search, and
walks its segments from the last to the first.  A unit cut by range
boundaries is merged by the block holding its end, from the partials of the
earlier blocks.  These tests restate that arithmetic in plain Python and
check what the merge relies on: every step is done exactly once; a cut
unit's pieces sit in consecutive blocks; each block publishes at most one
partial (the first segment it processes) and merges at most one unit (the
last segment it processes).
"""
import random

import pytest

TILE = 128


def tiles_of(pos0, C, t):
    """Key tiles visible to query tile t of a chunk of C queries starting at pos0."""
    return (pos0 + min(TILE * (t + 1), C) + TILE - 1) // TILE


def row_steps(C, L):
    """The kernel's closed form for the steps of one head of a row."""
    if C <= 0:
        return 0
    nt = (C + TILE - 1) // TILE
    a = (L - C + TILE - 1) // TILE
    return (nt - 1) * nt // 2 + (nt - 1) * a + (L + TILE - 1) // TILE


def owner_of(s, W, Ge):
    return ((s + 1) * Ge + W - 1) // W - 1


def split(chunks, lengths, hq, grid):
    """Per block: its segments (row, head, tile, U, nkt, k0, k1) in processing order."""
    C = [c if 0 <= c <= L else 0 for c, L in zip(chunks, lengths)]
    pos0 = [L - c for c, L in zip(C, lengths)]
    pre = [0]
    for c, L in zip(C, lengths):
        pre.append(pre[-1] + hq * row_steps(c, L))
    W = pre[-1]
    Ge = min(W, grid)
    blocks = []
    for cta in range(Ge):
        s0, s1 = W * cta // Ge, W * (cta + 1) // Ge
        x = s1 - 1
        lo, hi = 0, len(C) - 1
        while lo < hi:
            mid = (lo + hi + 1) >> 1
            if pre[mid] <= x:
                lo = mid
            else:
                hi = mid - 1
        r = lo
        wh = (pre[r + 1] - pre[r]) // hq
        off = x - pre[r]
        h, o2 = off // wh, off % wh
        a = (pos0[r] + TILE - 1) // TILE
        tl, th = 0, (C[r] + TILE - 1) // TILE - 1
        while tl < th:
            tm = (tl + th + 1) >> 1
            if tm * (tm + 1) // 2 + tm * a <= o2:
                tl = tm
            else:
                th = tm - 1
        t = tl
        U = pre[r] + h * wh + t * (t + 1) // 2 + t * a
        nkt = tiles_of(pos0[r], C[r], t)
        e, segs = s1, []
        while True:
            segs.append((r, h, t, U, nkt, max(s0 - U, 0), min(e - U, nkt)))
            if U <= s0:
                break
            e = U
            if t > 0:
                t -= 1
            elif h > 0:
                h -= 1
                t = (C[r] + TILE - 1) // TILE - 1
            else:
                r -= 1
                while C[r] == 0:
                    r -= 1
                h = hq - 1
                t = (C[r] + TILE - 1) // TILE - 1
            nkt = tiles_of(pos0[r], C[r], t)
            U -= nkt
        blocks.append(segs)
    return W, Ge, blocks, C, pos0


def check(chunks, lengths, hq, grid):
    W, Ge, blocks, C, pos0 = split(chunks, lengths, hq, grid)
    # the closed form equals the per-tile sum
    for c, L in zip(C, lengths):
        if c > 0:
            assert row_steps(c, L) == sum(tiles_of(L - c, c, t) for t in range((c + TILE - 1) // TILE))
    done = [0] * W
    pieces = {}
    for cta, segs in enumerate(blocks):
        s0, s1 = W * cta // Ge, W * (cta + 1) // Ge
        assert s1 > s0
        partials = merges = 0
        for k, (r, h, t, U, nkt, k0, k1) in enumerate(segs):
            assert 0 <= k0 < k1 <= nkt == tiles_of(pos0[r], C[r], t)
            for s in range(U + k0, U + k1):
                done[s] += 1
            pieces.setdefault((r, h, t), []).append((cta, k0, k1, k, len(segs)))
            if k1 < nkt:  # publishes a partial for the unit's last block
                partials += 1
                assert k == 0 and owner_of(U + nkt - 1, W, Ge) > cta
            elif k0 > 0:  # merges the unit
                merges += 1
                assert k == len(segs) - 1 and owner_of(U, W, Ge) < cta
        assert partials <= 1 and merges <= 1
    assert done == [1] * W
    for key, ps in pieces.items():
        ps.sort(key=lambda p: p[1])
        ctas = [p[0] for p in ps]
        assert ctas == list(range(ctas[0], ctas[0] + len(ctas)))
        assert ps[0][1] == 0
        for a, b in zip(ps, ps[1:]):
            assert a[2] == b[1]  # contiguous key ranges
    return W, Ge


def test_bench_launch_split():
    W, Ge = check([512] * 8, [4096] * 8, 12, 152)
    assert (W, Ge) == (11712, 152)


@pytest.mark.parametrize("seed", range(6))
def test_random_workloads(seed):
    rng = random.Random(seed)
    for _ in range(120):
        rows = rng.randint(1, 10)
        chunks, lengths = [], []
        for _ in range(rows):
            L = rng.choice([0, 1, 17, 128, 129, 300, 1000, 4096, rng.randint(0, 5000)])
            c = rng.choice([0, 1, 64, 128, 200, 512, L, rng.randint(0, max(L, 0))])
            if rng.random() < 0.05:
                c = L + 3  # a chunk longer than its row: skipped
            chunks.append(c)
            lengths.append(L)
        hq = rng.choice([1, 2, 4, 12])
        grid = rng.choice([1, 2, 5, 152, 300])
        if sum(row_steps(c if 0 <= c <= L else 0, L) for c, L in zip(chunks, lengths)) == 0:
            continue
        check(chunks, lengths, hq, grid)
