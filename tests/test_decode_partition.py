"""The decode kernel's stream-K work split and split-unit bookkeeping, restated on the CPU.

The kernel cuts every (row, KV head) unit into 16-token granules, lays all
granules out in (row, head, token) order and gives block b the range
[W*b/G, W*(b+1)/G).  A block whose range fits its twelve slots and covers at
most four pieces runs in burst mode: its seven consumer warps are dealt to the
pieces (one each, then one more at a time to the piece with the most granules
per warp while that is at least two).  Any other block runs in stream mode:
four warps take equal contiguous shares; a warp finishes a unit that lies
wholly in its share, parks its first unit when that started before its share
and ends inside it, and dumps its last one; after a barrier the warps that hold
a unit's states (a .. b) combine them, warp j taking chunks j, j + k, ...
A unit with pieces in P > 1 blocks is merged from one record per piece: the
first K = min(P, 8) pieces' blocks each merge the chunks c with c % K equal to
their index, and the unit's records live at record slot (first block + unit).

These tests restate that arithmetic in plain Python and check what the
kernel relies on: every granule is staged exactly once; burst warps get
non-empty shares of their piece within the ring; stream warps' states are
combined exactly once per unit and block, from slots that were written; each
split unit's eight chunks are merged exactly once; a block has at most two
split pieces; and record regions of different units never overlap and stay
inside the workspace the host sizes (blocks + rows x KV heads slots).
"""
import random

import numpy as np
import pytest

GRANULE, RING, BURST_PIECES, CONSUMERS, STREAM_WARPS, MERGE_WAYS = 16, 12, 4, 7, 4, 8
CHUNK, ML = 512, 64
REC = 8 * CHUNK + MERGE_WAYS * ML  # bytes of one record slot


def units_of(lengths, hk):
    """(unit id, first granule, granules) in (row, head) order, and W."""
    out, pos = [], 0
    for r, L in enumerate(lengths):
        n = (L + GRANULE - 1) // GRANULE
        for h in range(hk):
            out.append((r * hk + h, pos, n))
            pos += n
    return out, pos


def owner_of(g, W, G):
    """The kernel's closed form: the largest c with floor(c * W / G) <= g."""
    return ((g + 1) * G - 1) // W


def block_range(b, W, G):
    return W * b // G, W * (b + 1) // G


def burst_warps(sizes):
    """Warps per piece, dealt as the plan deals them."""
    wc = [1] * len(sizes)
    for _ in range(len(sizes), CONSUMERS):
        c = [(sz + w - 1) // w for sz, w in zip(sizes, wc)]
        best = max(c)
        if best <= 1:
            break
        wc[c.index(best)] += 1
    return wc


def stream_share(g0, g1, w):
    ng = g1 - g0
    return g0 + ng * w // STREAM_WARPS, g0 + ng * (w + 1) // STREAM_WARPS


def check_split(lengths, hk, G):
    units, W = units_of(lengths, hk)
    if W == 0:
        return
    Ge = min(G, W)
    unit_at = np.empty(W, dtype=np.int64)
    span = {}
    for u, us, n in units:
        if n:
            unit_at[us:us + n] = u
            span[u] = (us, n)
    # every granule's owner by the closed form is the block whose range holds it
    owners = [owner_of(g, W, Ge) for g in range(W)]
    for b in range(Ge):
        g0, g1 = block_range(b, W, Ge)
        assert all(owners[g] == b for g in range(g0, g1))
    staged = np.zeros(W, dtype=np.int64)
    merged = {}   # unit -> chunk -> times merged
    records = {}  # unit -> set of piece indices written
    for b in range(Ge):
        g0, g1 = block_range(b, W, Ge)
        ng = g1 - g0
        if ng == 0:
            continue
        pieces = []  # (unit, first, count) inside the block
        for g in range(g0, g1):
            u = int(unit_at[g])
            if pieces and pieces[-1][0] == u:
                pieces[-1][2] += 1
            else:
                pieces.append([u, g, 1])
        split = [p for p in pieces if span[p[0]][1] != p[2]]
        assert len(split) <= 2, "a block's split pieces are its first and its last"
        for u, a, cnt in split:
            us, n = span[u]
            cs = owner_of(us, W, Ge)
            P = owner_of(us + n - 1, W, Ge) - cs + 1
            assert P > 1 and cs <= b < cs + P
            records.setdefault(u, set()).add(b - cs)
            K = min(P, MERGE_WAYS)
            if b - cs < K:
                for c in range(b - cs, 8, K):
                    merged.setdefault(u, [0] * 8)[c] += 1
        if ng <= RING and len(pieces) <= BURST_PIECES:
            # burst: warps dealt to pieces, each a non-empty share of its piece
            wc = burst_warps([p[2] for p in pieces])
            assert sum(wc) <= CONSUMERS
            for (u, a, cnt), k in zip(pieces, wc):
                shares = [(a + i * cnt // k, a + (i + 1) * cnt // k) for i in range(k)]
                for wa, wb in shares:
                    assert wb > wa
                    assert 0 <= wa - g0 and wb - g0 <= RING
                    staged[wa:wb] += 1
            continue
        # stream: four shares; finish, park or dump; then combine
        shares = [stream_share(g0, g1, w) for w in range(STREAM_WARPS)]
        written = set()   # (warp, slot) holding a state
        finished = set()  # units a warp finished from registers
        for w, (wa, wb) in enumerate(shares):
            assert wb > wa
            staged[wa:wb] += 1
            seen = []
            for g in range(wa, wb):
                u = int(unit_at[g])
                if not seen or seen[-1] != u:
                    seen.append(u)
            for i, u in enumerate(seen):
                us, n = span[u]
                if us >= wa and us + n <= wb:
                    finished.add(u)
                elif i < len(seen) - 1:
                    assert i == 0, "only a warp's first unit can end before its share does"
                    written.add((w, 1))  # parked, reloaded into slot 1
                else:
                    written.add((w, 0))
        combined = {}  # unit -> list of (j, k)
        for w, (wa, wb) in enumerate(shares):
            first, last = int(unit_at[wa]), int(unit_at[wb - 1])
            for side, u in enumerate((first, last)):
                if side == 1 and u == first:
                    continue
                us, n = span[u]
                if us >= wa and us + n <= wb:
                    continue
                a, bb = 0, STREAM_WARPS - 1
                for x in range(STREAM_WARPS):
                    xa, xb = shares[x]
                    if xb <= us:
                        a = x + 1
                    if xa >= us + n and bb == STREAM_WARPS - 1 and x > 0:
                        bb = x - 1
                assert a <= w <= bb
                for x in range(a, bb + 1):
                    xa, xb = shares[x]
                    early = us < xa and us + n < xb
                    assert (x, 1 if early else 0) in written
                combined.setdefault(u, []).append((w - a, bb - a + 1))
        for u, js in combined.items():
            k = js[0][1]
            assert sorted(j for j, _ in js) == list(range(k)), "every holder combines once"
            chunks = sorted(c for j, _ in js for c in range(j, 8, k))
            assert chunks == list(range(8))
            assert u not in finished
    assert (staged == 1).all(), "every granule staged exactly once"
    # split units: all P records written, every chunk merged once
    for u, pieces in records.items():
        us, n = span[u]
        cs = owner_of(us, W, Ge)
        P = owner_of(us + n - 1, W, Ge) - cs + 1
        assert pieces == set(range(P))
        assert merged[u] == [1] * 8
    # record regions: [cs + u, cs + u + P) slots; disjoint; inside the workspace
    regions = []
    for u, pieces in records.items():
        us, n = span[u]
        cs = owner_of(us, W, Ge)
        P = len(pieces)
        K = min(P, MERGE_WAYS)
        start = (cs + u) * REC
        end = start + 8 * P * CHUNK + K * P * ML
        assert end <= (cs + u + P) * REC
        regions.append((start, end))
    regions.sort()
    for (s0, e0), (s1, e1) in zip(regions, regions[1:]):
        assert e0 <= s1, "record regions overlap"
    total = REC * (Ge + len(lengths) * hk)
    assert all(e <= total for _, e in regions)


def seeded_configs():
    """The benchmark's length mixes, drawn as the workloads draw them."""
    from paged_kv_cache_06_gb300 import workloads as wl
    out = []
    for name in ("tiny", "uniform", "mixed", "shared", "long"):
        case = wl.WORKLOADS[name](seed=0) if name not in ("mixed", "uniform") else \
            getattr(wl, name)(seed=0, layers=1)
        out.append((name, [int(x) for x in case.seq_lens]))
    return out


@pytest.mark.parametrize("grid", [152, 148, 37, 1])
def test_benchmark_length_mixes(grid):
    for name, lengths in seeded_configs():
        check_split(lengths, 2, grid)


def test_random_length_mixes():
    rnd = random.Random(7)
    for trial in range(400):
        rows = rnd.choice([1, 2, 3, 5, 8, 17, 32, 64, 96, 200])
        kind = rnd.random()
        if kind < 0.3:
            lengths = [rnd.randint(0, 600) for _ in range(rows)]
        elif kind < 0.6:
            lengths = [int(np.exp(rnd.uniform(np.log(1), np.log(40000)))) for _ in range(rows)]
        else:
            lengths = [rnd.choice([0, 1, 15, 16, 17, 300, 4096, 32769]) for _ in range(rows)]
        hk = rnd.choice([1, 2, 4])
        grid = rnd.choice([1, 2, 7, 64, 148, 152])
        check_split(lengths, hk, grid)


def test_burst_dealing_matches_hand_worked_cases():
    # one piece of 12 granules: all seven warps (ceil 12/6 = 2 > 1 still)
    assert burst_warps([12]) == [7]
    # pieces of 1 granule never get a second warp
    assert burst_warps([1, 1, 1, 1]) == [1, 1, 1, 1]
    # 3 and 2 granules: warps go to the piece with the most granules per warp
    # (ties to the first piece) until every warp holds one granule
    assert burst_warps([3, 2]) == [3, 2]
    # 12 and 1 granules: the long piece takes the six spare warps
    assert burst_warps([12, 1]) == [6, 1]
    # a share never empties: warps never exceed a piece's granules
    for sizes in ([1], [2], [5, 1], [4, 4, 3, 1]):
        assert all(k <= s for s, k in zip(sizes, burst_warps(sizes)))
