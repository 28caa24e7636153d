"""Host-side check of the decode schedule rule (the partitioning the metadata
kernel implements): cut the concatenated cost line of all problems (tiles of
tile_cost each + a fixed start-up cost) into `parts` equal pieces; a piece may
start or end inside a problem, and a piece shorter than a tile may be empty.
For any workload every tile must belong to exactly one piece, the
per-problem piece counts must equal the non-empty parts between the first and
the last part touching the problem (the closed form the kernel uses), each
piece's split index must be its rank among the pieces touching its first
problem, and the partial-result slots (the piece count of each split problem)
must total at most min(2 * parts, problems + parts).  Costs are in quarter
tiles: bf16 tiles 4, FP8 tiles 6, start-up 8.  The GPU test
test_schedule_covers_every_tile_once checks the kernel's own output."""
import numpy as np
import pytest

OVERHEAD = 8                      # start-up cost of a problem segment (quarter tiles)
TILE_COSTS = {"bf16": 4, "fp8": 6}


def schedule(tiles, parts, tile_cost=4, overhead=OVERHEAD):
    pre = [0]
    for n in tiles:
        pre.append(pre[-1] + (n * tile_cost + overhead if n > 0 else 0))
    total, np_ = pre[-1], len(tiles)

    def locate(x):
        if x >= total:
            return (np_, 0)
        lo, hi = 0, np_ - 1
        while lo < hi:
            mid = (lo + hi + 1) // 2
            if pre[mid] <= x:
                lo = mid
            else:
                hi = mid - 1
        t = max(x - pre[lo] - overhead, 0) // tile_cost
        return (lo + 1, 0) if t >= tiles[lo] else (lo, t)

    xs = [(total * k // parts) if total >= parts else min(k, total) for k in range(parts + 1)]
    starts = [locate(x) for x in xs]

    def part_of(pos):
        lo, hi = 0, parts - 1
        while lo < hi:
            mid = (lo + hi + 1) // 2
            if not pos < starts[mid]:
                lo = mid
            else:
                hi = mid - 1
        return lo

    ne_pre = [0]
    for k in range(parts):
        ne_pre.append(ne_pre[-1] + (1 if starts[k] < starts[k + 1] else 0))
    counts = [ne_pre[part_of((p, n - 1)) + 1] - ne_pre[part_of((p, 0))] if n > 0 else 0
              for p, n in enumerate(tiles)]
    split0 = [ne_pre[k] - ne_pre[part_of((starts[k][0], 0))] if starts[k] < starts[k + 1] and starts[k][0] < np_
              else 0 for k in range(parts)]
    return starts, counts, split0


def walk(tiles, starts, parts):
    """Enumerate (problem, tile, part) as the kernel's segment iterator does."""
    np_ = len(tiles)
    for k in range(parts):
        (p0, t0), (p1, t1) = starts[k], starts[k + 1]
        for p in range(p0, min(p1, np_ - 1) + 1):
            tb = t0 if p == p0 else 0
            te = min(t1 if p == p1 else tiles[p], tiles[p])
            for t in range(tb, te):
                yield p, t, k


@pytest.mark.parametrize("fmt", sorted(TILE_COSTS))
@pytest.mark.parametrize("seed", range(20))
def test_every_tile_once_and_split_bookkeeping(seed, fmt):
    rng = np.random.default_rng(seed)
    for _ in range(150):
        np_ = int(rng.integers(1, 14))
        parts = int(rng.integers(1, 200))
        tiles = [int(x) if rng.random() > 0.2 else 0 for x in rng.integers(0, 60, size=np_)]
        starts, counts, split0 = schedule(tiles, parts, TILE_COSTS[fmt])
        seen = {}
        touched = {}
        for p, t, k in walk(tiles, starts, parts):
            assert (p, t) not in seen
            seen[(p, t)] = k
            touched.setdefault(p, []).append(k)
        assert len(seen) == sum(tiles)
        for p, n in enumerate(tiles):
            ks = sorted(set(touched.get(p, [])))
            assert counts[p] == len(ks)
            for rank, k in enumerate(ks):
                if starts[k][0] == p:
                    assert split0[k] == rank
        # partial-result slots: split problems only, at most two per part
        slots = [c if c > 1 else 0 for c in counts]
        assert sum(slots) <= min(2 * parts, np_ + parts)


@pytest.mark.parametrize("fmt", sorted(TILE_COSTS))
def test_balance_on_a_ragged_mix(fmt):
    tc = TILE_COSTS[fmt]
    rng = np.random.default_rng(1002)
    lens = rng.integers(1024, 8193, size=128)
    tiles = [int((L + 63) // 64) for L in lens]
    parts = 152
    starts, counts, _ = schedule(tiles, parts, tc)
    load = np.zeros(parts)
    for p, t, k in walk(tiles, starts, parts):
        load[k] += tc
    for k in range(parts):
        load[k] += OVERHEAD * len({p for p, t, kk in walk(tiles, starts, parts) if kk == k})
    assert load.max() <= load.mean() * 1.15 + OVERHEAD + tc
    assert sum(counts) <= len(tiles) + parts


def test_parts_shorter_than_a_tile_are_empty_and_take_no_slot():
    """More parts than tiles: some cut points fall inside one tile, their parts are empty, and the
    problem's pieces (and slots) count only the non-empty parts."""
    tiles = [3, 1, 2]
    parts = 40
    starts, counts, split0 = schedule(tiles, parts, 6)
    nonempty = [k for k in range(parts) if starts[k] < starts[k + 1]]
    assert len(nonempty) == sum(tiles)  # one tile per non-empty part
    assert counts == [3, 1, 2]          # pieces: the non-empty parts only
    slots = [c if c > 1 else 0 for c in counts]
    assert slots == [3, 0, 2]           # a single piece takes no partial-result slot
    for p, t, k in walk(tiles, starts, parts):
        assert k in nonempty
