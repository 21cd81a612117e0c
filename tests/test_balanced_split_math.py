"""Host-side check of the balanced MLA split's arithmetic, restated from the
plan kernel and the decode kernel's run walk: row r has n_r tiles starting
at cum_r in the concatenation (T tiles in all); with C' = min(C, T) clusters,
cluster c takes [floor(c T / C'), floor((c+1) T / C')), tile x belongs to
cluster ((x + 1) C' - 1) // T, cluster c writes the partial of a cut row r to
slot c + r, and the reduce reads row r's partials from slots
c_first + r .. c_last + r.  Over random length mixes and cluster counts:
every tile is covered exactly once, every row's pieces are exactly its slot
range (so the reduce never reads an unwritten slot), a row with one piece is
written directly, slots stay below C + rows, and ranges differ by at most
one tile."""
import random


def plan(tiles, clusters):
    rows = len(tiles)
    cum, total = [], 0
    for n in tiles:
        cum.append(total)
        total += n
    C = min(clusters, total)
    ranges = [(0, 0, rows)] * clusters          # {x0, x1, first row}; no rows by default
    slots = [(0, 0)] * rows
    for r in range(rows):
        if tiles[r] == 0:
            continue
        first, last = cum[r], cum[r] + tiles[r] - 1
        cf = ((first + 1) * C - 1) // total
        cl = ((last + 1) * C - 1) // total
        slots[r] = (cf + r, cl - cf + 1)
        c = (first * C + total - 1) // total      # clusters whose range starts in row r
        while c < C and c * total // C <= last:
            ranges[c] = (c * total // C, (c + 1) * total // C, r)
            c += 1
    return cum, total, C, ranges, slots


def walk(cum, tiles, ranges, c):
    x0, x1, r = ranges[c]
    runs = []
    while r < len(cum):
        first, n = cum[r], tiles[r]
        row = r
        r += 1
        if first >= x1:
            break
        tb, te = max(x0 - first, 0), min(x1 - first, n)
        if tb >= te:
            continue
        runs.append((row, tb, te, tb == 0 and te == n, c + row))
    return runs


def test_balanced_split_covers_every_tile_once_and_slots_match():
    rng = random.Random(2024)
    for _ in range(4000):
        rows = rng.randint(1, 40)
        clusters = rng.randint(1, 80)
        tiles = [rng.choice([0, 0, 1, 2, 3, rng.randint(0, 200)]) for _ in range(rows)]
        cum, total, C, ranges, slots = plan(tiles, clusters)
        owner, pieces = {}, {}
        for c in range(clusters):
            for row, tb, te, direct, slot in walk(cum, tiles, ranges, c):
                for t in range(tb, te):
                    assert (row, t) not in owner
                    owner[(row, t)] = c
                pieces.setdefault(row, []).append((slot, direct))
        assert len(owner) == total
        for r in range(rows):
            got = pieces.get(r, [])
            first, count = slots[r]
            assert count == len(got)
            if count:
                assert sorted(s for s, _ in got) == list(range(first, first + count))
            assert all(d == (count == 1) for _, d in got)
            assert all(0 <= s < clusters + rows for s, _ in got)
        if total:
            sizes = [ranges[c][1] - ranges[c][0] for c in range(C)]
            assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
