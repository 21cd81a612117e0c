"""Host-side check of the balanced splits' arithmetic.  MLA (first part),
restated from the decode kernel's range search, run walk and slot table.  Row r has n_r tiles starting
at cum_r in the concatenation (T tiles in all).  Every row with tiles is
preceded by RUN_COST virtual tiles in a weighted concatenation (T_w
positions): row r occupies [W_r, W_r + RUN_COST + n_r), its real tile x sits
at W_r + RUN_COST + (x - cum_r).  With C' = min(C, T) clusters, cluster c
takes weighted positions [floor(c T_w / C'), floor((c+1) T_w / C')), i.e. the
real tiles from the image of its first position (a position in a virtual
block maps to the row's first tile) to the next cluster's; weighted position
y belongs to cluster ((y + 1) C' - 1) // T_w, cluster c writes the partial of
a cut row r to slot c + r, and the reduce reads row r's partials from slots
c_first + r .. c_last + r.  Over random length mixes and cluster counts:
every tile is covered exactly once, every row's pieces are exactly its slot
range (so the reduce never reads an unwritten slot), a row with one piece is
written directly, slots stay below C + rows, the weighted ranges differ by at
most one position, and a cluster's cost (its tiles plus RUN_COST per run it
opens) stays within RUN_COST of its weighted length.  GQA (second part):
the same weighting over (sequence, KV head) units, each CTA finding its range
from the lengths, the CTA holding a unit's first tile publishing the unit's
slot range."""
import random

RUN_COST = 8


def plan(tiles, clusters, run_cost=RUN_COST):
    rows = len(tiles)
    cum, wcum, total, wtotal = [], [], 0, 0
    for n in tiles:
        cum.append(total)
        wcum.append(wtotal)
        total += n
        wtotal += n + run_cost if n > 0 else 0
    C = min(clusters, total)
    ranges = [[0, 0, rows] for _ in range(clusters)]   # {x0, x1, first row}; no rows by default
    slots = [(0, 0)] * rows
    for r in range(rows):
        n = tiles[r]
        if n == 0:
            continue
        W = wcum[r]
        wf, wl = W + run_cost, W + run_cost + n - 1      # weighted first / last real tile
        cf = ((wf + 1) * C - 1) // wtotal
        cl = ((wl + 1) * C - 1) // wtotal
        slots[r] = (cf + r, cl - cf + 1)
        c = (W * C + wtotal - 1) // wtotal               # clusters whose range starts in row r
        while c < C and c * wtotal // C <= wl:
            y = c * wtotal // C
            x0 = cum[r] + min(max(y - wf, 0), n)
            ranges[c][0] = x0
            ranges[c][2] = r
            if c > 0:
                ranges[c - 1][1] = x0
            if c == C - 1:
                ranges[c][1] = total
            c += 1
    return cum, total, wtotal, C, [tuple(x) for x in ranges], slots


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
    for it in range(4000):
        rows = rng.randint(1, 40)
        clusters = rng.randint(1, 80)
        run_cost = RUN_COST if it % 4 else rng.choice([0, 1, 3, 8, 20])
        tiles = [rng.choice([0, 0, 1, 2, 3, rng.randint(0, 200)]) for _ in range(rows)]
        cum, total, wtotal, C, ranges, slots = plan(tiles, clusters, run_cost)
        owner, pieces = {}, {}
        for c in range(clusters):
            runs = walk(cum, tiles, ranges, c)
            for row, tb, te, direct, slot in runs:
                for t in range(tb, te):
                    assert (row, t) not in owner
                    owner[(row, t)] = c
                pieces.setdefault(row, []).append((slot, direct))
            if total and c < C:
                wlen = (c + 1) * wtotal // C - c * wtotal // C
                cost = sum(te - tb for _, tb, te, _, _ in runs) + run_cost * len(runs)
                assert wlen - run_cost <= cost <= wlen + run_cost
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
            wsizes = [(c + 1) * wtotal // C - c * wtotal // C for c in range(C)]
            assert min(wsizes) >= 1 and max(wsizes) - min(wsizes) <= 1
            assert all(ranges[c][0] <= ranges[c][1] for c in range(C))


def test_run_cost_zero_is_the_equal_tile_split():
    # with no cost per run the weighted split is the plain one: equal tile ranges
    rng = random.Random(7)
    for _ in range(500):
        tiles = [rng.randint(0, 50) for _ in range(rng.randint(1, 30))]
        clusters = rng.randint(1, 60)
        cum, total, wtotal, C, ranges, _ = plan(tiles, clusters, 0)
        assert wtotal == total
        for c in range(C):
            assert ranges[c][:2] == (c * total // C, (c + 1) * total // C)


def test_more_runs_get_fewer_tiles():
    # a cluster whose range meets many short rows holds fewer tiles than one
    # inside a long row
    tiles = [400] + [4] * 40
    cum, total, wtotal, C, ranges, _ = plan(tiles, 4)
    counts = [sum(te - tb for _, tb, te, _, _ in walk(cum, tiles, ranges, c)) for c in range(C)]
    runs = [len(walk(cum, tiles, ranges, c)) for c in range(C)]
    assert runs[0] == 1 and runs[-1] > 5
    assert counts[0] > counts[-1] + 5 * RUN_COST


# ---- the balanced GQA split (computed by every CTA from the lengths) --------

GQA_UNIT_COST = 2


def gqa_tile_of_position(cum, hkv, y, cost):
    """Real tile of weighted position y: sequence b by the last b with
    cum[b] + cost hkv b <= y, then the unit and the offset inside it (a
    position in a unit's virtual block maps to its first tile)."""
    batch = len(cum) - 1
    b = max(i for i in range(batch) if cum[i] + cost * hkv * i <= y)
    n = (cum[b + 1] - cum[b]) // hkv
    off = y - (cum[b] + cost * hkv * b)
    h = off // (n + cost)
    o = off - h * (n + cost) - cost
    return cum[b] + h * n + min(max(o, 0), n)


def gqa_plan(n_seq, hkv, grid, cost=GQA_UNIT_COST):
    cum = [0]
    for n in n_seq:
        cum.append(cum[-1] + n * hkv)
    T = cum[-1]
    Tw = T + cost * hkv * len(n_seq)
    C = min(grid, T)
    ranges = []
    for c in range(grid):
        if c >= C:
            ranges.append((0, 0))
            continue
        x0 = gqa_tile_of_position(cum, hkv, c * Tw // C, cost)
        x1 = T if c + 1 == C else gqa_tile_of_position(cum, hkv, (c + 1) * Tw // C, cost)
        ranges.append((x0, x1))
    return cum, T, Tw, C, ranges


def test_gqa_balanced_split_covers_every_tile_once_and_slots_match():
    rng = random.Random(99)
    for it in range(3000):
        batch = rng.randint(1, 24)
        hkv = rng.choice([1, 2, 4, 8])
        grid = rng.randint(1, 160)
        cost = GQA_UNIT_COST if it % 3 else rng.choice([0, 1, 5])
        n_seq = [max(1, rng.choice([1, 2, 3, rng.randint(1, 90)])) for _ in range(batch)]
        cum, T, Tw, C, ranges = gqa_plan(n_seq, hkv, grid, cost)
        units = [(b, h) for b in range(batch) for h in range(hkv)]
        ux = [cum[b] + h * n_seq[b] for b, h in units]         # first tile of each unit
        owner, pieces, published = {}, {}, {}
        for c in range(grid):
            x0, x1 = ranges[c]
            assert x0 <= x1
            for u, (b, h) in enumerate(units):
                tb, te = max(x0 - ux[u], 0), min(x1 - ux[u], n_seq[b])
                if tb >= te:
                    continue
                for t in range(tb, te):
                    assert (u, t) not in owner
                    owner[(u, t)] = c
                pieces.setdefault(u, []).append(c + u)           # the piece's slot
                if tb == 0:
                    # the CTA holding the first tile publishes the slot range
                    last = ux[u] + n_seq[b] - 1 + cost * (u + 1)
                    c_last = ((last + 1) * C - 1) // Tw
                    published[u] = (c + u, c_last - c + 1)
        assert len(owner) == T
        for u in range(len(units)):
            first, count = published[u]
            assert sorted(pieces[u]) == list(range(first, first + count))
        if T:
            wsizes = [(c + 1) * Tw // C - c * Tw // C for c in range(C)]
            assert max(wsizes) - min(wsizes) <= 1


def test_gqa_unit_cost_zero_is_the_equal_tile_split():
    rng = random.Random(5)
    for _ in range(300):
        n_seq = [rng.randint(1, 40) for _ in range(rng.randint(1, 16))]
        hkv, grid = rng.choice([1, 8]), rng.randint(1, 152)
        cum, T, Tw, C, ranges = gqa_plan(n_seq, hkv, grid, 0)
        for c in range(C):
            assert ranges[c] == (c * T // C, (c + 1) * T // C)


def decode_range(tiles, clusters, c, run_cost=RUN_COST, lanes=32):
    """The decode grid's own search for cluster c's range, restated: lane l
    sums the tiles and weighted tiles of its chunk of rows, a scan gives the
    chunk starts, and the lane whose weighted chunk holds the cluster's
    first (next cluster's first) position walks its rows to the real tile."""
    rows = len(tiles)
    per = (rows + lanes - 1) // lanes
    chunks = [range(min(l * per, rows), min(l * per + per, rows)) for l in range(lanes)]
    tl = [sum(tiles[r] for r in ch) for ch in chunks]
    wl = [sum(tiles[r] + run_cost for r in ch if tiles[r] > 0) for ch in chunks]
    T, Tw = sum(tl), sum(wl)
    C = min(clusters, T)
    if c >= C:
        return None

    def locate(y):
        cum0, w0 = 0, 0
        for l in range(lanes):
            if w0 <= y < w0 + wl[l]:
                cum, W = cum0, w0
                for r in chunks[l]:
                    n = tiles[r]
                    if n > 0 and y < W + run_cost + n:
                        return r, cum + min(max(y - W - run_cost, 0), n)
                    cum += n
                    W += n + run_cost if n > 0 else 0
            cum0 += tl[l]
            w0 += wl[l]
        raise AssertionError("position outside every chunk")

    r0, x0 = locate(c * Tw // C)
    x1 = T if c + 1 == C else locate((c + 1) * Tw // C)[1]
    return x0, x1, r0


def test_decode_grid_finds_the_plans_ranges():
    rng = random.Random(31)
    for it in range(1500):
        rows = rng.randint(1, 90)
        clusters = rng.randint(1, 80)
        run_cost = RUN_COST if it % 3 else rng.choice([0, 2, 11])
        tiles = [rng.choice([0, 1, 2, 5, rng.randint(0, 300)]) for _ in range(rows)]
        cum, total, wtotal, C, ranges, _ = plan(tiles, clusters, run_cost)
        for c in range(clusters):
            got = decode_range(tiles, clusters, c, run_cost)
            if c >= C:
                assert got is None
                continue
            x0, x1, r0 = got
            assert (x0, x1) == ranges[c][:2]
            # the walk from row r0 finds the same runs as from the plan's row
            mine = list(ranges)
            mine[c] = (x0, x1, r0)
            assert walk(cum, tiles, mine, c) == walk(cum, tiles, ranges, c)


def gqa_device_range(n_seq, hkv, grid, c, cost=GQA_UNIT_COST, lanes=32):
    """The GQA kernel's own search for CTA c's range, restated: lane l holds
    sequences [l m, (l+1) m) and their weighted positions (every sequence
    has hkv units of n + cost positions); the lane holding a range end walks
    its sequences to the unit and tile.  Returns (x0, x1, first unit, units)."""
    batch = len(n_seq)
    per = (batch + lanes - 1) // lanes
    T = sum(n * hkv for n in n_seq)
    Tw = T + cost * hkv * batch
    C = min(grid, T)
    if c >= C:
        return 0, 0, 0, 0

    def locate(y):
        xs, ws = 0, 0
        for l in range(lanes):
            seqs = range(min(l * per, batch), min(l * per + per, batch))
            w_lo = ws
            w_hi = ws + sum(hkv * (n_seq[b] + cost) for b in seqs)
            if w_lo <= y < w_hi:
                for b in seqs:
                    n = n_seq[b]
                    span = hkv * (n + cost)
                    if y < ws + span:
                        off = y - ws
                        h = off // (n + cost)
                        o = off - h * (n + cost) - cost
                        return xs + h * n + min(max(o, 0), n), b * hkv + h, o <= 0
                    xs += hkv * n
                    ws += span
                raise AssertionError("position not in the lane's sequences")
            xs += sum(hkv * n_seq[b] for b in seqs)
            ws = w_hi
        raise AssertionError("position outside every chunk")

    x0, u0, _ = locate(c * Tw // C)
    if c + 1 == C:
        x1, u_last = T, batch * hkv - 1
    else:
        x1, u1, f1 = locate((c + 1) * Tw // C)
        u_last = u1 - 1 if f1 else u1
    return x0, x1, u0, (u_last - u0 + 1 if x1 > x0 else 0)


def test_gqa_kernel_search_matches_the_split():
    rng = random.Random(77)
    for it in range(1500):
        batch = rng.randint(1, 80)
        hkv = rng.choice([1, 2, 8])
        grid = rng.randint(1, 160)
        cost = GQA_UNIT_COST if it % 3 else rng.choice([0, 1, 4])
        n_seq = [max(1, rng.choice([1, 2, rng.randint(1, 60)])) for _ in range(batch)]
        cum, T, Tw, C, ranges = gqa_plan(n_seq, hkv, grid, cost)
        ux = [cum[b] + h * n_seq[b] for b in range(batch) for h in range(hkv)]
        for c in range(grid):
            x0, x1, u0, count = gqa_device_range(n_seq, hkv, grid, c, cost)
            assert (x0, x1) == ranges[c]
            met = [u for u in range(batch * hkv)
                   if max(x0, ux[u]) < min(x1, ux[u] + n_seq[u // hkv])]
            assert count == len(met)
            if met:
                assert u0 == met[0] and met == list(range(u0, u0 + count))
