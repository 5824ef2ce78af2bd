"""The launch schedule (which CTA runs which unit and key-tile range), computed on
the host through the library's test hook; no GPU needed.

Every (unit, key tile) pair must be covered exactly once (masked forms: every
tile some row of the unit sees, found by brute force over the id vector); the
pieces of a tail unit must split its tiles in piece order; workspace slots and
arrival counters must stay inside what the library allocates (2 x SMs of
each); the tail must be shared out evenly."""
import collections

import numpy as np
import pytest

import non_causal_prefix_gb300 as ncp

MAX_PIECES = 8       # pieces one merge reads, plus one for a range boundary
MIN_PIECE_TILES = 4  # least key tiles per tail CTA
UNIT_COST = 3        # masked tails: item cost per tail unit, in visited key tiles

CASES = [
    # B, Nq, H, key tiles, SMs
    (1, 4096, 32, 32, 152),    # dense N=4096
    (2, 8192, 32, 64, 152),    # dense B=2 N=8192
    (1, 4096, 32, 40, 152),    # prefix 1024 + 4096
    (1, 32768, 32, 256, 152),  # dense N=32768
    (1, 128, 32, 1, 152),      # dense N=128
    (1, 256, 32, 256, 152),    # cross Nq=256, Nk=32768
    (1, 8192, 32, 4, 152),     # cross Nq=8192, Nk=512
    (1, 1000, 4, 8, 152),      # ragged: 16 units on 152 SMs
    (3, 777, 5, 13, 7),
    (1, 300, 1, 300, 148),     # one long unit and a ragged partner
    (2, 4096, 3, 17, 160),
]

# Masked forms: B, Nq, H, Np, id segments over the Np + Nq positions, SMs.
MASKED = [
    (1, 4448, 32, 0, ((-1, 333), (0, 2048), (-1, 19), (1, 2048)), 152),  # block-causal
    (1, 4096, 32, 1024, ((-1, 256), (0, 768), (1, 4096)), 152),          # masked prefix
    (2, 640, 3, 512, ((-1, 100), (3, 300), (-1, 500), (7, 252)), 13),
    (1, 3000, 4, 0, ((-1, 3000),), 40),                                   # causal text only
    (1, 1500, 2, 300, ((5, 1800),), 11),                                  # one image
    (3, 700, 2, 77, ((-1, 1), (2, 200), (-1, 300), (2, 276)), 9),         # ragged, repeated id
]


def masked_ids(Np, Nq, segments):
    ids = np.concatenate([np.full(n, k, dtype=np.int32) for k, n in segments])
    assert ids.size == Np + Nq
    return ids


def sched(B, Nq, H, T, sms):
    return ncp.debug_schedule(B, Nq, H, T, sms, False)


def masked_sched(B, Nq, H, Np, segments, sms):
    ids = masked_ids(Np, Nq, segments)
    return ncp.debug_schedule(B, Nq, H, 0, sms, True, ids, Np), ids


@pytest.fixture(scope="module", autouse=True)
def built():
    ncp.build(quiet=True)


@pytest.mark.parametrize("B,Nq,H,T,sms", CASES)
def test_schedule_covers_every_unit_tile_once(B, Nq, H, T, sms):
    rows, grid, slots = sched(B, Nq, H, T, sms)
    q_pairs = -(-Nq // 256)
    n_units = B * H * q_pairs
    assert 1 <= grid <= sms
    seen = np.zeros((n_units, T), dtype=np.int32)
    for cta, n, b, h, q0, two, tb, te, tail, piece, pieces, slot0 in rows:
        assert 0 <= cta < grid and 0 <= b < B and 0 <= h < H and q0 % 256 == 0 and q0 < Nq
        assert two == (q0 + 128 < Nq)
        assert 0 <= tb < te <= T
        unit = (b * H + h) * q_pairs + q0 // 256
        seen[unit, tb:te] += 1
    assert (seen == 1).all()


def needed_tiles(ids, Np, Nq, q0):
    """Key tiles (prefix tiles, then current ones) that some query row of the
    unit at q0 sees, by brute force over every (row, key) pair."""
    T0, T1 = -(-Np // 128), -(-Nq // 128)
    pos = np.arange(Np + Nq)
    rows = np.arange(q0, min(q0 + 256, Nq)) + Np
    vis = (pos[None, :] <= rows[:, None]) | (
        (ids[None, pos] >= 0) & (ids[None, pos] == ids[rows][:, None]))
    key_tile = np.where(pos < Np, pos // 128, T0 + (pos - Np) // 128)
    need = np.zeros(T0 + T1, dtype=bool)
    need[np.unique(key_tile[vis.any(axis=0)])] = True
    return need


@pytest.mark.parametrize("B,Nq,H,Np,segments,sms", MASKED)
def test_masked_schedule_covers_every_needed_tile_once(B, Nq, H, Np, segments, sms):
    check_masked_cover(B, Nq, H, Np, segments, sms)


def check_masked_cover(B, Nq, H, Np, segments, sms):
    (rows, grid, slots), ids = masked_sched(B, Nq, H, Np, segments, sms)
    T = -(-Np // 128) + -(-Nq // 128)
    q_pairs = -(-Nq // 256)
    assert 1 <= grid <= sms
    cover = collections.defaultdict(lambda: np.zeros(T, dtype=np.int32))
    for cta, n, b, h, q0, two, tb, te, tail, piece, pieces, slot0 in rows:
        assert 0 <= cta < grid and 0 <= b < B and 0 <= h < H and q0 % 256 == 0 and q0 < Nq
        assert 0 <= tb < te <= T
        cover[(b, h, q0)][tb:te] += 1
    assert len(cover) == B * H * q_pairs
    for (b, h, q0), c in cover.items():
        need = needed_tiles(ids, Np, Nq, q0)
        assert (c[need] == 1).all(), (b, h, q0)
        assert c.max() <= 1  # item ranges of one unit never overlap


def check_items_numbered(rows):
    per_cta = collections.defaultdict(list)
    for r in rows:
        per_cta[int(r[0])].append(int(r[1]))
    for cta, ns in per_cta.items():
        assert ns == list(range(len(ns)))


def check_tail(rows, grid, slots, T, sms):
    tail = rows[rows[:, 8] >= 0]
    whole = rows[rows[:, 8] < 0]
    assert (whole[:, 10] == 1).all()
    assert slots <= 2 * sms - 1  # the library allocates 2 x SMs slots
    used_slots = set()
    by_unit = collections.defaultdict(list)
    for r in tail:
        by_unit[int(r[8])].append(r)
    assert 2 * len(by_unit) <= 2 * sms  # arrival counters (2 per tail unit)
    for t_unit, items in by_unit.items():
        items.sort(key=lambda r: r[9])
        pieces = int(items[0][10])
        assert pieces >= 2
        assert [int(r[9]) for r in items] == list(range(pieces))
        assert len({(int(r[2]), int(r[3]), int(r[4])) for r in items}) == 1
        assert len({int(r[11]) for r in items}) == 1
        for a, b in zip(items, items[1:]):
            assert a[7] <= b[6]  # disjoint, in piece order
            assert b[0] == a[0] + 1  # consecutive CTAs
        for r in items:
            slot = int(r[11]) + int(r[9])
            assert 0 <= slot < max(slots, 1) and slot not in used_slots
            used_slots.add(slot)


@pytest.mark.parametrize("B,Nq,H,T,sms", CASES)
def test_items_are_numbered_per_cta(B, Nq, H, T, sms):
    check_items_numbered(sched(B, Nq, H, T, sms)[0])


@pytest.mark.parametrize("B,Nq,H,Np,segments,sms", MASKED)
def test_masked_items_are_numbered_per_cta(B, Nq, H, Np, segments, sms):
    check_items_numbered(masked_sched(B, Nq, H, Np, segments, sms)[0][0])


@pytest.mark.parametrize("B,Nq,H,T,sms", CASES)
def test_tail_pieces_partition_their_unit(B, Nq, H, T, sms):
    rows, grid, slots = sched(B, Nq, H, T, sms)
    check_tail(rows, grid, slots, T, sms)
    whole = rows[rows[:, 8] < 0]
    assert (whole[:, 6] == 0).all() and (whole[:, 7] == T).all()
    tail = rows[rows[:, 8] >= 0]
    for t_unit in set(tail[:, 8].tolist()):
        items = sorted(tail[tail[:, 8] == t_unit].tolist(), key=lambda r: r[9])
        assert items[0][6] == 0 and items[-1][7] == T
        assert all(a[7] == b[6] for a, b in zip(items, items[1:]))  # contiguous


@pytest.mark.parametrize("B,Nq,H,Np,segments,sms", MASKED)
def test_masked_tail_pieces(B, Nq, H, Np, segments, sms):
    (rows, grid, slots), _ = masked_sched(B, Nq, H, Np, segments, sms)
    T = -(-Np // 128) + -(-Nq // 128)
    check_tail(rows, grid, slots, T, sms)


PIECE_COST = 3  # the library's cost of an extra tail piece on a CTA, in key-tile times


def cta_costs(rows, T):
    """Per tail CTA: its tail tiles plus PIECE_COST for each tail item after
    its first."""
    tail = rows[rows[:, 8] >= 0]
    costs = {}
    for c in set(tail[:, 0].tolist()):
        mine = tail[tail[:, 0] == c]
        costs[c] = int((mine[:, 7] - mine[:, 6]).sum()) + PIECE_COST * (len(mine) - 1)
    return costs


def equal_range_cost(W, T, G):
    """The largest per-CTA cost of G equal ranges over W tail tiles."""
    worst = 0
    for c in range(G):
        lo, hi = c * W // G, (c + 1) * W // G
        if lo < hi:
            worst = max(worst, hi - lo + PIECE_COST * ((hi - 1) // T - lo // T))
    return worst


@pytest.mark.parametrize("B,Nq,H,T,sms", CASES)
def test_work_is_balanced(B, Nq, H, T, sms):
    rows, grid, _ = sched(B, Nq, H, T, sms)
    q_pairs = -(-Nq // 256)
    n_units = B * H * q_pairs
    work = np.zeros(grid, dtype=np.int64)
    for r in rows:
        work[r[0]] += r[7] - r[6]
    rounds = n_units // sms
    rem = n_units % sms
    if rem == 0:
        assert work.max() == T * -(-n_units // grid)
        return
    g_max = min(sms, rem * T // MIN_PIECE_TILES, rem * MAX_PIECES)
    tail = rows[rows[:, 8] >= 0]
    if g_max <= rem:  # not worth splitting: the last round runs whole units
        assert len(tail) == 0 and work.max() == T * (rounds + 1)
        return
    costs = cta_costs(rows, T)
    assert rem < len(costs) <= g_max
    # Every tail CTA works; the weighted ranges are no worse than equal ones,
    # and within one piece's cost of each other.
    assert all(v > 0 for v in costs.values())
    assert max(costs.values()) <= equal_range_cost(rem * T, T, g_max)
    assert max(costs.values()) - min(costs.values()) <= PIECE_COST + T


def test_masked_prefix_tail_is_shared_out():
    """Masked prefix workload (every unit visits all 40 tiles): 512 units on
    152 SMs leave 56 for the last round; their tiles go to every SM, and a CTA
    whose range crosses into a second unit (two tail items) pays that unit's
    UNIT_COST: it holds that many fewer tiles than the fullest one-item CTA."""
    (rows, grid, slots), _ = masked_sched(1, 4096, 32, 1024, ((-1, 256), (0, 768), (1, 4096)), 152)
    assert grid == 152
    rounds = 512 // 152
    tiles = np.zeros(grid, dtype=np.int64)
    items = np.zeros(grid, dtype=np.int64)
    for r in rows:
        if r[1] >= rounds:
            tiles[r[0]] += r[7] - r[6]
            items[r[0]] += 1
    assert tiles.sum() == 56 * 40 and (items >= 1).all()
    per_cta = 56 * (40 + UNIT_COST) / 152
    cost = tiles + UNIT_COST * (items - 1)
    assert cost.max() <= np.ceil(per_cta) and cost.min() >= np.floor(per_cta) - UNIT_COST
    assert tiles[items == 2].max() + UNIT_COST <= tiles[items == 1].max() + 1


def visited_tiles(ids, Np, Nq, q):
    """Key tiles the unit of query pair q visits, in order (the kernel's skip
    rule, as in visited_per_pair)."""
    T0, T1 = -(-Np // 128), -(-Nq // 128)
    pos0 = [t * 128 if t < T0 else Np + (t - T0) * 128 for t in range(T0 + T1)]
    ln = [min(128, (Np if t < T0 else Nq) - (t if t < T0 else t - T0) * 128) for t in range(T0 + T1)]
    lo, hi = [], []
    for t in range(T0 + T1):
        seg = ids[pos0[t]:pos0[t] + ln[t]]
        img = seg[seg >= 0]
        lo.append(int(img.min()) if img.size else 2**31 - 1)
        hi.append(int(img.max()) if img.size else -1)
    r_last = Np + min(q * 256 + 256, Nq) - 1
    qt0 = T0 + 2 * q
    qt1 = qt0 + 1 if q * 256 + 128 < Nq else qt0
    qlo, qhi = min(lo[qt0], lo[qt1]), max(hi[qt0], hi[qt1])
    return [t for t in range(T0 + T1) if pos0[t] <= r_last or (qlo <= hi[t] and lo[t] <= qhi)]


def visited_per_pair(ids, Np, Nq):
    """Key tiles each query pair's unit visits (the kernel's skip rule, restated:
    a tile is visited when it starts at or before the pair's last row, or when
    its image ids' range meets the pair's)."""
    T0, T1 = -(-Np // 128), -(-Nq // 128)
    pos0 = [t * 128 if t < T0 else Np + (t - T0) * 128 for t in range(T0 + T1)]
    ln = [min(128, (Np if t < T0 else Nq) - (t if t < T0 else t - T0) * 128) for t in range(T0 + T1)]
    lo, hi = [], []
    for t in range(T0 + T1):
        seg = ids[pos0[t]:pos0[t] + ln[t]]
        img = seg[seg >= 0]
        lo.append(int(img.min()) if img.size else 2**31 - 1)
        hi.append(int(img.max()) if img.size else -1)
    counts = []
    for q in range(-(-Nq // 256)):
        r_last = Np + min(q * 256 + 256, Nq) - 1
        qt0 = T0 + 2 * q
        qt1 = qt0 + 1 if q * 256 + 128 < Nq else qt0
        qlo, qhi = min(lo[qt0], lo[qt1]), max(hi[qt0], hi[qt1])
        counts.append(sum(1 for t in range(T0 + T1)
                          if pos0[t] <= r_last or (qlo <= hi[t] and lo[t] <= qhi)))
    return counts


def pair_costs(ids, Np, Nq):
    """Cost of each query pair's unit, restated: per visited key tile, 26 when
    the pair has two query tiles and 22 when it has one, plus 6 for each of its
    query tiles that sees only part of the key tile.  A query tile sees all of
    a key tile when the tile's last key is at or before the query tile's first
    position, or when both tiles hold one and the same image (no text)."""
    T0, T1 = -(-Np // 128), -(-Nq // 128)
    pos0 = [t * 128 if t < T0 else Np + (t - T0) * 128 for t in range(T0 + T1)]
    ln = [min(128, (Np if t < T0 else Nq) - (t if t < T0 else t - T0) * 128) for t in range(T0 + T1)]
    one_image = []
    for t in range(T0 + T1):
        seg = ids[pos0[t]:pos0[t] + ln[t]]
        one_image.append(int(seg[0]) if (seg >= 0).all() and (seg == seg[0]).all() else None)
    costs = []
    for q in range(-(-Nq // 256)):
        two = q * 256 + 128 < Nq
        c = 0
        for t in visited_tiles(ids, Np, Nq, q):
            c += 26 if two else 22
            for qt in range(2 if two else 1):
                first = Np + q * 256 + qt * 128
                tq = T0 + 2 * q + qt
                full = (pos0[t] + ln[t] - 1 <= first or
                        (one_image[tq] is not None and one_image[tq] == one_image[t]))
                c += 0 if full else 6
        costs.append(c)
    return costs


@pytest.mark.parametrize("B,Nq,H,Np,segments,sms", MASKED)
def test_masked_forms_deal_a_snake(B, Nq, H, Np, segments, sms):
    """Whole masked units: query pairs sorted by their cost (pair_costs; most
    first, the later pair first among equals); units level by level, head-major
    with the query pair fastest within a level; dealt in a snake."""
    (rows, grid, _), ids = masked_sched(B, Nq, H, Np, segments, sms)
    cnt = pair_costs(ids, Np, Nq)
    q_pairs = len(cnt)
    n_bh = B * H
    order = sorted(range(q_pairs), key=lambda q: (-cnt[q], -q))
    levels = [r for r in range(q_pairs) if r == 0 or cnt[order[r]] != cnt[order[r - 1]]]
    levels.append(q_pairs)
    whole_rounds = (n_bh * q_pairs) // grid
    for cta, n, b, h, q0, *_ in rows:
        if n >= whole_rounds:
            continue
        unit = n * grid + (grid - 1 - cta if n % 2 else cta)
        lv = max(i for i in range(len(levels) - 1) if levels[i] * n_bh <= unit)
        size = levels[lv + 1] - levels[lv]
        w = unit - levels[lv] * n_bh
        assert b * H + h == w // size
        assert q0 // 256 == order[levels[lv] + w % size]
    # Units of whole rounds come in non-increasing work.
    units = sorted((n * grid + (grid - 1 - cta if n % 2 else cta), q0 // 256)
                   for cta, n, b, h, q0, *_ in rows if n < whole_rounds)
    work = [cnt[q] for _, q in units]
    assert all(a >= b for a, b in zip(work, work[1:]))


@pytest.mark.parametrize("B,Nq,H,Np,segments,sms", MASKED)
def test_masked_tail_layout(B, Nq, H, Np, segments, sms):
    """The masked tail, restated: tail units in unit order, each worth
    UNIT_COST positions and then one per visited key tile; CTA c of G holds
    positions [c W / G, (c + 1) W / G) and one item per unit whose tiles meet
    that range, with the visited tiles that fall in it."""
    check_masked_tail_layout(B, Nq, H, Np, segments, sms)


def random_masked_case(seed):
    """A seeded masked shape: text and image segments over Np + Nq positions
    (ids -1..3, repeats allowed), a head count that leaves a partial last
    round, and an SM count from 8 to 160."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    Nq = int(rng.integers(100, 3000))
    Np = int(rng.integers(0, 2)) * int(rng.integers(1, 900))
    sms = int(rng.integers(8, 161))
    q_pairs = -(-Nq // 256)
    H = max(1, int(sms * rng.integers(1, 4) + rng.integers(1, sms)) // (B * q_pairs))
    n, pos, segs = Np + Nq, 0, []
    while pos < n:
        L = min(int(rng.integers(1, 700)), n - pos)
        segs.append((int(rng.integers(-1, 4)) if rng.random() < 0.7 else -1, L))
        pos += L
    return B, Nq, H, Np, tuple(segs), sms


@pytest.mark.parametrize("seed", range(12))
def test_masked_random_shapes(seed):
    """Coverage of every needed tile and the exact tail layout on seeded
    random masked shapes."""
    case = random_masked_case(4100 + seed)
    check_masked_cover(*case)
    check_masked_tail_layout(*case)


def check_masked_tail_layout(B, Nq, H, Np, segments, sms):
    (rows, grid, _), ids = masked_sched(B, Nq, H, Np, segments, sms)
    cnt = visited_per_pair(ids, Np, Nq)
    q_pairs, n_bh = len(cnt), B * H
    n_units = n_bh * q_pairs
    rem = n_units % grid if grid == sms else 0
    T = -(-Np // 128) + -(-Nq // 128)
    g_tail = min(sms, rem * T // MIN_PIECE_TILES, rem * MAX_PIECES)
    tail_rows = [r for r in rows if r[1] >= n_units // grid] if rem and g_tail > rem else []
    if not tail_rows:
        return
    cost = pair_costs(ids, Np, Nq)
    order = sorted(range(q_pairs), key=lambda q: (-cost[q], -q))
    levels = [r for r in range(q_pairs) if r == 0 or cost[order[r]] != cost[order[r - 1]]]
    levels.append(q_pairs)

    def unit_pair(u):
        lv = max(i for i in range(len(levels) - 1) if levels[i] * n_bh <= u)
        size = levels[lv + 1] - levels[lv]
        w = u - levels[lv] * n_bh
        return w // size, order[levels[lv] + w % size]

    tail = [unit_pair(u) for u in range(n_units - rem, n_units)]
    vis = [cnt[q] for _, q in tail]
    pos = np.concatenate([[0], np.cumsum(np.array(vis) + UNIT_COST)])
    W, G = int(pos[-1]), max(1, min(sum(vis) // MIN_PIECE_TILES, g_tail))
    expect = collections.defaultdict(list)
    for c in range(G):
        lo, hi = c * W // G, (c + 1) * W // G
        for r, (bh, q) in enumerate(tail):
            u0, u1 = pos[r] + UNIT_COST, pos[r + 1]
            if max(lo, u0) < min(hi, u1):
                expect[c].append((bh, q, max(lo, u0) - u0, min(hi, u1) - u0))
    # Visited tiles of a pair, in order (the kernel's skip rule), to turn an
    # item's tile range into visited indices.
    T0 = -(-Np // 128)
    got = collections.defaultdict(list)
    for cta, n, b, h, q0, two, tb, te, *_ in sorted(tail_rows, key=lambda r: (r[0], r[1])):
        q = q0 // 256
        seen = visited_tiles(ids, Np, Nq, q)
        v0 = seen.index(tb)
        v1 = seen.index(te - 1) + 1
        got[cta].append((b * H + h, q, v0, v1))
    assert dict(got) == dict(expect)


def random_dense_case(seed):
    """A seeded dense shape: units a little past a multiple of the SM count
    (or below it), any number of key tiles, 4 to 200 SMs."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    Nq = int(rng.integers(1, 9000))
    T = int(rng.integers(1, 300))
    sms = int(rng.integers(4, 201))
    q_pairs = -(-Nq // 256)
    target = sms * int(rng.integers(0, 4)) + int(rng.integers(1, sms + 1))
    H = max(1, target // (B * q_pairs))
    return B, Nq, H, T, sms


@pytest.mark.parametrize("seed", range(16))
def test_dense_random_shapes(seed):
    """Coverage, item numbering, tail pieces and balance on seeded random
    dense shapes."""
    case = random_dense_case(5200 + seed)
    test_schedule_covers_every_unit_tile_once(*case)
    test_items_are_numbered_per_cta(*case)
    test_tail_pieces_partition_their_unit(*case)
    test_work_is_balanced(*case)


def test_block_causal_tail_items_stay_few():
    """Block-causal N=4448 (text 333, image 2048, text 19, image 2048) on 152
    SMs: its 120 tail units include many short ones.  With plain visited-tile
    ranges some CTAs took 7 items and ended last; the unit cost keeps every
    tail CTA at 3 items or fewer."""
    (rows, grid, _), _ = masked_sched(1, 4448, 32, 0, ((-1, 333), (0, 2048), (-1, 19), (1, 2048)),
                                      152)
    rounds = (32 * 18) // 152
    items = collections.Counter(int(r[0]) for r in rows if r[1] >= rounds)
    assert grid == 152 and max(items.values()) <= 3

