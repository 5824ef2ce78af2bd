"""The launch schedule (which CTA runs which unit and key-tile range), computed on
the host through the library's test hook; no GPU needed.

Every (unit, key tile) pair must be covered exactly once; the pieces of a tail
unit must partition its key tiles in piece order; workspace slots and arrival
counters must stay inside what the library allocates (2 x SMs of each); the
tail must be shared out evenly."""
import collections

import numpy as np
import pytest

import non_causal_prefix_gb300 as ncp

MAX_PIECES = 8       # pieces one merge reads, plus one for a range boundary
MIN_PIECE_TILES = 4  # least key tiles per tail CTA

CASES = [
    # B, Nq, H, key tiles, SMs, masked
    (1, 4096, 32, 32, 152, False),    # dense N=4096
    (2, 8192, 32, 64, 152, False),    # dense B=2 N=8192
    (1, 4096, 32, 40, 152, False),    # prefix 1024 + 4096
    (1, 32768, 32, 256, 152, False),  # dense N=32768
    (1, 128, 32, 1, 152, False),      # dense N=128
    (1, 256, 32, 256, 152, False),    # cross Nq=256, Nk=32768
    (1, 8192, 32, 4, 152, False),     # cross Nq=8192, Nk=512
    (1, 1000, 4, 8, 152, False),      # ragged: 16 units on 152 SMs
    (3, 777, 5, 13, 7, False),
    (1, 300, 1, 300, 148, False),     # one long unit and a ragged partner
    (2, 4096, 3, 17, 160, False),
    (1, 4448, 32, 35, 152, True),     # block-causal: never split
    (1, 4096, 32, 40, 152, True),     # masked prefix-cached
    (2, 640, 3, 9, 13, True),
]


def sched(B, Nq, H, T, sms, masked):
    rows, grid, slots = ncp.debug_schedule(B, Nq, H, T, sms, masked)
    return rows, grid, slots


@pytest.fixture(scope="module", autouse=True)
def built():
    ncp.build(quiet=True)


@pytest.mark.parametrize("B,Nq,H,T,sms,masked", CASES)
def test_schedule_covers_every_unit_tile_once(B, Nq, H, T, sms, masked):
    rows, grid, slots = sched(B, Nq, H, T, sms, masked)
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


@pytest.mark.parametrize("B,Nq,H,T,sms,masked", CASES)
def test_items_are_numbered_per_cta(B, Nq, H, T, sms, masked):
    rows, grid, _ = sched(B, Nq, H, T, sms, masked)
    per_cta = collections.defaultdict(list)
    for r in rows:
        per_cta[int(r[0])].append(int(r[1]))
    for cta, ns in per_cta.items():
        assert ns == list(range(len(ns)))


@pytest.mark.parametrize("B,Nq,H,T,sms,masked", CASES)
def test_tail_pieces_partition_their_unit(B, Nq, H, T, sms, masked):
    rows, grid, slots = sched(B, Nq, H, T, sms, masked)
    tail = rows[rows[:, 8] >= 0]
    whole = rows[rows[:, 8] < 0]
    assert (whole[:, 6] == 0).all() and (whole[:, 7] == T).all() and (whole[:, 10] == 1).all()
    if masked:
        assert len(tail) == 0
        return
    assert slots <= 2 * sms - 1  # the library allocates 2 x SMs slots
    used_slots = set()
    by_unit = collections.defaultdict(list)
    for r in tail:
        by_unit[int(r[8])].append(r)
    assert sorted(by_unit) == list(range(len(by_unit)))
    assert 2 * len(by_unit) <= 2 * sms  # arrival counters
    for t_unit, items in by_unit.items():
        items.sort(key=lambda r: r[9])
        pieces = int(items[0][10])
        assert 2 <= pieces <= MAX_PIECES + 1
        assert [int(r[9]) for r in items] == list(range(pieces))
        assert len({(int(r[2]), int(r[3]), int(r[4])) for r in items}) == 1
        assert len({int(r[11]) for r in items}) == 1
        assert items[0][6] == 0 and items[-1][7] == T
        for a, b in zip(items, items[1:]):
            assert a[7] == b[6]  # contiguous, in piece order
            assert b[0] == a[0] + 1  # consecutive CTAs
        for r in items:
            slot = int(r[11]) + int(r[9])
            assert 0 <= slot < slots and slot not in used_slots
            used_slots.add(slot)


@pytest.mark.parametrize("B,Nq,H,T,sms,masked", CASES)
def test_work_is_balanced(B, Nq, H, T, sms, masked):
    rows, grid, _ = sched(B, Nq, H, T, sms, masked)
    q_pairs = -(-Nq // 256)
    n_units = B * H * q_pairs
    work = np.zeros(grid, dtype=np.int64)
    for r in rows:
        work[r[0]] += r[7] - r[6]
    rounds = n_units // sms
    rem = n_units % sms
    if masked or rem == 0:
        assert work.max() == T * -(-n_units // grid)
        return
    tail_ctas = min(sms, rem * T // MIN_PIECE_TILES, rem * MAX_PIECES)
    if tail_ctas <= rem:  # not worth splitting: the last round runs whole units
        assert work.max() == T * (rounds + 1)
        return
    share = work - rounds * T
    share = share[share > 0]
    assert len(share) == tail_ctas
    assert share.max() - share.min() <= 1
    assert share.max() == -(-(rem * T) // tail_ctas)


def test_masked_forms_deal_a_snake():
    B, Nq, H, T, sms = 1, 4448, 32, 35, 152
    rows, grid, _ = sched(B, Nq, H, T, sms, True)
    q_pairs = -(-Nq // 256)
    n_bh = B * H
    for cta, n, b, h, q0, *_ in rows:
        unit = n * grid + (grid - 1 - cta if n % 2 else cta)
        # longest first: last query pair over all heads, then the one before
        assert q0 // 256 == q_pairs - 1 - unit // n_bh
        assert b * H + h == unit % n_bh
