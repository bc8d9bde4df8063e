"""CPU check of the balanced grouped-head schedule's bookkeeping.

The kernel lays the work items (sequence, KV head, row block) end to end as their
ceil(L/64) key tiles, gives CTA c the tiles [c*W, (c+1)*W) with W = ceil(total/grid),
writes cut items' pieces to partial record (item + c) and lets the CTA holding an
item's first tile store {first record, count}. This re-derives that bookkeeping in
Python and checks the properties the kernel and the combine rely on: every tile is
covered exactly once, record ids are unique and below items + grid (the workspace
size), and the meta entry of each item lists exactly the records written for it.
"""
import random

import pytest


def tiles_of(L):
    return (L + 63) // 64 if L > 0 else 0


def schedule(seqlens, ips, grid):
    """Pieces (cta, item, t0, t1, record or None) and meta {item: (first, count)}."""
    total = sum(tiles_of(L) for L in seqlens) * ips
    W = -(-total // grid) if total else 0
    pieces, meta = [], {}
    for c in range(grid):
        pos, end = c * W, min(total, (c + 1) * W)
        base = 0
        for i, L in enumerate(seqlens):
            nt = tiles_of(L)
            while nt and base <= pos < base + nt * ips and pos < end:
                item_local, t0 = divmod(pos - base, nt)
                t1 = min(nt, t0 + (end - pos))
                item = i * ips + item_local
                first = base + item_local * nt
                c0, c1 = first // W, (first + nt - 1) // W
                if t0 == 0:
                    meta[item] = (item + c0, c1 - c0 + 1)
                pieces.append((c, item, t0, t1, None if c0 == c1 else item + c))
                pos += t1 - t0
            base += nt * ips
    return total, pieces, meta


@pytest.mark.parametrize("trial", range(40))
def test_balanced_schedule_bookkeeping(trial):
    rng = random.Random(trial)
    b = rng.randint(1, 40)
    seqlens = [rng.choice([0, 1, 63, 64, 65, rng.randint(0, 5000)]) for _ in range(b)]
    ips = rng.choice([1, 2, 4, 8, 24])  # KV heads x row blocks per sequence
    grid = rng.choice([1, 7, 148, 296, 444])
    total, pieces, meta = schedule(seqlens, ips, grid)
    # every tile of every item exactly once
    seen = {}
    for _, item, t0, t1, _ in pieces:
        assert 0 <= t0 < t1
        for t in range(t0, t1):
            assert (item, t) not in seen
            seen[(item, t)] = True
    expect = sum(tiles_of(seqlens[item // ips]) for item in range(b * ips))
    assert len(seen) == expect == total
    # records unique, inside the workspace
    recs = [r for *_, r in pieces if r is not None]
    assert len(recs) == len(set(recs))
    assert all(0 <= r < b * ips + grid for r in recs)
    # meta: one entry per non-empty item, listing exactly its records
    for item in range(b * ips):
        nt = tiles_of(seqlens[item // ips])
        mine = sorted(r for _, it, _, _, r in pieces if it == item and r is not None)
        whole = [p for p in pieces if p[1] == item and p[4] is None]
        if nt == 0:
            assert item not in meta and not mine and not whole
            continue
        first, count = meta[item]
        if count == 1:
            assert len(whole) == 1 and whole[0][2:4] == (0, nt) and not mine
        else:
            assert mine == list(range(first, first + count)) and not whole
