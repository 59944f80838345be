"""The decode split plans' index arithmetic, restated on the host and checked
by brute force (no GPU).  The kernels' own arithmetic is exercised by the
GPU parity tests; this pins the plans' invariants on many more batches than
a GPU run can afford.

Balanced plan (ragged batches): per KV head the batch's attended page
counts are laid end to end (prefix sums P_b), cut into N = min(B * S, T)
slots [floor(s T / N), floor((s + 1) T / N)); a slot's part inside sequence
b is a segment whose partial sits at id s + b; the combine reads, for
sequence b, ids slot_of(P_b) + b .. slot_of(P_{b+1} - 1) + b with
slot_of(x) = ceil((x + 1) N / T) - 1.  Checked: every id the combine reads
was written exactly once, ids stay below B * S + B - 1 (the workspace
block), every page of every sequence is covered once, and no slot holds
more than ceil(T / N) pages (the balance the plan exists for).

Per-sequence plan: S near-equal ranges of ceil(pages / S) pages per
sequence cover its pages exactly once."""
import random

import pytest


def balanced_segments(pages, S):
    B = len(pages)
    incl, t = [], 0
    for p in pages:
        t += p
        incl.append(t)
    T = t
    N = min(B * S, T)
    segs = []
    for slot in range(B * S):
        if slot >= N:
            continue
        pos, end = slot * T // N, (slot + 1) * T // N
        b = sum(1 for x in incl if x <= pos)
        while pos < end and b < B:
            if incl[b] <= pos:
                b += 1
                continue
            start = incl[b] - pages[b]
            stop = min(end, incl[b])
            segs.append(dict(slot=slot, b=b, k=slot + b, first=pos - start, n=stop - pos))
            pos = stop
            if stop == incl[b]:
                b += 1
    return segs, incl, T, N


def combine_range(b, pages, incl, T, N):
    if pages[b] == 0:
        return []

    def slot_of(x):
        return -(-((x + 1) * N) // T) - 1

    return list(range(slot_of(incl[b] - pages[b]) + b, slot_of(incl[b] - 1) + b + 1))


def check_balanced(pages, S):
    segs, incl, T, N = balanced_segments(pages, S)
    B = len(pages)
    ids = [(s["b"], s["k"]) for s in segs]
    assert len(ids) == len(set(ids)), "a segment id written twice"
    assert all(0 <= k < B * S + B - 1 for _, k in ids)
    slot_pages = {}
    for s in segs:
        slot_pages[s["slot"]] = slot_pages.get(s["slot"], 0) + s["n"]
    if T:
        assert max(slot_pages.values()) <= -(-T // N)
    for b in range(B):
        mine = sorted((s for s in segs if s["b"] == b), key=lambda s: s["first"])
        assert [s["k"] for s in mine] == combine_range(b, pages, incl, T, N)
        x = 0
        for s in mine:
            assert s["first"] == x and s["n"] > 0
            x += s["n"]
        assert x == pages[b]


def test_balanced_plan_worked_example():
    # 3 sequences of 5, 0 and 3 pages, S = 2: T = 8 pages over N = 6 slots
    pages = [5, 0, 3]
    segs, incl, T, N = balanced_segments(pages, 2)
    assert (T, N) == (8, 6)
    got = [(s["slot"], s["b"], s["first"], s["n"]) for s in segs]
    # slot bounds floor(8 s / 6): 0, 1, 2, 4, 5, 6, 8
    assert got == [(0, 0, 0, 1), (1, 0, 1, 1), (2, 0, 2, 2), (3, 0, 4, 1), (4, 2, 0, 1), (5, 2, 1, 2)]
    assert combine_range(0, pages, incl, T, N) == [0, 1, 2, 3]
    assert combine_range(1, pages, incl, T, N) == []
    assert combine_range(2, pages, incl, T, N) == [6, 7]


@pytest.mark.parametrize("seed", range(4))
def test_balanced_plan_random_batches(seed):
    rng = random.Random(seed)
    for _ in range(2500):
        B = rng.randint(2, 32)
        S = rng.randint(2, 24)
        pages = [rng.choice([0, 0, 1, 2, 3, rng.randint(0, 60), rng.randint(0, 4000)]) for _ in range(B)]
        check_balanced(pages, S)


def test_balanced_plan_fewer_pages_than_slots():
    for pages in ([1, 0, 0, 1], [0, 3], [1] * 32, [0] * 31 + [2]):
        for S in (2, 7, 57):
            check_balanced(pages, S)


def test_per_sequence_plan_covers_each_page_once():
    for L in range(0, 700, 7):
        for S in (1, 2, 3, 7, 57):
            last = (L + 15) // 16
            pps = (last + S - 1) // S if last else 0
            covered = []
            for split in range(S):
                pg0 = split * pps
                pg1 = min(pg0 + pps, last)
                covered += list(range(pg0, pg1)) if pg1 > pg0 else []
            assert covered == list(range(last))
