"""Properties of the split-KV plan arithmetic (host logic, CPU only).

The device planner cuts the concatenated page list of all sequences into
G_eff = min(G, max(1, P // 2)) contiguous splits, split c owning [floor(cP/G_eff),
floor((c+1)P/G_eff)), and gives split c's piece of sequence b the slot
slot_base[b] + c - first_split[b].  These integer formulas are restated
here and checked for coverage, balance, non-empty splits and slot bounds
over many length mixes.
"""
import numpy as np
import pytest


def plan(lens, page, G_max):
    pages = [(L + page - 1) // page for L in lens]
    prefix = np.concatenate([[0], np.cumsum(pages)]).astype(np.int64)
    P = int(prefix[-1])
    G = min(G_max, max(1, P // 2))

    def split_of(g):
        return ((g + 1) * G - 1) // P

    first = [split_of(prefix[b]) for b in range(len(lens))]
    last = [split_of(prefix[b + 1] - 1) for b in range(len(lens))]
    ns = [l - f + 1 for f, l in zip(first, last)]
    slot_base = np.concatenate([[0], np.cumsum(ns)]).astype(np.int64)
    return prefix, P, G, first, slot_base


def pieces(lens, page, G_max):
    prefix, P, G, first, slot_base = plan(lens, page, G_max)
    B = len(lens)
    out = []
    for c in range(G):
        g0, g1 = c * P // G, (c + 1) * P // G
        b = int(np.searchsorted(prefix, g0, side="right") - 1)
        while b < B and prefix[b] < g1:
            lo, hi = max(g0, prefix[b]), min(g1, prefix[b + 1])
            out.append((c, b, int(lo - prefix[b]), int(hi - prefix[b]),
                        int(slot_base[b] + c - first[b])))
            b += 1
    return out, P, G, slot_base


@pytest.mark.parametrize("seed", range(40))
def test_plan_covers_every_page_once_with_valid_slots(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    lens = [int(x) for x in rng.integers(1, 3000, B)]
    G_max = int(rng.integers(1, 300))
    out, P, G, slot_base = pieces(lens, 64, G_max)
    seen = {}
    for c, b, p0, p1, slot in out:
        assert p1 > p0, "empty piece"
        for p in range(p0, p1):
            assert (b, p) not in seen
            seen[(b, p)] = c
    assert len(seen) == P
    # every slot of sequence b is written exactly once, and slots are bounded
    slots = [s for *_, s in out]
    assert sorted(slots) == list(range(int(slot_base[-1])))
    assert slot_base[-1] <= G + B - 1
    # every split is non-empty and balanced to within one page
    sizes = [(c + 1) * P // G - c * P // G for c in range(G)]
    assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1


def test_more_splits_than_pages_is_clamped():
    out, P, G, slot_base = pieces([1, 1, 1, 65, 200, 1000], 64, 74)
    assert P == 25 and G == 12
    assert slot_base[-1] <= G + 6 - 1
    out, P, G, slot_base = pieces([1], 64, 74)
    assert P == 1 and G == 1
