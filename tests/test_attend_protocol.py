"""Model of the attention kernel's barrier protocol (CPU only).

The split-KV attention kernel runs five roles that meet only at mbarriers:
a TMA producer, a score-MMA issuer, a value-MMA issuer, the softmax warps
and (implicitly) the tensor pipe.  Every wait is a parity wait, which cannot
tell phase F from phase F + 2.  This file restates each role's loop (the
order of its waits and arrivals, nothing of the arithmetic) and drives the
roles in many interleavings over the split plans of the five workloads.  A
wait that passes while its barrier is not exactly at the awaited phase is a
failure, and so is a state where no role can move.

Copies, MMAs and commits complete as soon as they are issued: they never
wait on anything once issued, so this can only hide delays, not orderings.
The model follows the kernel's loops one for one; a change to the order of
waits or arrivals in the kernel must be made here too.
"""
from __future__ import annotations

import random

import pytest

from synth import workloads as W

RING, TILE, PAGE = 5, 128, 64


class Bar:
    def __init__(self, name: str, count: int = 1):
        self.name, self.count, self.pending, self.done = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.done += 1
            self.pending = self.count

    def ready(self, phase: int) -> bool:
        """Parity semantics of mbarrier.try_wait.parity for phase `phase`;
        raises if the parity test passes on the wrong phase."""
        ok = (self.done & 1) != (phase & 1)
        if ok and self.done != phase + 1:
            raise AssertionError(f"{self.name}: wait for phase {phase} passed at done={self.done}")
        return ok


class Ring:
    def __init__(self):
        self.s = self.n = 0

    def next(self):
        self.n += 1
        self.s = (self.s + 1) % RING

    def skip(self, m: int):
        for _ in range(m):
            self.next()


def ntiles(p0, p1):
    return (p1 - p0 + TILE - 1) // TILE if p1 > p0 else 0


def nslabs(ts, p1):
    v = p1 - ts
    return 4 if v >= TILE else (v + 31) // 32


def split_segments(seq_lens, T, t, G):
    """(sequence, first token, visible end) of each split, as the kernel's
    segment iterator yields them: splits cut the concatenated page list
    evenly, G_eff = min(G, max(1, pages // 2))."""
    pages = [(L + PAGE - 1) // PAGE for L in seq_lens]
    prefix = [0]
    for p in pages:
        prefix.append(prefix[-1] + p)
    P = prefix[-1]
    Geff = min(G, max(1, P // 2))
    out = []
    for c in range(Geff):
        g0, g1 = c * P // Geff, (c + 1) * P // Geff
        b = max(i for i in range(len(pages)) if prefix[i] <= g0)
        segs = []
        while b < len(pages) and prefix[b] < g1:
            lo, hi = max(g0, prefix[b]), min(g1, prefix[b + 1])
            vis = seq_lens[b] - T + t + 1
            segs.append((b, (lo - prefix[b]) * PAGE, min((hi - prefix[b]) * PAGE, vis)))
            b += 1
        out.append(segs)
    return out


def run_protocol(segs, rescale: bool, seed: int | None, guard: bool = True,
                 seg_guard: bool = True):
    """Returns None when every role finishes, else the blocked roles.
    `guard` = False drops the value-MMA role's wait for S(x+1), `seg_guard`
    = False the score-MMA role's wait for the previous segment's last PV.
    Issued copies complete in random order (a separate copy-engine role)."""
    rnd = random.Random(seed)
    pending = []
    full = [Bar(f"full{i}") for i in range(RING)]
    empty = [Bar(f"empty{i}") for i in range(RING)]
    s_full = [Bar("s_full0"), Bar("s_full1")]
    p_full = [Bar("p_full0"), Bar("p_full1")]
    pv_done = [Bar("pv_done0"), Bar("pv_done1")]
    q_full, q_empty, o_free = Bar("q_full"), Bar("q_empty"), Bar("o_free")

    def producer():
        rp, k = Ring(), 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            if k > 0:
                yield q_empty, k - 1
            q_full.arrive()
            for i in range(n + 1):
                nsc = 9 if i < n else 0
                nv = nslabs(p0 + (i - 1) * TILE, p1) if i >= 1 else 0
                for _ in range(nsc + nv):
                    if rp.n >= RING:
                        yield empty[rp.s], rp.n // RING - 1
                    pending.append(full[rp.s])
                    rp.next()
            k += 1

    def score_mma():
        rp, g, k = Ring(), 0, 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            yield q_full, k
            for i in range(n + 1):
                if i < n:
                    gs = g + i
                    if gs >= 2:
                        yield pv_done[gs & 1], (gs - 2) >> 1
                    if i == 0 and k > 0 and seg_guard:
                        yield pv_done[(gs - 1) & 1], (gs - 1) >> 1
                    for _ in range(9):
                        yield full[rp.s], rp.n // RING
                        empty[rp.s].arrive()
                        rp.next()
                    s_full[gs & 1].arrive()
                    if i == n - 1:
                        q_empty.arrive()
                if i >= 1:
                    rp.skip(nslabs(p0 + (i - 1) * TILE, p1))
            g += n
            k += 1

    def value_mma():
        rp, g, k = Ring(), 0, 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            for i in range(n + 1):
                if i < n:
                    rp.skip(9)
                if i >= 1:
                    gv = g + i - 1
                    if i == 1 and k > 0:
                        yield o_free, k - 1
                    yield p_full[gv & 1], gv >> 1
                    if guard and i < n:
                        yield s_full[(gv + 1) & 1], (gv + 1) >> 1
                    for _ in range(nslabs(p0 + (i - 1) * TILE, p1)):
                        yield full[rp.s], rp.n // RING
                        empty[rp.s].arrive()
                        rp.next()
                    pv_done[gv & 1].arrive()
            g += n
            k += 1

    def softmax():
        g = 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            for i in range(n):
                yield s_full[g & 1], g >> 1
                if i > 0 and rescale:
                    yield pv_done[(g - 1) & 1], (g - 1) >> 1
                p_full[g & 1].arrive()
                g += 1
            yield pv_done[(g - 1) & 1], (g - 1) >> 1
            o_free.arrive()

    roles = {"score": score_mma(), "value": value_mma(), "softmax": softmax(),
             "producer": producer()}
    waiting = {r: None for r in roles}
    alive = list(roles)
    while alive:
        cand = [r for r in alive if waiting[r] is None or waiting[r][0].ready(waiting[r][1])]
        if pending and (not cand or rnd.random() < 0.5):
            pending.pop(rnd.randrange(len(pending))).arrive()
            continue
        if not cand:
            return {r: (waiting[r][0].name, waiting[r][1]) for r in alive}
        r = rnd.choice(cand) if seed is not None else cand[0]
        try:
            waiting[r] = next(roles[r])
        except StopIteration:
            alive.remove(r)
            waiting[r] = None
    return None


@pytest.mark.parametrize("n_tiles", [1, 2, 3, 5, 8])
def test_single_and_multi_segment(n_tiles):
    segs = [(0, 0, n_tiles * TILE), (1, 0, 3 * TILE - 40), (2, 0, 64), (3, 0, 0), (4, 64, 200)]
    for seed in range(12):
        assert run_protocol(segs, seed % 2 == 0, seed) is None


@pytest.mark.parametrize("name", ["b1-l4096", "b64-paged", "b4-l128k", "b128-l16k-t2"])
def test_workload_split_plans(name):
    wl = W.config(name)
    G = 148 // (2 * wl.T)
    for t in range(wl.T):
        plans = split_segments(wl.seq_lens, wl.T, t, G)
        for c, segs in enumerate(plans):
            if name == "b128-l16k-t2" and c % 4:
                continue   # long splits: every fourth keeps the test short
            for rescale, seed in ((False, None), (True, 7), (False, 11)):
                assert run_protocol(segs, rescale, seed) is None, (t, c)


def test_model_catches_segment_start_aliasing():
    """Without the score-MMA role's wait for the previous segment's last PV,
    a one-tile segment followed by another lets that role pass a parity wait
    on a slot whose value-stage fill of the lap before has not landed."""
    segs = [(0, 0, TILE), (1, 0, 3 * TILE - 40)]
    failures = 0
    for seed in range(40):
        try:
            failures += run_protocol(segs, seed % 2 == 0, seed, seg_guard=False) is not None
        except AssertionError:
            failures += 1
    assert failures > 0


def test_model_catches_lap_aliasing():
    """Without its wait on S(x+1) the value-MMA role can pass a parity wait
    on a slot one lap behind: some interleaving of a 3-tile segment shows it,
    so the checks above are not vacuous."""
    failures = 0
    for seed in range(20):
        try:
            failures += run_protocol([(0, 0, 3 * TILE)], False, seed, guard=False) is not None
        except AssertionError:
            failures += 1
    assert failures > 0


# ---------------------------------------------------------------------------
# Paired kernel (even T): a cluster of two CTAs, one per query token, shares
# every cache tile.  The even CTA issues all MMAs with cta_group::2; each CTA
# loads its half of each stage into its own 10-slot ring, and both halves
# complete the even CTA's `ready` barrier (modelled as one arrival per CTA).
# A value slab past the visible end is the exception: the odd CTA loads it
# against a local barrier and its relay warp completes it on `ready` after
# zeroing stale rows; the relay also forwards the odd CTA's query image.
# Commits reach both CTAs (multicast); the softmax warps of both CTAs arrive
# on the even CTA's p_full and o_free.  Ring step i of a segment holds score
# blocks 0-4 of tile i, the value slabs of tile i-1, then score blocks 5-8 of
# tile i, so PV(i-1) overlaps S(i).

PRING = 10


def step_items(i, n, nv_prev):
    """('S', b) / ('V', v) items of ring step i (i = 0..n) in ring order."""
    nsc = 9 if i < n else 0
    head = 5 if nsc else 0
    out = [("S", b) for b in range(head)]
    out += [("V", v) for v in range(nv_prev if i >= 1 else 0)]
    out += [("S", b) for b in range(head, nsc)]
    return out


class Ring10(Ring):
    def next(self):
        self.n += 1
        self.s = (self.s + 1) % PRING


def run_pair_protocol(segs, rescale: bool, seed: int | None, seg_guard: bool = True):
    """seg_guard: the score role waits for PV of the previous tile before the
    first tile of a later segment."""
    rnd = random.Random(seed)
    ready = [Bar(f"ready{i}", 2) for i in range(PRING)]
    zb = Bar("zb")
    empty = {r: [Bar(f"empty{r}{i}") for i in range(PRING)] for r in "LP"}
    s_full = {r: [Bar(f"s_full{r}0"), Bar(f"s_full{r}1")] for r in "LP"}
    pv_done = {r: [Bar(f"pv_done{r}0"), Bar(f"pv_done{r}1")] for r in "LP"}
    q_empty = {r: Bar(f"q_empty{r}") for r in "LP"}
    p_full = [Bar("p_full0", 2), Bar("p_full1", 2)]
    q_ready, q_full_p, o_free = Bar("q_ready", 2), Bar("q_fullP"), Bar("o_free", 2)

    def steps(n, p0, p1):
        for i in range(n + 1):
            yield i, step_items(i, n, nslabs(p0 + (i - 1) * TILE, p1) if i >= 1 else 0)

    def partial(i, item, p0, p1):
        kind, v = item
        return kind == "V" and p1 - (p0 + (i - 1) * TILE + 32 * v) < 32

    def producer(side):
        rp, k = Ring10(), 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            if k > 0:
                yield q_empty[side], k - 1
            (q_ready if side == "L" else q_full_p).arrive()
            for i, items in steps(n, p0, p1):
                for item in items:
                    if rp.n >= PRING:
                        yield empty[side][rp.s], rp.n // PRING - 1
                    if side == "P" and partial(i, item, p0, p1):
                        zb.arrive()
                    else:
                        ready[rp.s].arrive()
                    rp.next()
            k += 1

    def relay():
        rp, k, nz = Ring10(), 0, 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            yield q_full_p, k
            q_ready.arrive()
            for i, items in steps(n, p0, p1):
                for item in items:
                    if partial(i, item, p0, p1):
                        yield zb, nz
                        ready[rp.s].arrive()
                        nz += 1
                    rp.next()
            k += 1

    def both(bars):
        for b in bars:
            b.arrive()

    def score_mma():
        rp, g, k = Ring10(), 0, 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            yield q_ready, k
            for i, items in steps(n, p0, p1):
                gs = g + i
                if i < n:
                    if gs >= 2:
                        yield pv_done["L"][gs & 1], (gs - 2) >> 1
                    if seg_guard and i == 0 and gs >= 1:
                        yield pv_done["L"][(gs - 1) & 1], (gs - 1) >> 1
                for kind, _ in items:
                    if kind == "S":
                        yield ready[rp.s], rp.n // PRING
                        both([empty["L"][rp.s], empty["P"][rp.s]])
                    rp.next()
                if i < n:
                    both([s_full["L"][gs & 1], s_full["P"][gs & 1]])
                    if i == n - 1:
                        both([q_empty["L"], q_empty["P"]])
            g += n
            k += 1

    def value_mma():
        rp, g, k = Ring10(), 0, 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            for i, items in steps(n, p0, p1):
                gv = g + i - 1
                if i >= 1:
                    if i == 1 and k > 0:
                        yield o_free, k - 1
                    yield p_full[gv & 1], gv >> 1
                for kind, _ in items:
                    if kind == "V":
                        yield ready[rp.s], rp.n // PRING
                        both([empty["L"][rp.s], empty["P"][rp.s]])
                    rp.next()
                if i >= 1:
                    both([pv_done["L"][gv & 1], pv_done["P"][gv & 1]])
            g += n
            k += 1

    def softmax(side):
        g = 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            for i in range(n):
                yield s_full[side][g & 1], g >> 1
                if i > 0 and rescale:
                    yield pv_done[side][(g - 1) & 1], (g - 1) >> 1
                p_full[g & 1].arrive()
                g += 1
            yield pv_done[side][(g - 1) & 1], (g - 1) >> 1
            o_free.arrive()

    roles = {"producerL": producer("L"), "producerP": producer("P"), "relay": relay(),
             "score": score_mma(), "value": value_mma(), "softmaxL": softmax("L"),
             "softmaxP": softmax("P")}
    waiting = {r: None for r in roles}
    alive = list(roles)
    while alive:
        cand = [r for r in alive if waiting[r] is None or waiting[r][0].ready(waiting[r][1])]
        if not cand:
            return {r: (waiting[r][0].name, waiting[r][1]) for r in alive}
        r = rnd.choice(cand) if seed is not None else cand[0]
        try:
            waiting[r] = next(roles[r])
        except StopIteration:
            alive.remove(r)
            waiting[r] = None
    return None


@pytest.mark.parametrize("n_tiles", [1, 2, 3, 5, 8, 13])
def test_pair_single_and_multi_segment(n_tiles):
    segs = [(0, 0, n_tiles * TILE), (1, 0, 3 * TILE - 40), (2, 0, 64), (3, 0, 0), (4, 64, 200),
            (5, 0, 2 * TILE), (6, 0, TILE)]
    for seed in range(16):
        assert run_pair_protocol(segs, seed % 2 == 0, seed) is None


def test_pair_workload_split_plan():
    for name in ("b128-l16k-t2", "b64-paged"):
        wl = W.config(name)
        G = 148 // 4
        plans = split_segments(wl.seq_lens, 2, 1, G)
        for c, segs in enumerate(plans):
            if c % 3:
                continue
            for rescale, seed in ((False, None), (True, 5)):
                assert run_pair_protocol(segs, rescale, seed) is None, (name, c)


# Paired kernel, 16 KB stages: a stage carries two score blocks (or the last
# one) or two value slabs (or the last one) of this CTA's half, in a 5-slot
# ring.  Ring step i: score stages {0,1}, {2,3}, the value stages of tile
# i-1, then score stages {4,5}, {6,7}, {8}.

PRING2 = 5


def step_items2(i, n, nv_prev):
    """('S', first block) / ('V', first slab) stages of ring step i."""
    score = [("S", b) for b in (0, 2, 4, 6, 8)] if i < n else []
    vals = [("V", v) for v in range(0, nv_prev, 2)] if i >= 1 else []
    return score[:2] + vals + score[2:] if score else vals


class Ring5(Ring):
    pass


def run_pair16_protocol(segs, rescale: bool, seed: int | None, items_fn=None,
                        slabs_per_stage: int = 2, in_order: bool = False):
    """items_fn / slabs_per_stage: the step layout (default: two slabs per
    value stage, step_items2).  Issued copies complete in random order (a
    separate copy-engine role), unless in_order."""
    items_fn = items_fn or step_items2
    rnd = random.Random(seed)
    pending = []   # barriers of issued, not yet completed copies
    R = PRING2
    ready = [Bar(f"ready{i}", 2) for i in range(R)]
    zb = Bar("zb")
    empty = {r: [Bar(f"empty{r}{i}") for i in range(R)] for r in "LP"}
    s_full = {r: [Bar(f"s_full{r}0"), Bar(f"s_full{r}1")] for r in "LP"}
    pv_done = {r: [Bar(f"pv_done{r}0"), Bar(f"pv_done{r}1")] for r in "LP"}
    q_empty = {r: Bar(f"q_empty{r}") for r in "LP"}
    p_full = [Bar("p_full0", 2), Bar("p_full1", 2)]
    q_ready, q_full_p, o_free = Bar("q_ready", 2), Bar("q_fullP"), Bar("o_free", 2)

    def steps(n, p0, p1):
        for i in range(n + 1):
            yield i, items_fn(i, n, nslabs(p0 + (i - 1) * TILE, p1) if i >= 1 else 0)

    def partial(i, item, p0, p1):
        kind, v = item
        if kind != "V":
            return False
        last = min(v + slabs_per_stage, nslabs(p0 + (i - 1) * TILE, p1)) - 1
        return p1 - (p0 + (i - 1) * TILE + 32 * last) < 32

    def producer(side):
        rp, k = Ring(), 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            if k > 0:
                yield q_empty[side], k - 1
            (q_ready if side == "L" else q_full_p).arrive()
            for i, items in steps(n, p0, p1):
                for item in items:
                    if rp.n >= R:
                        yield empty[side][rp.s], rp.n // R - 1
                    if side == "P" and partial(i, item, p0, p1):
                        pending.append(zb)
                    else:
                        pending.append(ready[rp.s])
                    if in_order:
                        pending.pop(0).arrive()
                    rp.next()
            k += 1

    def copy_engine():
        while True:
            if pending:
                pending.pop(rnd.randrange(len(pending))).arrive()
            yield None

    def relay():
        rp, k, nz = Ring(), 0, 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            yield q_full_p, k
            q_ready.arrive()
            for i, items in steps(n, p0, p1):
                for item in items:
                    if partial(i, item, p0, p1):
                        yield zb, nz
                        ready[rp.s].arrive()
                        nz += 1
                    rp.next()
            k += 1

    def both(bars):
        for b in bars:
            b.arrive()

    def score_mma():
        rp, g, k = Ring(), 0, 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            yield q_ready, k
            for i, items in steps(n, p0, p1):
                gs = g + i
                if i < n:
                    if gs >= 2:
                        yield pv_done["L"][gs & 1], (gs - 2) >> 1
                    if i == 0 and gs >= 1:
                        yield pv_done["L"][(gs - 1) & 1], (gs - 1) >> 1
                for kind, _ in items:
                    if kind == "S":
                        yield ready[rp.s], rp.n // R
                        both([empty["L"][rp.s], empty["P"][rp.s]])
                    rp.next()
                if i < n:
                    both([s_full["L"][gs & 1], s_full["P"][gs & 1]])
                    if i == n - 1:
                        both([q_empty["L"], q_empty["P"]])
            g += n
            k += 1

    def value_mma():
        rp, g, k = Ring(), 0, 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            for i, items in steps(n, p0, p1):
                gv = g + i - 1
                if i >= 1:
                    if i == 1 and k > 0:
                        yield o_free, k - 1
                    yield p_full[gv & 1], gv >> 1
                for kind, _ in items:
                    if kind == "V":
                        yield ready[rp.s], rp.n // R
                        both([empty["L"][rp.s], empty["P"][rp.s]])
                    rp.next()
                if i >= 1:
                    both([pv_done["L"][gv & 1], pv_done["P"][gv & 1]])
            g += n
            k += 1

    def softmax(side):
        g = 0
        for _, p0, p1 in segs:
            n = ntiles(p0, p1)
            if n == 0:
                continue
            for i in range(n):
                yield s_full[side][g & 1], g >> 1
                if i > 0 and rescale:
                    yield pv_done[side][(g - 1) & 1], (g - 1) >> 1
                p_full[g & 1].arrive()
                g += 1
            yield pv_done[side][(g - 1) & 1], (g - 1) >> 1
            o_free.arrive()

    roles = {"producerL": producer("L"), "producerP": producer("P"), "relay": relay(),
             "score": score_mma(), "value": value_mma(), "softmaxL": softmax("L"),
             "softmaxP": softmax("P")}
    engine = copy_engine()
    waiting = {r: None for r in roles}
    alive = list(roles)
    while alive:
        cand = [r for r in alive if waiting[r] is None or waiting[r][0].ready(waiting[r][1])]
        if pending and (not cand or rnd.random() < 0.5):
            next(engine)
            continue
        if not cand:
            return {r: (waiting[r][0].name, waiting[r][1]) for r in alive}
        r = rnd.choice(cand) if seed is not None else cand[0]
        try:
            waiting[r] = next(roles[r])
        except StopIteration:
            alive.remove(r)
            waiting[r] = None
    return None


@pytest.mark.parametrize("n_tiles", [1, 2, 3, 5, 8, 13])
def test_pair16_single_and_multi_segment(n_tiles):
    segs = [(0, 0, n_tiles * TILE), (1, 0, 3 * TILE - 40), (2, 0, 64), (3, 0, 0), (4, 64, 200),
            (5, 0, 2 * TILE), (6, 0, TILE), (7, 0, 100)]
    for seed in range(16):
        assert run_pair16_protocol(segs, seed % 2 == 0, seed) is None


def test_pair16_workload_split_plan():
    for name in ("b128-l16k-t2", "b64-paged"):
        wl = W.config(name)
        plans = split_segments(wl.seq_lens, 2, 1, 148 // 4)
        for c, segs in enumerate(plans):
            if c % 3:
                continue
            for rescale, seed in ((False, None), (True, 5)):
                assert run_pair16_protocol(segs, rescale, seed) is None, (name, c)


# A ring order that is unsafe when copies complete out of order: value slabs
# all between score stages {2,3} and {4,5} with one slab per stage.  The
# last slab's slot was last used by this step's first score stage, which
# the value role's waits do not cover.

def step_items_unsafe(i, n, nv_prev):
    score = [("S", b) for b in (0, 2, 4, 6, 8)] if i < n else []
    vals = [("V", v) for v in range(nv_prev)] if i >= 1 else []
    return score[:2] + vals + score[2:] if score else vals


def test_model_catches_out_of_order_hazard():
    """With step_items_unsafe a slow copy lets the value role pass a parity
    wait a lap early: the model, whose copies complete in random order,
    reports it."""
    failures = 0
    for seed in range(60):
        try:
            failures += run_pair16_protocol([(0, 0, 6 * TILE)], False, seed,
                                            step_items_unsafe, 1) is not None
        except AssertionError:
            failures += 1
    assert failures > 0
