"""Model of the attention kernel's barrier protocol (CPU only).

The split-KV attention kernel (attend_sv.cu) runs, per cluster, a score side
(TMA producer, score-MMA issuer, softmax warps) and a value side (TMA
producer, value-MMA issuer, correction/epilogue warps, and for token pairs a
relay warp in the odd value CTA).  They meet only at mbarriers, and every
wait is a parity wait, which cannot tell phase F from phase F + 2.

This file restates each role's loop (the order of its waits, arrivals and
buffer accesses, nothing of the arithmetic) and drives the roles in many
random interleavings over the split plans of the workloads.  Besides
deadlock and a parity wait passing on the wrong phase, it tracks what every
buffer holds and fails when a role reads a buffer that does not hold what
it expects: a ring slot (stage number), an S buffer (tile), a landing buffer
(tile), q~ and the RoPE block (segment), and O (which value MMAs, rescales
and read-outs have happened).

Copies complete in random order, and only when a separate copy-engine role
runs; MMAs complete when issued (they wait on nothing once issued), so this
can only hide delays, not orderings.  A change to the order of waits,
arrivals or buffer accesses in the kernel must be made here too.
"""
from __future__ import annotations

import random

import pytest

from synth import workloads as W

SRING, VRING, TILE, PAGE = 13, 9, 128, 64


class Bar:
    def __init__(self, name: str, count: int = 1):
        self.name, self.count, self.pending, self.done = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: too many arrivals"
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


class RingPos:
    def __init__(self, R: int):
        self.R, self.s, self.n = R, 0, 0

    @property
    def ph(self):
        return (self.n // self.R) & 1

    def next(self):
        self.n += 1
        self.s = (self.s + 1) % self.R


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


class Hazard(AssertionError):
    pass


def expect(cond, what):
    if not cond:
        raise Hazard(what)


def run_sv_protocol(segs, pair: bool, rescale: bool, seed: int | None, drop: str = "",
                    slow: str = ""):
    """Returns None when every role finishes, else the blocked roles.

    pair: the four-CTA form (sides L = leader, P = peer on both the score
    and the value side); else the two-CTA form (side L only).  rescale: the
    correction warps rescale O at every tile after the first.  drop names a
    wait to leave out (planted mistakes): "s_free", "pvd_land", "stg_free",
    "q_empty", "pvd_rescale", "zdone".  slow: roles whose names start with it
    run only when nothing else can (a slow role widens the windows in which
    the others race ahead)."""
    rnd = random.Random(seed)
    sides = "LP" if pair else "L"
    nside = len(sides)
    pending = []            # copies issued, not yet landed: (callback)
    nst_s = 5 if pair else 9
    # ---- barriers (one object per CTA where each CTA has its own)
    full_s = [Bar(f"full_s{i}", 1) for i in range(SRING)]          # leader's
    empty_s = {x: [Bar(f"empty_s{x}{i}") for i in range(SRING)] for x in sides}
    s_full = {x: [Bar(f"s_full{x}0"), Bar(f"s_full{x}1")] for x in sides}
    s_free = [Bar("s_free0", nside), Bar("s_free1", nside)]        # leader's
    q_ready = Bar("q_ready", nside)
    qr = {x: Bar(f"qr{x}") for x in sides}
    q_empty = {x: Bar(f"q_empty{x}") for x in sides}
    pvd_s = {x: [Bar(f"pvd_s{x}0"), Bar(f"pvd_s{x}1")] for x in sides}
    full_v = [Bar(f"full_v{i}", 1) for i in range(VRING)]          # leader's
    empty_v = {x: [Bar(f"empty_v{x}{i}") for i in range(VRING)] for x in sides}
    land = {x: [Bar(f"land{x}0"), Bar(f"land{x}1")] for x in sides}
    o_ok = [Bar("o_ok0", nside), Bar("o_ok1", nside)]              # leader's
    pvd_v = {x: [Bar(f"pvd_v{x}0"), Bar(f"pvd_v{x}1")] for x in sides}
    zb, zdone = Bar("zb"), Bar("zdone")
    # ---- buffer contents
    ring_s = {x: [None] * SRING for x in sides}     # stage number held
    ring_v = {x: [None] * VRING for x in sides}
    sbuf = {x: [None, None] for x in sides}         # tile whose S is held
    landing = {x: [None, None] for x in sides}      # tile whose P is held
    landing_read = {x: [None, None] for x in sides}  # last tile whose P the PV consumed
    staging = {x: [None, None] for x in sides}      # tile whose P each staging buffer holds
    staging_sent = {x: [None, None] for x in sides}  # last tile whose staged P has landed
    stg_free = {x: Bar(f"stg_free{x}") for x in sides}
    qc = {x: None for x in sides}                   # segment whose q~ is in TMEM
    qr_data = {x: None for x in sides}              # segment whose RoPE block landed
    o_state = {x: {"seg": None, "last": None, "read": None} for x in sides}

    seg_list = [(i, s) for i, s in enumerate(segs) if ntiles(s[1], s[2]) > 0]

    # -------------------------------------------------------------- score side
    def producer_s(x):
        rp = RingPos(SRING)
        for k, (_, (_, p0, p1)) in enumerate(seg_list):
            n = ntiles(p0, p1)
            if k > 0 and "q_empty" not in drop:
                yield q_empty[x], k - 1

            def land_qr(x=x, k=k):
                qr_data[x] = k
                qr[x].arrive()
            pending.append(land_qr)
            for _ in range(n):
                for _ in range(nst_s):
                    if rp.n >= SRING:
                        yield empty_s[x][rp.s], rp.n // SRING - 1
                    stage, slot = rp.n, rp.s

                    def land_s(x=x, slot=slot, stage=stage):
                        ring_s[x][slot] = stage
                        if not pair:
                            full_s[slot].arrive()
                        else:
                            land_pair_s[slot].append(x)
                            if len(land_pair_s[slot]) == 2:
                                land_pair_s[slot].clear()
                                full_s[slot].arrive()
                    pending.append(land_s)
                    rp.next()

    land_pair_s = [[] for _ in range(SRING)]   # pair: both halves complete the leader's barrier

    def issuer_s():
        rp, g = RingPos(SRING), 0
        for k, (_, (_, p0, p1)) in enumerate(seg_list):
            n = ntiles(p0, p1)
            yield q_ready, k
            for i in range(n):
                gs = g + i
                if gs >= 2 and "s_free" not in drop:
                    yield s_free[gs & 1], (gs - 2) >> 1
                for _ in range(nst_s):
                    yield full_s[rp.s], rp.n // SRING
                    for x in sides:
                        expect(ring_s[x][rp.s] == rp.n, f"score slot {rp.s} of {x} holds "
                               f"{ring_s[x][rp.s]}, MMA wants stage {rp.n}")
                        expect(qc[x] == k, f"q~ of {x} holds segment {qc[x]}, S wants {k}")
                        expect(qr_data[x] == k, f"RoPE block of {x} holds {qr_data[x]}, want {k}")
                    for x in sides:
                        empty_s[x][rp.s].arrive()
                    rp.next()
                for x in sides:
                    expect(sbuf[x][gs & 1] is None or sbuf[x][gs & 1] == "read",
                           f"S buffer {gs & 1} of {x} overwritten before it was read")
                    sbuf[x][gs & 1] = gs
                    s_full[x][gs & 1].arrive()
                if i == n - 1:
                    for x in sides:
                        q_empty[x].arrive()
            g += n

    def softmax(x):
        g = 0
        for k, (_, (_, p0, p1)) in enumerate(seg_list):
            n = ntiles(p0, p1)
            if k > 0 and "q_empty" not in drop:
                yield q_empty[x], k - 1
            qc[x] = k          # q~ into TMEM while the RoPE block lands
            yield qr[x], k
            q_ready.arrive()
            for i in range(n):
                yield s_full[x][g & 1], g >> 1
                expect(sbuf[x][g & 1] == g, f"softmax {x} wants S({g}), buffer holds "
                       f"{sbuf[x][g & 1]}")
                sbuf[x][g & 1] = "read"
                s_free[g & 1].arrive()
                # a single token stages P in one buffer, freed when the
                # copy of P(g - 1) lands; a pair in two, buffer g & 1 freed
                # with landing buffer g & 1 (PV(g - 2) done)
                if not pair and g >= 1 and "stg_free" not in drop:
                    yield stg_free[x], g - 1
                if g >= 2 and "pvd_land" not in drop:
                    yield pvd_s[x][g & 1], (g - 2) >> 1
                sb = (g & 1) if pair else 0
                # P(g) into the local staging buffer, then one bulk copy to
                # the value CTA's landing buffer g & 1; the copy reads the
                # staging buffer and lands some time later
                expect(staging[x][sb] is None or staging_sent[x][sb] == staging[x][sb],
                       f"staging of {x} rewritten before its copy of P({staging[x][sb]}) landed")
                staging[x][sb] = g

                def copy_lands(x=x, g=g, sb=sb):
                    expect(staging[x][sb] == g, f"copy of P({g}) from {x} read a staging "
                           f"buffer holding P({staging[x][sb]})")
                    staging_sent[x][sb] = g
                    expect(landing[x][g & 1] is None or
                           landing_read[x][g & 1] == landing[x][g & 1],
                           f"landing {g & 1} of {x} rewritten before PV read "
                           f"P({landing[x][g & 1]})")
                    landing[x][g & 1] = g
                    land[x][g & 1].arrive()
                pending.append(copy_lands)
                g += 1

    # -------------------------------------------------------------- value side
    def partial(ts, v, p1):
        return p1 - (ts + 32 * v) < 32

    land_pair_v = [[] for _ in range(VRING)]

    def producer_v(x):
        rp, nz = RingPos(VRING), 0
        for _, (_, p0, p1) in seg_list:
            n = ntiles(p0, p1)
            for i in range(n):
                ts = p0 + i * TILE
                for v in range(nslabs(ts, p1)):
                    for _ in range(1 if pair else 2):
                        if rp.n >= VRING:
                            yield empty_v[x][rp.s], rp.n // VRING - 1
                        part = pair and x == "P" and partial(ts, v, p1)
                        if part and nz > 0 and "zdone" not in drop:
                            yield zdone, nz - 1
                        stage, slot = rp.n, rp.s

                        def land_v(x=x, slot=slot, stage=stage, part=part):
                            ring_v[x][slot] = stage
                            if part:
                                zb.arrive()
                            elif pair:
                                land_pair_v[slot].append(x)
                                if len(land_pair_v[slot]) == 2:
                                    land_pair_v[slot].clear()
                                    full_v[slot].arrive()
                            else:
                                full_v[slot].arrive()
                        pending.append(land_v)
                        if part:
                            nz += 1
                        rp.next()

    def relay():
        rp, nz = RingPos(VRING), 0
        for _, (_, p0, p1) in seg_list:
            n = ntiles(p0, p1)
            for i in range(n):
                ts = p0 + i * TILE
                for v in range(nslabs(ts, p1)):
                    if partial(ts, v, p1):
                        yield zb, nz
                        expect(ring_v["P"][rp.s] == rp.n, "relay zeroes the wrong stage")
                        land_pair_v[rp.s].append("P")
                        if len(land_pair_v[rp.s]) == 2:
                            land_pair_v[rp.s].clear()
                            full_v[rp.s].arrive()
                        zdone.arrive()
                        nz += 1
                    rp.next()

    def issuer_v():
        rp, g = RingPos(VRING), 0
        for k, (_, (_, p0, p1)) in enumerate(seg_list):
            n = ntiles(p0, p1)
            for i in range(n):
                gv = g + i
                # o_ok of a segment's first tile comes from the correction
                # warps after their read-out of the previous segment's O
                yield o_ok[gv & 1], gv >> 1
                for x in sides:
                    expect(landing[x][gv & 1] == gv, f"PV({gv}) reads landing of {x} holding "
                           f"P({landing[x][gv & 1]})")
                    st = o_state[x]
                    if i == 0:
                        expect(k == 0 or st["read"] == k - 1,
                               f"O of {x} reset for segment {k} before segment {k - 1} was read")
                        st["seg"], st["last"] = k, None
                    else:
                        expect(st["last"] == gv - 1, f"PV({gv}) on O of {x} after PV({st['last']})")
                    expect(st.get("rescaled_for", gv) == gv,
                           f"O of {x} rescaled for tile {st.get('rescaled_for')} before PV({gv})")
                for _ in range(nslabs(p0 + i * TILE, p1)):
                    for _ in range(1 if pair else 2):
                        yield full_v[rp.s], rp.n // VRING
                        for x in sides:
                            expect(ring_v[x][rp.s] == rp.n, f"value slot {rp.s} of {x} holds "
                                   f"{ring_v[x][rp.s]}, MMA wants stage {rp.n}")
                        for x in sides:
                            empty_v[x][rp.s].arrive()
                        rp.next()
                for x in sides:
                    landing_read[x][gv & 1] = gv
                    o_state[x]["last"] = gv
                    o_state[x].pop("rescaled_for", None)
                    pvd_v[x][gv & 1].arrive()
                    pvd_s[x][gv & 1].arrive()
            g += n

    def correction(x):
        g = 0
        for k, (_, (_, p0, p1)) in enumerate(seg_list):
            n = ntiles(p0, p1)
            for i in range(n):
                yield land[x][g & 1], g >> 1
                expect(landing[x][g & 1] == g, f"correction {x} reads f, l of "
                       f"P({landing[x][g & 1]}) for tile {g}")
                if not pair:
                    stg_free[x].arrive()
                if rescale and i > 0:
                    if "pvd_rescale" not in drop:
                        yield pvd_v[x][(g - 1) & 1], (g - 1) >> 1
                    st = o_state[x]
                    expect(st["seg"] == k and st["last"] == g - 1,
                           f"rescale of O of {x} for tile {g} after PV({st['last']})")
                    st["rescaled_for"] = g
                o_ok[g & 1].arrive()
                g += 1
            yield pvd_v[x][(g - 1) & 1], (g - 1) >> 1
            st = o_state[x]
            expect(st["seg"] == k and st["last"] == g - 1,
                   f"epilogue of {x} reads O after PV({st['last']}), segment ends at {g - 1}")
            st["read"] = k

    roles = {"issuer_s": issuer_s(), "issuer_v": issuer_v()}
    for x in sides:
        roles[f"producer_s{x}"] = producer_s(x)
        roles[f"softmax{x}"] = softmax(x)
        roles[f"producer_v{x}"] = producer_v(x)
        roles[f"correction{x}"] = correction(x)
    if pair:
        roles["relay"] = relay()
    waiting = {r: None for r in roles}
    alive = list(roles)
    while alive:
        cand = [r for r in alive if waiting[r] is None or waiting[r][0].ready(waiting[r][1])]
        if pending and (not cand or rnd.random() < 0.4):
            pending.pop(rnd.randrange(len(pending)))()
            continue
        if not cand:
            return {r: (waiting[r][0].name, waiting[r][1]) for r in alive}
        fast = [r for r in cand if not (slow and r.startswith(slow))]
        pick = fast if fast and rnd.random() < 0.97 else cand
        r = rnd.choice(pick) if seed is not None else pick[0]
        try:
            waiting[r] = next(roles[r])
        except StopIteration:
            alive.remove(r)
            waiting[r] = None
    return None


SEGS = [(0, 0, 5 * TILE), (1, 0, 3 * TILE - 40), (2, 0, 64), (3, 0, 0), (4, 64, 200),
        (5, 0, 2 * TILE), (6, 0, TILE), (7, 0, 100), (8, 0, 33), (9, 0, 31)]


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("n_tiles", [1, 2, 3, 8, 13])
def test_single_and_multi_segment(pair, n_tiles):
    segs = [(0, 0, n_tiles * TILE)] + SEGS[1:]
    for seed in range(10):
        assert run_sv_protocol(segs, pair, seed % 2 == 0, seed) is None


@pytest.mark.parametrize("name", ["b1-l4096", "b64-paged", "b4-l128k", "b128-l16k-t2"])
def test_workload_split_plans(name):
    wl = W.config(name)
    pair = wl.T % 2 == 0
    G = 148 // (2 * wl.T)
    t = wl.T - 1 if pair else 0   # a pair iterates its odd token's range
    plans = split_segments(wl.seq_lens, wl.T, t, G)
    for c, segs in enumerate(plans):
        if c % 5:
            continue   # every fifth split keeps the test short
        for rescale, seed in ((False, None), (True, 7)):
            assert run_sv_protocol(segs, pair, rescale, seed) is None, (name, c)


# the role that falls behind when a wait is missing, for each planted mistake
SLOW_FOR = {"s_free": "softmax", "pvd_land": "issuer_v", "q_empty": "issuer_s",
            "pvd_rescale": "issuer_v", "stg_free": "correction"}


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("drop", list(SLOW_FOR))
def test_model_catches_dropped_waits(pair, drop):
    if pair and drop == "stg_free":
        pytest.skip("a pair stages P in two buffers and does not wait on stg_free")
    """Leaving out any one of these waits lets some interleaving read or
    overwrite a buffer at the wrong time: the checks above are not vacuous."""
    failures = 0
    for seed in range(40):
        try:
            failures += run_sv_protocol(SEGS, pair, True, seed, drop=drop,
                                        slow=SLOW_FOR[drop]) is not None
        except AssertionError:
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("slow", ["softmax", "issuer_v", "issuer_s", "correction", "producer"])
def test_slow_roles(pair, slow):
    """The full protocol under the same adversarial schedules."""
    for seed in range(8):
        assert run_sv_protocol(SEGS, pair, seed % 2 == 0, seed, slow=slow) is None


def test_model_catches_dropped_relay_wait():
    """Without the producer's wait for the relay, two partial value slabs of
    one-tile segments can both land on the local barrier before the relay
    waits: a parity wait passes a phase late."""
    segs = [(b, 0, 20 + b) for b in range(8)]
    failures = 0
    for seed in range(60):
        try:
            failures += run_sv_protocol(segs, True, False, seed, drop="zdone",
                                        slow="relay") is not None
        except AssertionError:
            failures += 1
    assert failures > 0
