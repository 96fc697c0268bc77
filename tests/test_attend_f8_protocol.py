"""Model of the FP8 attention kernel's barrier protocol (CPU only).

attend_f8.cu runs one CTA per (KV split, query token, latent half) with a
TMA producer, a score-MMA issuer (the score MMAs of each tile on the four
latent blocks and the RoPE block), two converter warps (this half's codes of
a tile, loaded from the pool into registers, widened to bf16 into one value
buffer once the previous value MMA has read it, then the tile's value MMAs
issued by one of their threads) and four softmax warps.  They meet only at
mbarriers, and every wait is a parity wait.  As for the bf16 kernel's model
(test_attend_protocol.py), each role's loop is restated -- the order of its
waits, arrivals and buffer accesses, none of the arithmetic -- and driven in
many random interleavings; the model fails on deadlock, on a parity wait
passing on the wrong phase, and when a role reads a buffer that does not
hold what it expects (ring slot, row scales, S buffer, value buffer, query
image, O).  A change to the order of waits, arrivals or buffer accesses in
the kernel must be made here too.
"""
from __future__ import annotations

import random

import pytest

from synth import workloads as W
from test_attend_protocol import TILE, Bar, expect, ntiles, split_segments

RING = 4


def run_f8_protocol(segs, half: int, rescale: bool, seed: int | None, drop: str = "",
                    slow: str = ""):
    """Returns None when every role finishes, else the blocked roles.
    drop names a wait to leave out (planted mistakes); slow: roles whose
    names start with it run only when nothing else can."""
    rnd = random.Random(seed)
    pending = []
    vb = (2 * half, 2 * half + 1)
    full = [Bar(f"full{i}") for i in range(RING)]
    empty = [Bar(f"empty{i}") for i in range(RING)]
    s_full = [Bar("s_full0"), Bar("s_full1")]
    p_full = [Bar("p_full0", 4), Bar("p_full1", 4)]
    pv_done = [Bar("pv_done0"), Bar("pv_done1")]
    v_full = [Bar("v_full0"), Bar("v_full1")]
    c_full = [Bar("c_full0"), Bar("c_full1")]
    c_empty = [Bar("c_empty0", 4), Bar("c_empty1", 4)]
    q_full, q_empty, o_free = Bar("q_full"), Bar("q_empty", 5), Bar("o_free", 4)
    ring = [None] * RING          # stage number a slot holds (landed)
    scales = [None, None]         # tile whose scales a buffer holds
    s_buf = [None, None]          # ("S" | "P", tile)
    v_buf = [None]                # tile whose values the buffer holds
    v_read = [-1]                 # last tile whose value MMAs ran
    q_img = [None]                # segment whose query image is loaded
    o_state = {"seg": None, "last": None}
    live = [(k, s) for k, s in enumerate(segs) if ntiles(s[1], s[2]) > 0]

    def land(fn):
        pending.append(fn)

    def producer():
        g = 0
        for kk, (_, (_, p0, p1)) in enumerate(live):
            if kk > 0 and "q_empty" not in drop:
                yield q_empty, kk - 1
            land(lambda kk=kk: (q_img.__setitem__(0, kk), q_full.arrive()))
            for i in range(ntiles(p0, p1)):
                if g >= 2 and "c_empty" not in drop:
                    yield c_empty[g & 1], (g >> 1) - 1
                land(lambda g=g: (scales.__setitem__(g & 1, g), c_full[g & 1].arrive()))
                for kb in range(5):
                    nr = 5 * g + kb
                    s = nr % RING
                    if nr >= RING:
                        yield empty[s], nr // RING - 1
                    land(lambda s=s, nr=nr: (ring.__setitem__(s, nr), full[s].arrive()))
                g += 1

    def mma():
        g = 0
        for kk, (k, (_, p0, p1)) in enumerate(live):
            n = ntiles(p0, p1)
            yield q_full, kk
            for i in range(n):
                if g >= 2 and "pv_s" not in drop:
                    yield pv_done[g & 1], (g - 2) >> 1
                expect(s_buf[g & 1] is None or s_buf[g & 1] == ("P", g - 2),
                       f"S({g}) over {s_buf[g & 1]}")
                for kb in range(5):
                    nr = 5 * g + kb
                    yield full[nr % RING], nr // RING
                    expect(ring[nr % RING] == nr, f"S({g}) block {kb}: slot holds "
                           f"{ring[nr % RING]}")
                    expect(q_img[0] == kk, f"S({g}) with the query of segment {q_img[0]}")
                    empty[nr % RING].arrive()
                s_buf[g & 1] = ("S", g)
                s_full[g & 1].arrive()
                if i == n - 1:
                    q_empty.arrive()
                g += 1

    def converter():
        g = 0
        for kk, (_, (_, p0, p1)) in enumerate(live):
            for i in range(ntiles(p0, p1)):
                # the codes come from the pool (no ring stage), then wait for
                # the value buffer
                if g >= 1 and "pv_v" not in drop:
                    yield pv_done[(g - 1) & 1], (g - 1) >> 1
                expect(v_read[0] >= g - 1, f"values of tile {g} written over those of "
                       f"tile {v_buf[0]} before PV({g - 1}) ran")
                v_buf[0] = g
                # the value MMAs of tile g, issued by a converter thread
                if i == 0 and kk > 0 and "o_free" not in drop:
                    yield o_free, kk - 1
                yield p_full[g & 1], g >> 1

                # issued here, executed later: the MMAs read P, the value
                # buffer and O when they run (a pending event)
                def run_pv(g=g, i=i, kk=kk):
                    expect(s_buf[g & 1] == ("P", g), f"PV({g}) reads {s_buf[g & 1]}")
                    expect(v_buf[0] == g, f"PV({g}) reads values of tile {v_buf[0]}")
                    st = o_state
                    if i == 0:
                        expect(st["seg"] is None or st.get("read") == st["seg"],
                               f"PV({g}) overwrites O of segment {st['seg']} before its read")
                        st.clear()
                        st.update(seg=kk, last=None)
                    else:
                        expect(st["last"] == g - 1, f"PV({g}) after PV({st['last']})")
                    expect(st.get("rescaled_for", g) == g, "rescale raced a PV")
                    st["last"] = g
                    st.pop("rescaled_for", None)
                    v_read[0] = g
                    pv_done[g & 1].arrive()
                land(run_pv)
                g += 1

    def softmax(w):
        g = 0
        for kk, (k, (_, p0, p1)) in enumerate(live):
            n = ntiles(p0, p1)
            yield q_full, kk
            expect(q_img[0] == kk, f"softmax {w} reads the scale of segment {q_img[0]}")
            q_empty.arrive()
            for i in range(n):
                yield s_full[g & 1], g >> 1
                yield c_full[g & 1], g >> 1
                expect(s_buf[g & 1] in (("S", g), ("P", g)), f"softmax {w} reads {s_buf[g & 1]}")
                expect(scales[g & 1] == g, f"softmax {w} reads scales of {scales[g & 1]}")
                if rescale and i > 0 and w == 0:
                    if "pv_rescale" not in drop:
                        yield pv_done[(g - 1) & 1], (g - 1) >> 1
                    expect(o_state["last"] == g - 1, f"rescale for tile {g} after PV({o_state['last']})")
                    o_state["rescaled_for"] = g
                c_empty[g & 1].arrive()
                s_buf[g & 1] = ("P", g)
                p_full[g & 1].arrive()
                g += 1
            yield pv_done[(g - 1) & 1], (g - 1) >> 1
            expect(o_state["last"] == g - 1, f"epilogue reads O after PV({o_state['last']})")
            if w == 0:
                o_state["read"] = kk
            o_free.arrive()

    roles = {"producer": producer(), "mma": mma(), "converter": converter()}
    for w in range(4):
        roles[f"softmax{w}"] = softmax(w)
    waiting = {r: None for r in roles}
    alive = list(roles)

    def ready(r):
        return waiting[r] is None or waiting[r][0].ready(waiting[r][1])

    while alive:
        cand = [r for r in alive if ready(r)]
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


@pytest.mark.parametrize("half", [0, 1])
@pytest.mark.parametrize("n_tiles", [1, 2, 3, 8])
def test_single_and_multi_segment(half, n_tiles):
    segs = [(0, 0, n_tiles * TILE)] + SEGS[1:]
    for seed in range(10):
        assert run_f8_protocol(segs, half, seed % 2 == 0, seed) is None


@pytest.mark.parametrize("name", ["b1-l4096", "b64-paged", "b4-l128k", "b128-l16k-t2"])
def test_workload_split_plans(name):
    wl = W.config(name)
    G = 148 // (2 * wl.T)
    for t in range(wl.T):
        plans = split_segments(wl.seq_lens, wl.T, t, G)
        for c, segs in enumerate(plans):
            if c % 7:
                continue
            assert run_f8_protocol(segs, c % 2, c % 3 == 0, c) is None, (name, t, c)


# The kernel also keeps a wait that the ordering already implies, so that
# leaving it out is no hazard here: the wait for the epilogue before a
# segment's first PV (that PV also waits for P from all four softmax warps,
# which write the epilogue first).  The value MMAs are issued by the thread
# that wrote the value buffer, so the buffer needs no barrier of its own.
SLOW_FOR = {"pv_v": "converter", "pv_s": "softmax", "c_empty": "softmax", "q_empty": "mma",
            "pv_rescale": "converter"}


@pytest.mark.parametrize("drop", list(SLOW_FOR))
def test_model_catches_dropped_waits(drop):
    """Leaving out any one of these waits lets some interleaving read or
    overwrite a buffer at the wrong time: the checks are not vacuous."""
    failures = 0
    for seed in range(40):
        try:
            failures += run_f8_protocol(SEGS, seed % 2, True, seed, drop=drop,
                                        slow=SLOW_FOR[drop]) is not None
        except AssertionError:
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("slow", ["softmax", "mma", "converter", "producer"])
def test_slow_roles(slow):
    for seed in range(8):
        assert run_f8_protocol(SEGS, seed % 2, seed % 2 == 0, seed, slow=slow) is None
