"""Model of the explicit-form prefill attention kernel's barrier protocol (CPU only).

prefill.cu's attention runs one CTA per (128-query tile, head, sequence)
with a TMA producer (the Q tile once, then K and V tiles through separate
two-stage rings, K one tile ahead of V), an MMA issuer (S(j) into S buffer
j & 1 once PV(j - 2) has read P(j - 2) from it, then PV(j - 1)) and the
softmax warps (S row into registers, maximum, lazy rescale of O after
PV(j - 1), P written over S).  The eight softmax warps meet at named
barriers and act together, so they are one role here.  As for the decode
kernels' models, each role's loop is restated -- the order of its waits,
arrivals and buffer accesses, none of the arithmetic -- and driven in many
random interleavings: copies land in random order, MMAs complete when
issued.  The model fails on deadlock, on a parity wait passing on the wrong
phase, and when a role reads a buffer that does not hold what it expects
(K or V stage, S buffer, O).  A change to the order of waits, arrivals or
buffer accesses in the kernel must be made here too.
"""
from __future__ import annotations

import random

import pytest

from test_attend_protocol import Bar, expect


def run_prefill_protocol(n: int, rescale: bool, seed: int | None, drop: str = "",
                         slow: str = ""):
    """n key tiles; rescale: the softmax rescales O at every tile after the
    first.  Returns None when every role finishes, else the blocked roles."""
    rnd = random.Random(seed)
    pending = []
    kfull, kempty = [Bar("kfull0"), Bar("kfull1")], [Bar("kempty0"), Bar("kempty1")]
    vfull, vempty = [Bar("vfull0"), Bar("vfull1")], [Bar("vempty0"), Bar("vempty1")]
    s_full, p_full = [Bar("s_full0"), Bar("s_full1")], [Bar("p_full0"), Bar("p_full1")]
    pv_done = [Bar("pv_done0"), Bar("pv_done1")]
    q_full = Bar("q_full")
    kbuf, vbuf = [None, None], [None, None]      # tile a stage holds (landed)
    sbuf = [None, None]                          # ("S" | "P", tile)
    q = [False]
    o = {"last": None, "rescaled_for": None}

    def producer():
        def land_q():
            q[0] = True
            q_full.arrive()
        pending.append(land_q)
        for j in range(n + 1):
            if j < n:
                s = j & 1
                if j >= 2 and "kempty" not in drop:
                    yield kempty[s], (j >> 1) - 1

                def land_k(s=s, j=j):
                    kbuf[s] = j
                    kfull[s].arrive()
                pending.append(land_k)
            if j >= 1:
                jv = j - 1
                s = jv & 1
                if jv >= 2 and "vempty" not in drop:
                    yield vempty[s], (jv >> 1) - 1

                def land_v(s=s, jv=jv):
                    vbuf[s] = jv
                    vfull[s].arrive()
                pending.append(land_v)

    def mma():
        yield q_full, 0
        for j in range(n + 1):
            if j < n:
                s = j & 1
                if j >= 2 and "pv_s" not in drop:
                    yield pv_done[s], (j - 2) >> 1
                yield kfull[s], j >> 1
                expect(q[0], f"S({j}) before the Q tile landed")
                expect(kbuf[s] == j, f"S({j}) reads the K stage holding tile {kbuf[s]}")
                expect(sbuf[s] is None or sbuf[s] == ("done", j - 2),
                       f"S({j}) written over {sbuf[s]}")
                sbuf[s] = ("S", j)
                kempty[s].arrive()
                s_full[s].arrive()
            if j >= 1:
                jv = j - 1
                s = jv & 1
                yield p_full[s], jv >> 1
                yield vfull[s], jv >> 1
                expect(sbuf[s] == ("P", jv), f"PV({jv}) reads {sbuf[s]}")
                expect(vbuf[s] == jv, f"PV({jv}) reads the V stage holding tile {vbuf[s]}")
                expect(o["last"] == (jv - 1 if jv > 0 else None),
                       f"PV({jv}) after PV({o['last']})")
                expect(jv == 0 or not rescale or o["rescaled_for"] == jv,
                       f"PV({jv}) before the rescale of O for it")
                o["last"] = jv
                sbuf[s] = ("done", jv)
                pv_done[s].arrive()
                vempty[s].arrive()

    def softmax():
        for j in range(n):
            s = j & 1
            yield s_full[s], j >> 1
            expect(sbuf[s] == ("S", j), f"softmax wants S({j}), buffer holds {sbuf[s]}")
            if rescale and j > 0:
                if "pv_rescale" not in drop:
                    yield pv_done[(j - 1) & 1], (j - 1) >> 1
                expect(o["last"] == j - 1, f"rescale for tile {j} after PV({o['last']})")
                o["rescaled_for"] = j
            sbuf[s] = ("P", j)
            p_full[s].arrive()
        if n > 0:
            yield pv_done[(n - 1) & 1], (n - 1) >> 1
            expect(o["last"] == n - 1, f"epilogue reads O after PV({o['last']})")

    roles = {"producer": producer(), "mma": mma(), "softmax": softmax()}
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


@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 32])
def test_prefill_tiles(n):
    for seed in range(20):
        assert run_prefill_protocol(n, seed % 2 == 0, seed) is None


@pytest.mark.parametrize("slow", ["producer", "mma", "softmax"])
def test_slow_roles(slow):
    for seed in range(10):
        assert run_prefill_protocol(9, seed % 2 == 1, seed, slow=slow) is None


# The MMA issuer also waits for PV(j - 2) before S(j) overwrites the buffer
# holding P(j - 2).  Here its own earlier MMAs complete when issued, so the
# loop order already implies that wait and leaving it out is no hazard in
# the model; in the kernel it orders the asynchronous MMAs explicitly.
SLOW_FOR = {"kempty": "mma", "vempty": "mma", "pv_rescale": "mma"}


@pytest.mark.parametrize("drop", list(SLOW_FOR))
def test_model_catches_dropped_waits(drop):
    """Leaving out any one of these waits lets some interleaving read or
    overwrite a buffer at the wrong time: the checks are not vacuous."""
    failures = 0
    for seed in range(60):
        try:
            failures += run_prefill_protocol(8, True, seed, drop=drop,
                                             slow=SLOW_FOR[drop]) is not None
        except AssertionError:
            failures += 1
    assert failures > 0
