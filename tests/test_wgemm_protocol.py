"""Model of the weight-streaming GEMM's protocol (wgemm.cu), CPU only.

One CTA of the GEMM runs a TMA producer (weight tiles of the first ring
stages requested before the wait on the previous kernel, activation tiles
after it, then both for every later K chunk once the stage is free), an MMA
issuer (waits for a stage's bytes, issues its MMAs, commits the stage back
to the producer, and after the last chunk commits the accumulator-done
barrier) and the epilogue warps (wait on the previous kernel before writing
outputs, wait for the accumulator, reuse the ring's shared memory as a
staging buffer).  With several K splits the CTAs of one output tile write
fp32 partials, fence, and count themselves on a per-tile counter; the CTA
that makes the count complete resets it for the next launch and sums the
partials in split order.

As for the attention kernels' models, each role's order of waits, arrivals
and buffer accesses is restated (none of the arithmetic) and driven in many
random interleavings.  Copies land in random order; MMAs execute in issue
order on a tensor pipe that runs at random times, and a commit arrives once
every MMA issued before it has executed.  The model fails on deadlock, on a
parity wait passing on the wrong phase, when a copy is issued into a stage
whose previous chunk has not been consumed, when an MMA reads a stage
missing either half of its chunk, when activations or outputs are touched
before the previous kernel is done, when the epilogue reads the accumulator
before the last MMA or reuses the ring while a copy is in flight, and when
a split-K reduction reads a partial not yet written.  A change to the order
of waits, arrivals or accesses in the kernel must be made here too.
"""
from __future__ import annotations

import random

import pytest

from test_attend_protocol import Bar, expect

KA, KB = 16384, 32768   # bytes of a stage's weight and activation halves (NT = 256)


class TxBar:
    """mbarrier with one expected arrival per phase plus a transaction count:
    the phase completes when the arrival came and every expected byte landed."""

    def __init__(self, name: str):
        self.name, self.arrived, self.tx, self.done = name, False, 0, 0

    def arrive_expect_tx(self, nbytes: int):
        expect(not self.arrived, f"{self.name}: second arrival in one phase")
        self.arrived, self.tx = True, self.tx + nbytes
        self._maybe_complete()

    def complete_tx(self, nbytes: int):
        self.tx -= nbytes
        self._maybe_complete()

    def _maybe_complete(self):
        if self.arrived and self.tx == 0:
            self.done += 1
            self.arrived = False

    def ready(self, phase: int) -> bool:
        ok = (self.done & 1) != (phase & 1)
        if ok and self.done != phase + 1:
            raise AssertionError(f"{self.name}: wait for phase {phase} passed at done={self.done}")
        return ok


def run_cta(nk: int, S: int, seed: int | None, drop: str = "", slow: str = ""):
    """One CTA over nk K chunks with an S-stage ring.  Returns None when every
    role finishes, else the blocked roles."""
    rnd = random.Random(seed)
    full = [TxBar(f"full{s}") for s in range(S)]
    empty = [Bar(f"empty{s}") for s in range(S)]
    done = Bar("done")
    prev_kernel = {"done": False}
    stage = [{"A": None, "B": None} for _ in range(S)]
    consumed = set()          # chunks whose MMAs executed
    copies = []               # copies in flight: (kind, chunk, stage)
    pipe = []                 # tensor pipe queue: ("mma", chunk) | ("commit", bar)
    acc = {"mmas": 0}

    def issue_copy(kind, i):
        s = i % S
        expect(i < S or (i - S) in consumed,
               f"{kind} copy of chunk {i} into stage {s} before chunk {i - S} was consumed")
        if kind == "B":
            expect(prev_kernel["done"], f"activation copy of chunk {i} before the previous kernel")
        copies.append((kind, i, s))

    def land(c):
        kind, i, s = c
        stage[s][kind] = i
        if not (kind == "B" and "b_bytes" in drop):
            full[s].complete_tx(KA if kind == "A" else KB)

    def producer():
        pre = min(nk, S)
        per_stage = KA if "b_bytes" in drop else KA + KB
        for i in range(pre):
            full[i].arrive_expect_tx(per_stage)
            issue_copy("A", i)
            if "grid_wait" in drop:
                issue_copy("B", i)
        if "grid_wait" not in drop:
            while not prev_kernel["done"]:
                yield None, None       # griddepcontrol.wait
            for i in range(pre):
                issue_copy("B", i)
        for i in range(pre, nk):
            s = i % S
            if "empty" not in drop:
                yield empty[s], (i // S) - 1
            full[s].arrive_expect_tx(per_stage)
            issue_copy("A", i)
            issue_copy("B", i)

    def mma():
        for i in range(nk):
            s = i % S
            if "full" not in drop:
                yield full[s], i // S
            pipe.append(("mma", i))
            pipe.append(("commit", empty[s]))
        pipe.append(("commit", done))

    def epilogue():
        while not prev_kernel["done"]:
            yield None, None           # griddepcontrol.wait before writing outputs
        if "done" not in drop:
            yield done, 0
        expect(acc["mmas"] == nk, f"epilogue reads the accumulator after {acc['mmas']} of {nk} MMAs")
        expect(not copies, f"staging reuses the ring with copies in flight: {copies}")

    def execute_pipe():
        op = pipe.pop(0)
        if op[0] == "mma":
            i = op[1]
            s = i % S
            expect(stage[s]["A"] == i and stage[s]["B"] == i,
                   f"MMA of chunk {i} reads stage {s} holding {stage[s]}")
            consumed.add(i)
            acc["mmas"] += 1
        else:
            op[1].arrive()

    roles = {"producer": producer(), "mma": mma(), "epilogue": epilogue()}
    waiting = {r: None for r in roles}
    alive = list(roles)
    while alive:
        def can_run(r):
            w = waiting[r]
            if w is None:
                return True
            if w[0] is None:
                return prev_kernel["done"]
            return w[0].ready(w[1])
        cand = [r for r in alive if can_run(r)]
        events = []
        if copies:
            events.append("copy")
        if pipe:
            events.append("pipe")
        if not prev_kernel["done"]:
            events.append("prev")
        if events and (not cand or rnd.random() < 0.45):
            e = rnd.choice(events)
            if e == "copy":
                land(copies.pop(rnd.randrange(len(copies))))
            elif e == "pipe":
                execute_pipe()
            else:
                prev_kernel["done"] = True
            continue
        if not cand:
            return {r: (waiting[r][0].name if waiting[r][0] else "grid", waiting[r][1])
                    for r in alive}
        fast = [r for r in cand if not (slow and r == slow)]
        pick = fast if fast and rnd.random() < 0.97 else cand
        r = rnd.choice(pick) if seed is not None else pick[0]
        try:
            waiting[r] = next(roles[r])
        except StopIteration:
            alive.remove(r)
            waiting[r] = None
    return None


def run_split_k(splits: int, launches: int, seed: int, drop: str = ""):
    """The split-K reduction of one output tile over back-to-back launches
    sharing the tile counter.  Each CTA: write partial, fence, count; the
    CTA completing the count resets it and reads every partial.  A launch's
    epilogues start only after the previous launch has finished (they wait
    on it first).  Returns the number of reducing CTAs per launch."""
    rnd = random.Random(seed)
    counter = [0]
    reducers = []
    for launch in range(launches):
        written = set()
        steps = {z: 0 for z in range(splits)}
        last_ctas = 0
        flags = {}
        while steps:
            z = rnd.choice(list(steps))
            k = steps[z]
            if k == 0:
                written.add(z)                    # partial stored, then __threadfence
            elif k == 1:
                prev = counter[0]
                counter[0] += 1                   # atomicAdd
                target = splits - 2 if "off_by_one" in drop else splits - 1
                flags[z] = prev == target
                if flags[z] and "reset" not in drop:
                    counter[0] = 0
            else:
                if flags[z]:
                    last_ctas += 1
                    expect(written == set(range(splits)),
                           f"launch {launch}: reduction with partials {sorted(written)} written")
                del steps[z]
                continue
            steps[z] = k + 1
        reducers.append(last_ctas)
    return reducers


@pytest.mark.parametrize("nk,S", [(1, 4), (2, 2), (3, 4), (4, 4), (9, 4), (37, 4), (8, 3),
                                  (85, 4), (2, 6), (13, 6), (40, 5)])
def test_ring(nk, S):
    for seed in range(25):
        assert run_cta(nk, S, seed) is None


@pytest.mark.parametrize("slow", ["producer", "mma", "epilogue"])
def test_slow_roles(slow):
    for seed in range(15):
        assert run_cta(11, 4, seed, slow=slow) is None


@pytest.mark.parametrize("splits", [2, 3, 7, 16])
def test_split_k_reduction(splits):
    for seed in range(40):
        assert run_split_k(splits, 3, seed) == [1, 1, 1]


# Each dropped wait or miscounted byte lets some interleaving touch a buffer
# at the wrong time; the slow role is the one whose lag exposes it.
RING_SLIPS = {"empty": "mma", "full": "producer", "done": "mma", "b_bytes": "",
              "grid_wait": ""}


@pytest.mark.parametrize("drop", list(RING_SLIPS))
def test_model_catches_ring_slips(drop):
    failures = 0
    for seed in range(80):
        try:
            failures += run_cta(12, 4, seed, drop=drop, slow=RING_SLIPS[drop]) is not None
        except AssertionError:
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("drop", ["off_by_one", "reset"])
def test_model_catches_split_k_slips(drop):
    failures = 0
    for seed in range(40):
        try:
            failures += run_split_k(4, 3, seed, drop=drop) != [1, 1, 1]
        except AssertionError:
            failures += 1
    assert failures > 0
