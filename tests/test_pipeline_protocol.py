"""A model of the stage-ring protocol of the warp-specialised MHA decode
kernel, run under random interleavings on the CPU.

One producer warp fills S stages (full / empty mbarriers, a phase parity per
use) and a ring of 4 item slots; the 4 consumer warps merge each item through
a double-buffered exchange.  The stages are one sub-ring of S / 4 per consumer
warp, and block j of every item goes to sub-ring j % 4 (so a warp sums the
same blocks of an item whatever the CTA ran before).  The model
checks that no wait passes before its own data landed, that no stage, slot or
exchange buffer is overwritten while in use, and that nothing deadlocks.

It also keeps the design of an earlier build, one ring whose stage t belongs
to warp t % 4: there parity waits alias when one stage passes between warps
(a stage count that is not a multiple of 4), which once corrupted an 8-bit
kernel's barrier accounting; that case stays as a negative check.
"""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.phase = 0  # phases completed

    def arrive(self, tx=0):
        self.tx += tx
        self.pending -= 1
        assert self.pending >= 0, "over-arrival"
        self._maybe_complete()

    def complete_tx(self, n):
        self.tx -= n
        assert self.tx >= 0, "tx underflow"
        self._maybe_complete()

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def try_wait(self, parity):
        # true when the phase with this parity has completed: current phase parity != parity
        return (self.phase & 1) != parity


def simulate(items, S, W=4, slots=4, seed=0, design="subrings"):
    """design: "subrings" (the MHA kernel: one sub-ring of S / W stages per
    consumer warp, block j of every item in sub-ring j % W) or "ring" (stage
    t of one ring belongs to warp t % W, the item's first block to whichever
    warp owns the next stage; the 8-bit kernel of an earlier build)."""
    rng = random.Random(seed)
    full = [Bar(1) for _ in range(S)]
    empty = [Bar(1) for _ in range(S)]
    ifull = [Bar(1) for _ in range(slots)]
    iempty = [Bar(W) for _ in range(slots)]
    mfull = [Bar(W) for _ in range(2)]
    mempty = [Bar(W) for _ in range(2)]
    stage_owner = [None] * S    # (t) whose data the stage holds / is landing
    stage_landed = [False] * S
    slot_item = [None] * slots
    slot_q_landed = [False] * slots
    item_info = [None] * slots
    copies = []                 # pending async copies: (kind, index, value)

    S4 = S // W
    cw = [0] * W  # blocks issued into each warp's sub-ring

    def producer():
        t = 0
        pstage = 0
        pphase = 0
        for k, nb in enumerate(items + [None]):
            slot = k % slots
            while not iempty[slot].try_wait(((k // slots) & 1) ^ 1):
                yield "wait iempty"
            if nb is None:
                item_info[slot] = ("end",)
                ifull[slot].arrive()
                return
            item_info[slot] = ("item", k, nb, t)
            slot_item[slot] = k
            slot_q_landed[slot] = False
            if nb > 0:
                ifull[slot].arrive(tx=1)
                copies.append(("q", slot, k))
            else:
                ifull[slot].arrive()
            for j in range(nb):
                if design == "subrings":
                    w = j % W
                    c = cw[w]
                    cw[w] += 1
                    stage = w * S4 + c % S4
                    while not empty[stage].try_wait(((c // S4) & 1) ^ 1):
                        yield "wait empty"
                else:
                    while not empty[pstage].try_wait(pphase ^ 1):
                        yield "wait empty"
                    stage = pstage
                    pstage += 1
                    if pstage == S:
                        pstage = 0
                        pphase ^= 1
                # refill only a stage whose previous use was consumed
                assert stage_owner[stage] is None, f"stage {stage} refilled while holding t={stage_owner[stage]}"
                stage_owner[stage] = t
                stage_landed[stage] = False
                full[stage].arrive(tx=1)
                copies.append(("tile", stage, t))
                t += 1
                yield "issued"

    def consumer(warp):
        k = 0
        c = 0  # blocks this warp took from its sub-ring
        while True:
            slot = k % slots
            while not ifull[slot].try_wait((k // slots) & 1):
                yield "wait ifull"
            info = item_info[slot]
            if info[0] == "end":
                return
            _, kk, nb, t_first = info
            assert kk == k, f"warp {warp} read item {kk} expecting {k}"
            if nb > 0:
                assert slot_q_landed[slot] and slot_item[slot] == k, "q not landed"
            iempty[slot].arrive()
            yield "read item"
            if design == "subrings":
                j = warp  # the same blocks of every item: the warp's sums do not depend on history
                while j < nb:
                    stage = warp * S4 + c % S4
                    while not full[stage].try_wait((c // S4) & 1):
                        yield "wait full"
                    t = t_first + j
                    assert stage_owner[stage] == t and stage_landed[stage], \
                        f"warp {warp} t={t}: stage {stage} holds {stage_owner[stage]} landed={stage_landed[stage]}"
                    yield "compute"
                    stage_owner[stage] = None
                    empty[stage].arrive()
                    j += W
                    c += 1
            else:
                j = (warp - t_first % W + W) % W
                t0 = t_first + j
                stage = t0 % S
                phase = (t0 // S) & 1
                while j < nb:
                    while not full[stage].try_wait(phase):
                        yield "wait full"
                    t = t_first + j
                    assert stage_owner[stage] == t and stage_landed[stage], \
                        f"warp {warp} t={t}: stage {stage} holds {stage_owner[stage]} landed={stage_landed[stage]}"
                    yield "compute"
                    stage_owner[stage] = None
                    empty[stage].arrive()
                    j += W
                    stage += W
                    if stage >= S:
                        stage -= S
                        phase ^= 1
            b = k & 1
            use = (k >> 1) & 1
            while not mempty[b].try_wait(use ^ 1):
                yield "wait mempty"
            mbuf[b][warp] = k
            mfull[b].arrive()
            while not mfull[b].try_wait(use):
                yield "wait mfull"
            for w2 in range(W):
                assert mbuf[b][w2] == k, f"merge buffer {b} warp {w2} holds {mbuf[b][w2]} expecting {k}"
            yield "merge"
            mempty[b].arrive()
            k += 1

    mbuf = [[None] * W for _ in range(2)]
    actors = [producer()] + [consumer(w) for w in range(W)]
    alive = list(range(len(actors)))
    idle_rounds = 0
    steps = 0
    while alive or copies:
        progressed = False
        choices = alive[:] + (["copy"] if copies else [])
        rng.shuffle(choices)
        for c in choices:
            if c == "copy":
                i = rng.randrange(len(copies))
                kind, idx, val = copies.pop(i)
                if kind == "q":
                    slot_q_landed[idx] = True
                    ifull[idx].complete_tx(1)
                else:
                    stage_landed[idx] = True
                    full[idx].complete_tx(1)
                progressed = True
                break
            try:
                r = next(actors[c])
                if not r.startswith("wait"):
                    progressed = True
                    break
            except StopIteration:
                alive.remove(c)
                progressed = True
                break
        steps += 1
        if not progressed:
            idle_rounds += 1
            if idle_rounds > 50:
                raise AssertionError(f"deadlock after {steps} steps; alive={alive} copies={len(copies)}")
        else:
            idle_rounds = 0
    return steps


def _trial(rng, S):
    items = [rng.choice([0, 1, 2, 3, 5, 8, 17, 32]) for _ in range(rng.randint(1, 30))]
    return items


@pytest.mark.parametrize("design", ["subrings", "ring"])
@pytest.mark.parametrize("S", [4, 8, 12, 16])
def test_stage_counts_the_launchers_choose_are_safe(S, design):
    rng = random.Random(S)
    for trial in range(150):
        simulate(_trial(rng, S), S, seed=trial, design=design)


def test_a_stage_count_off_the_warp_multiple_aliases_phases():
    # the count an 8-bit launch at block 16 would take from its 48 KB budget
    # without rounding: 48 KB / (2 * 16 * 132 B) = 11 stages
    rng = random.Random(11)
    failures = 0
    for trial in range(60):
        items = [rng.choice([8, 17, 32]) for _ in range(rng.randint(5, 30))]
        try:
            simulate(items, 11, seed=trial, design="ring")
        except AssertionError:
            failures += 1
    assert failures > 0
