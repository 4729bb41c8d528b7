"""A model of the synchronisation protocol of the tensor-core E4M3 decode
kernel (pa_decode_q8t), run under random interleavings on the CPU.

Actors: the producer warp (item records, K / V copies into a ring of S
stages), the query converter (claims items and builds each item's query
operand), the S issuer, the P V issuer, four softmax warps and four epilogue
warps; the tensor core executes MMAs in issue order and TMA copies land in any
order.  Barriers carry a completed-phase count: a wait for phase n passes on
the parity test and then asserts that the barrier completed exactly phase n,
so parity aliasing shows up as a failed assertion or a deadlock.  Buffer
hazards are checked directly: the softmax of tile g overwrites P buffer g & 1
only after P V of tile g - 2 has finished, and the factor slot g & 3 only after
the epilogue of tile g - 4; a stage is refilled only after its tile was fully
consumed.

The epilogue of an item's last tile merges the four quarters from the item's
final softmax state, which the softmax warps leave in slot g & 3; the model
checks that the slot still holds that tile's state when the merge has read it.

The query converter claims item k only once the producer has at most four
tiles of item k - 1 left to issue, so a CTA holds at most one claimed item it
has not started, and only near its current item's end (claimed up to four
items ahead, the launch's last items sat queued behind other items in a few
CTAs while the rest had none).

Three variants that were tried on the way are kept as negative checks: an
epilogue that waits on the 2-deep P barrier (the softmax warps may complete it
twice before the epilogue looks), a single MMA thread that defers each tile's
P V behind the next S without issuing it before it blocks on an item (empty
items then fill every item slot), and an epilogue that frees its O buffer
before the merge has read the final state (P V of tile g + 2, then S and the
softmax of tile g + 4 may go ahead and rewrite the slot: outputs of a kv head
came out wrong now and then on the GPU before this was found).
"""
import random

import pytest


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.cp = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: over-arrival"
        if self.pending == 0:
            self.cp += 1
            self.pending = self.count

    def ready(self, n):
        # try_wait.parity(n & 1): the phase of that parity is the last completed
        return (self.cp & 1) != (n & 1)

    def check(self, n, who):
        assert self.cp == n + 1, f"{who}: waited {self.name} phase {n}, barrier completed {self.cp} phases"


class Deadlock(AssertionError):
    pass


def simulate(items, S, design="final", seed=0):
    """items: tiles per item (0 = an empty item).  design: "final" (the
    kernel), "claim_ahead", "pfull_epilogue", "single_issuer_no_flush" or
    "ofree_before_merge".  Returns the most items the converter had claimed
    beyond the one the producer was on."""
    rng = random.Random(seed)
    SL = 4
    two_issuers = design != "single_issuer_no_flush"
    full = [Bar(f"full{i}", 1) for i in range(S)]
    empty = [Bar(f"empty{i}", 1) for i in range(S)]
    ifull = [Bar(f"ifull{i}", 2 if two_issuers else 1) for i in range(SL)]
    iempty = [Bar(f"iempty{i}", 10 if two_issuers else 9) for i in range(SL)]
    sfull = [Bar(f"sfull{i}", 1) for i in range(2)]
    sfree = [Bar(f"sfree{i}", 4) for i in range(2)]
    pfull = [Bar(f"pfull{i}", 4) for i in range(2)]
    afull = [Bar(f"afull{i}", 4) for i in range(4)]
    ofull = [Bar(f"ofull{i}", 1) for i in range(2)]
    ofree = [Bar(f"ofree{i}", 4) for i in range(2)]
    NEAR = 4  # tiles of an item still to issue when the next item is claimed
    pnear = [Bar(f"pnear{i}", 1) for i in range(SL)]
    tc = []      # tensor core queue, in issue order
    copies = []  # copies in flight, any order
    pv_done, epi_done, stage_done = set(), set(), set()
    stage_tile = [None] * S
    first = []
    producer_at, claimed = [-1], [-1]  # items the producer started and the converter claimed
    lead = [0]  # most items claimed beyond the producer's
    t = 0
    for nt in items:
        first.append(t)
        t += nt

    def wait(bar, n, who):
        while not bar.ready(n):
            yield "wait"
        bar.check(n, who)

    def producer():
        t = 0
        for k, nt in enumerate(items + [None]):
            slot = k % SL
            if k >= SL:
                yield from wait(iempty[slot], k // SL - 1, "producer iempty")
            ifull[slot].arrive()
            producer_at[0] = k
            if nt is None:
                return
            if nt <= NEAR:
                pnear[slot].arrive()
            for ti in range(nt):
                st = t % S
                if t >= S:
                    yield from wait(empty[st], t // S - 1, "producer empty")
                    assert t - S in stage_done, f"stage {st} refilled before tile {t - S} was consumed"
                stage_tile[st] = t
                copies.append(st)
                t += 1
                yield "issue"
                if ti == nt - 1 - NEAR:
                    pnear[slot].arrive()

    def converter():
        for k, nt in enumerate(items + [None]):
            slot = k % SL
            if k >= SL:
                yield from wait(iempty[slot], k // SL - 1, "converter iempty")
            if k > 0 and design != "claim_ahead":
                # item k is claimed once the producer has at most NEAR tiles of
                # item k - 1 left to issue
                yield from wait(pnear[(k - 1) % SL], (k - 1) // SL, "converter pnear")
                assert producer_at[0] >= k - 1
            claimed[0] = k
            lead[0] = max(lead[0], claimed[0] - producer_at[0])
            yield "convert"
            ifull[slot].arrive()
            if nt is None:
                return

    def pv(g, st):
        b = g & 1
        yield from wait(pfull[b], g // 2, "pv pfull")
        if g >= 2:
            yield from wait(ofree[b], g // 2 - 1, "pv ofree")
        tc.append(("PV", g, b, st))

    def s_issuer():
        g = 0
        for k, nt in enumerate(items):
            slot = k % SL
            yield from wait(ifull[slot], k // SL, "s ifull")
            if nt == 0:
                iempty[slot].arrive()
                continue
            for ti in range(nt):
                t = first[k] + ti
                b = g & 1
                yield from wait(full[t % S], t // S, "s full")
                if g >= 2:
                    yield from wait(sfree[b], g // 2 - 1, "s sfree")
                    yield from wait(ofull[b], g // 2 - 1, "s ofull")
                tc.append(("S", g, b))
                if ti == nt - 1:
                    tc.append(("iempty", slot))
                g += 1

    def pv_issuer():
        g = 0
        for k, nt in enumerate(items):
            slot = k % SL
            yield from wait(ifull[slot], k // SL, "pv ifull")
            iempty[slot].arrive()
            for ti in range(nt):
                yield from pv(g, (first[k] + ti) % S)
                g += 1

    def single_issuer():  # S(g) then the deferred P V(g - 1), never flushed
        g = 0
        prev = None
        for k, nt in enumerate(items):
            slot = k % SL
            yield from wait(ifull[slot], k // SL, "mma ifull")
            if nt == 0:
                iempty[slot].arrive()
                continue
            for ti in range(nt):
                t = first[k] + ti
                b = g & 1
                yield from wait(full[t % S], t // S, "mma full")
                if g >= 2:
                    yield from wait(sfree[b], g // 2 - 1, "mma sfree")
                tc.append(("S", g, b))
                if ti == nt - 1:
                    tc.append(("iempty", slot))
                if prev is not None:
                    yield from pv(*prev)
                prev = (g, t % S)
                g += 1
        if prev is not None:
            yield from pv(*prev)

    def softmax():
        g = 0
        for k, nt in enumerate(items):
            slot = k % SL
            yield from wait(ifull[slot], k // SL, "softmax ifull")
            iempty[slot].arrive()
            for ti in range(nt):
                t = first[k] + ti
                b = g & 1
                yield from wait(full[t % S], t // S, "softmax full")
                assert stage_tile[t % S] == t
                yield from wait(sfull[b], g // 2, "softmax sfull")
                sfree[b].arrive()
                assert g < 2 or g - 2 in pv_done, f"P buffer {b} overwritten while P V({g - 2}) is pending"
                assert g < 4 or g - 4 in epi_done, f"factor slot {g & 3} overwritten before epilogue({g - 4})"
                yield "compute"
                if ti == nt - 1:
                    final_slot[g & 3] = g  # the item's final softmax state
                pfull[b].arrive()
                afull[g & 3].arrive()
                g += 1

    epi_count = {}
    final_slot = [None] * 4  # tile whose item's final softmax state each slot holds

    def epilogue():
        g = 0
        for k, nt in enumerate(items):
            slot = k % SL
            yield from wait(ifull[slot], k // SL, "epilogue ifull")
            iempty[slot].arrive()
            for ti in range(nt):
                b = g & 1
                if design == "pfull_epilogue":
                    yield from wait(pfull[b], g // 2, "epilogue pfull")
                else:
                    yield from wait(afull[g & 3], g // 4, "epilogue afull")
                yield from wait(ofull[b], g // 2, "epilogue ofull")
                assert g in pv_done
                yield "read"
                last = ti == nt - 1
                if not last or design == "ofree_before_merge":
                    ofree[b].arrive()
                if last:
                    # the item's merge reads its final state from slot g & 3
                    yield "merge"
                    assert final_slot[g & 3] == g, f"final-state slot {g & 3} rewritten during the merge of tile {g}"
                    if design != "ofree_before_merge":
                        ofree[b].arrive()
                epi_count[g] = epi_count.get(g, 0) + 1
                if epi_count[g] == 4:
                    epi_done.add(g)
                g += 1

    if two_issuers:
        actors = [producer(), converter(), s_issuer(), pv_issuer()]
    else:
        actors = [producer(), single_issuer()]
    actors += [softmax() for _ in range(4)] + [epilogue() for _ in range(4)]
    alive = list(range(len(actors)))
    idle = 0
    while alive or copies or tc:
        choices = alive[:] + (["copy"] if copies else []) + (["tc"] if tc else [])
        rng.shuffle(choices)
        progressed = False
        for c in choices:
            if c == "copy":
                full[copies.pop(rng.randrange(len(copies)))].arrive()
                progressed = True
                break
            if c == "tc":
                op = tc.pop(0)
                if op[0] == "S":
                    sfull[op[2]].arrive()
                elif op[0] == "iempty":
                    iempty[op[1]].arrive()
                else:
                    _, g, b, st = op
                    pv_done.add(g)
                    stage_done.add(stage_tile[st])
                    ofull[b].arrive()
                    empty[st].arrive()
                progressed = True
                break
            try:
                if next(actors[c]) != "wait":
                    progressed = True
                    break
            except StopIteration:
                alive.remove(c)
                progressed = True
                break
        if progressed:
            idle = 0
        else:
            idle += 1
            if idle > 200:
                raise Deadlock(f"deadlock; actors alive {alive}")
    return lead[0]


def _cases(n, seed):
    rng = random.Random(seed)
    for trial in range(n):
        items = [rng.choice([0, 1, 1, 2, 3, 5, 8, 16]) for _ in range(rng.randint(1, 25))]
        yield items, rng.choice([2, 3, 4, 5, 8]), trial


def test_final_protocol_never_deadlocks_aliases_or_overwrites():
    for items, S, trial in _cases(400, 7):
        assert simulate(items, S, "final", seed=trial) <= 1


def test_converter_claims_at_most_one_item_ahead_of_the_producer():
    leads = [simulate(items, S, "claim_ahead", seed=trial) for items, S, trial in _cases(200, 7)]
    assert max(leads) > 1  # without the wait it runs further ahead
    assert max(simulate(items, S, "final", seed=trial) for items, S, trial in _cases(200, 7)) == 1


def _fails(design, n=300):
    bad = 0
    for items, S, trial in _cases(n, 7):
        try:
            simulate(items, S, design, seed=trial)
        except AssertionError:
            bad += 1
    return bad


@pytest.mark.parametrize("design", ["pfull_epilogue", "single_issuer_no_flush", "ofree_before_merge"])
def test_the_rejected_variants_fail_in_the_model(design):
    assert _fails(design) > 0
