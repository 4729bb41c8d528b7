"""A model of the synchronisation protocol of the 16-bit tensor-core
grouped-query decode kernel (pa_decode_gqa), run under random interleavings on
the CPU.

Actors: the K producer warp (item ring, the K half of a ring of S stages, a
record per stage of the tile's blocks), the V producer warp (reads the
records in tile order, fills the V half of each stage), the MMA thread (S of
tile g, then P V of tile g - 1), and four softmax warps (score tile g, then
the epilogue of tile g - 1).  The tensor core runs MMAs in issue order and
copies land in any order.  Barriers carry a completed-phase count: a wait for
phase n passes on the parity test and then asserts that the barrier completed
exactly phase n, so parity aliasing shows up as a failed assertion or a
deadlock.  Buffer hazards are checked directly:

  - a stage's K half is refilled only after S of its tile finished and every
    softmax warp read the tile's block mask;
  - its V half only after P V of its tile finished;
  - a record is rewritten only after the V producer read it;
  - P buffer g & 1 only after P V of tile g - 2;
  - the rescale slot g & 3 only after every warp's epilogue of tile g - 4.

Two variants are kept as negative checks: a K producer that does not wait for
the V producer to hand a record back, and a K half released by the S commit
alone (before the softmax warps read the block mask).
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
    kernel), "no_record_release" or "k_free_at_s"."""
    rng = random.Random(seed)
    SL, NW = 4, 4
    kfull = [Bar(f"kfull{i}", 1) for i in range(S)]
    vfull = [Bar(f"vfull{i}", 1) for i in range(S)]
    kempty = [Bar(f"kempty{i}", 1 if design == "k_free_at_s" else 1 + NW) for i in range(S)]
    vempty = [Bar(f"vempty{i}", 1) for i in range(S)]
    zfull = [Bar(f"zfull{i}", 1) for i in range(S)]
    zfree = [Bar(f"zfree{i}", 1) for i in range(S)]
    ifull = [Bar(f"ifull{i}", 1) for i in range(SL)]
    iempty = [Bar(f"iempty{i}", NW + 1) for i in range(SL)]
    sfull = [Bar(f"sfull{i}", 1) for i in range(2)]
    sfree = [Bar(f"sfree{i}", NW) for i in range(2)]
    pfull = [Bar(f"pfull{i}", NW) for i in range(2)]
    ofull = [Bar(f"ofull{i}", 1) for i in range(2)]
    ofree = [Bar(f"ofree{i}", NW) for i in range(2)]
    tc, copies = [], []
    done = {"S": set(), "PV": set()}
    mask_of = [None] * S    # tile whose block mask the stage's mask word holds
    record = [None] * S     # the V producer's record: ("tile", t) or ("end",)
    k_half = [None] * S
    v_half = [None] * S
    mask_reads, epi = {}, {}
    first = []
    t = 0
    for nt in items:
        first.append(t)
        t += nt
    total = t

    def wait(bar, n, who):
        while not bar.ready(n):
            yield "wait"
        bar.check(n, who)

    def k_producer():
        tk = 0
        for k, nt in enumerate(items + [None]):
            slot = k % SL
            if k >= SL:
                yield from wait(iempty[slot], k // SL - 1, "K producer iempty")
            ifull[slot].arrive()
            if nt is None:
                break
            for _ in range(nt):
                st = tk % S
                if tk >= S:
                    yield from wait(kempty[st], tk // S - 1, "K producer kempty")
                    assert tk - S in done["S"], f"K half {st} refilled before S({tk - S})"
                    assert mask_reads.get(tk - S, 0) == NW, f"mask of stage {st} rewritten before every softmax read"
                    if design != "no_record_release":
                        yield from wait(zfree[st], tk // S - 1, "K producer zfree")
                mask_of[st] = tk
                record[st] = ("tile", tk)
                k_half[st] = tk
                copies.append(("K", st))
                zfull[st].arrive()
                tk += 1
                yield "issue"
        st = tk % S
        if tk >= S and design != "no_record_release":
            yield from wait(zfree[st], tk // S - 1, "K producer zfree (end)")
        record[st] = ("end",)
        zfull[st].arrive()

    def v_producer():
        tv = 0
        while True:
            st = tv % S
            yield from wait(zfull[st], tv // S, "V producer zfull")
            rec = record[st]
            if rec[0] == "end":
                assert tv == total, f"end record after {tv} of {total} tiles"
                return
            assert rec == ("tile", tv), f"V producer read {rec} for tile {tv}"
            zfree[st].arrive()  # the record is in registers
            yield "read"
            if tv >= S:
                yield from wait(vempty[st], tv // S - 1, "V producer vempty")
                assert tv - S in done["PV"], f"V half {st} refilled before P V({tv - S})"
            v_half[st] = tv
            copies.append(("V", st))
            tv += 1

    def mma():
        g = 0
        prev = None

        def pv(gp, tp):
            b = gp & 1
            yield from wait(pfull[b], gp // 2, "P V pfull")
            if gp >= 2:
                yield from wait(ofree[b], gp // 2 - 1, "P V ofree")
            yield from wait(vfull[tp % S], tp // S, "P V vfull")
            assert v_half[tp % S] == tp
            tc.append(("PV", gp, b, tp))

        for k, nt in enumerate(items):
            slot = k % SL
            yield from wait(ifull[slot], k // SL, "MMA ifull")
            if nt == 0:
                iempty[slot].arrive()
                continue
            for ti in range(nt):
                t = first[k] + ti
                b = g & 1
                yield from wait(kfull[t % S], t // S, "S kfull")
                assert k_half[t % S] == t
                if g >= 2:
                    yield from wait(sfree[b], g // 2 - 1, "S sfree")
                tc.append(("S", g, b, t))
                if ti == nt - 1:
                    tc.append(("iempty", slot))
                if prev is not None:
                    yield from pv(*prev)
                prev = (g, t)
                g += 1
        if prev is not None:
            yield from pv(*prev)

    def softmax():
        g = 0
        pend = None

        def epilogue(gp):
            b = gp & 1
            yield from wait(pfull[b], gp // 2, "epilogue pfull")
            yield from wait(ofull[b], gp // 2, "epilogue ofull")
            assert gp in done["PV"]
            yield "read"
            epi[gp] = epi.get(gp, 0) + 1
            ofree[b].arrive()

        for k, nt in enumerate(items):
            slot = k % SL
            yield from wait(ifull[slot], k // SL, "softmax ifull")
            iempty[slot].arrive()
            for ti in range(nt):
                t = first[k] + ti
                b = g & 1
                yield from wait(kfull[t % S], t // S, "softmax kfull")
                yield from wait(sfull[b], g // 2, "softmax sfull")
                assert g in done["S"]
                assert mask_of[t % S] == t, f"softmax({t}) read the mask of tile {mask_of[t % S]}"
                mask_reads[t] = mask_reads.get(t, 0) + 1
                sfree[b].arrive()
                if design != "k_free_at_s":
                    kempty[t % S].arrive()
                if rng.random() < 0.5:  # a row past the attended tokens: its V row is zeroed once V landed
                    yield from wait(vfull[t % S], t // S, "softmax vfull")
                    assert v_half[t % S] == t
                assert g < 2 or g - 2 in done["PV"], f"P buffer {b} rewritten while P V({g - 2}) is pending"
                assert g < 4 or epi.get(g - 4, 0) == NW, f"rescale slot {g & 3} rewritten before epilogue({g - 4})"
                yield "compute"
                pfull[b].arrive()
                if pend is not None:
                    yield from epilogue(pend)
                pend = g
                g += 1
        if pend is not None:
            yield from epilogue(pend)

    actors = [k_producer(), v_producer(), mma()] + [softmax() for _ in range(NW)]
    alive = list(range(len(actors)))
    idle = 0
    while alive or copies or tc:
        choices = alive[:] + (["copy"] if copies else []) + (["tc"] if tc else [])
        rng.shuffle(choices)
        progressed = False
        for c in choices:
            if c == "copy":
                kind, st = copies.pop(rng.randrange(len(copies)))
                (kfull if kind == "K" else vfull)[st].arrive()
                progressed = True
                break
            if c == "tc":
                op = tc.pop(0)
                if op[0] == "S":
                    done["S"].add(op[1])
                    sfull[op[2]].arrive()
                    kempty[op[3] % S].arrive()
                elif op[0] == "iempty":
                    iempty[op[1]].arrive()
                else:
                    done["PV"].add(op[1])
                    ofull[op[2]].arrive()
                    vempty[op[3] % S].arrive()
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
            if idle > 300:
                raise Deadlock(f"deadlock; actors alive {alive}")


def _cases(n, seed):
    rng = random.Random(seed)
    for trial in range(n):
        items = [rng.choice([0, 0, 1, 1, 2, 3, 5, 8]) for _ in range(rng.randint(1, 25))]
        yield items, rng.choice([2, 3, 4]), trial


def test_final_protocol_never_deadlocks_aliases_or_overwrites():
    for items, S, trial in _cases(300, 11):
        simulate(items, S, "final", seed=trial)


@pytest.mark.parametrize("design", ["no_record_release", "k_free_at_s"])
def test_the_rejected_variants_fail_in_the_model(design):
    bad = 0
    for items, S, trial in _cases(200, 11):
        try:
            simulate(items, S, design, seed=trial)
        except AssertionError:
            bad += 1
    assert bad > 0
