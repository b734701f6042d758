"""CPU model of the mbarrier protocol of the tcgen05 batched GEMV (ql_batched.cu, tc::gemv_tc_kernel).

Each role of the kernel is a generator that waits and arrives as the kernel does: the producer
lane (copies into kS shared-memory stages), 4 dequantisation groups of 4 warps (stage codes in,
A slots out), the MMA lane (A slots and accumulators in, commits out) and 4 epilogue warps.
Copies and commits complete at random later times. A hardware parity wait passes when the
barrier's current phase parity differs from the one waited on, so it cannot tell phase k - 1
from phase k + 1; every wait here names the phase index it means and the model fails when a
wait passes before that phase has completed (the fault this protocol was changed to exclude),
or when no role can move.
"""
import random

import pytest

kS, kA, kPair, kRB, kGroups = 16, 3, 2, 8, 4


class Bar:
    def __init__(self, count, name):
        self.count, self.pending, self.phase, self.name = count, count, 0, name

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: more arrivals than its count"
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def wait_passes(self, k):
        passed = (self.phase & 1) != (k & 1)
        assert not (passed and self.phase <= k), f"{self.name}: phase {k} waited, {self.phase} completed"
        return passed


def simulate(T, kwu, seed, per_group_free=True):
    rnd = random.Random(seed)
    nrb = (T + kRB - 1) // kRB
    nstage = nrb * kwu
    ps = kPair if kwu % kPair == 0 else 1
    npr = kwu // ps
    npair = nrb * npr
    sfull = [Bar(1, f"SFull{i}") for i in range(kS)]
    sfree = [Bar(4, f"SFree{i}") for i in range(kS)]
    afull = [Bar(4, f"AFull{i}") for i in range(kA)]
    afree = [Bar(1, f"AFree{i}") for i in range(kGroups if per_group_free else kA)]
    dfull = [Bar(1, "DFull0"), Bar(1, "DFull1")]
    dfree = [Bar(4, "DFree0"), Bar(4, "DFree1")]
    copies, commits = [], []

    def producer():
        for s in range(nstage):
            if s >= kS:
                while not sfree[s % kS].wait_passes(s // kS - 1):
                    yield False
            copies.append(sfull[s % kS])
            yield True

    def dequant(j):
        nfree = 0
        for g in range(j, npair, kGroups):
            rb, pp, a = g // npr, g % npr, g % kA
            if g >= kA:
                if per_group_free:
                    while not afree[j].wait_passes(nfree):
                        yield False
                    nfree += 1
                else:
                    while not afree[a].wait_passes(g // kA - 1):
                        yield False
            for u in range(ps):
                st = rb * kwu + ps * pp + u
                while not sfull[st % kS].wait_passes(st // kS):
                    yield False
                sfree[st % kS].arrive()
                yield True
            afull[a].arrive()
            yield True

    def mma():
        rb = pp = 0
        for g in range(npair):
            d, a = rb & 1, g % kA
            if pp == 0 and rb >= 2:
                while not dfree[d].wait_passes((rb >> 1) - 1):
                    yield False
            while not afull[a].wait_passes(g // kA):
                yield False
            if per_group_free:
                if g + kA < npair:
                    commits.append(afree[(g + kA) % kGroups])
            else:
                commits.append(afree[a])
            if ps * pp + ps == kwu:
                commits.append(dfull[d])
            yield True
            pp += 1
            if pp == npr:
                pp, rb = 0, rb + 1

    def epilogue():
        for rb in range(nrb):
            d = rb & 1
            while not dfull[d].wait_passes(rb >> 1):
                yield False
            dfree[d].arrive()
            yield True

    # one generator per warp: the 4 quarter warps of a group run the same schedule
    live = [producer(), mma()] + [dequant(j) for j in range(kGroups) for _ in range(4)] + [epilogue() for _ in range(4)]
    idle = 0
    while live:
        moved = False
        if copies and rnd.random() < 0.5:
            copies.pop(0).arrive()
            moved = True
        if commits and rnd.random() < 0.5:
            commits.pop(0).arrive()
            moved = True
        r = rnd.choice(live)
        try:
            moved = next(r) or moved
        except StopIteration:
            live.remove(r)
            moved = True
        idle = 0 if moved else idle + 1
        assert idle < 20000, f"no role can move (T={T}, kwu={kwu})"


@pytest.mark.parametrize("kwu", [8, 7, 3, 1])
@pytest.mark.parametrize("T", [1, 9, 21, 41, 250])
def test_protocol_never_aliases_or_stalls(T, kwu):
    for seed in range(6):
        simulate(T, kwu, seed)


def test_model_catches_shared_slot_waits():
    """Non-vacuity: the earlier protocol (one slot-free barrier per A slot, waited by whichever
    group takes the slot next) aliases on some schedule."""
    hits = 0
    for seed in range(20):
        try:
            simulate(41, 8, seed, per_group_free=False)
        except AssertionError as e:
            assert "waited" in str(e)
            hits += 1
    assert hits > 0
