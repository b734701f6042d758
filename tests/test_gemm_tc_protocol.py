"""CPU model of the mbarrier protocol of the tcgen05 prompt GEMM (ql_gemm.cu, gemm_tc_kernel).

Each role of the kernel is a generator that waits, arrives and issues as the kernel does:
* the code producer lane: one copy per unit into kSW stages, the first kSW before any wait;
* the activation producer lane: per unit an expect-tx arrival and two half copies into kSB
  stages, after the commit that frees the stage;
* the MMA lane: one wait per unit, its MMAs, one commit that frees the unit's activation stage
  and A slot, a commit for the accumulator after the last unit, a last commit it waits for;
* 16 dequantisation warps: the A slot's free phase, the code stage, an arrival that frees the
  code stage, the store into the A slot, an arrival on the unit's ready barrier; then the
  accumulator's phase and the epilogue.

Copies complete at random later times in any order. Commits complete in the order issued, each
one after all the MMAs issued before it. Besides the phase checks, the model tracks the data:
* a wait that passes before the phase it names has completed fails;
* so does an arrival that lands in another phase than the one it is meant for;
* and a schedule on which no role can move.
A code stage, an activation stage and an A slot each hold one unit at a time. A copy or a store
that overwrites a buffer another role has not finished with fails, and so does a read of a
buffer that does not hold the unit yet.
"""
import random

import pytest

kDW = 16                                        # dequantisation warps
kCodeBytes, kBHalfPerToken = 9216, 128          # one unit of 8 tiles; 64 f16 of K per token
RINGS = {256: (3, 3), 128: (3, 6), 32: (4, 7)}  # token tile -> (code stages, activation stages)


class Bar:
    """An mbarrier: a phase completes when its arrivals and its expected bytes are all in."""

    def __init__(self, count, name):
        self.count, self.pending, self.tx, self.phase, self.name = count, count, 0, 0, name

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, k, tx=0):
        assert self.phase == k, f"{self.name}: arrival for phase {k} landed in phase {self.phase}"
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: more arrivals than its count"
        self.tx += tx
        self._complete()

    def complete_tx(self, k, n):
        assert self.phase == k, f"{self.name}: bytes for phase {k} landed in phase {self.phase}"
        self.tx -= n
        self._complete()

    def wait_passes(self, k):
        passed = (self.phase & 1) != (k & 1)
        assert not (passed and self.phase <= k), f"{self.name}: phase {k} waited, {self.phase} completed"
        return passed


def simulate(NT, nst, seed, defect=None):
    kSW, kSB = RINGS[NT]
    kA = kSB
    rnd = random.Random(seed)
    half = NT * kBHalfPerToken
    wfull = [Bar(1, f"WFull{s}") for s in range(kSW)]
    wempty = [Bar(kDW, f"WEmpty{s}") for s in range(kSW)]
    ready = [Bar(kDW + (0 if defect == "ready_without_producer" else 1), f"Ready{s}") for s in range(kSB)]
    free = [Bar(1, f"Free{s}") for s in range(kSB)]
    dfull, done = Bar(1, "DFull"), Bar(1, "Done")

    # the buffers: which unit each holds, and who still uses it
    wst = [dict(unit=None, landed=False, reads=kDW) for _ in range(kSW)]
    bst = [dict(unit=None, halves=0, busy=False) for _ in range(kSB)]
    asl = [dict(unit=None, stored=set(), busy=False) for _ in range(kA)]
    mma_done = [-1]                  # the last unit whose MMAs have completed
    copies, commits = [], []         # in flight: copies land in any order, commits in issue order

    def copy_w(u):
        s = u % kSW
        assert wst[s]["reads"] == kDW, f"code stage {s} overwritten by unit {u} before every warp read unit {wst[s]['unit']}"
        wst[s].update(unit=u, landed=False, reads=0)
        wfull[s].arrive(u // kSW, tx=kCodeBytes)

        def land():
            wst[s]["landed"] = True
            wfull[s].complete_tx(u // kSW, kCodeBytes)
        copies.append(land)

    def code_producer():
        prew = min(nst, kSW)
        for u in range(prew):
            copy_w(u)
        yield True
        for u in range(prew, nst):
            while not wempty[u % kSW].wait_passes(u // kSW - 1):
                yield False
            copy_w(u)
            yield True

    def act_producer():
        for u in range(nst):
            s = u % kSB
            if u >= kSB and defect != "producer_skips_free":
                while not free[s].wait_passes(u // kSB - 1):
                    yield False
            b = bst[s]
            assert not b["busy"], f"activation stage {s} overwritten by unit {u} while MMAs of unit {b['unit']} read it"
            assert b["unit"] is None or b["unit"] == u - kSB, f"activation stage {s}: unit {b['unit']} never read"
            b.update(unit=u, halves=0)
            if defect == "ready_without_producer":
                tx = 0
            else:
                ready[s].arrive(u // kSB, tx=2 * half)
                tx = 2 * half
            for _ in range(2):
                def land(s=s, u=u, tx=tx):
                    bst[s]["halves"] += 1
                    if tx:
                        ready[s].complete_tx(u // kSB, half)
                copies.append(land)
            yield True

    def mma():
        for u in range(nst):
            s, a = u % kSB, u % kA
            while not ready[s].wait_passes(u // kSB):
                yield False
            b, sl = bst[s], asl[a]
            assert b["unit"] == u and b["halves"] == 2, f"MMAs of unit {u} read activation stage {s} before it landed"
            assert sl["unit"] == u and len(sl["stored"]) == kDW, f"MMAs of unit {u} read A slot {a} before every warp stored"
            b["busy"] = sl["busy"] = True

            def complete(u=u, s=s, a=a):
                bst[s]["busy"] = asl[a]["busy"] = False
                mma_done[0] = u
                free[s].arrive(u // kSB)
            commits.append(complete)
            if u == nst - 1:
                commits.append(lambda: dfull.arrive(0))
            yield True
        commits.append(lambda: done.arrive(0))
        while not done.wait_passes(0):
            yield False
        assert mma_done[0] == nst - 1, "tensor memory released before the MMAs completed"

    def dequant(w):
        for u in range(nst):
            s, a = u % kSW, u % kA
            if u >= kA and defect != "dequant_skips_free":
                while not free[a].wait_passes(u // kA - 1):
                    yield False
            while not wfull[s].wait_passes(u // kSW):
                yield False
            c = wst[s]
            assert c["unit"] == u and c["landed"], f"warp {w} read code stage {s} for unit {u} before it landed"
            c["reads"] += 1
            wempty[s].arrive(u // kSW)
            yield True
            sl = asl[a]
            assert not sl["busy"], f"warp {w} stored unit {u} into A slot {a} while MMAs of unit {sl['unit']} read it"
            if sl["unit"] != u:
                assert sl["unit"] is None or len(sl["stored"]) == kDW, f"A slot {a}: unit {sl['unit']} only partly stored"
                sl.update(unit=u, stored=set())
            sl["stored"].add(w)
            ready[u % kSB].arrive(u // kSB)
            yield True
        while not dfull.wait_passes(0):
            yield False
        assert mma_done[0] == nst - 1, f"warp {w} read the accumulator before the last MMAs completed"

    # slow copies or slow commits on some seeds, so that every order of landing gets explored
    p_copy, p_commit = rnd.choice([0.5, 0.1, 0.01]), rnd.choice([0.5, 0.1, 0.01])
    live = [code_producer(), act_producer(), mma()] + [dequant(w) for w in range(kDW)]
    idle = 0
    while live or copies or commits:
        moved = False
        if copies and rnd.random() < p_copy:
            copies.pop(rnd.randrange(len(copies)))()
            moved = True
        if commits and rnd.random() < p_commit:
            commits.pop(0)()
            moved = True
        if live:
            r = rnd.choice(live)
            try:
                moved = next(r) or moved
            except StopIteration:
                live.remove(r)
                moved = True
        idle = 0 if moved else idle + 1
        assert idle < 20000, f"no role can move (NT={NT}, units={nst})"


@pytest.mark.parametrize("NT", sorted(RINGS))
@pytest.mark.parametrize("nst", [1, 2, 3, 4, 7, 8, 13, 32])
def test_protocol_never_aliases_or_stalls(NT, nst):
    for seed in range(5):
        simulate(NT, nst, seed)


# what the model reports (a planted defect shows up as whichever comes first on a schedule)
DETECTIONS = ("before it landed", "before every warp", "while MMAs", "never read", "partly stored",
              "landed in phase", "waited", "more arrivals", "no role can move")


@pytest.mark.parametrize("NT", sorted(RINGS))
@pytest.mark.parametrize("defect", ["ready_without_producer", "producer_skips_free", "dequant_skips_free"])
def test_model_catches_planted_defects(NT, defect):
    """Non-vacuity: each step the protocol relies on, left out, fails on some schedule."""
    hits = 0
    for seed in range(40):
        try:
            simulate(NT, 13, seed, defect=defect)
        except AssertionError as e:
            assert any(m in str(e) for m in DETECTIONS), str(e)
            hits += 1
    assert hits > 0
