"""Host model of the one-CTA blockscale kernel's TMEM buffer protocol on the band
path (gemm_blockscale.cu: BufSeq, the tile park and the store warps).

Three roles share two TMEM K-block buffers through mbarriers:
- the MMA warp fills a buffer per K-step once the buffer's empty barrier has
  completed;
- the eight epilogue warps read it after its full barrier.  They release it, or,
  at a tile's last K-step, write the tile's sums back into it (the park) and
  arrive on the park barrier;
- the four store warps copy a park out and release its buffer, two arrivals
  each.

The model follows the kernel's buffer sequence and mbarrier parity rule: a wait
for parity p passes once the barrier's current phase parity differs from p.  It
runs random interleavings and checks three things: no role waits forever, the
MMA never overwrites a buffer that is still being read or still holds a park,
and the store warps find their tile in the buffer they expect.  It also checks
that two plausible protocol mistakes fail it: a lead that is not capped at the
tile's K-steps minus one, and a store warp that releases the buffer before it
has read the park."""
import random

import pytest

PARK_LEAD = 2   # kParkLead in gemm_blockscale.cu


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0

    def arrive(self, n=1):
        self.pending -= n
        assert self.pending >= 0, "more arrivals than the barrier's count"
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def passes(self, parity):
        return (self.phase & 1) != parity


class BufSeq:
    """The kernel's BufSeq::next."""

    def __init__(self, lead_cap=True):
        self.use = [0, 0]
        self.last = 1
        self.lead_cap = lead_cap

    def next(self, ks, nks, park):
        lead = min(PARK_LEAD, nks - 1) if self.lead_cap else PARK_LEAD
        if not park:
            b = (self.use[0] + self.use[1]) & 1
        else:
            b = (1 - self.last) if ks < lead else self.last ^ ((ks - lead) & 1)
        n = self.use[b]
        self.use[b] += 1
        if ks == nks - 1:
            self.last = b
        return b, n


def run_model(ntiles, nks, park, seed, lead_cap=True, early_release=False, max_steps=200_000):
    """True if every role finishes; an AssertionError on an overwrite or a wrong park."""
    rnd = random.Random(seed)
    tfull = [Barrier(1), Barrier(1)]
    tempty = [Barrier(8), Barrier(8)]
    park_full = Barrier(8)
    tmem = [None, None]   # ('kb', tile, ks) or ('park', tile) or None

    def mma():
        seq = BufSeq(lead_cap)
        for t in range(ntiles):
            for ks in range(nks):
                b, n = seq.next(ks, nks, park)
                while not tempty[b].passes((n & 1) ^ 1):
                    yield
                assert tmem[b] is None, f"MMA overwrites {tmem[b]} with tile {t} K-step {ks}"
                tmem[b] = ("kb", t, ks)
                tfull[b].arrive()
                yield

    def epilogue():
        seq = BufSeq(lead_cap)
        for t in range(ntiles):
            for ks in range(nks):
                b, n = seq.next(ks, nks, park)
                while not tfull[b].passes(n & 1):
                    yield
                assert tmem[b] == ("kb", t, ks), f"epilogue expected tile {t} K-step {ks}, found {tmem[b]}"
                yield   # the TMEM loads
                if park and ks == nks - 1:
                    tmem[b] = ("park", t)
                    park_full.arrive(8)
                else:
                    tmem[b] = None
                    tempty[b].arrive(8)
                yield

    def store_warps():
        if not park:
            return
        seq = BufSeq(lead_cap)
        parked = 0
        for t in range(ntiles):
            b = None
            for ks in range(nks):
                b, _ = seq.next(ks, nks, True)
            while not park_full.passes(parked & 1):
                yield
            parked += 1
            assert tmem[b] == ("park", t), f"store warps expected the park of tile {t}, found {tmem[b]}"
            if early_release:
                for _ in range(4):
                    tempty[b].arrive(2)
                yield
                tmem[b] = None
            else:
                for _ in range(rnd.randint(0, 6)):   # a slow drain
                    yield
                tmem[b] = None
                for _ in range(4):
                    tempty[b].arrive(2)
            yield

    alive = [mma(), epilogue(), store_warps()]
    steps = 0
    while alive:
        role = rnd.choice(alive)
        try:
            next(role)
        except StopIteration:
            alive.remove(role)
        steps += 1
        if steps > max_steps:
            return False
    return True


@pytest.mark.parametrize("nks", [1, 2, 3, 4, 16, 17])
@pytest.mark.parametrize("park", [False, True])
def test_protocol_completes_without_overwrites(nks, park):
    for seed in range(25):
        assert run_model(5, nks, park, seed), f"a role waited forever: K-steps {nks}, park {park}, seed {seed}"


def test_uncapped_lead_is_caught():
    # with fewer K-steps per tile than the lead, a second park can complete before the store
    # warps have waited for the first, and their parity wait then misses a phase
    outcomes = [run_model(5, 2, True, seed, lead_cap=False) for seed in range(60)]
    assert not all(outcomes)


def test_early_release_is_caught():
    with pytest.raises(AssertionError, match="MMA overwrites"):
        for seed in range(60):
            run_model(5, 16, True, seed, early_release=True)
