"""A model of the reverse walk's dO-slice handshake, checked over random
interleavings (CPU).

On 32-column slices the reverse walk's store warp requests each chunk's dO
slice by TMA into one of two buffers; the compute threads read chunk c + 1's
slice (after the slice barrier) to write its (gamma dO)^T image and then
arrive on barO; P^T dO of chunk c + 1 reads the slice itself once barO says
the images are written, and the compute threads wait for it (barY) before they
form Y of that chunk and write the next chunk's image.  The store warp waits on
barO's phases in order before it requests the slice two chunks on, into the
buffer that slice c used.

The model keeps the mbarrier's parity semantics (a parity wait passes while the
barrier's current phase parity differs from the one asked for) and checks, for
every chunk count and many random schedules, that:
- no slice is read before it has landed, and the reader sees the right chunk;
- no slice buffer is refilled before both its readers (the image writer and
  P^T dO) are done with it;
- nothing deadlocks, and no request is still in flight at the end.
A variant that waits for barO's phase c + 1 without first waiting for phase 0
must fail the model: that parity wait passes while phase 0 is still open.
"""
import random

import pytest


class Bar:
    """An mbarrier: arrival count per phase, transaction bytes, phase number."""

    def __init__(self, count):
        self.count, self.pending, self.phase, self.tx = count, count, 0, 0

    def arrive(self, tx=0):
        self.pending -= 1
        self.tx += tx
        assert self.pending >= 0, "more arrivals than the count in one phase"
        self._maybe()

    def complete_tx(self, b):
        self.tx -= b
        self._maybe()

    def _maybe(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def test(self, parity):
        return (self.phase & 1) != parity


def run(n, seed, first_wait=True):
    rnd = random.Random(seed)
    barO, barDO, barQ, barY = Bar(1), Bar(1), Bar(1), Bar(1)
    buf = {0: None, 1: None}       # chunk whose slice each buffer holds
    readers = {}                   # chunk -> set of readers done
    inflight = []                  # (chunk, buffer) requested, not landed

    def read(chunk, who):
        assert buf[chunk & 1] == chunk, (who, "read the wrong slice", chunk, buf)
        readers.setdefault(chunk, set()).add(who)

    def compute():
        buf[0] = 0                 # chunk 0's rows come by plain loads
        read(0, "image")
        barO.arrive()
        for ci in range(n):
            while not barY.test(ci & 1):   # Y of chunk ci: P^T dO has completed
                yield
            if ci + 1 < n:
                while not barQ.test(ci & 1):
                    yield
                while not barDO.test(ci & 1):
                    yield
                read(ci + 1, "image")
                yield
                barO.arrive()
            yield

    def do_issuer():               # P^T dO reads the slice, then Q^T (gamma dO)
        for ci in range(n):
            while not barO.test(ci & 1):
                yield
            read(ci, "P")
            barY.arrive()              # (its completion; K dh' is left out of the model)
            yield
            barQ.arrive()

    def store():
        def request(k):
            old = buf[k & 1]
            if old is not None:
                assert readers.get(old, set()) >= {"image", "P"}, ("refilled before read", k, old)
            barDO.arrive(tx=1)
            inflight.append((k, k & 1))
        if n > 1:
            if first_wait:
                while not barO.test(0):
                    yield
            request(1)
        for ci in range(n):
            if ci + 2 < n:
                while not barO.test((ci + 1) & 1):
                    yield
                request(ci + 2)
            yield

    def tma():
        while True:
            if inflight and rnd.random() < 0.3:
                k, b = inflight.pop(0)
                buf[b] = k
                barDO.complete_tx(1)
            yield

    actors = [compute(), do_issuer(), store()]
    t = tma()
    done = [False] * 3
    steps = 0
    while not all(done):
        steps += 1
        assert steps < 200000, "deadlock"
        i = rnd.randrange(4)
        if i == 3:
            next(t)
        elif not done[i]:
            try:
                next(actors[i])
            except StopIteration:
                done[i] = True
    assert not inflight, "a request still in flight at the end"


@pytest.mark.parametrize("n", range(1, 12))
def test_slice_handshake_holds(n):
    for seed in range(200):
        run(n, seed)


def test_without_the_first_phase_wait_the_model_fails():
    failed = 0
    for seed in range(200):
        try:
            run(6, seed, first_wait=False)
        except AssertionError:
            failed += 1
    assert failed > 0
