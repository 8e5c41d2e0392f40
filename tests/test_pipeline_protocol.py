"""A model of the logits kernels' shared-memory hand-offs, run under random interleavings
on the CPU.

The kernels pass buffers between warps through mbarriers, waited on by phase parity: a
wait for parity P succeeds while the barrier's current phase index has the other parity.
Such a wait cannot tell a phase from the one two later, so every waiter must be at most
one phase behind the barrier it waits on.  The model keeps the kernels' ownership rules
(producer warp pw fills the stages with kctr % producers == pw; MMA issuer m reads those
with kctr % issuers == m; every issuer releases each item's query buffer once; an
accumulator slot is rewritten only after every epilogue warp released its previous use)
and checks that no reader ever sees a buffer that holds another stage's, item's or use's
data, with the reads of an MMA or a tensor-memory load spanning other warps' steps.

Three failures are planted in the model's configuration, not in any kernel: a stage ring
whose size is not a multiple of the producer count, the earlier query-buffer release (an
issuer with no stage in an item arrived on the release barrier without waiting for the
item's rows), and a slot reused after all but one epilogue warp released it.  All must be
found; the configurations the two kernels use must run clean and never deadlock."""
import numpy as np
import pytest


class Violation(Exception):
    pass


class Deadlock(Exception):
    pass


class Bar:
    """mbarrier: `count` arrivals complete the current phase."""

    def __init__(self, count):
        self.count, self.pending, self.phase = count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.phase += 1

    def parity_done(self, parity):
        return (self.phase & 1) != parity


def schedule(actors, rng):
    """Run generator actors to completion.  Each yields the condition it waits on next
    (None = no wait); a random ready actor steps each time."""
    cond = {}
    for a in actors:
        try:
            cond[a] = next(a)
        except StopIteration:
            pass
    while cond:
        ready = [a for a, c in cond.items() if c is None or c()]
        if not ready:
            raise Deadlock()
        a = ready[int(rng.integers(len(ready)))]
        try:
            cond[a] = next(a)
        except StopIteration:
            del cond[a]


def stage_ring(n_stages, n_producers, n_issuers, total, rng):
    """Producers fill stage buffers, issuers read them (an in-flight read spans a step)."""
    kfull = [Bar(1) for _ in range(n_stages)]
    kempty = [Bar(1) for _ in range(n_stages)]
    ring = [None] * n_stages

    def producer(pw):
        for kctr in range(total):
            if kctr % n_producers != pw:
                continue
            s, n = kctr % n_stages, kctr // n_stages
            yield lambda: kempty[s].parity_done((n & 1) ^ 1)
            ring[s] = kctr
            kfull[s].arrive()

    def issuer(m):
        for kctr in range(total):
            if kctr % n_issuers != m:
                continue
            s, n = kctr % n_stages, kctr // n_stages
            yield lambda: kfull[s].parity_done(n & 1)
            if ring[s] != kctr:
                raise Violation("stage %d read as use %d holds %r" % (s, kctr, ring[s]))
            yield None  # MMAs in flight
            if ring[s] != kctr:
                raise Violation("stage %d overwritten under use %d" % (s, kctr))
            kempty[s].arrive()

    schedule([producer(p) for p in range(n_producers)] + [issuer(m) for m in range(n_issuers)], rng)


def query_buffers(n_buf, stages_per_item, wait_before_release, rng, n_issuers=2):
    """One producer loads each item's query rows into buffer item % n_buf; the issuers
    take the item's stages alternately and release the buffer once each."""
    qfull = [Bar(1) for _ in range(n_buf)]
    qempty = [Bar(n_issuers) for _ in range(n_buf)]
    buf = [None] * n_buf

    def producer():
        for i in range(len(stages_per_item)):
            b, u = i % n_buf, i // n_buf
            yield lambda: qempty[b].parity_done((u & 1) ^ 1)
            buf[b] = i
            qfull[b].arrive()

    def issuer(m):
        kctr = 0
        for i, n_st in enumerate(stages_per_item):
            b, u = i % n_buf, i // n_buf
            waited = False
            for _ in range(n_st):
                if kctr % n_issuers == m:
                    if not waited:
                        yield lambda: qfull[b].parity_done(u & 1)
                        waited = True
                    if buf[b] != i:
                        raise Violation("buffer %d read for item %d holds %r" % (b, i, buf[b]))
                    yield None  # MMAs in flight
                    if buf[b] != i:
                        raise Violation("buffer %d overwritten under item %d" % (b, i))
                kctr += 1
            if not waited and wait_before_release:
                yield lambda: qfull[b].parity_done(u & 1)
            qempty[b].arrive()

    schedule([producer()] + [issuer(m) for m in range(n_issuers)], rng)


def acc_slots(n_slots, n_issuers, n_epi, items, rng, need_releases=None):
    """Accumulator slots in tensor memory: per (stage, query row) a use u writes slot
    u % n_slots once every epilogue warp has released the slot's previous use (a release
    counter that only grows), and completes it on the slot's barrier; every epilogue warp
    reads every use in order.  items: list of (stages, rows)."""
    need = n_epi if need_releases is None else need_releases
    accfull = [Bar(1) for _ in range(n_slots)]
    released = [0] * n_slots
    acc = [None] * n_slots

    def issuer(m):
        kctr = ucnt = 0
        for n_st, rows in items:
            for _ in range(n_st):
                if kctr % n_issuers == m:
                    for r in range(rows):
                        u = ucnt + r
                        slot = u % n_slots
                        yield lambda: released[slot] >= need * (u // n_slots)
                        acc[slot] = u  # the MMAs of this use start writing
                        yield None
                        accfull[slot].arrive()
                kctr += 1
                ucnt += rows

    def epilogue():
        u = 0
        for n_st, rows in items:
            for _ in range(n_st * rows):
                slot = u % n_slots
                yield lambda: accfull[slot].parity_done((u // n_slots) & 1)
                if acc[slot] != u:
                    raise Violation("slot %d read as use %d holds %r" % (slot, u, acc[slot]))
                yield None  # tensor-memory load in flight
                if acc[slot] != u:
                    raise Violation("slot %d overwritten under use %d" % (slot, u))
                released[slot] += 1
                u += 1

    schedule([issuer(m) for m in range(n_issuers)] + [epilogue() for _ in range(n_epi)], rng)


def runs(fn, trials, seed):
    """(violations, deadlocks) over `trials` random schedules of fn(rng)."""
    rng = np.random.default_rng(seed)
    v = d = 0
    for _ in range(trials):
        try:
            fn(rng)
        except Violation:
            v += 1
        except Deadlock:
            d += 1
    return v, d


@pytest.mark.parametrize("n_stages,n_producers", [(8, 2), (4, 4)])  # the FP4 and FP8 kernels
def test_stage_ring_of_the_kernels_is_safe(n_stages, n_producers):
    assert runs(lambda rng: stage_ring(n_stages, n_producers, 2, 40, rng), 300, 1) == (0, 0)


def test_stage_ring_not_a_multiple_of_the_producers_is_caught():
    v, _ = runs(lambda rng: stage_ring(3, 4, 2, 40, rng), 300, 2)
    assert v > 0


def _items(rng):
    # short items (one or two stages) make an issuer with no stage in an item common
    return list(rng.integers(1, 4, size=int(rng.integers(4, 12))))


@pytest.mark.parametrize("n_buf", [2, 1])  # the FP4 and FP8 kernels
def test_query_release_after_the_rows_landed_is_safe(n_buf):
    assert runs(lambda rng: query_buffers(n_buf, _items(rng), True, rng), 400, 3) == (0, 0)


@pytest.mark.parametrize("n_buf", [2, 1])
def test_early_query_release_is_caught(n_buf):
    v, _ = runs(lambda rng: query_buffers(n_buf, _items(rng), False, rng), 400, 4)
    assert v > 0


def _groups(rng):
    # (stages, query rows) per item: decode items (one row) and draft groups (up to six)
    n = int(rng.integers(3, 8))
    return [(int(rng.integers(1, 4)), int(rng.integers(1, 7))) for _ in range(n)]


def test_accumulator_slots_of_the_kernels_are_safe():
    # both kernels: three slots, two issuers, eight epilogue warps (four here keep it small)
    assert runs(lambda rng: acc_slots(3, 2, 4, _groups(rng), rng), 200, 5) == (0, 0)


def test_accumulator_slot_reused_before_every_release_is_caught():
    v, _ = runs(lambda rng: acc_slots(3, 2, 4, _groups(rng), rng, need_releases=3), 200, 6)
    assert v > 0
