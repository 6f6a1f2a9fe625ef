"""Host-side model of the jagged backward kernel's mbarrier protocol.

Each warp role of the kernel (TMA producer, MMA issuer, compute warps, dQ
warps) is written as a generator of the waits and signals it performs, in
the kernel's order, for one CTA's list of (key tile, query blocks). A random
scheduler interleaves the roles many times over random tile lists and checks:

* no deadlock: some role can always make progress until all are done;
* no parity aliasing: a barrier never completes phase k + 2 while a role
  that waits on it has not yet passed its wait for phase k (mbarrier waits
  only see the phase parity, so that would let the wait pass early);
* the reuse of each TMEM / shared-memory buffer is ordered after the last
  read of its previous contents, through the barriers.

Negative controls show that each check has teeth: one dQ^T TMEM buffer
with the reduction three blocks behind deadlocks at a tile switch; a producer
that refills stages without waiting for their release is flagged as parity
aliasing; an MMA thread that rewrites a dQ^T buffer without waiting for its
drain is flagged as early reuse. The scheduler is adversarial (roles are
held back at random for whole rounds) so that rare interleavings occur.
"""

import random

import pytest

NSTAGE = 3  # Q/dO stages at D = 128


class Roles:
    """Waits and signals of the committed kernel; `dq_bufs` and `lag` select
    the dQ^T buffering (2 and 2 in the kernel)."""

    def __init__(self, tiles, dq_bufs=2, lag=2):
        self.tiles, self.dq_bufs, self.lag = tiles, dq_bufs, lag

    def stage(self, n):  # per-slot barrier: (name, slot), phase
        return n % NSTAGE, n // NSTAGE

    def producer(self):
        n = 0
        for t, nq in enumerate(self.tiles):
            for i in range(nq):
                s, ph = self.stage(n)
                if n >= NSTAGE:
                    yield "wait", ("stage_empty", s), ph - 1
                yield "sig", ("stage_full", s), ph
                n += 1
                if i == 0:  # K and V after the tile's first stage
                    if t > 0:
                        yield "wait", ("kv_empty", 0), t - 1
                    yield "sig", ("kv_full", 0), t

    def mma(self):
        n = 0
        for t, nq in enumerate(self.tiles):
            yield "wait", ("kv_full", 0), t
            for i in range(nq):
                s, ph = self.stage(n)
                if i == 0:
                    yield "wait", ("stage_full", s), ph
                    yield "sig", ("s_full", 0), n
                    yield "sig", ("dp_full", 0), n
                yield "wait", ("p_ready", 0), n
                if i == 0 and t > 0:
                    yield "wait", ("dkdv_free", 0), t - 1
                yield "use", "dV", t  # dV accumulator written
                more = i + 1 < nq
                if more:
                    s2, ph2 = self.stage(n + 1)
                    yield "wait", ("stage_full", s2), ph2
                    yield "sig", ("s_full", 0), n + 1
                yield "wait", ("ds_ready", 0), n
                yield "sig", ("stage_empty_mma", s), ph
                b = n % self.dq_bufs
                if n >= self.dq_bufs:
                    yield "wait", ("dq_free", b), n // self.dq_bufs - 1
                yield "use", ("dQ", b), n  # dQ^T TMEM buffer written
                yield "sig", ("dq_full", b), n // self.dq_bufs
                yield "sig", ("ds_free", 0), n
                if more:
                    yield "sig", ("dp_full", 0), n + 1
                n += 1
            yield "sig", ("dkdv_full", 0), t
            yield "sig", ("kv_empty", 0), t

    def compute(self):
        n = 0
        for t, nq in enumerate(self.tiles):
            for _ in range(nq):
                s, ph = self.stage(n)
                yield "wait", ("aux_full", s), ph
                yield "wait", ("s_full", 0), n
                yield "sig", ("p_ready", 0), n
                yield "wait", ("dp_full", 0), n
                if n > 0:
                    yield "wait", ("ds_free", 0), n - 1
                yield "sig", ("ds_ready", 0), n
                yield "sig", ("stage_empty_cmp", s), ph
                n += 1
            yield "wait", ("dkdv_full", 0), t
            yield "read", "dV", t  # epilogue reads the accumulators
            yield "sig", ("dkdv_free", 0), t

    def reducer(self):
        n = 0

        def drain(m):
            b = m % self.dq_bufs
            yield "wait", ("dq_full", b), m // self.dq_bufs
            yield "read", ("dQ", b), m
            yield "sig", ("dq_free", b), m // self.dq_bufs

        for nq in self.tiles:
            for _ in range(nq):
                s, ph = self.stage(n)
                yield "wait", ("stage_full", s), ph
                yield "sig", ("aux_full", s), ph
                if n >= self.lag:
                    yield from drain(n - self.lag)
                n += 1
        for m in range(max(0, n - self.lag), n):
            yield from drain(m)


# stage_empty completes when both the MMA commit and the compute warps arrived
JOINED = {"stage_empty": ("stage_empty_mma", "stage_empty_cmp")}


def simulate(tiles, rng, roles_cls=Roles, **kw):
    R = roles_cls(tiles, **kw)
    gens = {"producer": R.producer(), "mma": R.mma(), "compute": R.compute(),
            "reducer": R.reducer()}
    done = {}        # (name, slot) -> number of completed phases
    part = {}        # partial arrivals of joined barriers
    passed = {}      # (role, (name, slot)) -> highest phase waited for
    waiters = {}     # (name, slot) -> roles that wait on it
    last_read = {}   # buffer -> last index read
    errors = []
    # who waits on what (for the aliasing check), from a dry run
    for role in gens:
        for op, key, _ in getattr(roles_cls(tiles, **kw), role)():
            if op == "wait":
                waiters.setdefault(key, set()).add(role)

    def complete(key, ph):
        if done.get(key, 0) != ph:
            errors.append("phase order %s: %d after %d" % (key, ph, done.get(key, 0)))
        done[key] = ph + 1
        for role in waiters.get(key, ()):
            if ph >= 2 and passed.get((role, key), -1) < ph - 2:
                errors.append("aliasing: %s phase %d completes before %s waited for %d"
                              % (key, ph, role, ph - 2))

    pending = {r: None for r in gens}
    alive = set(gens)
    # Adversarial schedule: each round a role may be held back (with a
    # probability drawn per run) and otherwise takes 1-8 steps; a round that
    # holds nobody back and still makes no progress is a deadlock.
    p_hold = rng.choice((0.0, 0.3, 0.6, 0.85))
    hold_all_off = False
    while alive:
        progress = False
        order = list(alive)
        rng.shuffle(order)
        for role in order:
            if not hold_all_off and rng.random() < p_hold:
                continue
            for _ in range(rng.randint(1, 8)):
                if pending[role] is None:
                    try:
                        pending[role] = next(gens[role])
                    except StopIteration:
                        alive.discard(role)
                        progress = True
                        break
                op, key, idx = pending[role]
                if op == "wait":
                    if done.get(key, 0) <= idx:
                        break
                    passed[(role, key)] = idx
                elif op == "sig":
                    name, slot = key
                    joined = next((j for j, parts in JOINED.items() if name in parts), None)
                    if joined is None:
                        complete(key, idx)
                    else:
                        arrived = part.setdefault((joined, slot, idx), set())
                        arrived.add(name)
                        if len(arrived) == len(JOINED[joined]):
                            complete((joined, slot), idx)
                elif op == "use":
                    # a buffer is rewritten: its previous contents must have been read
                    if isinstance(key, tuple):  # dQ^T buffer b holds block idx
                        prev = idx - R.dq_bufs
                        if prev >= 0 and last_read.get(key, -1) < prev:
                            errors.append("dQ^T buffer %d rewritten before block %d was read"
                                          % (key[1], prev))
                    else:  # dV/dK accumulators of tile idx
                        if idx > 0 and last_read.get(key, -1) < idx - 1:
                            errors.append("accumulators rewritten before tile %d's epilogue"
                                          % (idx - 1))
                elif op == "read":
                    last_read[key] = max(last_read.get(key, -1), idx)
                pending[role] = None
                progress = True
        if not progress:
            if hold_all_off:
                return "deadlock", {r: pending[r] for r in alive}
            hold_all_off = True
        else:
            hold_all_off = False
    return ("errors", errors) if errors else None


def _random_tiles(rng):
    return [rng.randint(1, 6) for _ in range(rng.randint(1, 7))]


def test_committed_protocol_has_no_deadlock_aliasing_or_early_reuse():
    rng = random.Random(11)
    for _ in range(3000):
        tiles = _random_tiles(rng)
        assert simulate(tiles, rng) is None, tiles


@pytest.mark.parametrize("tiles", [[1], [1, 1, 1, 1], [6, 1, 5], [2, 2, 2, 2, 2]])
def test_committed_protocol_fixed_cases(tiles):
    rng = random.Random(12)
    for _ in range(200):
        assert simulate(tiles, rng) is None


def test_negative_control_single_dq_buffer_three_blocks_behind_deadlocks():
    # The MMA thread's dQ^T of a tile's last block then waits for a drain that
    # the dQ warps only reach after staging the next tile's second block, whose
    # Q/dO load the producer issues only after the next tile's K/V load, which
    # waits for this tile's products to finish.
    rng = random.Random(13)
    results = [simulate(_random_tiles(rng), rng, dq_bufs=1, lag=3) for _ in range(300)]
    assert any(r is not None and r[0] == "deadlock" for r in results)


def test_single_dq_buffer_two_blocks_behind_is_safe():
    # With the next tile's first stage loaded ahead of its K and V, the drain
    # that a tile's last dQ^T waits for no longer depends on that tile ending.
    rng = random.Random(16)
    for _ in range(1000):
        assert simulate(_random_tiles(rng), rng, dq_bufs=1, lag=2) is None


def test_single_dq_buffer_one_block_behind_is_safe():
    rng = random.Random(14)
    for _ in range(1000):
        assert simulate(_random_tiles(rng), rng, dq_bufs=1, lag=1) is None


class NoStageEmptyWait(Roles):
    """Negative control: the producer refills stages without waiting for
    their release."""

    def producer(self):
        for op, key, idx in Roles.producer(self):
            if not (op == "wait" and key[0] == "stage_empty"):
                yield op, key, idx


class NoDqFreeWait(Roles):
    """Negative control: the MMA thread rewrites a dQ^T buffer without
    waiting for its drain."""

    def mma(self):
        for op, key, idx in Roles.mma(self):
            if not (op == "wait" and key[0] == "dq_free"):
                yield op, key, idx


def test_negative_control_missing_release_wait_is_flagged_as_aliasing():
    rng = random.Random(15)
    results = [simulate([12, 12], rng, roles_cls=NoStageEmptyWait) for _ in range(300)]
    assert any(r is not None and r[0] == "errors" and any("aliasing" in e for e in r[1])
               for r in results)


def test_negative_control_missing_drain_wait_is_flagged_as_early_reuse():
    rng = random.Random(16)
    results = [simulate([6, 6], rng, roles_cls=NoDqFreeWait) for _ in range(300)]
    assert any(r is not None and r[0] == "errors" and any("rewritten" in e for e in r[1])
               for r in results)
