"""A CPU model of the mainloop's barrier protocol, run under random
interleavings of its roles and asynchronous operations.

It follows the kernel's bookkeeping exactly: stage index s and phase ph per
role, full[s] / empty[s] (count 1), acc_full[b] (count 1), acc_empty[b]
(count 4 x CTAs), the producer waiting empty[s] at parity ph ^ 1 (so its
first pass through the ring does not wait), the consumer waiting full[s] at
parity ph. mbarrier semantics: a phase completes when its pending arrivals
reach zero and its transaction count is zero; try_wait.parity(P) succeeds
once the phase of parity P has completed. TMA loads land (complete_tx) in any
order; tcgen05 MMAs and commits complete in issue order.

Checks ("B200 Tma Pipeline Designer", step 8, protocol): no deadlock; every
completed phase of every barrier saw exactly its designated arrivals (one
producer and one consumer per stage phase); no stage is overwritten while an
MMA may still read it and no accumulator is overwritten before the epilogue
read it; every output tile carries exactly its own K blocks. Planted bugs --
the arrival coming from a lane other than the TMA issuer (CUTLASS issue
#3722), a wrong initial phase, a missing wait -- must each be caught.
"""
import random

import pytest


class MBarrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending, self.tx, self.phase = count, 0, 0
        self.cur, self.done = [], []

    def arrive(self, who, tx=0):
        self.tx += tx
        self.cur.append(who)
        self.pending -= 1
        self._check()

    def complete_tx(self, n):
        self.tx -= n
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.done.append(self.cur)
            self.cur = []
            self.phase ^= 1
            self.pending = self.count

    def waited(self, parity):
        return parity != self.phase


class Violation(Exception):
    pass


class Deadlock(Exception):
    pass


def simulate(CG, STAGES, tiles, KB, seed, bug=None, epi_warps=4, out=None):
    """Runs the protocol; `out` (a dict), if given, receives the barriers
    (keys full, empty, accf, acce: per CTA rank, per stage / accumulator)."""
    rng = random.Random(seed)
    full = [[MBarrier(f"full{r}[{s}]", 1) for s in range(STAGES)] for r in range(CG)]
    empty = [[MBarrier(f"empty{r}[{s}]", 1) for s in range(STAGES)] for r in range(CG)]
    accf = [[MBarrier(f"accf{r}[{b}]", 1) for b in range(2)] for r in range(CG)]
    acce = [[MBarrier(f"acce{r}[{b}]", epi_warps * CG) for b in range(2)] for r in range(CG)]
    smem = [[None] * STAGES for _ in range(CG)]      # tag held by each stage buffer
    readers = [[0] * STAGES for _ in range(CG)]      # MMAs in flight reading it
    tmem = [[None, None] for _ in range(CG)]         # accumulator contents
    unread = [[0, 0] for _ in range(CG)]             # epilogue warps still to read
    outputs = {}
    tma_inflight = []                                # (rank, stage, tag, bytes)
    tensor_fifo = []                                 # in-order MMA / commit ops

    def producer(r):
        s, ph = 0, 0
        for t in tiles:
            for kb in range(KB):
                if bug != "no_empty_wait":
                    want = ph if bug == "wrong_initial_phase" else ph ^ 1
                    yield empty[r][s], want
                if r == 0 and bug != "arrive_from_other_lane":
                    full[0][s].arrive(f"producer{r}", tx=CG)   # expect_tx covers the pair
                tma_inflight.append((r, s, (t, kb, r), 1))
                s += 1
                if s == STAGES:
                    s, ph = 0, ph ^ 1

    def mma():
        s, ph = 0, 0
        for lt, t in enumerate(tiles):
            b, aph = lt & 1, (lt >> 1) & 1
            if bug != "no_acc_empty_wait":
                yield acce[0][b], aph ^ 1
            for kb in range(KB):
                yield full[0][s], ph
                for r in range(CG):
                    readers[r][s] += 1
                tensor_fifo.append(("mma", s, t, kb, b))
                tensor_fifo.append(("commit", [empty[r][s] for r in range(CG)], "mma"))
                s += 1
                if s == STAGES:
                    s, ph = 0, ph ^ 1
            tensor_fifo.append(("commit", [accf[r][b] for r in range(CG)], "mma"))

    def epilogue(r, w):
        for lt, t in enumerate(tiles):
            b, aph = lt & 1, (lt >> 1) & 1
            yield accf[r][b], aph
            got = tmem[r][b]
            if got != (t, tuple(range(KB))):
                raise Violation(f"epilogue {r}.{w} read {got} for tile {t}")
            outputs.setdefault((t, r), []).append(w)
            unread[r][b] -= 1
            acce[0][b].arrive(f"epilogue{r}.{w}")

    def run_tensor_op():
        op = tensor_fifo.pop(0)
        if op[0] == "mma":
            _, s, t, kb, b = op
            for r in range(CG):
                if smem[r][s] != (t, kb, r):
                    raise Violation(f"MMA read stage {s} of CTA {r}: {smem[r][s]}, wanted {(t, kb, r)}")
                if kb == 0:
                    if unread[r][b] > 0:
                        raise Violation(f"accumulator {b} of CTA {r} overwritten before the epilogue read it")
                    tmem[r][b] = (t, ())
                    unread[r][b] = epi_warps
                cur = tmem[r][b]
                tmem[r][b] = (t, cur[1] + (kb,))
                readers[r][s] -= 1
        else:
            for bar in op[1]:
                bar.arrive(op[2])

    roles = [producer(r) for r in range(CG)] + [mma()] + \
        [epilogue(r, w) for r in range(CG) for w in range(epi_warps)]
    waits = {i: None for i in range(len(roles))}   # (barrier, parity) each role waits on
    steps = 0
    while waits or tma_inflight or tensor_fifo:
        steps += 1
        ready = [i for i, w in waits.items() if w is None or w[0].waited(w[1])]
        choices = [("role", i) for i in ready]
        choices += [("tma", j) for j in range(len(tma_inflight))]
        if tensor_fifo:
            choices.append(("tensor", 0))
        if not choices:
            raise Deadlock("blocked: " + ", ".join(f"{w[0].name}@{w[1]}" for w in waits.values()))
        kind, j = rng.choice(choices)
        if kind == "role":
            try:
                waits[j] = next(roles[j])
            except StopIteration:
                del waits[j]
        elif kind == "tma":
            r, s, tag, nbytes = tma_inflight.pop(j)
            if readers[r][s] > 0:
                raise Violation(f"stage {s} of CTA {r} overwritten while an MMA may read it")
            smem[r][s] = tag
            full[0][s].complete_tx(nbytes)
        else:
            run_tensor_op()
    # Every completed phase saw exactly its designated arrivals.
    for r in range(CG):
        for s in range(STAGES):
            if r == 0:
                assert all(a == ["producer0"] for a in full[0][s].done), full[0][s].done
            assert all(a == ["mma"] for a in empty[r][s].done)
        for b in range(2):
            assert all(a == ["mma"] for a in accf[r][b].done)
    for b in range(2):
        for a in acce[0][b].done:
            assert sorted(a) == sorted(f"epilogue{r}.{w}" for r in range(CG) for w in range(epi_warps))
    for t in tiles:
        for r in range(CG):
            assert sorted(outputs[(t, r)]) == list(range(epi_warps))
    if out is not None:
        out.update(full=full, empty=empty, accf=accf, acce=acce)
    return steps


def run_until_stable(CG, STAGES, tiles, KB, seed, bug=None):
    try:
        simulate(CG, STAGES, tiles, KB, seed, bug)
        return "ok"
    except Violation as e:
        return f"violation: {e}"
    except Deadlock as e:
        return f"deadlock: {e}"


@pytest.mark.parametrize("CG", [1, 2])
@pytest.mark.parametrize("STAGES", [2, 3, 5, 8, 9])
def test_protocol_holds_under_random_interleavings(CG, STAGES):
    for seed in range(12):
        rng = random.Random(seed * 31 + STAGES)
        KB = rng.randint(1, 3 * STAGES)
        ntiles = rng.randint(1, 5)
        tiles = list(range(seed, seed + ntiles))
        assert run_until_stable(CG, STAGES, tiles, KB, seed) == "ok", (CG, STAGES, KB, ntiles, seed)


@pytest.mark.parametrize("CG", [1, 2])
def test_arrival_from_another_lane_hangs(CG):
    # The lane that issues the TMA is not the one that posts expect_tx: the
    # stage's only arrival never comes and the pipeline cannot advance.
    res = run_until_stable(CG, 4, [0, 1], 6, 3, bug="arrive_from_other_lane")
    assert res.startswith("deadlock")


def test_wrong_initial_phase_hangs():
    assert run_until_stable(1, 4, [0], 5, 1, bug="wrong_initial_phase").startswith("deadlock")


def test_missing_empty_wait_is_caught():
    # A producer that never waits for a free stage refills stages the MMA has
    # not consumed: either it overwrites data in use or the surplus arrivals
    # wedge the barrier.
    results = [run_until_stable(1, 2, [0, 1], 5, seed, bug="no_empty_wait") for seed in range(20)]
    assert all(r != "ok" for r in results), results


def test_missing_accumulator_wait_is_caught():
    # An MMA issuer that does not wait for acc_empty overwrites an
    # accumulator the epilogue has not read yet.
    results = [run_until_stable(1, 4, list(range(8)), 1, seed, bug="no_acc_empty_wait") for seed in range(40)]
    assert any(r.startswith("violation") for r in results), results[:3]
