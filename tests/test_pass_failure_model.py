"""The failure path of the tensor-core state pass (csrc/gdn_prefill_tc.cu, pass_tc_kernel) in the
randomised CPU model of tests/test_pass_protocol_model.py: every mbarrier wait of the kernel is
bounded, and one of them, chosen at random, gives up. After that, a wait gives up only when
nothing in the CTA can make progress any more (no copy or MMA group outstanding, every warp
blocked) -- what a time bound does. The roles then follow the kernel's failure handling:

- a compute or MMA warp whose wait gave up skips the work that needed it, and the named
  barrier's OR tells the other eight of these warps, which leave the chunk loop together;
- the copy warp, which is not part of the named barrier, stops issuing when one of its own
  waits gives up, and in every case waits (bounded) for the last phase it issued on each
  copy barrier, so no copy is in flight -- another warp's failure can leave copies that
  nobody else waits for;
- the MMA warp waits (bounded) for its last committed MMA groups;
- then all ten warps meet at the CTA barrier before tensor memory is freed.

Checked over many schedules, chunk counts and failure points: every warp finishes (the
unbounded named and CTA barriers stay matched), and when tensor memory is freed no bulk copy
is in flight and no MMA group is queued or running. The buffer-version checks of the
success-path model keep holding. Planted mistakes each fail some schedule:
the copy warp's drain left out, or done only after its own failure; the MMA warp's drain left
out -- a failure reported at the barrier after the state update leaves the warps to exit while
the second part of group 2 (O2, which only the output waits for) may still run. Host logic
only.
"""
import random

import pytest

import test_pass_protocol_model as base
from test_pass_protocol_model import (N_COMPUTE, g1_reads, g1_writes, o2_reads, o2_rmw, par,
                                      u_bufs, upd_reads, upd_writes, xp)


class FailSim(base.Sim):
    def __init__(self, nch, rng, fail_at, mutant=None):
        super().__init__(nch, rng, mutant)
        self.fail_at = fail_at     # the index of the bounded wait that gives up first
        self.n_waits = 0
        self.failed = False
        self.giveup = set()        # ids of blocked waits told to give up (quiescence)
        self.blocked_waits = {}    # wait id -> actor index
        self.freed = False

    def bounded(self, bar, k, actor):
        """Generator returning True when phase k of `bar` completes, False when it gives up."""
        idx = self.n_waits
        self.n_waits += 1
        b = self.bars[bar]
        if idx == self.fail_at:
            self.failed = True
            return False
        wid = (actor, idx)
        b.waiting.append(k)
        while (b.c & 1) == (k & 1):
            assert b.c <= k + 1
            self.blocked_waits[wid] = actor
            yield lambda: (b.c & 1) != (k & 1) or wid in self.giveup
            if wid in self.giveup:
                self.blocked_waits.pop(wid, None)
                b.waiting.remove(k)
                self.failed = True
                return False
        self.blocked_waits.pop(wid, None)
        b.waiting.remove(k)
        return True

    def or_sync(self, name, n, flag, out):
        """Named barrier with an OR reduction (bar.red.or): out[0] = any arrival's flag."""
        gen = self.sync_arrived.setdefault(name, [0, 0, False, {}])
        g = gen[1]
        gen[0] += 1
        gen[2] = gen[2] or flag
        if gen[0] == n:
            gen[3][g] = gen[2]
            gen[0], gen[1], gen[2] = 0, g + 1, False
        else:
            yield lambda: gen[1] != g
        out[0] = gen[3][g]

    def arrive_odone(self, phase):
        b = self.bars["oDone"]
        if self.failed and b.c != phase:   # after a failure nobody waits for these phases
            return
        b.arrive(phase)

    def outstanding(self):
        return bool(self.events) or bool(self.mma_queue) or self.mma_busy is not None

    def free_tmem(self):
        assert not self.outstanding(), "tensor memory freed with copies or MMA groups outstanding"
        self.freed = True


def copy_warp(s, me):
    nch = s.nch
    nA = nBU = 0
    if nch > 0:
        s.copy("fullA", ["W", "Q", ("vec", 0)], 0)
        s.copy("fullB", ["P", "Kt"], 0)
        s.copy("fullU", u_bufs(), ("U", 0))
        nA = nBU = 1
    yield from s.sync("cta", 10)
    ok = True
    if nch > 0:
        s.arrive_odone(0)
        if nch > 1:
            if (yield from s.bounded("mma1", 0, me)):
                s.copy("fullA", ["W", "Q", ("vec", 1)], 1)
                nA = 2
            else:
                ok = False
        for it in range(nch - 1):
            if not ok:
                break
            if not (yield from s.bounded("mma2", it, me)):
                ok = False
                break
            s.copy("fullB", ["P", "Kt"], it + 1)
            s.copy("fullU", u_bufs(), ("U", it + 1))
            nBU = it + 2
            if it + 2 < nch:
                if not (yield from s.bounded("oDone", it, me)):
                    ok = False
                    break
                s.arrive_odone(it + 1)
                if not (yield from s.bounded("mma1", it + 1, me)):
                    ok = False
                    break
                s.copy("fullA", ["W", "Q", ("vec", par(it + 2))], it + 2)
                nA = it + 3
        if s.mutant != "no copy drain" and not (ok and s.mutant == "drain only on own failure"):
            # the last issued phase of each copy barrier, whatever happened (another warp's
            # failure leaves copies nobody else waits for); one already waited for returns at once
            yield from s.bounded("fullA", nA - 1, me)
            yield from s.bounded("fullB", nBU - 1, me)
            yield from s.bounded("fullU", nBU - 1, me)
    yield from s.sync("cta", 10)


def mma_warp(s, me):
    nch = s.nch
    yield from s.sync("cta", 10)
    mine = False
    n1 = n2 = 0

    def issue1(k):
        nonlocal n1
        if not (yield from s.bounded("fullA", k, me)):
            return False
        s.mma(f"mma1({k})", g1_reads(k), g1_writes(s, k), "mma1", k)
        n1 = k + 1
        return True

    if nch > 0:
        mine = not (yield from issue1(0))
    bad = [False]
    for it in range(nch):
        yield from s.or_sync("named", N_COMPUTE + 1, mine, bad)            # B1
        if bad[0]:
            break
        if (yield from s.bounded("fullB", it, me)):
            s.mma(f"upd({it})", upd_reads(it), upd_writes(s, it), "upd", it)
            if (yield from s.bounded("scaled", it, me)):
                s.mma(f"mma2({it})", o2_reads(it), [], "mma2", it, o2_rmw(s, it))
            else:
                mine = True
                s.mma(f"commit mma2({it})", [], [], "mma2", it)
            n2 = it + 1
        else:
            mine = True
        yield from s.or_sync("named", N_COMPUTE + 1, mine, bad)            # B2
        if bad[0]:
            break
        if it + 1 < nch:
            mine = not (yield from issue1(it + 1))
    yield from s.or_sync("named", N_COMPUTE + 1, bad[0] or mine, bad)      # after the loop
    if bad[0] and s.mutant != "no MMA drain":
        if n1 > 0:
            yield from s.bounded("mma1", n1 - 1, me)
        if n2 > 0:
            yield from s.bounded("mma2", n2 - 1, me)
    yield from s.sync("cta", 10)


def compute_warp(s, w, me):
    nch = s.nch
    s.write(("S", w), 0)
    yield from s.sync("cta", 10)
    bad = [False]
    mine = False
    for it in range(nch):
        ok1 = yield from s.bounded("mma1", it, me)
        ok2 = yield from s.bounded("fullU", it, me)
        mine = mine or not (ok1 and ok2)
        tag = f"warp{w} chunk {it}"
        x = xp(s, it)
        if not mine:
            s.read(("Xd", x), ("raw", it), tag)
            s.read(("U", w), ("U", it), tag)
            s.read(("vec", par(it)), it, tag)
            yield lambda: True
            s.write(("D", w), it)
            s.write(("E", w), it)
        yield from s.or_sync("named", N_COMPUTE + 1, mine, bad)            # B1
        if bad[0]:
            break
        s.read(("Xo", x, w), ("O1", it), tag)       # f_t O1 in place (no wait failed before B1)
        yield lambda: True
        s.write(("Xo", x, w), ("fO1", it))
        s.bars["scaled"].arrive(it)
        if not (yield from s.bounded("upd", it, me)):
            mine = True
        if not mine:
            s.read(("Xd", 1 - x), ("dS", it), tag)
            s.read(("Xo", 1 - x, w), ("dS", it), tag)
            s.read(("vec", par(it)), it, tag)
            s.write(("S", w), it + 1)
        yield from s.or_sync("named", N_COMPUTE + 1, mine, bad)            # B2
        if bad[0]:
            break
        if not (yield from s.bounded("mma2", it, me)):
            mine = True                  # the output is skipped; reported at the next barrier
        if not mine:
            s.read_begin(("Xo", x, w), ("O", it), tag)
            s.read_begin(("vec", par(it)), it, tag)
            yield lambda: True
            s.read_end(("Xo", x, w), ("O", it), tag)
            s.read_end(("vec", par(it)), it, tag)
        s.arrive_odone(it)
    yield from s.or_sync("named", N_COMPUTE + 1, bad[0] or mine, bad)
    yield from s.sync("cta", 10)
    if w == 0:
        s.free_tmem()      # warp 0 frees tensor memory after the final CTA barrier


def run(nch, seed, fail_at, mutant=None):
    rng = random.Random(seed)
    s = FailSim(nch, rng, fail_at, mutant)
    actors = [copy_warp(s, 0), mma_warp(s, 1)] + [compute_warp(s, w, 2 + w)
                                                   for w in range(N_COMPUTE)]
    blocked = [None] * len(actors)
    done = [False] * len(actors)
    for _ in range(400_000):
        if all(done):
            assert s.freed
            return s
        ready = [i for i, a in enumerate(actors)
                 if not done[i] and (blocked[i] is None or blocked[i]())]
        if not ready:
            if s.outstanding():
                s.tick()
                continue
            # nothing can progress: the oldest blocked bounded wait runs out of time
            assert s.blocked_waits, f"deadlock on an unbounded barrier: nch={nch} done={done}"
            s.giveup.add(min(s.blocked_waits, key=lambda wid: wid[1]))
            continue
        if rng.random() < 0.3:
            s.tick()
            continue
        i = rng.choice(ready)
        try:
            blocked[i] = next(actors[i])
        except StopIteration:
            done[i] = True
    raise AssertionError(f"no progress: nch={nch} seed={seed} done={done}")


def waits_in_clean_run(nch):
    s = run(nch, 0, fail_at=-1)
    return s.n_waits


@pytest.mark.parametrize("nch", [1, 2, 3, 5])
def test_pass_failure_path_drains_and_finishes(nch):
    total = waits_in_clean_run(nch)
    assert total > 0
    for seed in range(40):
        fail_at = random.Random(1000 + seed).randrange(total)
        s = run(nch, seed, fail_at)
        assert s.failed


@pytest.mark.parametrize("mutant", ["no copy drain", "drain only on own failure", "no MMA drain"])
def test_failure_model_catches_missing_drains(mutant):
    """Leaving out the copy warp's drain, or draining only after its own failure, lets the CTA
    free tensor memory (and exit) with copies still landing in its shared memory; leaving out
    the MMA warp's drain lets it free tensor memory under a running MMA group."""
    caught = 0
    total = waits_in_clean_run(5)
    for seed in range(80):
        fail_at = random.Random(2000 + seed).randrange(total)
        try:
            run(5, seed, fail_at, mutant)
        except AssertionError:
            caught += 1
    assert caught > 0, mutant
