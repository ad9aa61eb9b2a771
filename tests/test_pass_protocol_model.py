"""A randomised CPU model of the tensor-core state pass's synchronisation (csrc/gdn_prefill_tc.cu,
pass_tc_kernel): a copy warp, an MMA warp and eight compute warps, in the order each of them
executes its steps, over mbarriers with the hardware's parity semantics (a wait for phase k
returns once the barrier's current phase has a different parity), transaction-counted
barriers completed when a bulk copy lands, MMA groups that run in issue order and complete
their commit barrier when done (group 2 in two parts: the state update, committed on its own
barrier, then O2), a named barrier over the compute and MMA warps, and the CTA
barriers. Copies and MMA groups take random times and the scheduler interleaves the warps at
random. The buffers are shared-memory tiles (W, q, P, k, the U image, vec) and tensor-memory
regions: the bf16 operand parts of the state and of D / D' (each warp its rows), and two
accumulator regions that alternate by chunk parity -- a chunk's raw D^T and O1^T in one (the
compute warps scale O1^T by f_t in place, and O2^T is then added onto it, giving the output),
its state update in the other. Over many schedules and chunk counts it checks that

- no parity wait can alias: while a thread waits for phase k the barrier never completes
  phase k + 1 (else the wait would miss phase k and hang);
- every arrival on the output barrier lands in the phase it is meant for;
- each shared buffer or tensor-memory region is read only at the version it must hold, and
  no copy or MMA rewrites it while a reader may still use it;
- every warp finishes.

Planted mistakes (a missing wait, a buffer reused early, an early arrival, a group issued
before its barrier, one accumulator set instead of two, the output read before the second
part of group 2 is done, O2 added before the compute warps have scaled O1) each fail some
schedule, so the
checks have teeth. The model is host logic only; the GPU tests run the kernel itself.
"""
import random

import pytest

N_COMPUTE = 8


class Bar:
    """An mbarrier: `c` completed phases; arrival-counted (`count`) or transaction-counted."""

    def __init__(self, name, count=None):
        self.name, self.count, self.c, self.pending = name, count, 0, 0
        self.waiting = []  # phases some thread is waiting for

    def complete(self):
        for k in self.waiting:
            assert self.c < k + 1, f"{self.name}: phase {self.c} completes while a wait for {k} is pending"
        self.c += 1

    def arrive(self, phase):
        assert self.c == phase, f"{self.name}: arrival for phase {phase} while phase {self.c} is open"
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.complete()


class Sim:
    def __init__(self, nch, rng, mutant=None):
        self.nch, self.rng, self.mutant = nch, rng, mutant
        self.bars = {n: Bar(n) for n in ("fullA", "fullB", "fullU", "mma1", "upd", "mma2")}
        self.bars["oDone"] = Bar("oDone", N_COMPUTE + 1)
        self.bars["scaled"] = Bar("scaled", N_COMPUTE)
        self.events = []      # [countdown, callable]
        self.mma_queue = []   # MMA groups in issue order: (name, start_fn, finish_fn)
        self.mma_busy = None  # [countdown, finish_fn]
        self.buf = {}         # buffer -> version it holds
        self.readers = {}     # buffer -> set of open reader tags
        self.sync_arrived = {}

    # ---- buffers
    def write(self, b, version):
        assert not self.readers.get(b), f"{b} rewritten to {version} while read by {self.readers[b]}"
        self.buf[b] = version

    def read_begin(self, b, version, tag):
        assert self.buf.get(b) == version, f"{b} holds {self.buf.get(b)}, {tag} needs {version}"
        self.readers.setdefault(b, set()).add(tag)

    def read_end(self, b, version, tag):
        assert self.buf.get(b) == version, f"{b} changed under {tag}"
        self.readers[b].discard(tag)

    def read(self, b, version, tag):
        self.read_begin(b, version, tag)
        self.read_end(b, version, tag)

    # ---- asynchronous work
    def later(self, fn):
        self.events.append([self.rng.randint(1, 12), fn])

    def copy(self, bar, bufs, version):
        """A bulk copy: its destination is being written from issue until it lands."""
        for b in bufs:
            self.write(b, ("in flight", version))
        def land():
            for b in bufs:
                self.write(b, version)
            self.bars[bar].complete()
        self.later(land)

    def mma(self, name, reads, writes, bar, k, rmw=()):
        """An MMA group: it reads `reads`, writes `writes`, and reads then rewrites each
        (buffer, version in, version out) of `rmw` (an accumulator it adds onto)."""
        def start():
            for b, v in reads:
                self.read_begin(b, v, name)
            for b, vin, vout in rmw:
                assert self.buf.get(b) == vin, f"{b} holds {self.buf.get(b)}, {name} adds onto {vin}"
                self.write(b, ("mma", name))
            for b, v in writes:
                self.write(b, ("mma", name))
        def finish():
            for b, v in reads:
                self.read_end(b, v, name)
            for b, vin, vout in rmw:
                self.write(b, vout)
            for b, v in writes:
                self.write(b, v)
            self.bars[bar].complete()
        self.mma_queue.append((start, finish))

    def tick(self):
        for e in self.events:
            e[0] -= 1
        due = [e for e in self.events if e[0] <= 0]
        self.events = [e for e in self.events if e[0] > 0]
        for _, fn in due:
            fn()
        if self.mma_busy is not None:
            self.mma_busy[0] -= 1
            if self.mma_busy[0] <= 0:
                self.mma_busy[1]()
                self.mma_busy = None
        if self.mma_busy is None and self.mma_queue:
            start, finish = self.mma_queue.pop(0)
            start()
            self.mma_busy = [self.rng.randint(1, 40), finish]  # at times longer than a copy

    # ---- thread-side waits (generators yield predicates)
    def wait(self, bar, k):
        b = self.bars[bar]
        b.waiting.append(k)
        while (b.c & 1) == (k & 1):   # the hardware's parity test
            assert b.c <= k + 1
            yield lambda: (b.c & 1) != (k & 1)
        assert b.c == k + 1, f"{bar}: wait for phase {k} returned at {b.c}"
        b.waiting.remove(k)

    def sync(self, name, n):
        gen = self.sync_arrived.setdefault(name, [0, 0])  # [arrived, generation]
        g = gen[1]
        gen[0] += 1
        if gen[0] == n:
            gen[0], gen[1] = 0, g + 1
        else:
            yield lambda: gen[1] != g


def par(k):
    return k & 1


def xp(s, k):
    """The accumulator region of chunk k (X0 or X1, by parity): its raw D^T, then O2^T, in the
    "d" half and O1^T in the "o" half; the other region takes chunk k's state update."""
    return 0 if s.mutant == "one D/O1 set" else par(k)


def u_bufs():
    """The U^T image in shared memory: every compute warp's rows."""
    return [("U", w) for w in range(N_COMPUTE)]


def g1_reads(k):
    """Group 1 of chunk k: the state's hi / lo parts (tensor memory, each warp's rows), W, q."""
    return [(("S", w), k) for w in range(N_COMPUTE)] + [("W", k), ("Q", k)]


def g1_writes(s, k):
    """The raw D^T half, and the O1^T half in pieces: each compute warp's rows and columns."""
    x = xp(s, k)
    return [(("Xd", x), ("raw", k))] + [(("Xo", x, w), ("O1", k)) for w in range(N_COMPUTE)]


def upd_reads(k):
    """Group 2 of chunk k, first part (committed on its own barrier): the state update from
    D' hi / lo (tensor memory, each warp's rows) and the k tile."""
    return [(("E", w), k) for w in range(N_COMPUTE)] + [("Kt", k)]


def upd_writes(s, k):
    x = xp(s, k)
    return [(("Xd", 1 - x), ("dS", k))] + [(("Xo", 1 - x, w), ("dS", k)) for w in range(N_COMPUTE)]


def o2_reads(k):
    """Group 2 of chunk k, second part: O2^T from D hi / lo and the P tiles..."""
    return [(("D", w), k) for w in range(N_COMPUTE)] + [("P", k)]


def o2_rmw(s, k):
    """... added onto f_t O1^T, which the compute warps left in the O1 columns."""
    return [(("Xo", xp(s, k), w), ("fO1", k), ("O", k)) for w in range(N_COMPUTE)]


def copy_warp(s):
    nch = s.nch
    if nch > 0:
        s.copy("fullA", ["W", "Q", ("vec", 0)], 0)
        s.copy("fullB", ["P", "Kt"], 0)
        s.copy("fullU", u_bufs(), ("U", 0))
    yield from s.sync("cta", 10)
    if nch == 0:
        yield from s.sync("cta", 10)
        return
    s.bars["oDone"].arrive(0)
    early_u = s.mutant == "U after group 1"  # planted: U(k) once group 1 of chunk k-1 is done
    if nch > 1:
        yield from s.wait("mma1", 0)
        s.copy("fullA", ["W", "Q", ("vec", 1)], 1)
        if early_u:
            s.copy("fullU", u_bufs(), ("U", 1))
    for it in range(nch - 1):
        yield from s.wait("mma2", it)
        s.copy("fullB", ["P", "Kt"], it + 1)
        if not early_u:
            s.copy("fullU", u_bufs(), ("U", it + 1))
        if it + 2 < nch:
            if s.mutant == "arrive early":
                s.bars["oDone"].arrive(it + 1)
                yield from s.wait("oDone", it)
            elif s.mutant != "no output barrier":
                yield from s.wait("oDone", it)
                s.bars["oDone"].arrive(it + 1)
            yield from s.wait("mma1", it + 1)
            s.copy("fullA", ["W", "Q", ("vec", par(it + 2))], it + 2)
            if early_u:
                s.copy("fullU", u_bufs(), ("U", it + 2))
    yield from s.sync("cta", 10)


def mma_warp(s):
    nch = s.nch
    yield from s.sync("cta", 10)

    def issue1(k):
        yield from s.wait("fullA", k)
        s.mma(f"mma1({k})", g1_reads(k), g1_writes(s, k), "mma1", k)

    if nch > 0:
        yield from issue1(0)
    for it in range(nch):
        yield from s.sync("named", N_COMPUTE + 1)                          # B1
        yield from s.wait("fullB", it)
        s.mma(f"upd({it})", upd_reads(it), upd_writes(s, it), "upd", it)
        if s.mutant != "O2 before the scaling":
            yield from s.wait("scaled", it)
        s.mma(f"mma2({it})", o2_reads(it), [], "mma2", it, o2_rmw(s, it))
        if s.mutant == "group 1 before the state barrier" and it + 1 < nch:
            yield from issue1(it + 1)
        yield from s.sync("named", N_COMPUTE + 1)                          # B2
        if it + 1 < nch and s.mutant != "group 1 before the state barrier":
            yield from issue1(it + 1)
    yield from s.sync("named", N_COMPUTE + 1)                              # after the loop
    yield from s.sync("cta", 10)


def compute_warp(s, w):
    nch = s.nch
    s.write(("S", w), 0)                                                   # this warp's rows
    yield from s.sync("cta", 10)
    for it in range(nch):
        yield from s.wait("mma1", it)
        yield from s.wait("fullU", it)
        tag = f"warp{w} chunk {it}"
        x = xp(s, it)
        s.read(("Xd", x), ("raw", it), tag)
        s.read(("U", w), ("U", it), tag)                                   # its rows of U
        s.read(("vec", par(it)), it, tag)
        yield lambda: True                                                 # other warps may run
        s.write(("D", w), it)                                              # its D, D' rows
        s.write(("E", w), it)
        yield from s.sync("named", N_COMPUTE + 1)                          # B1
        s.read(("Xo", x, w), ("O1", it), tag)                              # f_t O1 in place
        yield lambda: True
        s.write(("Xo", x, w), ("fO1", it))
        s.bars["scaled"].arrive(it)
        yield from s.wait("upd", it)
        s.read(("Xd", 1 - x), ("dS", it), tag)                             # the state update
        s.read(("Xo", 1 - x, w), ("dS", it), tag)
        s.read(("vec", par(it)), it, tag)
        s.write(("S", w), it + 1)                                          # next chunk's S rows
        yield from s.sync("named", N_COMPUTE + 1)                          # B2
        if s.mutant != "output before O2":
            yield from s.wait("mma2", it)
        s.read_begin(("Xo", x, w), ("O", it), tag)                         # under group 1
        s.read_begin(("vec", par(it)), it, tag)
        yield lambda: True
        s.read_end(("Xo", x, w), ("O", it), tag)
        s.read_end(("vec", par(it)), it, tag)
        s.bars["oDone"].arrive(it)
    yield from s.sync("named", N_COMPUTE + 1)
    yield from s.sync("cta", 10)


def run(nch, seed, mutant=None):
    rng = random.Random(seed)
    s = Sim(nch, rng, mutant)
    actors = [copy_warp(s), mma_warp(s)] + [compute_warp(s, w) for w in range(N_COMPUTE)]
    blocked = [None] * len(actors)
    done = [False] * len(actors)
    for _ in range(200_000):
        if all(done):
            return True
        ready = [i for i, a in enumerate(actors)
                 if not done[i] and (blocked[i] is None or blocked[i]())]
        if not ready or rng.random() < 0.3:
            s.tick()
            continue
        i = rng.choice(ready)
        try:
            blocked[i] = next(actors[i])
        except StopIteration:
            done[i] = True
    raise AssertionError(f"no progress: nch={nch} seed={seed} done={done}")


@pytest.mark.parametrize("nch", [0, 1, 2, 3, 5, 8])
def test_pass_protocol_over_random_schedules(nch):
    for seed in range(60):
        assert run(nch, seed)


@pytest.mark.parametrize("mutant", ["no output barrier", "U after group 1", "arrive early",
                                    "group 1 before the state barrier", "one D/O1 set",
                                    "output before O2", "O2 before the scaling"])
def test_model_catches_planted_mistakes(mutant):
    """Each mistake, planted in the model, fails some schedule."""
    caught = 0
    for seed in range(60):
        try:
            run(5, seed, mutant)
        except AssertionError:
            caught += 1
    assert caught > 0, mutant
