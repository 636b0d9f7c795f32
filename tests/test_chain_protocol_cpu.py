"""Host-side check of the reverse chain's synchronisation protocol (the
tcgen05 backward chain of csrc/delta_bwd_tc.cu), by a model of its roles run
under many random interleavings:

  issuer      the one thread issuing products and record copies, in the
              kernel's order of waits, products, commits and copies;
  readback    warps moving dS' and du between TMEM and their operand tiles
              (two here, arriving on barriers that expect two);
  staging     warps writing the scale * dO tiles (two, likewise);
  tensor pipe executes issued products in order; a commit arrives once
              every product issued before it has completed;
  copy engine completes record copies in any order.

mbarrier waits are modelled as the hardware's parity test: a wait for phase
k succeeds when the completed-phase count n has n - k odd, so a waiter that
let its barrier run two phases ahead would block on the wrong phase.  Each
run asserts that no waiter ever falls that far behind, that the run never
deadlocks, and that no product reads a tile (or TMEM region) while a thread
or a copy writes it, nor the other way round."""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count, self.arrived, self.done = count, 0, 0   # done = completed phases

    def arrive(self):
        self.arrived += 1
        assert self.arrived <= self.count
        if self.arrived == self.count:
            self.arrived, self.done = 0, self.done + 1


class Model:
    def __init__(self, nc, NB, gated, n_rb=2, n_do=2, rng=None):
        self.nc, self.NB, self.gated, self.rng = nc, NB, gated, rng
        b = Barrier
        self.bar = {"DSREADY": b(n_rb), "DU": b(1), "DUREADY": b(n_rb), "DS": b(1), "END": b(1)}
        for i in range(NB):
            self.bar[f"REC{i}"], self.bar[f"DO{i}"], self.bar[f"FREE{i}"] = b(1), b(n_do), b(1)
        self.waiting = {}        # role -> (barrier, phase) it waits on
        self.pipe = []           # in-order tensor pipe: products and commits
        self.copies = []         # record copies in flight: (step, buffer)
        self.reads = {}          # resource -> products in flight reading it
        self.writes = {}         # resource -> products in flight writing it
        self.gend_read = {}      # step -> readback warps that have read its e^{b_L}
        self.du_read = {}        # step -> readback warps that have read du from TMEM
        self.ds_done = {}        # step -> readback warps done with TMEM dS for that step
        self.roles = {"issuer": self.issuer(), "tensor": self.tensor(), "copy": self.copy()}
        for r in range(n_rb):
            self.roles[f"rb{r}"] = self.readback(r)
        for s in range(n_do):
            self.roles[f"stage{s}"] = self.staging(s)
        self.n_rb = n_rb

    # ---------------------------------------------------------- primitives
    def parity_ok(self, name, k):
        n = self.bar[name].done
        assert n <= k + 1, f"{name}: phase {k} awaited after {n} completions (aliasing)"
        return (n - k) % 2 == 1

    def wait(self, role, name, k):
        self.waiting[role] = (name, k)
        return lambda: self.parity_ok(name, k)

    def product(self, tag, reads, writes):
        for r in reads:
            assert not self.writes.get(r), f"{tag} reads {r} while it is written"
            self.reads.setdefault(r, set()).add(tag)
        for w in writes:
            self.writes.setdefault(w, set()).add(tag)
        self.pipe.append(("mma", tag, reads, writes))

    def commit(self, name):
        self.pipe.append(("commit", name))

    def thread_write(self, res, who):
        assert not self.reads.get(res), f"{who} writes {res} while products read it"
        assert not self.writes.get(res), f"{who} writes {res} while products write it"

    def thread_read(self, res, who):
        assert not self.writes.get(res), f"{who} reads {res} while products write it"

    def issue_copy(self, step):
        b = step % self.NB
        self.thread_write(f"rec{b}", "record copy")
        if step >= self.NB:   # the buffer's previous step: every e^{b_L} read done
            assert self.gend_read.get(step - self.NB, 0) == (self.n_rb if self.gated else 0)
        self.writes.setdefault(f"rec{b}", set()).add(f"copy{step}")
        self.copies.append((step, b))

    # ---------------------------------------------------------- roles
    def issuer(self):
        nc, NB = self.nc, self.NB
        if nc == 0:
            return
        issued = 0
        while issued < NB and issued < nc:
            self.issue_copy(issued)
            issued += 1
        for i in range(nc):
            b, u = i % NB, i // NB
            yield self.wait("issuer", f"REC{b}", u)
            yield self.wait("issuer", f"DO{b}", u)
            # du = Aq^T dO' (DU overwritten: every warp has read du of step i - 1)
            assert i == 0 or self.du_read.get(i - 1, 0) == self.n_rb
            self.product(f"A{i}", [f"rec{b}", f"do{b}"], ["DU"])
            yield self.wait("issuer", "DSREADY", i)
            assert self.ds_done.get(i, 0) == self.n_rb
            self.product(f"K{i}", [f"rec{b}", "sds"], ["DU"])
            self.commit("DU")
            self.product(f"Q{i}", [f"rec{b}", f"do{b}"], ["DS"])
            if i >= 1 and issued < nc:
                self.issue_copy(issued)
                issued += 1
            yield self.wait("issuer", "DUREADY", i)
            self.product(f"W{i}", [f"rec{b}", "sdu"], ["DS"])
            self.commit("DS")
            self.commit(f"FREE{b}")
        self.commit("END")
        yield self.wait("issuer", "END", 0)

    def readback(self, r):
        nc, NB = self.nc, self.NB
        who = f"rb{r}"
        for i in range(nc):
            if i > 0:
                yield self.wait(who, "DS", i - 1)
            self.thread_read("DS", who)
            self.thread_write("sds", who)
            if self.gated:
                yield self.wait(who, f"REC{i % NB}", i // NB)
                self.thread_read(f"rec{i % NB}", who)
                self.gend_read[i] = self.gend_read.get(i, 0) + 1
                self.thread_write("DS", who)          # dS' * e^{b_L} back into TMEM
            elif i == 0:
                self.thread_write("DS", who)          # the final state's gradient
            self.ds_done[i] = self.ds_done.get(i, 0) + 1
            self.bar["DSREADY"].arrive()
            yield self.wait(who, "DU", i)
            self.thread_read("DU", who)
            self.du_read[i] = self.du_read.get(i, 0) + 1
            self.thread_write("sdu", who)
            self.bar["DUREADY"].arrive()
        if nc > 0:
            yield self.wait(who, "DS", nc - 1)
            self.thread_read("DS", who)

    def staging(self, s):
        NB = self.NB
        who = f"stage{s}"
        for j in range(self.nc):
            b = j % NB
            if j >= NB:
                yield self.wait(who, f"FREE{b}", j // NB - 1)
            self.thread_write(f"do{b}", who)
            self.bar[f"DO{b}"].arrive()

    def tensor(self):
        while True:
            yield lambda: bool(self.pipe)
            op = self.pipe.pop(0)
            if op[0] == "mma":
                _, tag, reads, writes = op
                for res in reads:
                    self.reads[res].discard(tag)
                for res in writes:
                    self.writes[res].discard(tag)
            else:
                self.bar[op[1]].arrive()

    def copy(self):
        while True:
            yield lambda: bool(self.copies)
            step, b = self.copies.pop(self.rng.randrange(len(self.copies)))
            self.writes[f"rec{b}"].discard(f"copy{step}")
            self.bar[f"REC{b}"].arrive()

    # ---------------------------------------------------------- scheduler
    def run(self):
        ready = {n: (lambda: True) for n in self.roles}
        finished = set()
        # every role runs at a speed drawn per run (some 50 times slower than
        # others), so that schedules starving one role are common
        speed = {n: self.rng.choice((0.02, 1.0)) for n in self.roles}
        for _ in range(400000):
            live = [n for n in self.roles if n not in finished and ready[n]()]
            workers = [n for n in self.roles if n not in finished and n not in ("tensor", "copy")]
            if not workers:
                assert not self.copies
                return
            assert live, f"deadlock: {self.waiting}"
            n = self.rng.choices(live, weights=[speed[x] for x in live])[0]
            self.waiting.pop(n, None)
            try:
                ready[n] = next(self.roles[n])
            except StopIteration:
                finished.add(n)
        raise AssertionError("did not finish")


@pytest.mark.parametrize("NB", [2, 4])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("nc", [0, 1, 2, 3, 5, 9])
def test_chain_protocol_random_interleavings(NB, gated, nc):
    for seed in range(60):
        Model(nc, NB, gated, rng=random.Random(1000 * nc + 10 * NB + seed)).run()


def test_model_catches_a_missing_free_wait():
    """The check is not vacuous: staging warps that skip the wait for the
    buffer's previous use overwrite a dO tile that products still read."""
    class NoFree(Model):
        def staging(self, s):
            for j in range(self.nc):
                b = j % self.NB
                self.thread_write(f"do{b}", f"stage{s}")
                self.bar[f"DO{b}"].arrive()
                yield lambda: True

    caught = 0
    for seed in range(40):
        try:
            NoFree(6, 2, False, rng=random.Random(seed)).run()
        except AssertionError:
            caught += 1
    assert caught > 0


def test_model_catches_phase_aliasing():
    """A single DO barrier shared by all buffers (so a fast staging role can
    complete two phases before the issuer waits) is reported as aliasing or
    as a deadlock."""
    class SharedDo(Model):
        def __init__(self, *a, **k):
            super().__init__(*a, **k)
            for i in range(self.NB):
                self.bar[f"DO{i}"] = self.bar["DO0"]

    caught = 0
    for seed in range(40):
        try:
            SharedDo(6, 4, False, rng=random.Random(seed)).run()
        except AssertionError:
            caught += 1
    assert caught > 0


def test_model_catches_an_early_record_copy():
    """An issuer that starts each record copy one step early (before the
    buffer's previous products, and its e^{b_L} reads, are done) is caught."""
    class EarlyCopy(Model):
        def issuer(self):
            nc, NB = self.nc, self.NB
            issued = 0
            while issued < NB and issued < nc:
                self.issue_copy(issued)
                issued += 1
            for i in range(nc):
                b, u = i % NB, i // NB
                if issued < nc:              # not after this step's DSREADY
                    self.issue_copy(issued)
                    issued += 1
                yield self.wait("issuer", f"REC{b}", u)
                yield self.wait("issuer", f"DO{b}", u)
                self.product(f"A{i}", [f"rec{b}", f"do{b}"], ["DU"])
                yield self.wait("issuer", "DSREADY", i)
                self.product(f"K{i}", [f"rec{b}", "sds"], ["DU"])
                self.commit("DU")
                self.product(f"Q{i}", [f"rec{b}", f"do{b}"], ["DS"])
                yield self.wait("issuer", "DUREADY", i)
                self.product(f"W{i}", [f"rec{b}", "sdu"], ["DS"])
                self.commit("DS")
                self.commit(f"FREE{b}")
            self.commit("END")
            yield self.wait("issuer", "END", 0)

    caught = 0
    for seed in range(40):
        try:
            EarlyCopy(6, 2, True, rng=random.Random(seed)).run()
        except AssertionError:
            caught += 1
    assert caught > 0
