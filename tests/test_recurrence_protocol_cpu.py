"""Host-side check of the forward recurrence's synchronisation protocol (the
tcgen05 state scan of csrc/delta_inter_tc.cu), the same way as the reverse
chain's (test_chain_protocol_cpu.py): a model of its roles under random
interleavings, with mbarrier waits as the hardware's parity test.

  issuer    per chunk c: u product into accumulator c % 2 (on top of the
            preloaded U), commit "u"; after the u tile is ready, the state
            product S += K~^T u, commit "s"; the output product into the
            same accumulator, then (once chunk c - 1's output is taken)
            commit "o"
  state     warps turning u into its bf16 tile (half of them), then the new
            S into its bf16 tile (and, gated, decaying it by the next
            chunk's e^{b_end})
  preload   warps writing U of chunk c into accumulator c % 2
  output    warps taking O out of accumulator c % 2 and zeroing it; one of
            them starts the record copy of chunk c + NB into chunk c's buffer

Each run asserts no phase aliasing, no deadlock, no product reading a tile
or TMEM region that a thread or copy is writing (and the other way round),
and that a record buffer is refilled only after every read of its previous
record (products, the U preload, the e^{b_end} reads) is done."""
import random

import pytest

from test_chain_protocol_cpu import Barrier, Model as _ChainModel


class Recurrence(_ChainModel):
    def __init__(self, nc, NB, gated, n_state=2, n_pre=2, n_out=2, rng=None):
        self.nc, self.NB, self.gated, self.rng = nc, NB, gated, rng
        b = Barrier
        self.bar = {"U": b(1), "S": b(1), "O": b(1), "SREADY": b(n_state),
                    "UREADY": b(n_state), "UPRE": b(n_pre), "OFREE0": b(n_out),
                    "OFREE1": b(n_out)}
        for i in range(NB):
            self.bar[f"REC{i}"] = b(1)
        self.waiting, self.pipe, self.copies = {}, [], []
        self.reads, self.writes = {}, {}
        self.rec_reads = {}      # chunk -> generic reads of its record done (U preload, gend)
        self.n_state, self.n_pre = n_state, n_pre
        self.roles = {"issuer": self.issuer(), "tensor": self.tensor(), "copy": self.copy()}
        for r in range(n_state):
            self.roles[f"state{r}"] = self.state(r)
        for r in range(n_pre):
            self.roles[f"pre{r}"] = self.preload(r)
        for r in range(n_out):
            self.roles[f"out{r}"] = self.output(r)

    def issue_copy(self, c):
        b = c % self.NB
        self.thread_write(f"rec{b}", "record copy")
        if c >= self.NB:   # every generic read of the buffer's previous record done
            prev = c - self.NB
            want = self.n_pre + (self.n_state if self.gated and prev >= 1 else 0)
            assert self.rec_reads.get(prev, 0) == want, (c, self.rec_reads.get(prev, 0), want)
        self.writes.setdefault(f"rec{b}", set()).add(f"copy{c}")
        self.copies.append((c, b))

    def issuer(self):
        nc, NB = self.nc, self.NB
        if nc == 0:
            return
        for c in range(min(NB, nc)):
            self.issue_copy(c)
        for c in range(nc):
            b, a = c % NB, f"acc{c & 1}"
            yield self.wait("issuer", "SREADY", c)
            yield self.wait("issuer", "UPRE", c)
            yield self.wait("issuer", f"REC{b}", c // NB)
            self.product(f"u{c}", [f"rec{b}", "sb", a], [a])
            self.commit("U")
            yield self.wait("issuer", "UREADY", c)
            self.product(f"s{c}", [f"rec{b}", "ut"], ["S"])
            self.commit("S")
            self.product(f"o{c}", [f"rec{b}", "ut", a], [a])
            if c >= 1:
                yield self.wait("issuer", f"OFREE{(c - 1) & 1}", ((c - 1) >> 1) + 1)
            self.commit("O")

    def state(self, r):
        nc, NB = self.nc, self.NB
        who = f"state{r}"
        u_warp = r == 0          # half of the state warps also move u
        if self.gated and nc > 0:
            yield self.wait(who, "REC0", 0)
            self.thread_read("rec0", who)
        self.thread_write("sb", who)
        self.thread_write("S", who)
        self.bar["SREADY"].arrive()
        for c in range(nc):
            if u_warp:
                yield self.wait(who, "U", c)
                self.thread_read(f"acc{c & 1}", who)
                self.thread_write("ut", who)
            self.bar["UREADY"].arrive()
            yield self.wait(who, "S", c)
            if c + 1 < nc:
                self.thread_read("S", who)
                self.thread_write("sb", who)
                self.bar["SREADY"].arrive()
                if self.gated:
                    b = (c + 1) % NB
                    yield self.wait(who, f"REC{b}", (c + 1) // NB)
                    self.thread_read(f"rec{b}", who)
                    self.rec_reads[c + 1] = self.rec_reads.get(c + 1, 0) + 1
                    self.thread_write("S", who)       # decayed in TMEM
        if nc > 0:
            self.thread_read("S", who)

    def preload(self, r):
        nc, NB = self.nc, self.NB
        who = f"pre{r}"
        for c in range(nc):
            if c >= 1:
                yield self.wait(who, "U", c - 1)
            yield self.wait(who, f"OFREE{c & 1}", c >> 1)
            yield self.wait(who, f"REC{c % NB}", c // NB)
            self.thread_read(f"rec{c % NB}", who)
            self.rec_reads[c] = self.rec_reads.get(c, 0) + 1
            self.thread_write(f"acc{c & 1}", who)
            self.bar["UPRE"].arrive()

    def output(self, r):
        nc, NB = self.nc, self.NB
        who = f"out{r}"
        for a in ("acc0", "acc1"):
            self.thread_write(a, who)
        self.bar["OFREE0"].arrive()
        self.bar["OFREE1"].arrive()
        for c in range(nc):
            yield self.wait(who, "O", c)
            self.thread_read(f"acc{c & 1}", who)
            self.thread_write(f"acc{c & 1}", who)     # O lanes zeroed
            self.bar[f"OFREE{c & 1}"].arrive()
            if r == 0 and c + NB < nc:
                self.issue_copy(c + NB)
        if False:
            yield


@pytest.mark.parametrize("NB", [1, 2, 4])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("nc", [0, 1, 2, 3, 5, 9])
def test_recurrence_protocol_random_interleavings(NB, gated, nc):
    for seed in range(60):
        Recurrence(nc, NB, gated, rng=random.Random(1000 * nc + 10 * NB + seed)).run()


def test_recurrence_model_catches_a_missing_output_hand_off():
    """An issuer that commits "o" without waiting for the output warps to
    take the previous chunk lets a commit run ahead of its waiters: the
    check reports aliasing, a hazard or a deadlock."""
    class NoHandOff(Recurrence):
        def issuer(self):
            nc, NB = self.nc, self.NB
            for c in range(min(NB, nc)):
                self.issue_copy(c)
            for c in range(nc):
                b, a = c % NB, f"acc{c & 1}"
                yield self.wait("issuer", "SREADY", c)
                yield self.wait("issuer", "UPRE", c)
                yield self.wait("issuer", f"REC{b}", c // NB)
                self.product(f"u{c}", [f"rec{b}", "sb", a], [a])
                self.commit("U")
                yield self.wait("issuer", "UREADY", c)
                self.product(f"s{c}", [f"rec{b}", "ut"], ["S"])
                self.commit("S")
                self.product(f"o{c}", [f"rec{b}", "ut", a], [a])
                self.commit("O")

    caught = 0
    for seed in range(60):
        try:
            NoHandOff(9, 4, False, n_state=1, rng=random.Random(seed)).run()
        except AssertionError:
            caught += 1
    assert caught > 0


def test_recurrence_model_catches_an_early_preload():
    """Preload warps that skip waiting for the issuer to take the previous
    chunk's U overwrite an accumulator that a product still uses."""
    class EarlyPreload(Recurrence):
        def preload(self, r):
            nc, NB = self.nc, self.NB
            who = f"pre{r}"
            for c in range(nc):
                yield self.wait(who, f"REC{c % NB}", c // NB)
                self.thread_read(f"rec{c % NB}", who)
                self.rec_reads[c] = self.rec_reads.get(c, 0) + 1
                self.thread_write(f"acc{c & 1}", who)
                self.bar["UPRE"].arrive()

    caught = 0
    for seed in range(60):
        try:
            EarlyPreload(9, 4, False, rng=random.Random(seed)).run()
        except AssertionError:
            caught += 1
    assert caught > 0
