"""The dense GEMM's pipeline protocol with both operands expanded, simulated on
the CPU under random schedules.

Roles and barriers follow the kernel: a producer fills a ring of RAW stages
(full_raw), the MMA issuer waits for a stage's copies at its first block and for
a free TMEM buffer (tm_empty, NBUF buffers), commits each block (tm_full) and
releases a stage after its last block (empty_raw); two converter warps publish
each stage's scales into slot s mod NSC once its copies have landed
(sc_ready); eight workers wait for a stage's scales at its first block and for
each block's accumulator, and hand the buffer back after loading it.  Copies and
MMAs complete asynchronously after random delays, as on the GPU.

Checked on every step of every schedule:
* each parity wait finds its barrier 0 or 1 phases past the phase it waits for
  (a barrier 2 phases ahead, or 1 behind, would alias on the parity bit);
* no scale slot is read before its stage was published, nor rewritten while a
  worker still reads the stage before;
* no raw stage is refilled while an MMA of its previous stage is pending;
* no TMEM buffer is written by an MMA while a worker has not yet loaded the block
  before it;
* every schedule finishes (no deadlock), each worker folding every block in order.
"""
import random

import pytest

KB = 4          # blocks per stage
RAW = 3         # raw stages in flight
NSC = RAW + 1   # scale slots
NBUF = 2        # TMEM accumulator buffers
WORKERS = 8
CONV = 2


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.completed = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: more arrivals than expected"
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count


def run_schedule(nstages, seed):
    rng = random.Random(seed)
    nblocks = nstages * KB
    full_raw = [Barrier(f"full_raw{i}", 1) for i in range(RAW)]
    empty_raw = [Barrier(f"empty_raw{i}", 1) for i in range(RAW)]
    tm_full = [Barrier(f"tm_full{i}", 1) for i in range(NBUF)]
    tm_empty = [Barrier(f"tm_empty{i}", WORKERS) for i in range(NBUF)]
    sc_ready = [Barrier(f"sc_ready{i}", CONV) for i in range(NSC)]

    state = {"loaded": [0] * WORKERS, "folded": [0] * WORKERS, "mma_done": 0, "mma_issued": 0,
             "published": [0] * nstages}
    async_events = []  # (remaining ticks, action)

    def wait(bar, phase):
        """Generator helper: poll until phase completes (one poll per scheduler step)."""
        while True:
            if phase < 0:
                return
            # a fresh barrier has completed no phase; waiting for phase -1 passes
            assert bar.completed >= phase, (bar.name, "behind by more than one phase", phase, bar.completed)
            assert bar.completed <= phase + 1, (bar.name, "two phases ahead", phase, bar.completed)
            if bar.completed == phase + 1:
                return
            yield

    def producer():
        for g in range(nstages):
            yield from wait(empty_raw[g % RAW], g // RAW - 1)
            # refilling the slot: the MMAs of stage g - RAW have all completed
            assert state["mma_done"] >= (g - RAW + 1) * KB if g >= RAW else True
            async_events.append([rng.randint(1, 30), lambda g=g: full_raw[g % RAW].arrive()])
            yield

    def mma():
        for b in range(nblocks):
            s, kb = divmod(b, KB)
            if kb == 0:
                yield from wait(full_raw[s % RAW], s // RAW)
            tb = b % NBUF
            yield from wait(tm_empty[tb], b // NBUF - 1)
            # writing buffer tb: every worker has loaded block b - NBUF
            assert all(n >= b - NBUF + 1 for n in state["loaded"]), ("tmem overwritten", b, state["loaded"])
            state["mma_issued"] += 1

            def complete(b=b, tb=tb, s=s, kb=kb):
                state["mma_done"] = b + 1  # MMAs complete in order
                tm_full[tb].arrive()
                if kb == KB - 1:
                    empty_raw[s % RAW].arrive()
            delay = rng.randint(1, 20)
            # in-order completion: never before the previous MMA's
            pend = [e[0] for e in async_events if getattr(e[1], "is_mma", False)]
            delay = max([delay] + [d + 1 for d in pend])
            complete.is_mma = True
            async_events.append([delay, complete])
            yield

    def converter(cw):
        for s in range(nstages):
            yield from wait(full_raw[s % RAW], s // RAW)
            for _ in range(rng.randint(0, 6)):  # the scale loads
                yield
            # rewriting slot s % NSC: every worker is past stage s - NSC
            if s >= NSC:
                assert all(n >= (s - NSC + 1) * KB for n in state["folded"]), ("scale slot overwritten", s)
            state["published"][s] += 1
            sc_ready[s % NSC].arrive()
            yield

    def worker(w):
        for b in range(nblocks):
            s, kb = divmod(b, KB)
            if kb == 0:
                yield from wait(sc_ready[s % NSC], s // NSC)
            tb = b % NBUF
            yield from wait(tm_full[tb], b // NBUF)
            # the fold reads stage s's scales: both converters have published them
            assert state["published"][s] == CONV, ("scales read before they were published", b)
            for _ in range(rng.randint(1, 8)):  # TMEM loads
                yield
            state["loaded"][w] = b + 1
            tm_empty[tb].arrive()  # early release: the block is in registers
            for _ in range(rng.randint(1, 8)):  # the fold of the last piece
                yield
            assert state["folded"][w] == b
            state["folded"][w] = b + 1
            yield

    roles = [producer(), mma()] + [converter(i) for i in range(CONV)] + [worker(i) for i in range(WORKERS)]
    live = list(roles)
    steps = 0
    while live or async_events:
        steps += 1
        assert steps < 10_000_000, "no progress"
        # advance asynchronous completions by one tick
        for e in list(async_events):
            e[0] -= 1
        for e in [e for e in async_events if e[0] <= 0]:
            async_events.remove(e)
            e[1]()
        if live:
            r = rng.choice(live)
            try:
                next(r)
            except StopIteration:
                live.remove(r)
        elif not async_events:
            break
    assert state["folded"] == [nblocks] * WORKERS
    assert state["mma_done"] == nblocks


@pytest.mark.parametrize("nstages", [1, 2, 3, 4, 5, 9, 17])
@pytest.mark.parametrize("seed", range(12))
def test_expanded_pipeline_protocol(nstages, seed):
    run_schedule(nstages, seed)
