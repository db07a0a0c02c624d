"""A discrete-event model of the tensor-core prefill kernel's synchronisation:
the TMA producer, the MMA-issuing warp, the softmax warpgroups and the
epilogue, talking through mbarriers; TMA copies and the tensor pipe complete
asynchronously after random delays (the pipe in issue order, as one thread's
tcgen05 MMAs do).

Every parity wait and probe states the absolute phase it means. The model
checks that a wait passes only once that phase has completed and never on an
older one (a parity wait cannot tell phase k from k - 2 or k + 2), that a
waiter is never overtaken by two phases (it would then wait for a phase that
cannot come), and that every schedule ends without a deadlock. The roles
follow the kernel's loops step by step (the producer, the MMA warp with its
waits placed inside MMA groups and its probes, the softmax and the epilogue),
so a change of the kernel's protocol is mirrored here and checked on the CPU
before it runs on a GPU.
"""
from __future__ import annotations

import heapq
import random


class ProtocolError(AssertionError):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.completed = 0   # phases completed so far
        self.arrived = 0     # arrivals in the current phase
        self.tx = 0          # bytes still expected in the current phase

    def _maybe_complete(self):
        if self.arrived == self.count and self.tx == 0:
            self.completed += 1
            self.arrived = 0

    def arrive(self):
        self.arrived += 1
        self._maybe_complete()

    def expect_tx_arrive(self, nbytes):
        self.tx += nbytes
        self.arrive()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        if self.tx < 0:
            raise ProtocolError(f"{self.name}: more bytes landed than expected")
        self._maybe_complete()

    def parity_done(self, parity):
        # try_wait.parity / test_wait.parity: the phase of this parity has completed
        return (self.completed & 1) != parity


def _check(bar, parity, k, what):
    """A parity test on `bar` that means phase k (parity k & 1)."""
    if parity != (k & 1):
        raise ProtocolError(f"{what}: parity {parity} does not name phase {k}")
    done = bar.parity_done(parity)
    if done and bar.completed < k + 1:
        raise ProtocolError(f"{what}: {bar.name} passed on an older phase "
                            f"(completed {bar.completed}, meant phase {k})")
    if not done and bar.completed >= k + 1:
        raise ProtocolError(f"{what}: {bar.name} is two phases past phase {k} "
                            f"(completed {bar.completed}); the wait would never end")
    return done


class Model:
    """One CTA: NT heads, STAGES K/V stages, nk non-empty key tiles; spec_miss
    when the first non-empty tile is not tile 0 (the speculative tile-0 loads
    are then wasted). `rng` drives every delay."""

    def __init__(self, NT, STAGES, nk, spec_miss, rng, variant="kernel"):
        self.NT, self.STAGES, self.nk, self.spec_miss = NT, STAGES, nk, spec_miss
        self.rng, self.variant = rng, variant
        B = Barrier
        self.q = B("q", 1)
        self.kfull = [B(f"kfull{s}", 1) for s in range(STAGES)]
        self.vfull = [B(f"vfull{s}", 1) for s in range(STAGES)]
        self.kempty = [B(f"kempty{s}", 1) for s in range(STAGES)]
        self.vempty = [B(f"vempty{s}", 1) for s in range(STAGES)]
        self.sfull = [B(f"sfull{t}", 1) for t in range(NT)]
        self.pfull = [B(f"pfull{t}", 1) for t in range(NT)]
        self.odone = [B(f"odone{t}", 1) for t in range(NT)]
        self.spec = B("spec", 1)
        self.t = 0.0
        self.events = []      # (time, seq, fn)
        self.seq = 0
        self.pipe_done = 0.0  # completion time of the last issued MMA

    # ---- asynchronous agents
    def at(self, dt, fn):
        self.seq += 1
        heapq.heappush(self.events, (self.t + dt, self.seq, fn))

    def tma(self, bar, nbytes):
        self.at(self.rng.expovariate(1.0) * self.rng.choice([0.1, 1.0, 5.0]),
                lambda: bar.complete_tx(nbytes))

    def mma(self, n_ops=1):
        start = max(self.t, self.pipe_done)
        self.pipe_done = start + n_ops * self.rng.uniform(0.5, 1.5)

    def commit(self, bar):
        # arrives once every MMA this thread issued before it has completed
        self.seq += 1
        heapq.heappush(self.events, (max(self.t, self.pipe_done) + 1e-9, self.seq, bar.arrive))

    # ---- the roles, as generators of ("wait", bar, parity, k, what) / ("test", ...) /
    # ("delay", dt); everything else happens inline
    def producer(self):
        m, S = self, self.STAGES
        # kernel start: Q and the speculative key/value tile 0
        m.q.expect_tx_arrive(2); m.tma(m.q, 2)
        m.kfull[0].expect_tx_arrive(1); m.tma(m.kfull[0], 1)
        m.vfull[0].expect_tx_arrive(1); m.tma(m.vfull[0], 1)
        yield ("delay", m.rng.uniform(0, 3))  # classification
        if m.nk == 0 or m.spec_miss:
            yield ("wait", m.q, 0, 0, "producer q")
            yield ("wait", m.kfull[0], 0, 0, "producer spec k")
            yield ("wait", m.vfull[0], 0, 0, "producer spec v")
            if m.variant != "old-speculation":
                m.spec.arrive()
        for n in range(m.nk):
            st, use = n % S, n // S
            if n == 0 and not m.spec_miss:
                continue
            if n >= S:
                yield ("wait", m.kempty[st], (use - 1) & 1, use - 1, f"producer kempty n={n}")
            m.kfull[st].expect_tx_arrive(1); m.tma(m.kfull[st], 1)
            if n >= S:
                yield ("wait", m.vempty[st], (use - 1) & 1, use - 1, f"producer vempty n={n}")
            m.vfull[st].expect_tx_arrive(1); m.tma(m.vfull[st], 1)
            yield ("delay", m.rng.uniform(0, 0.5))

    def mma_warp(self):
        m, S, NT, nk = self, self.STAGES, self.NT, self.nk
        if nk == 0:
            return
        shift = 1 if m.spec_miss else 0

        def fill(st, use):  # absolute phase of a stage's use-th real fill
            return use + (shift if st == 0 else 0)

        def issue_s(t, st, k0, k1, D16):
            m.mma(k1 - k0)
            if k1 == D16:
                m.commit(m.sfull[t])
                if t == NT - 1:
                    m.commit(m.kempty[st])

        D16, kLate = 8, 7
        yield ("delay", m.rng.uniform(0, 3))
        if m.spec_miss:
            if m.variant == "old-speculation":
                yield ("wait", m.kfull[0], 0, 0, "mma spec k (old)")
                yield ("wait", m.vfull[0], 0, 0, "mma spec v (old)")
            else:
                yield ("wait", m.spec, 0, 0, "mma spec")
        yield ("wait", m.q, 0, 0, "mma q")
        yield ("wait", m.kfull[0], fill(0, 0) & 1, fill(0, 0), "mma k0")
        yield ("wait", m.vfull[0], fill(0, 0) & 1, fill(0, 0), "mma v0")
        for t in range(NT):
            issue_s(t, 0, 0, D16, D16)
        p0_seen = False
        for n in range(nk):
            st = n % S
            has_next = n + 1 < nk
            st1, use1 = (n + 1) % S, (n + 1) // S
            p1_seen = False
            for t in range(NT):
                if not (p0_seen if t == 0 else p1_seen):
                    yield ("wait", m.pfull[t], n & 1, n, f"mma pfull{t} n={n}")
                m.mma(4)
                if has_next:
                    f1 = fill(st1, use1)
                    if t == 0:
                        yield ("wait", m.kfull[st1], f1 & 1, f1, f"mma kfull n+1={n + 1}")
                    if t == NT - 1:
                        yield ("wait", m.vfull[st1], f1 & 1, f1, f"mma vfull n+1={n + 1}")
                m.mma(4)
                if n == nk - 1:
                    m.commit(m.odone[t])
                if t == NT - 1:
                    m.commit(m.vempty[st])
                if has_next:
                    if NT > 1 and t == NT - 1:
                        issue_s(t, st1, 0, kLate, D16)
                        p0_seen = yield ("test", m.pfull[0], (n + 1) & 1, n + 1, "mma probe p0")
                        issue_s(t, st1, kLate, D16, D16)
                    elif NT > 1:
                        issue_s(t, st1, 0, kLate, D16)
                        p1_seen = yield ("test", m.pfull[1], n & 1, n, "mma probe p1")
                        issue_s(t, st1, kLate, D16, D16)
                    else:
                        issue_s(t, st1, 0, D16, D16)
                yield ("delay", m.rng.uniform(0, 0.3))
        for s in range(min(S, nk)):
            last_use = (nk - 1 - s) // S
            yield ("wait", m.kempty[s], last_use & 1, last_use, f"mma drain kempty{s}")
            yield ("wait", m.vempty[s], last_use & 1, last_use, f"mma drain vempty{s}")

    def softmax(self, t):
        m = self
        for n in range(m.nk):
            yield ("wait", m.sfull[t], n & 1, n, f"softmax{t} sfull n={n}")
            yield ("delay", m.rng.uniform(0.2, 4.0))
            m.pfull[t].arrive()
        if m.nk > 0:
            yield ("wait", m.odone[t], 0, 0, f"epilogue{t} odone")
        else:
            yield ("wait", m.q, 0, 0, f"epilogue{t} q")

    def _check_end_state(self):
        # every barrier completed exactly the phases the protocol gives it
        S, nk, NT = self.STAGES, self.nk, self.NT
        for st in range(S):
            real = len(range(st, nk, S)) if nk else 0
            if st == 0 and not (nk > 0 and not self.spec_miss):
                real += 1  # the speculative phase, waited for separately
            for bars in (self.kfull, self.vfull):
                if bars[st].completed != real:
                    raise ProtocolError(f"{bars[st].name}: {bars[st].completed} phases, expected {real}")
            uses = len(range(st, nk, S))
            for bars in (self.kempty, self.vempty):
                if bars[st].completed != uses:
                    raise ProtocolError(f"{bars[st].name}: {bars[st].completed} phases, expected {uses}")
        for t in range(NT):
            for bar, want in ((self.sfull[t], nk), (self.pfull[t], nk), (self.odone[t], 1 if nk else 0)):
                if bar.completed != want:
                    raise ProtocolError(f"{bar.name}: {bar.completed} phases, expected {want}")
        want_spec = 1 if (nk == 0 or self.spec_miss) and self.variant != "old-speculation" else 0
        if self.spec.completed != want_spec:
            raise ProtocolError(f"spec: {self.spec.completed} phases, expected {want_spec}")

    # ---- scheduler
    def run(self, max_steps=100000):
        actors = [self.producer(), self.mma_warp()] + [self.softmax(t) for t in range(self.NT)]
        state = {i: ("ready", None) for i in range(len(actors))}

        def step(i, value=None):
            try:
                op = actors[i].send(value)
            except StopIteration:
                state[i] = ("done", None)
                return
            state[i] = ("op", op)

        for i in range(len(actors)):
            step(i)
        for _ in range(max_steps):
            progressed = True
            while progressed:
                progressed = False
                for i, (kind, op) in list(state.items()):
                    if kind != "op":
                        continue
                    if op[0] == "wait":
                        _, bar, parity, k, what = op
                        if _check(bar, parity, k, what):
                            step(i); progressed = True
                    elif op[0] == "test":
                        _, bar, parity, k, what = op
                        step(i, _check(bar, parity, k, what)); progressed = True
                    elif op[0] == "delay":
                        state[i] = ("sleep", None)
                        self.at(op[1], lambda i=i: step(i))
                        progressed = True
            if all(kind == "done" for kind, _ in state.values()) and not self.events:
                self._check_end_state()
                return
            if not self.events:
                blocked = [op[4] for kind, op in state.values() if kind == "op"]
                raise ProtocolError(f"deadlock: blocked on {blocked}")
            self.t, _, fn = heapq.heappop(self.events)
            fn()
        raise ProtocolError("schedule did not finish")
