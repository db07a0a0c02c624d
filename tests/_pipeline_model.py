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

With ``stop_at`` set the model runs the kernel's failure path instead: the
producer issues no load from that non-empty tile on (the debug library's
injected stall), every wait is bounded (a waiter that can no longer make
progress gives up, as the kernel's timed waits do), and the roles follow the
kernel's code after a wait gave up. The run must then end, with no copy in
flight when the roles are done (the CTA exits) and no MMA in flight when the
tensor memory is freed.
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


def _check(bar, parity, k, what, strict=True):
    """A parity test on `bar` that means phase k (parity k & 1). With
    strict=False (the failure path) only the hardware's answer is returned."""
    if not strict:
        return bar.parity_done(parity)
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

    def __init__(self, NT, STAGES, nk, spec_miss, rng, variant="kernel", stop_at=None, rope=False):
        self.NT, self.STAGES, self.nk, self.spec_miss = NT, STAGES, nk, spec_miss
        self.rope = rope  # the fused rotary embedding: q_rot[t] before head t's first product
        self.rng, self.variant = rng, variant
        self.stop_at = stop_at          # producer stall (failure path) or None
        self.strict = stop_at is None   # protocol checks only on the normal path
        self.timeouts = []              # waits that gave up (failure path)
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
        self.drain = B("drain", 1)
        self.qrot = [B(f"qrot{t}", 1) for t in range(NT)]
        self.t = 0.0
        self.events = []      # (time, seq, fn)
        self.seq = 0
        self.pipe_done = 0.0  # completion time of the last issued MMA

    # ---- asynchronous agents
    def at(self, dt, fn, kind="step"):
        self.seq += 1
        heapq.heappush(self.events, (self.t + dt, self.seq, fn, kind))

    def tma(self, bar, nbytes):
        self.at(self.rng.expovariate(1.0) * self.rng.choice([0.1, 1.0, 5.0]),
                lambda: bar.complete_tx(nbytes), "tma")

    def mma(self, n_ops=1):
        start = max(self.t, self.pipe_done)
        self.pipe_done = start + n_ops * self.rng.uniform(0.5, 1.5)

    def commit(self, bar):
        # arrives once every MMA this thread issued before it has completed
        self.seq += 1
        heapq.heappush(self.events, (max(self.t, self.pipe_done) + 1e-9, self.seq, bar.arrive, "mma"))

    @staticmethod
    def W(bar, k, what):
        """A bounded wait on `bar` for its phase k; evaluates to False when the
        wait gave up (failure path only)."""
        r = yield ("wait", bar, k & 1, k, what)
        return r

    # ---- the roles, as generators of ("wait", bar, parity, k, what) / ("test", ...) /
    # ("delay", dt); everything else happens inline
    def producer(self):
        m, S, W = self, self.STAGES, self.W
        # kernel start: Q and the speculative key/value tile 0
        m.q.expect_tx_arrive(2); m.tma(m.q, 2)
        m.kfull[0].expect_tx_arrive(1); m.tma(m.kfull[0], 1)
        m.vfull[0].expect_tx_arrive(1); m.tma(m.vfull[0], 1)
        yield ("delay", m.rng.uniform(0, 3))  # classification
        ok = True
        k_issued = 1 if (m.nk > 0 and not m.spec_miss) else 0
        v_issued = k_issued
        extra0 = 1 if (m.nk == 0 or m.spec_miss) else 0
        if m.nk == 0 or m.spec_miss:
            ok = yield from W(m.q, 0, "producer q")
            ok = ok and (yield from W(m.kfull[0], 0, "producer spec k"))
            ok = ok and (yield from W(m.vfull[0], 0, "producer spec v"))
            if m.variant != "old-speculation":
                m.spec.arrive()
        for n in range(m.nk):
            if not ok:
                break
            st, use = n % S, n // S
            if n == 0 and not m.spec_miss:
                continue
            if n == m.stop_at:
                break
            if n >= S:
                ok = yield from W(m.kempty[st], use - 1, f"producer kempty n={n}")
                if not ok:
                    break
            m.kfull[st].expect_tx_arrive(1); m.tma(m.kfull[st], 1)
            k_issued = n + 1
            if n >= S:
                ok = yield from W(m.vempty[st], use - 1, f"producer vempty n={n}")
                if not ok:
                    break
            m.vfull[st].expect_tx_arrive(1); m.tma(m.vfull[st], 1)
            v_issued = n + 1
            yield ("delay", m.rng.uniform(0, 0.5))
        # the kernel's exit drain: the last armed phase of every full barrier
        def arms(issued, st):
            return (extra0 if st == 0 else 0) + ((issued - 1 - st) // S + 1 if issued > st else 0)
        m.armed_k = [arms(k_issued, st) for st in range(S)]
        m.armed_v = [arms(v_issued, st) for st in range(S)]
        yield from W(m.q, 0, "producer drain q")
        for st in range(S):
            if m.armed_k[st]:
                yield from W(m.kfull[st], m.armed_k[st] - 1, f"producer drain kfull{st}")
            if m.armed_v[st]:
                yield from W(m.vfull[st], m.armed_v[st] - 1, f"producer drain vfull{st}")

    def mma_warp(self):
        m, S, NT, nk, W = self, self.STAGES, self.NT, self.nk, self.W
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
        ok = True
        if m.spec_miss:
            if m.variant == "old-speculation":
                yield ("wait", m.kfull[0], 0, 0, "mma spec k (old)")
                yield ("wait", m.vfull[0], 0, 0, "mma spec v (old)")
            else:
                ok = yield from W(m.spec, 0, "mma spec")
        ok = ok and (yield from W(m.q, 0, "mma q"))
        ok = ok and (yield from W(m.kfull[0], fill(0, 0), "mma k0"))
        ok = ok and (yield from W(m.vfull[0], fill(0, 0), "mma v0"))
        for t in range(NT):
            if not ok:
                break
            if m.rope:
                ok = yield from W(m.qrot[t], 0, f"mma qrot{t}")
                if not ok:
                    break
            issue_s(t, 0, 0, D16, D16)
        p0_seen = False
        for n in range(nk):
            if not ok:
                break
            st = n % S
            has_next = n + 1 < nk
            st1, use1 = (n + 1) % S, (n + 1) // S
            p1_seen = False
            for t in range(NT):
                if not ok:
                    break
                if not (p0_seen if t == 0 else p1_seen):
                    ok = yield from W(m.pfull[t], n, f"mma pfull{t} n={n}")
                    if not ok:
                        break
                m.mma(4)
                if has_next:
                    f1 = fill(st1, use1)
                    if t == 0:
                        ok = yield from W(m.kfull[st1], f1, f"mma kfull n+1={n + 1}")
                        if not ok:
                            break
                    if t == NT - 1:
                        ok = yield from W(m.vfull[st1], f1, f"mma vfull n+1={n + 1}")
                        if not ok:
                            break
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
            if not ok:
                break
            last_use = (nk - 1 - s) // S
            ok = yield from W(m.kempty[s], last_use, f"mma drain kempty{s}")
            ok = ok and (yield from W(m.vempty[s], last_use, f"mma drain vempty{s}"))
        if not ok and m.variant != "no-failure-drain":
            # every MMA issued completes before the tensor memory is freed
            m.commit(m.drain)
            yield from W(m.drain, 0, "mma failure drain")

    def softmax(self, t):
        m, W = self, self.W
        ok = True
        if m.rope:  # rotate the head's query tile once Q has landed
            ok = yield from W(m.q, 0, f"softmax{t} q for rotation")
            if ok:
                yield ("delay", m.rng.uniform(0.5, 3.0))
            m.qrot[t].arrive()
        for n in range(m.nk):
            if ok:
                ok = yield from W(m.sfull[t], n, f"softmax{t} sfull n={n}")
            if ok:  # after a failed wait the tile pass is skipped
                yield ("delay", m.rng.uniform(0.2, 4.0))
            m.pfull[t].arrive()
        if m.nk > 0:
            if ok:
                yield from W(m.odone[t], 0, f"epilogue{t} odone")
        elif ok:
            yield from W(m.q, 0, f"epilogue{t} q")

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
        for t in range(NT):
            if self.qrot[t].completed != (1 if self.rope else 0):
                raise ProtocolError(f"qrot{t}: {self.qrot[t].completed} phases")
        want_spec = 1 if (nk == 0 or self.spec_miss) and self.variant != "old-speculation" else 0
        if self.spec.completed != want_spec:
            raise ProtocolError(f"spec: {self.spec.completed} phases, expected {want_spec}")

    # ---- scheduler
    def run(self, max_steps=100000):
        actors = [self.producer(), self.mma_warp()] + [self.softmax(t) for t in range(self.NT)]
        state = {i: ("ready", None) for i in range(len(actors))}
        since = {}  # actor -> time its current wait began

        def step(i, value=None):
            try:
                op = actors[i].send(value)
            except StopIteration:
                state[i] = ("done", None)
                return
            state[i] = ("op", op)
            since[i] = self.t

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
                        if _check(bar, parity, k, what, self.strict):
                            step(i, True); progressed = True
                    elif op[0] == "test":
                        _, bar, parity, k, what = op
                        step(i, _check(bar, parity, k, what, self.strict)); progressed = True
                    elif op[0] == "delay":
                        state[i] = ("sleep", None)
                        self.at(op[1], lambda i=i: step(i))
                        progressed = True
            if all(kind == "done" for kind, _ in state.values()):
                # the CTA exits: nothing of it may still be in flight
                pending = sorted({kind for _, _, _, kind in self.events})
                if "tma" in pending:
                    raise ProtocolError("a copy is still in flight when the CTA exits")
                if "mma" in pending or self.pipe_done > self.t + 1e-6:
                    raise ProtocolError("an MMA is still in flight when the tensor memory is freed")
                if self.strict:
                    self._check_end_state()
                return
            if not self.events:
                blocked = [(since[i], i, op[4]) for i, (kind, op) in state.items()
                           if kind == "op" and op[0] == "wait"]
                if self.strict or not blocked:
                    raise ProtocolError(f"deadlock: blocked on {[b[2] for b in blocked]}")
                # failure path: the longest-waiting wait runs out of time first
                _, i, what = min(blocked)
                self.timeouts.append(what)
                step(i, False)
                continue
            self.t, _, fn, _ = heapq.heappop(self.events)
            fn()
        raise ProtocolError("schedule did not finish")
