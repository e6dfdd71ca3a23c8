"""Simulator of the mbarrier full/empty staging ring.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages describe the protocol in prose only:

* "Producer-Consumer Warp Specialization for TMA Operations": each staging
  buffer has a "full" and an "empty" mbarrier; tile i goes through a buffer
  chosen from i; each barrier flips phase when its buffer fills / drains; a
  waiter names the phase it waits for by a parity bit computed from the tile
  index (the page gives parity(i / 2) for two buffers).
* "pwwt.cn news/4436243", section 2.2: an mbarrier is a counter of expected
  arrivals; a TMA copy registers its byte count on the barrier (expected
  transaction count) and the copy engine's completion counts it down, so no
  thread has to arrive for the data.  Section 3.4: producer and consumer loops
  over ``slot = tile % stages``; one barrier per slot is not enough.
* "gpu_warp_specialization" (aicassindra.com), "End-to-end flow": producers
  fill stages ahead, consumers release them, fill/steady state/drain.

Readings taken where the pages are garbled or silent (each is a knob of
``Rules`` so the tests can show the other reading fails):

* slot = i % S (the S = 2 example on the TMA page lists 0,1,0,1; its formula
  "i/2" contradicts its own example).
* full wait parity = (i // S) & 1 (the page's parity(i/2) for S = 2).
* empty wait parity = ((i // S) & 1) ^ 1: the producer's first lap waits on the
  phase preceding a fresh barrier, which PTX reports as complete.
* only the consumer arrives on "empty" and only the producer waits on it (the
  section 3.4 pseudocode has both roles arrive-and-wait, which cannot start).

The mbarrier model follows the PTX ISA: a barrier holds the parity of its
current phase, a pending-arrival count and a transaction count; the phase
completes when both counts reach zero, then the parity flips and the arrival
count is re-armed; ``test_wait.parity(p)`` succeeds iff the phase with parity
p is no longer the current one.

Agents are generators that yield a predicate to block on; a seeded scheduler
steps a random ready agent, so asynchronous engines (TMA copies, tensor-core
commits, store reads) complete in random order and after random delays.
"""
from __future__ import annotations

import random
from dataclasses import dataclass, field
from typing import Callable, List, Optional


class ProtocolError(Exception):
    """Base class for a broken protocol run."""


class Deadlock(ProtocolError):
    """No agent can make progress but work remains (invariant I3)."""


class Violation(ProtocolError):
    """A safety invariant (I1, I2 or I4) failed."""


class MBarrier:
    """PTX mbarrier state: phase parity, pending arrivals, tx-count."""

    def __init__(self, count: int, name: str = ""):
        if count < 1:
            raise ValueError("an mbarrier needs an expected count >= 1")
        self.count = count
        self.pending = count
        self.tx = 0
        self.phase = 0          # parity of the current, incomplete phase
        self.completed = 0      # phases completed so far
        self.name = name

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase ^= 1
            self.completed += 1
            self.pending = self.count

    def arrive(self, n: int = 1):
        if n > self.pending:
            raise Violation("%s: more arrivals than expected in one phase" % self.name)
        self.pending -= n
        self._maybe_complete()

    def arrive_expect_tx(self, nbytes: int):
        """expect-tx(nbytes) followed by one arrive-on, as one operation."""
        self.tx += nbytes
        self.arrive(1)

    def complete_tx(self, nbytes: int):
        self.tx -= nbytes
        self._maybe_complete()

    def test_wait_parity(self, parity: int) -> bool:
        return self.phase != (parity & 1)


@dataclass
class Rules:
    slot: Callable[[int, int], int] = lambda i, S: i % S
    full_parity: Callable[[int, int], int] = lambda i, S: (i // S) & 1
    empty_parity: Callable[[int, int], int] = lambda i, S: ((i // S) & 1) ^ 1
    single_barrier: bool = False            # one barrier per slot for both signals
    both_arrive_on_empty: bool = False      # literal section 3.4 pseudocode


def schedule(i: int, S: int, rules: Rules = Rules()):
    """(slot, full-wait parity, empty-wait parity) of item i in an S-stage ring."""
    return rules.slot(i, S), rules.full_parity(i, S), rules.empty_parity(i, S)


@dataclass
class Event:
    agent: str
    what: str
    item: int
    slot: int
    parity: Optional[int] = None
    phases_done: Optional[int] = None


@dataclass
class Trace:
    events: List[Event] = field(default_factory=list)
    steps: int = 0
    max_lead: int = 0           # largest (issued - released) observed

    def of(self, agent: str, what: str):
        return [e for e in self.events if e.agent == agent and e.what == what]


class _Agent:
    def __init__(self, name, gen):
        self.name = name
        self.gen = gen
        self.pred = None
        self.done = False
        self._advance(None)

    def _advance(self, _):
        try:
            self.pred = next(self.gen)
        except StopIteration:
            self.done = True
            self.pred = None

    def ready(self) -> bool:
        return (not self.done) and (self.pred is None or self.pred())

    def step(self):
        self._advance(None)


class _Engine:
    """Asynchronous unit: completes submitted jobs in random or FIFO order."""

    def __init__(self, name, rng, ordered=False):
        self.name = name
        self.rng = rng
        self.ordered = ordered
        self.jobs = []
        self.done = False

    def submit(self, fn):
        self.jobs.append(fn)

    def ready(self) -> bool:
        return bool(self.jobs)

    def step(self):
        k = 0 if self.ordered else self.rng.randrange(len(self.jobs))
        self.jobs.pop(k)()


def _run(agents, engines, rng, max_steps, trace):
    units = list(agents) + list(engines)
    while True:
        live = [a for a in agents if not a.done]
        if not live and not any(e.jobs for e in engines):
            return trace
        ready = [u for u in units if u.ready()]
        if not ready:
            raise Deadlock("no agent can progress: " + ", ".join(
                "%s waiting" % a.name for a in live))
        rng.choice(ready).step()
        trace.steps += 1
        if trace.steps > max_steps:
            raise Deadlock("step bound %d exceeded" % max_steps)


def simulate_ring(n_items: int, stages: int, n_consumers: int = 1,
                  rules: Rules = Rules(), seed: int = 0,
                  store_lag: Optional[int] = None, tile_bytes: int = 32768,
                  max_steps: Optional[int] = None) -> Trace:
    """One producer feeding an S-slot ring read by ``n_consumers`` consumers.

    ``store_lag`` None: each consumer reads the slot synchronously and then
    arrives on empty (the FFMA consumers).  ``store_lag`` = L: a single
    consumer hands the slot to an asynchronous store engine (TMA store) and
    releases a slot once every store but the newest L has finished reading
    shared memory (``cp.async.bulk.wait_group.read L``), as in the staged copy.
    """
    rng = random.Random(seed)
    S = stages
    trace = Trace()
    if max_steps is None:
        max_steps = 200 * (n_items + 1) * (n_consumers + 2)
    full = [MBarrier(1, "full%d" % s) for s in range(S)]
    if rules.single_barrier:
        empty = full
    else:
        cnt = n_consumers + (1 if rules.both_arrive_on_empty else 0)
        empty = [MBarrier(cnt, "empty%d" % s) for s in range(S)]
    state = ["free"] * S             # free / loading / full
    tile_in = [None] * S
    done_readers = [set() for _ in range(S)]
    counters = {"issued": 0, "released": 0}
    tma = _Engine("tma", rng)
    store = _Engine("store", rng)

    def producer():
        for i in range(n_items):
            s = rules.slot(i, S)
            if rules.both_arrive_on_empty:
                target = empty[s].completed + 1
                empty[s].arrive()
                yield lambda: empty[s].completed >= target
            else:
                p = rules.empty_parity(i, S)
                yield lambda: empty[s].test_wait_parity(p)
                trace.events.append(Event("producer", "empty_ok", i, s, p, empty[s].completed))
            if state[s] != "free":                                     # I1
                raise Violation("I1: item %d issued into slot %d still %s (item %s)"
                                % (i, s, state[s], tile_in[s]))
            state[s] = "loading"
            tile_in[s] = i
            done_readers[s] = set()
            full[s].arrive_expect_tx(tile_bytes)
            counters["issued"] += 1
            trace.max_lead = max(trace.max_lead, counters["issued"] - counters["released"])
            trace.events.append(Event("producer", "issue", i, s))

            def land(s=s, i=i):
                if tile_in[s] != i or state[s] != "loading":
                    raise Violation("I1: copy of item %d landed in a reused slot" % i)
                state[s] = "full"
                full[s].complete_tx(tile_bytes)
            tma.submit(land)

    def release(s, i):
        state[s] = "free"
        counters["released"] += 1
        trace.events.append(Event("consumer", "release", i, s))

    def consumer(c):
        for i in range(n_items):
            s = rules.slot(i, S)
            p = rules.full_parity(i, S)
            yield lambda: full[s].test_wait_parity(p)
            if tile_in[s] != i or state[s] != "full":                  # I2
                raise Violation("I2: consumer %d read slot %d for item %d but it holds "
                                "item %s (%s)" % (c, s, i, tile_in[s], state[s]))
            trace.events.append(Event("consumer%d" % c, "full_ok", i, s, p, full[s].completed))
            for _ in range(rng.randrange(3)):
                yield None                                             # compute
            if tile_in[s] != i:
                raise Violation("I1: slot %d overwritten while item %d was read" % (s, i))
            done_readers[s].add(c)
            if len(done_readers[s]) == n_consumers:
                release(s, i)
            if rules.both_arrive_on_empty:
                target = empty[s].completed + 1
                empty[s].arrive()
                yield lambda: empty[s].completed >= target
            else:
                empty[s].arrive()

    def storer():
        L = store_lag
        pending = []          # items whose store has not finished reading smem
        unreleased = []       # items stored but whose slot is not yet released
        for i in range(n_items):
            s = rules.slot(i, S)
            p = rules.full_parity(i, S)
            yield lambda: full[s].test_wait_parity(p)
            if tile_in[s] != i or state[s] != "full":                  # I2
                raise Violation("I2: store of item %d from slot %d holding %s"
                                % (i, s, tile_in[s]))
            trace.events.append(Event("consumer0", "full_ok", i, s, p, full[s].completed))
            pending.append(i)
            unreleased.append(i)

            def read_done(i=i, s=s):
                if tile_in[s] != i:
                    raise Violation("I1: slot %d overwritten while item %d was stored" % (s, i))
                pending.remove(i)
            store.submit(read_done)
            # wait_group.read L: every store but the newest L has finished reading
            yield lambda i=i: all(j > i - L for j in pending)
            while unreleased and unreleased[0] not in pending:
                j = unreleased.pop(0)
                sj = rules.slot(j, S)
                release(sj, j)
                empty[sj].arrive()
        yield lambda: not pending                                      # wait_group.read 0
        while unreleased:
            j = unreleased.pop(0)
            release(rules.slot(j, S), j)

    agents = [_Agent("producer", producer())]
    if store_lag is None:
        agents += [_Agent("consumer%d" % c, consumer(c)) for c in range(n_consumers)]
    else:
        if n_consumers != 1:
            raise ValueError("the store path has one storer")
        agents.append(_Agent("storer", storer()))
    return _run(agents, [tma, store], rng, max_steps, trace)


def simulate_gemm(n_tiles: int, k_blocks: int, stages: int, acc_slots: int = 2,
                  epi_warps: int = 4, rules: Rules = Rules(), seed: int = 0,
                  stage_bytes: int = 49152, max_steps: Optional[int] = None) -> Trace:
    """The persistent tensor-core GEMM: TMA producer -> S-slot smem ring ->
    MMA issuer (commits release slots asynchronously, in issue order) ->
    ``acc_slots``-slot accumulator ring -> ``epi_warps`` epilogue warps.

    Every role walks the same tile sequence; the producer and MMA issuer keep
    one k-block counter running across tiles, so phases carry over tile
    boundaries.
    """
    rng = random.Random(seed)
    S, A = stages, acc_slots
    trace = Trace()
    if max_steps is None:
        max_steps = 400 * (n_tiles * (k_blocks + 2) + 1) * (epi_warps + 3)
    full = [MBarrier(1, "full%d" % s) for s in range(S)]
    empty = full if rules.single_barrier else [MBarrier(1, "empty%d" % s) for s in range(S)]
    acc_full = [MBarrier(1, "acc_full%d" % a) for a in range(A)]
    acc_empty = [MBarrier(epi_warps, "acc_empty%d" % a) for a in range(A)]
    state = ["free"] * S
    tag = [None] * S
    acc_tile = [None] * A
    acc_kdone = [0] * A
    acc_state = ["free"] * A          # free / accumulating / ready
    epi_done = [set() for _ in range(A)]
    tma = _Engine("tma", rng)
    tc = _Engine("tensor", rng, ordered=True)

    def producer():
        it = 0
        for t in range(n_tiles):
            for kb in range(k_blocks):
                s = rules.slot(it, S)
                p = rules.empty_parity(it, S)
                yield lambda: empty[s].test_wait_parity(p)
                if state[s] != "free":
                    raise Violation("I1: k-block %d issued into busy slot %d" % (it, s))
                state[s], tag[s] = "loading", (t, kb)
                full[s].arrive_expect_tx(stage_bytes)
                trace.events.append(Event("producer", "issue", it, s, p, empty[s].completed))

                def land(s=s, tk=(t, kb)):
                    if tag[s] != tk:
                        raise Violation("I1: copy landed in a reused slot")
                    state[s] = "full"
                    full[s].complete_tx(stage_bytes)
                tma.submit(land)
                it += 1

    def mma():
        it = 0
        for t in range(n_tiles):
            a = t % A
            pa = ((t // A) & 1) ^ 1
            yield lambda: acc_empty[a].test_wait_parity(pa)
            if acc_state[a] != "free":
                raise Violation("accumulator %d reused before the epilogue drained it" % a)
            acc_state[a], acc_tile[a], acc_kdone[a] = "accumulating", t, 0
            for kb in range(k_blocks):
                s = rules.slot(it, S)
                p = rules.full_parity(it, S)
                yield lambda: full[s].test_wait_parity(p)
                if tag[s] != (t, kb) or state[s] != "full":
                    raise Violation("I2: MMA of (%d,%d) read slot %d holding %s"
                                    % (t, kb, s, tag[s]))
                trace.events.append(Event("mma", "full_ok", it, s, p, full[s].completed))

                def mma_done(s=s, a=a, tk=(t, kb)):
                    if tag[s] != tk:
                        raise Violation("I1: slot overwritten during its MMA")
                    acc_kdone[a] += 1
                    state[s] = "free"
                    empty[s].arrive()                                  # tcgen05.commit
                tc.submit(mma_done)
                it += 1

            def acc_done(a=a, t=t):
                if acc_kdone[a] != k_blocks or acc_tile[a] != t:
                    raise Violation("accumulator committed before its MMAs finished")
                acc_state[a] = "ready"
                acc_full[a].arrive()
            tc.submit(acc_done)

    def epilogue(w):
        for t in range(n_tiles):
            a = t % A
            p = (t // A) & 1
            yield lambda: acc_full[a].test_wait_parity(p)
            if acc_tile[a] != t or acc_state[a] != "ready":
                raise Violation("epilogue %d read accumulator %d holding tile %s"
                                % (w, a, acc_tile[a]))
            trace.events.append(Event("epi%d" % w, "acc_ok", t, a, p, acc_full[a].completed))
            for _ in range(rng.randrange(3)):
                yield None
            epi_done[a].add((t, w))
            if sum(1 for (tt, _) in epi_done[a] if tt == t) == epi_warps:
                acc_state[a] = "free"
            acc_empty[a].arrive()

    agents = [_Agent("producer", producer()), _Agent("mma", mma())]
    agents += [_Agent("epi%d" % w, epilogue(w)) for w in range(epi_warps)]
    return _run(agents, [tma, tc], rng, max_steps, trace)


# ---------------------------------------------------------------------------
# Replay of an event trace recorded on the GPU.
#
# A trace event is a tuple (t, ev, item, slot, parity): t a timestamp, ev one
# of "wait" (a wait returned; recorded after it), "issued" (a producer issued
# an item's copies, or the MMA lane committed a tile to its accumulator;
# recorded before) or "released" (a consumer released a slot; recorded
# before).  Events are replayed in time order, with "issued"/"released"
# before "wait" at equal times, through the MBarrier model above:
#
# * a producer's "issued" registers the item on full[slot] (the first
#   producer of a unit registers every producer's bytes, as one arrive with
#   expect-tx) and puts its copy in flight;
# * a consumer's "wait" on full first lands the item's copies in flight, then
#   must find the phase it names complete (I4); its item must be the one the
#   slot holds and every producer must have issued it (I2);
# * a "released" arrives on empty[slot] of every producer (on the CTA pair the
#   commit reaches both CTAs' empty barriers); a producer's "wait" on empty
#   must find its phase complete, which is what keeps a slot from being
#   refilled before it was released (I1);
# * the accumulator ring likewise: the MMA lane waits on acc_empty and
#   commits to every epilogue role's acc_full; each epilogue role waits on its
#   acc_full and arrives on acc_empty.
#
# Slot and parity of every wait must also follow ``rules``.

def replay(producers, consumer, stages: int, mma_acc=None, epilogues=None,
           rules: Rules = Rules(), acc_slots: int = 2) -> Trace:
    """Replays one unit's GPU trace; raises Violation at the first event the
    model contradicts.  producers: one event list per producing CTA;
    consumer: the consuming role's events; mma_acc / epilogues: the
    accumulator ring's events (optional)."""
    S, P = stages, len(producers)
    if P < 1:
        raise ValueError("need at least one producer")
    full = [MBarrier(1, "full%d" % s) for s in range(S)]
    empty = [[MBarrier(1, "empty%d.%d" % (p, s)) for s in range(S)] for p in range(P)]
    holds = [None] * S              # item the slot was last registered for
    issuers = [set() for _ in range(S)]
    in_flight = {}                  # item -> producers whose copy has not landed
    trace = Trace()
    stream = []
    kinds = {"issued": 0, "released": 0, "wait": 1}
    for p, evs in enumerate(producers):
        stream += [(t, kinds[ev], "producer", p, ev, i, s, par) for (t, ev, i, s, par) in evs]
    stream += [(t, kinds[ev], "consumer", 0, ev, i, s, par) for (t, ev, i, s, par) in consumer]
    E = len(epilogues or [])
    if mma_acc is not None:
        acc_full = [[MBarrier(1, "acc_full%d.%d" % (e, a)) for a in range(acc_slots)]
                    for e in range(E)]
        acc_empty = [MBarrier(E, "acc_empty%d" % a) for a in range(acc_slots)]
        committed = {}              # accumulator item -> epilogue roles not yet signalled
        stream += [(t, kinds[ev], "mma_acc", 0, ev, i, s, par) for (t, ev, i, s, par) in mma_acc]
        for e, evs in enumerate(epilogues):
            stream += [(t, kinds[ev], "epilogue", e, ev, i, s, par) for (t, ev, i, s, par) in evs]
    stream.sort(key=lambda x: (x[0], x[1]))

    for t, _, role, who, ev, i, s, par in stream:
        trace.steps += 1
        if role == "producer":
            if s != rules.slot(i, S):
                raise Violation("producer %d: item %d in slot %d" % (who, i, s))
            if ev == "wait":
                if par != rules.empty_parity(i, S):
                    raise Violation("producer %d: item %d waited empty parity %d" % (who, i, par))
                if not empty[who][s].test_wait_parity(par):
                    raise Violation("I1/I4: producer %d passed empty[%d] (parity %d) for item %d "
                                    "before the slot's previous item was released" % (who, s, par, i))
                trace.events.append(Event("producer%d" % who, "empty_ok", i, s, par,
                                          empty[who][s].completed))
            elif ev == "issued":
                if holds[s] != i:
                    if holds[s] is not None and issuers[s] and holds[s] in in_flight:
                        raise Violation("I1: item %d issued into slot %d while item %d is still "
                                        "in flight" % (i, s, holds[s]))
                    if full[s].completed != i // S:
                        raise Violation("I1: item %d issued into slot %d in phase %d"
                                        % (i, s, full[s].completed))
                    holds[s], issuers[s] = i, set()
                    full[s].arrive_expect_tx(P)     # one unit of bytes per producer's copy
                issuers[s].add(who)
                in_flight.setdefault(i, set()).add(who)
                trace.events.append(Event("producer%d" % who, "issue", i, s))
        elif role == "consumer":
            if s != rules.slot(i, S):
                raise Violation("consumer: item %d in slot %d" % (i, s))
            if ev == "wait":
                if par != rules.full_parity(i, S):
                    raise Violation("consumer: item %d waited full parity %d" % (i, par))
                if holds[s] != i or len(issuers[s]) != P:
                    raise Violation("I2: consumer passed full[%d] for item %d, which holds item %s "
                                    "issued by %d of %d producers"
                                    % (s, i, holds[s], len(issuers[s]), P))
                for _ in in_flight.pop(i, set()):
                    full[s].complete_tx(1)
                if not full[s].test_wait_parity(par):
                    raise Violation("I4: consumer passed full[%d] (parity %d) for item %d before "
                                    "the phase completed" % (s, par, i))
                trace.events.append(Event("consumer", "full_ok", i, s, par, full[s].completed))
            elif ev == "released":
                if holds[s] != i:
                    raise Violation("consumer released slot %d for item %d, which holds item %s"
                                    % (s, i, holds[s]))
                for p in range(P):
                    empty[p][s].arrive()
                trace.events.append(Event("consumer", "release", i, s))
        elif role == "mma_acc":
            if s != i % acc_slots:
                raise Violation("MMA lane: accumulator item %d in slot %d" % (i, s))
            if ev == "wait":
                want = ((i // acc_slots) & 1) ^ 1
                if par != want or not acc_empty[s].test_wait_parity(par):
                    raise Violation("MMA lane passed acc_empty[%d] (parity %d) for item %d before "
                                    "the epilogue released it" % (s, par, i))
            elif ev == "issued":
                committed[i] = set(range(E))
        else:   # epilogue role `who`
            if s != i % acc_slots:
                raise Violation("epilogue %d: accumulator item %d in slot %d" % (who, i, s))
            if ev == "wait":
                if par != (i // acc_slots) & 1:
                    raise Violation("epilogue %d: item %d waited parity %d" % (who, i, par))
                if who in committed.get(i, ()):
                    committed[i].discard(who)
                    acc_full[who][s].arrive()
                if not acc_full[who][s].test_wait_parity(par):
                    raise Violation("epilogue %d passed acc_full[%d] for item %d before its commit"
                                    % (who, s, i))
            elif ev == "released":
                acc_empty[s].arrive()
    return trace
