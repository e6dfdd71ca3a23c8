"""Pins for the mbarrier ring simulator (oracle/ring_sim.py).

The printed S = 2 example of "Producer-Consumer Warp Specialization for TMA
Operations" is a golden fixture; the protocol invariants are checked under
random interleavings, and each garbled or literal reading of the pages is shown
to fail.
"""
import os

import pytest

from oracle import ring_sim as rs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "p2_double_buffer_schedule.txt")


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(tuple(int(x) for x in line.split()))
    return rows


def test_golden_schedule_closed_form():
    rows = _golden_rows()
    assert len(rows) == 4
    for S, i, slot, parity in rows:
        s, pf, pe = rs.schedule(i, S)
        assert (s, pf) == (slot, parity)
        assert pe == parity ^ 1


def test_golden_schedule_simulated():
    """The slots and parities a simulated run actually used match the page."""
    rows = _golden_rows()
    for seed in range(20):
        tr = rs.simulate_ring(4, 2, seed=seed)
        got = {(e.item, e.slot, e.parity) for e in tr.of("consumer0", "full_ok")}
        assert got == {(i, slot, parity) for _, i, slot, parity in rows}
        issued = [(e.item, e.slot) for e in tr.of("producer", "issue")]
        assert issued == [(i, slot) for _, i, slot, _ in rows]


def test_mbarrier_phase_semantics():
    b = rs.MBarrier(1)
    assert b.test_wait_parity(1)          # the phase before a fresh barrier counts as done
    assert not b.test_wait_parity(0)
    b.arrive_expect_tx(100)               # arrival alone does not finish the phase
    assert not b.test_wait_parity(0)
    b.complete_tx(60)
    assert not b.test_wait_parity(0)
    b.complete_tx(40)                     # tx reaches zero: phase 0 completes
    assert b.test_wait_parity(0) and not b.test_wait_parity(1)
    assert b.completed == 1
    with pytest.raises(rs.Violation):
        rs.MBarrier(1).arrive(2)


def _check_phases(tr, S, consumers):
    """I4: a successful wait saw exactly the phase count the parity rule implies."""
    for c in consumers:
        for e in tr.of(c, "full_ok"):
            assert e.phases_done == e.item // S + 1
    for e in tr.of("producer", "empty_ok"):
        assert e.phases_done == e.item // S


@pytest.mark.parametrize("S", range(1, 9))
@pytest.mark.parametrize("n_consumers", [1, 8])
def test_invariants_consumer_ring(S, n_consumers):
    for seed in range(6):
        n = 3 * S + 5
        tr = rs.simulate_ring(n, S, n_consumers=n_consumers, seed=seed)
        _check_phases(tr, S, ["consumer%d" % c for c in range(n_consumers)])
        assert 1 <= tr.max_lead <= S
        assert len(tr.of("consumer0", "release")) + len(tr.of("consumer", "release")) >= n


@pytest.mark.parametrize("S", range(1, 9))
@pytest.mark.parametrize("lag", [0, 1])
def test_invariants_store_ring(S, lag):
    if lag >= S:
        pytest.skip("a store lag must leave one slot to load into")
    for seed in range(6):
        tr = rs.simulate_ring(3 * S + 4, S, store_lag=lag, seed=seed)
        _check_phases(tr, S, ["consumer0"])


def test_producer_runs_up_to_S_ahead():
    """With S stages the producer can have S items in flight before a release
    ("gpu_warp_specialization", end-to-end flow: stage 3 issued while stage 0 is
    being computed)."""
    for S in (2, 4, 6):
        leads = {rs.simulate_ring(4 * S, S, seed=s).max_lead for s in range(40)}
        assert max(leads) == S


@pytest.mark.parametrize("S", [1, 2, 3, 4, 6])
@pytest.mark.parametrize("acc", [1, 2])
def test_invariants_gemm(S, acc):
    for seed in range(4):
        tr = rs.simulate_gemm(n_tiles=5, k_blocks=3, stages=S, acc_slots=acc, seed=seed)
        for e in tr.of("mma", "full_ok"):
            assert e.phases_done == e.item // S + 1
        for w in range(4):
            for e in tr.of("epi%d" % w, "acc_ok"):
                assert e.phases_done == e.item // acc + 1


def test_gemm_k_iterations_carry_phase_across_tiles():
    """A per-tile (rather than running) k counter would reuse parities wrongly
    when S does not divide the k-block count; the running counter is checked
    to complete for such shapes."""
    for seed in range(10):
        rs.simulate_gemm(n_tiles=7, k_blocks=5, stages=4, seed=seed)
        rs.simulate_gemm(n_tiles=4, k_blocks=1, stages=3, seed=seed)


# --- negative tests: each reading the pages rule out must fail ------------------

def _fails(fn, exc=rs.ProtocolError, seeds=range(30)):
    failures = 0
    for s in seeds:
        try:
            fn(s)
        except exc:
            failures += 1
    return failures


def test_slot_i_div_2_fails():
    rules = rs.Rules(slot=lambda i, S: i // 2)
    assert _fails(lambda s: rs.simulate_ring(6, 2, rules=rules, seed=s)) == 30


def test_unflipped_empty_parity_deadlocks():
    rules = rs.Rules(empty_parity=lambda i, S: (i // S) & 1)
    for S in (1, 2, 4):
        assert _fails(lambda s: rs.simulate_ring(8, S, rules=rules, seed=s), rs.Deadlock) == 30


def test_single_barrier_per_slot_fails():
    rules = rs.Rules(single_barrier=True)
    assert _fails(lambda s: rs.simulate_ring(8, 2, rules=rules, seed=s)) == 30
    assert _fails(lambda s: rs.simulate_gemm(3, 3, 2, rules=rules, seed=s)) == 30


def test_both_roles_arrive_and_wait_on_empty_deadlocks():
    rules = rs.Rules(both_arrive_on_empty=True)
    assert _fails(lambda s: rs.simulate_ring(6, 2, rules=rules, seed=s), rs.Deadlock) == 30


def test_gemm_full_parity_not_flipped_per_lap_fails():
    rules = rs.Rules(full_parity=lambda i, S: 0)
    assert _fails(lambda s: rs.simulate_gemm(3, 4, 2, rules=rules, seed=s)) == 30


hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402


@settings(max_examples=60, deadline=None)
@given(S=st.integers(1, 8), n=st.integers(0, 40), c=st.integers(1, 4),
       seed=st.integers(0, 2 ** 31 - 1))
def test_property_ring(S, n, c, seed):
    tr = rs.simulate_ring(n, S, n_consumers=c, seed=seed)
    _check_phases(tr, S, ["consumer%d" % k for k in range(c)])


@settings(max_examples=40, deadline=None)
@given(S=st.integers(1, 6), tiles=st.integers(0, 6), kb=st.integers(1, 6),
       acc=st.integers(1, 3), seed=st.integers(0, 2 ** 31 - 1))
def test_property_gemm(S, tiles, kb, acc, seed):
    rs.simulate_gemm(tiles, kb, S, acc_slots=acc, seed=seed)


# ------------------------------------------------------------------ replay
# The replay entry point feeds a recorded event trace through the same
# mbarrier model.  A run of the simulator, written out as such a trace, must
# replay cleanly; each planted mistake must be reported.

def _as_trace(tr):
    """The simulator's own events as a replay input (list order = time)."""
    prod, cons = [], []
    for t, e in enumerate(tr.events):
        if e.agent == "producer":
            prod.append((t, "wait" if e.what == "empty_ok" else "issued", e.item, e.slot,
                         e.parity or 0))
        elif e.what == "full_ok":
            cons.append((t, "wait", e.item, e.slot, e.parity))
        elif e.what == "release":
            cons.append((t, "released", e.item, e.slot, 0))
    return prod, cons


@pytest.mark.parametrize("S", [1, 2, 3, 5])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_replay_of_a_simulated_run_passes(S, seed):
    tr = rs.simulate_ring(23, S, seed=seed)
    prod, cons = _as_trace(tr)
    assert len(prod) == 2 * 23 and len(cons) == 2 * 23
    rep = rs.replay([prod], cons, S)
    assert len(rep.of("consumer", "full_ok")) == 23


def _unit(n, S, pair=False, tiles_k=4):
    """A valid trace of one unit: item i is issued once item i - S is released;
    tiles of tiles_k items go through a two-slot accumulator ring read by one
    epilogue role per CTA."""
    P = 2 if pair else 1
    prods = [[] for _ in range(P)]
    cons, mma, epis = [], [], [[] for _ in range(P)]
    t = 0
    for i in range(n):
        t += 10
        for p in range(P):
            prods[p] += [(t, "wait", i, i % S, ((i // S) & 1) ^ 1), (t + 1, "issued", i, i % S, 0)]
        cons += [(t + 5, "wait", i, i % S, (i // S) & 1), (t + 6, "released", i, i % S, 0)]
        if i % tiles_k == tiles_k - 1:
            tl = i // tiles_k
            mma += [(t + 2, "wait", tl, tl % 2, ((tl // 2) & 1) ^ 1), (t + 7, "issued", tl, tl % 2, 0)]
            for e in range(P):
                epis[e] += [(t + 8, "wait", tl, tl % 2, (tl // 2) & 1), (t + 9, "released", tl, tl % 2, 0)]
    return prods, cons, mma, epis


@pytest.mark.parametrize("S,pair", [(1, False), (2, False), (4, False), (3, True), (6, True)])
def test_replay_of_a_valid_unit_passes(S, pair):
    prods, cons, mma, epis = _unit(24, S, pair)
    rs.replay(prods, cons, S, mma_acc=mma, epilogues=epis)


def test_replay_reports_a_refill_before_release():
    prods, cons, mma, epis = _unit(12, 2)
    # the release of item 3 moves after the producer's wait for item 5
    k = [j for j, ev in enumerate(cons) if ev[1] == "released" and ev[2] == 3][0]
    wait5 = [ev for ev in prods[0] if ev[1] == "wait" and ev[2] == 5][0]
    cons[k] = (wait5[0] + 3,) + cons[k][1:]
    cons.sort()
    with pytest.raises(rs.Violation, match="before the slot's previous item was released"):
        rs.replay(prods, cons, 2)


def test_replay_reports_a_wrong_parity():
    prods, cons, _, _ = _unit(8, 2)
    k = [j for j, ev in enumerate(cons) if ev[1] == "wait" and ev[2] == 3][0]
    cons[k] = cons[k][:4] + (0,)                 # item 3 must wait on parity 1
    with pytest.raises(rs.Violation, match="parity"):
        rs.replay(prods, cons, 2)


def test_replay_reports_a_stage_seen_before_the_peer_issued_it():
    prods, cons, _, _ = _unit(8, 3, pair=True)
    prods[1] = [ev for ev in prods[1] if not (ev[1] == "issued" and ev[2] == 4)]
    with pytest.raises(rs.Violation, match="I2"):
        rs.replay(prods, cons, 3)


def test_replay_reports_a_wrong_slot():
    prods, cons, _, _ = _unit(8, 3)
    k = [j for j, ev in enumerate(prods[0]) if ev[1] == "issued" and ev[2] == 4][0]
    prods[0][k] = prods[0][k][:3] + (0, 0)
    with pytest.raises(rs.Violation, match="slot"):
        rs.replay(prods, cons, 3)


def test_replay_reports_an_accumulator_read_before_its_commit():
    prods, cons, mma, epis = _unit(16, 2)
    k = [j for j, ev in enumerate(mma) if ev[1] == "issued" and ev[2] == 1][0]
    w = [ev for ev in epis[0] if ev[1] == "wait" and ev[2] == 1][0]
    mma[k] = (w[0] + 1,) + mma[k][1:]
    with pytest.raises(rs.Violation, match="before its commit"):
        rs.replay(prods, cons, 2, mma_acc=mma, epilogues=epis)


def test_replay_reports_an_accumulator_reused_before_release():
    prods, cons, mma, epis = _unit(24, 2, pair=True)
    # tile 0's release by the odd CTA's epilogue comes after the MMA lane's wait for tile 2
    w2 = [ev for ev in mma if ev[1] == "wait" and ev[2] == 2][0]
    k = [j for j, ev in enumerate(epis[1]) if ev[1] == "released" and ev[2] == 0][0]
    epis[1][k] = (w2[0] + 1,) + epis[1][k][1:]
    with pytest.raises(rs.Violation, match="before the epilogue released it"):
        rs.replay(prods, cons, 2, mma_acc=mma, epilogues=epis)
