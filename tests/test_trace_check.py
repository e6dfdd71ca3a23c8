"""The trace checker itself, on synthetic traces: a trace that follows the
ring protocol passes, and each planted mistake (wrong slot, wrong parity, a
slot refilled before its release, a consumer seeing a stage before it was
issued, a lost release) is reported.  No GPU."""
import numpy as np
import pytest

from mbarrier_gemm_pipelines_gb300 import trace
from trace_check import check


def _recs(rows):
    a = np.zeros(len(rows), dtype=trace.RECORD)
    for k, (t, item, role, ev, slot, par) in enumerate(rows):
        a[k] = (t, item, role, ev, slot, par)
    return a


def _valid(n, S):
    """Producer fills item i once item i - S is released; everything in order."""
    prod, cons = [], []
    t = 0
    for i in range(n):
        t += 10
        prod += [(t, i, 0, 0, i % S, ((i // S) & 1) ^ 1), (t + 1, i, 0, 1, i % S, 0)]
        cons += [(t + 5, i, 1, 0, i % S, (i // S) & 1), (t + 6, i, 1, 2, i % S, 0)]
    return {(0, 0): _recs(prod), (0, 1): _recs(cons)}, {(0, 0): 2 * n, (0, 1): 2 * n}


@pytest.mark.parametrize("S", [1, 2, 3, 6])
def test_valid_trace_passes(S):
    ev, cnt = _valid(20, S)
    assert check(ev, cnt, S) == []


def _mutate(S, role, idx, field, value):
    ev, cnt = _valid(12, S)
    ev[(0, role)][idx][field] = value
    return check(ev, cnt, S)


def test_wrong_slot_is_reported():
    assert any("slot" in e for e in _mutate(3, 0, 8, "slot", 0))


def test_wrong_parity_is_reported():
    assert any("parity" in e for e in _mutate(2, 1, 6, "parity", 0))   # item 3 waits on parity 1


def test_refill_before_release_is_reported():
    ev, cnt = _valid(12, 2)
    rel = ev[(0, 1)]
    # item 3's release happens after the producer's wait for item 5
    rel[7]["t"] = ev[(0, 0)][10]["t"] + 3
    assert any("before the release" in e for e in check(ev, cnt, 2))


def test_consumer_before_issue_is_reported():
    ev, cnt = _valid(6, 2)
    ev[(0, 0)][5]["t"] = ev[(0, 1)][4]["t"] + 1          # item 2 issued after it was seen full
    assert any("before producer" in e for e in check(ev, cnt, 2))


def test_lost_release_is_reported():
    ev, cnt = _valid(8, 2)
    cons = ev[(0, 1)]
    keep = np.ones(len(cons), bool)
    keep[3] = False                                       # release of item 1
    ev[(0, 1)] = cons[keep]
    assert any("before item 1 was released" in e for e in check(ev, cnt, 2))


def test_truncated_trace_is_reported():
    ev, cnt = _valid(4, 2)
    cnt[(0, 1)] = 100
    assert any("only" in e for e in check(ev, cnt, 2))


def test_decode_layout():
    cap = 3
    raw = np.zeros(trace.bytes_for(cap), dtype=np.uint8)
    counts = raw[:trace.HEADER_BYTES].view("<u4").reshape(trace.MAX_CTAS, trace.ROLES)
    counts[5, 1] = 2
    recs = raw[trace.HEADER_BYTES:].view(trace.RECORD).reshape(trace.MAX_CTAS, trace.ROLES, cap)
    recs[5, 1, 0] = (123, 7, 1, 0, 3, 1)
    recs[5, 1, 1] = (130, 7, 1, 2, 3, 0)
    ev, cnt = trace.decode(raw)
    assert cnt == {(5, 1): 2}
    assert list(ev[(5, 1)]["t"]) == [123, 130] and int(ev[(5, 1)][0]["slot"]) == 3
