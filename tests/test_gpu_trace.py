"""The pipelines follow the ring protocol on the GPU: every kernel runs with
the event trace on, and the trace is checked (slot and parity of every wait,
no slot refilled before its release, no stage consumed before it was issued,
the tensor-core accumulator ring likewise).  Outputs are checked too, so the
trace does not change results."""
import pytest
import torch

import oracle
from oracle import ring_sim
from mbarrier_gemm_pipelines_gb300 import inputs, trace
from gpu_helpers import (TOL, load_library, rel_frobenius, require_gpu, split_tail, to_host_f64,
                         tuned)
import trace_check as roles
from trace_check import check

pytestmark = pytest.mark.gpu

EVENT_KIND = {trace.WAIT_DONE: "wait", trace.ISSUED: "issued", trace.RELEASED: "released"}


def _tuples(recs):
    return [(int(r["t"]), EVENT_KIND[int(r["ev"])], int(r["item"]), int(r["slot"]),
             int(r["parity"])) for r in recs]


def replay_units(ev, S, cta_group=1, accumulator=False):
    """Replays every unit's recorded events through the ring simulator's
    mbarrier model (it raises at the first contradiction); returns the
    number of units replayed."""
    n = 0
    for u in sorted({cta // cta_group for cta, _ in ev}):
        lead = u * cta_group
        if (lead, roles.CONSUMER) not in ev:
            continue
        members = range(lead, lead + cta_group)
        prods = [_tuples(ev[(c, roles.PRODUCER)]) for c in members]
        cons = _tuples(ev[(lead, roles.CONSUMER)])
        mma = epis = None
        if accumulator:
            mma = _tuples(ev[(lead, roles.MMA_ACC)])
            epis = [_tuples(ev[(c, roles.EPILOGUE)]) for c in members]
        ring_sim.replay(prods, cons, S, mma_acc=mma, epilogues=epis)
        n += 1
    return n


@pytest.fixture(scope="module")
def gbr():
    require_gpu()
    return load_library()


@pytest.mark.parametrize("S,lag", [(1, 0), (2, 0), (2, 1), (4, 1), (7, 1)])
def test_copy_trace(gbr, S, lag):
    src = torch.randn(8192, 1024, device="cuda")           # 1024 tiles, ~7 per CTA
    gbr.copy_tuning(lag, 1)
    try:
        with trace.Recorder(cap=256) as rec:
            dst = gbr.staged_copy(src, tile=(128, 64), stages=S)
            ev, cnt = rec.events()
    finally:
        gbr.copy_tuning(-1, -1)
    gbr.check_device()
    assert torch.equal(dst, src)
    assert len(ev) >= 2 * 100
    errs = check(ev, cnt, S)
    assert errs == [], errs[:5]
    assert replay_units(ev, S) >= 100


@pytest.mark.parametrize("dtype", ["ffma", "ffma_cpasync"])
@pytest.mark.parametrize("S", [1, 2, 3, 4])
def test_ffma_trace(gbr, dtype, S):
    A, B, bias = inputs.gemm_normal(512, 512, 1024, seed=31)   # 16 tiles x 32 k-blocks
    with trace.Recorder(cap=256) as rec:
        C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype=dtype, stages=S)
        ev, cnt = rec.events()
    gbr.check_device()
    assert rel_frobenius(to_host_f64(C), oracle.gemm_bias_relu(A, B, bias)) <= TOL[dtype]
    errs = check(ev, cnt, S)
    assert errs == [], errs[:5]
    assert replay_units(ev, S) >= 16


def test_ffma_trace_keeps_one_launch(gbr):
    """With the split tail forced on, an FFMA call under the event trace still
    runs as one launch (a split call's second launch would overwrite the first
    one's trace): 256 tiles x 32 k-blocks, every ring item consumed once in
    the record."""
    A, B, bias = inputs.gemm_normal(2048, 2048, 1024, seed=32)
    with split_tail(gbr, 1):
        with trace.Recorder(cap=256) as rec:
            C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype="ffma", stages=3)
            ev, cnt = rec.events()
    gbr.check_device()
    assert rel_frobenius(to_host_f64(C), oracle.gemm_bias_relu(A, B, bias)) <= TOL["ffma"]
    assert check(ev, cnt, 3) == []
    released = sum(int((r["ev"] == trace.RELEASED).sum()) for (cta, role), r in ev.items()
                   if role == roles.CONSUMER)
    assert released == 256 * 32


@pytest.mark.parametrize("dtype,pair,ks,S,split", [
    ("bf16", 2, 2, 3, -1), ("bf16", 2, 1, 6, 0), ("bf16", 1, 1, 4, -1), ("bf16", 1, 2, 2, 1),
    ("tf32", 2, 2, 3, 1), ("tf32", 1, 1, 3, 0),
])
def test_umma_trace(gbr, dtype, pair, ks, S, split):
    # 2048 x 2048 x 1024: 64 tiles of 256 x 256 on 76 pairs, or 128 of
    # 128 x 256 on 152 CTAs; 8 to 16 k-blocks per tile, so the stage ring wraps
    # on every unit; split forced on, off, and auto.
    A, B, bias = inputs.gemm_normal(2048, 2048, 1024, seed=32)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    with tuned(gbr, pair, ks), split_tail(gbr, split):
        with trace.Recorder(cap=512) as rec:
            C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype=dtype, stages=S)
            ev, cnt = rec.events()
    gbr.check_device()
    ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    assert rel_frobenius(to_host_f64(C), ref) <= TOL[dtype]
    errs = check(ev, cnt, S, cta_group=pair, accumulator=True)
    assert errs == [], errs[:5]
    assert replay_units(ev, S, cta_group=pair, accumulator=True) >= 64 // pair


def test_umma_trace_many_tiles_per_unit(gbr):
    """4096 x 4096 x 512 on the pair: 256 tiles, 3-4 per unit, so the
    two-slot accumulator ring wraps."""
    A, B, bias = inputs.gemm_normal(4096, 4096, 512, seed=33)
    A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    with trace.Recorder(cap=512) as rec:
        C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype="bf16", stages=3)
        ev, cnt = rec.events()
    gbr.check_device()
    assert rel_frobenius(to_host_f64(C), oracle.gemm_bias_relu(A.float(), B.float(), bias)) <= TOL["bf16"]
    errs = check(ev, cnt, 3, cta_group=2, accumulator=True)
    assert errs == [], errs[:5]
    assert max(len(v) for (cta, role), v in ev.items() if role == 2) >= 6   # >= 3 tiles
    assert replay_units(ev, 3, cta_group=2, accumulator=True) == 76


@pytest.mark.parametrize("pair", [1, 2])
def test_grouped_trace(gbr, pair):
    counts = [300, 0, 513, 77]
    cnt_, X, W, b = inputs.grouped(tokens=sum(counts), experts=4, K=512, N=1032, seed=34)
    with tuned(gbr, pair), trace.Recorder(cap=512) as rec:
        C = gbr.gemm_bias_relu_grouped(X.cuda(), W.cuda(), b.cuda(), counts, stages=3)
        ev, cnt = rec.events()
    gbr.check_device()
    ref = oracle.gemm_bias_relu_grouped(X.float(), W.float(), b, counts)
    assert rel_frobenius(to_host_f64(C), ref) <= TOL["bf16"]
    errs = check(ev, cnt, 3, cta_group=pair, accumulator=True)
    assert errs == [], errs[:5]
    assert replay_units(ev, 3, cta_group=pair, accumulator=True) >= 1


@pytest.mark.parametrize("counts,pair", [([2048, 1024, 512, 256, 128, 64, 32, 32], 2),
                                         ([100, 64, 128, 1], 1)])
def test_grouped_auto_pair_choice(gbr, counts, pair):
    """The automatic choice between one CTA and the CTA pair: the pair as soon
    as an expert spans more than one 128-row tile (skewed experts included),
    one CTA when every expert fits one.  Seen in the trace: a pair launch runs
    its MMA lane on even CTAs only."""
    cnt_, X, W, b = inputs.grouped(tokens=sum(counts), experts=len(counts), K=256, N=520,
                                   seed=35)
    with trace.Recorder(cap=1024) as rec:
        C = gbr.gemm_bias_relu_grouped(X.cuda(), W.cuda(), b.cuda(), counts, stages=3)
        ev, cnt = rec.events()
    gbr.check_device()
    ref = oracle.gemm_bias_relu_grouped(X.float(), W.float(), b, counts)
    assert rel_frobenius(to_host_f64(C), ref) <= TOL["bf16"]
    mma_ctas = {cta for (cta, role) in ev if role == roles.CONSUMER}
    assert mma_ctas
    if pair == 2:
        assert all(c % 2 == 0 for c in mma_ctas)
    else:
        assert any(c % 2 == 1 for c in mma_ctas)


def test_trace_off_leaves_buffer_untouched(gbr):
    buf = torch.zeros(trace.bytes_for(1), dtype=torch.uint8, device="cuda")
    src = torch.randn(1024, 512, device="cuda")
    gbr.staged_copy(src, tile=(128, 64), stages=2)     # tracing is off
    gbr.check_device()
    assert int(buf.sum()) == 0
    from mbarrier_gemm_pipelines_gb300 import _binding as bb
    assert bb.lib().gbr_trace_buffer(buf.data_ptr(), 100) == bb.ERR_INVALID
    assert bb.lib().gbr_trace_buffer(buf.data_ptr() + 4, buf.numel() - 4) == bb.ERR_INVALID
