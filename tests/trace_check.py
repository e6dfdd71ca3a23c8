"""Checks a decoded pipeline event trace against the ring protocol.

The protocol (slot = i mod S; a wait on "full" for item i uses parity
(i / S) & 1, a wait on "empty" uses ((i / S) & 1) ^ 1; a slot is refilled only
after its previous occupant was released; a consumer sees a stage only after
its producer issued it) is restated here from the pages, independently of both
the kernels and the oracle.  Times are %globaltimer values recorded by the
kernels: "issued" and "released" before the operation they announce, "wait
done" after the wait returned, so every ordering below must hold with <=.
"""
from collections import defaultdict

WAIT_DONE, ISSUED, RELEASED = 0, 1, 2
PRODUCER, CONSUMER, EPILOGUE, MMA_ACC = 0, 1, 2, 3


def _split(recs):
    waits, issued, released = [], {}, {}
    for r in recs:
        ev, item, t = int(r["ev"]), int(r["item"]), int(r["t"])
        if ev == WAIT_DONE:
            waits.append((item, int(r["slot"]), int(r["parity"]), t))
        elif ev == ISSUED:
            issued[item] = (int(r["slot"]), t)
        elif ev == RELEASED:
            if item in released:
                released[item] = None          # released twice: flagged below
            else:
                released[item] = (int(r["slot"]), t)
    return waits, issued, released


def _ring(errors, tag, S, producers, consumer):
    """producers: list of record arrays (one per CTA of the unit); consumer: the
    unit's consumer records."""
    cw, _, crel = _split(consumer)
    for i, (item, slot, par, _) in enumerate(cw):
        if item != i:
            errors.append("%s: consumer wait %d is for item %d" % (tag, i, item))
            return
        if slot != i % S or par != (i // S) & 1:
            errors.append("%s: consumer item %d used slot %d parity %d" % (tag, i, slot, par))
    for item, v in crel.items():
        if v is None:
            errors.append("%s: item %d released twice" % (tag, item))
        elif v[0] != item % S:
            errors.append("%s: item %d released slot %d" % (tag, item, v[0]))
    full_t = {item: t for item, _, _, t in cw}
    for p, recs in enumerate(producers):
        pw, piss, _ = _split(recs)
        if len(pw) != len(cw):
            errors.append("%s: producer %d waited %d times, consumer %d" % (tag, p, len(pw), len(cw)))
        for i, (item, slot, par, t) in enumerate(pw):
            if item != i:
                errors.append("%s: producer %d wait %d is for item %d" % (tag, p, i, item))
                return
            if slot != i % S or par != ((i // S) & 1) ^ 1:
                errors.append("%s: producer %d item %d used slot %d parity %d" % (tag, p, i, slot, par))
            if i >= S:
                prev = crel.get(i - S)
                if prev is None:
                    errors.append("%s: slot %d refilled for item %d before item %d was released"
                                  % (tag, i % S, i, i - S))
                elif prev[1] > t:
                    errors.append("%s: producer %d refilled slot %d for item %d at %d, before the "
                                  "release of item %d at %d" % (tag, p, i % S, i, t, i - S, prev[1]))
            if item not in piss:
                errors.append("%s: producer %d never issued item %d" % (tag, p, item))
            elif item in full_t and piss[item][1] > full_t[item]:
                errors.append("%s: consumer saw item %d full before producer %d issued it"
                              % (tag, item, p))


def _acc_ring(errors, tag, mma_acc, epilogues):
    aw, aiss, _ = _split(mma_acc)
    for j, (tl, slot, par, _) in enumerate(aw):
        if tl != j or slot != j & 1 or par != ((j >> 1) & 1) ^ 1:
            errors.append("%s: accumulator empty wait %d: item %d slot %d parity %d"
                          % (tag, j, tl, slot, par))
    acc_empty_t = {tl: t for tl, _, _, t in aw}
    for e, recs in enumerate(epilogues):
        ew, _, erel = _split(recs)
        if len(ew) != len(aw):
            errors.append("%s: epilogue %d saw %d accumulators, MMA lane filled %d"
                          % (tag, e, len(ew), len(aw)))
        for j, (tl, slot, par, t) in enumerate(ew):
            if tl != j or slot != j & 1 or par != (j >> 1) & 1:
                errors.append("%s: epilogue %d full wait %d: item %d slot %d parity %d"
                              % (tag, e, j, tl, slot, par))
            if tl in aiss and aiss[tl][1] > t:
                errors.append("%s: epilogue %d saw accumulator %d before its commit" % (tag, e, tl))
            rel = erel.get(tl)
            if rel is None:
                errors.append("%s: epilogue %d never released accumulator %d" % (tag, e, tl))
            elif tl + 2 in acc_empty_t and rel[1] > acc_empty_t[tl + 2]:
                errors.append("%s: accumulator %d reused before epilogue %d released it"
                              % (tag, tl & 1, e))


def check(events, counted, S, cta_group=1, accumulator=False):
    """events/counted: as returned by trace.decode.  cta_group: CTAs per unit
    (2 for the CTA-pair tensor-core kernel: both CTAs produce, the even one
    consumes).  accumulator: also check the tensor-core accumulator ring.
    Returns a list of violations (empty: the trace follows the protocol)."""
    errors = []
    for key, n in counted.items():
        if key in events and len(events[key]) < n:
            errors.append("CTA %d role %d: %d events, only %d recorded (enlarge the buffer)"
                          % (key[0], key[1], n, len(events[key])))
    ctas = sorted({cta for cta, _ in events})
    units = defaultdict(list)
    for cta in ctas:
        units[cta // cta_group].append(cta)
    for u, members in units.items():
        lead = u * cta_group
        tag = "unit %d" % u
        consumer = events.get((lead, CONSUMER))
        producers = [events[(c, PRODUCER)] for c in range(lead, lead + cta_group)
                     if (c, PRODUCER) in events]
        if consumer is None and not producers:
            continue
        if consumer is None or len(producers) != cta_group:
            errors.append("%s: missing producer or consumer events" % tag)
            continue
        _ring(errors, tag, S, producers, consumer)
        if accumulator:
            epis = [events[(c, EPILOGUE)] for c in range(lead, lead + cta_group)
                    if (c, EPILOGUE) in events]
            if (lead, MMA_ACC) not in events or len(epis) != cta_group:
                errors.append("%s: missing accumulator-ring events" % tag)
                continue
            _acc_ring(errors, tag, events[(lead, MMA_ACC)], epis)
    return errors
