"""Event trace of the ring protocol (``gbr_trace_buffer`` in include/gbr.h).

Usage::

    with trace.Recorder() as rec:           # allocates a device buffer, turns tracing on
        gbr.staged_copy(src, dst, tile=(128, 64), stages=4)
        torch.cuda.synchronize()
    events = rec.events()                    # {(cta, role): numpy record array}

Each record holds the %globaltimer time (ns), the ring item, the event, the
slot and the parity the wait used.  Decoding is all this module does; it
computes nothing of the operators.
"""
from __future__ import annotations

import numpy as np

MAX_CTAS = 512
ROLES = 4
HEADER_BYTES = MAX_CTAS * ROLES * 4
REGION_BYTES = MAX_CTAS * ROLES * 16

ROLE_NAMES = {0: "producer", 1: "consumer", 2: "epilogue", 3: "mma_acc"}
EVENT_NAMES = {0: "wait_done", 1: "issued", 2: "released"}
WAIT_DONE, ISSUED, RELEASED = 0, 1, 2

RECORD = np.dtype([("t", "<u8"), ("item", "<u4"), ("role", "u1"), ("ev", "u1"), ("slot", "u1"),
                   ("parity", "u1")])


def bytes_for(cap: int) -> int:
    """Buffer size that holds `cap` records per (CTA, role)."""
    return HEADER_BYTES + REGION_BYTES * int(cap)


def decode(raw: np.ndarray) -> tuple[dict, dict]:
    """raw: the whole trace buffer as uint8.  Returns ({(cta, role): records},
    {(cta, role): events counted}); a role with more events than the region
    holds keeps its first `cap` records."""
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    cap = (raw.size - HEADER_BYTES) // REGION_BYTES
    counts = raw[:HEADER_BYTES].view("<u4").reshape(MAX_CTAS, ROLES)
    recs = raw[HEADER_BYTES:HEADER_BYTES + REGION_BYTES * cap].view(RECORD)
    recs = recs.reshape(MAX_CTAS, ROLES, cap)
    events, counted = {}, {}
    for cta, role in zip(*np.nonzero(counts)):
        n = int(counts[cta, role])
        counted[(int(cta), int(role))] = n
        events[(int(cta), int(role))] = recs[cta, role, :min(n, cap)].copy()
    return events, counted


class Recorder:
    """Turns tracing on for the with-block, into a zeroed device buffer."""

    def __init__(self, cap: int = 4096, device=None):
        self.cap = int(cap)
        self.device = device
        self.buf = None

    def __enter__(self):
        import torch
        from . import _binding
        self.buf = torch.zeros(bytes_for(self.cap), dtype=torch.uint8,
                               device=self.device or "cuda")
        _binding.check(_binding.lib().gbr_trace_buffer(self.buf.data_ptr(), self.buf.numel()))
        return self

    def __exit__(self, *exc):
        from . import _binding
        _binding.lib().gbr_trace_buffer(None, 0)
        return False

    def events(self):
        import torch
        torch.cuda.synchronize()
        return decode(self.buf.cpu().numpy())
