"""Plain reference of the decode-loop commit (TEST INFRASTRUCTURE ONLY).

Arc PR #217, "device decode loop", section "What this does" (step 3: the
commit scatters the token into the buffer the next forward reads, bumps the
device position and publishes the token into a pinned host ring) and section
"Fault detection replaces the sync rather than dropping it" (the commit
range-checks the token and the position before it writes anything and
latches a code into a sticky fault word); Arc PR #220 (a parked token must
never reach another sequence: records carry the row's owner).  The pages fix
no layout; the record here is (token, position before the commit, owner,
stamp = record index + 1), a refused row publishes token -1, and fault bits
are BAD_TOKEN = 1, BAD_POSITION = 2.
"""
from __future__ import annotations

import numpy as np

BAD_TOKEN = 0x1
BAD_POSITION = 0x2


def commit(tokens, V: int, next_ids, positions, max_position: int, owners, head: int, capacity: int, ring,
           fault: int = 0):
    """One commit of len(tokens) rows, row by row.  Returns the new (next_ids,
    positions, ring, head, fault); the inputs are not modified.  ring is a
    list of capacity records (token, position, owner, stamp)."""
    next_ids = list(next_ids)
    positions = list(positions)
    ring = list(ring)
    for r, tok in enumerate(tokens):
        tok = int(tok)
        pos = int(positions[r])
        bad = 0
        if not 0 <= tok < V:
            bad |= BAD_TOKEN
        if not 0 <= pos < max_position:
            bad |= BAD_POSITION
        if bad == 0:
            next_ids[r] = tok
            positions[r] = pos + 1
        fault |= bad
        idx = head + r
        owner = 0 if owners is None else int(owners[r])
        ring[idx % capacity] = (-1 if bad else tok, pos, owner, (idx + 1) % (1 << 32))
    return next_ids, positions, ring, head + len(tokens), fault


def empty_ring(capacity: int):
    return [(0, 0, 0, 0)] * capacity


def as_records(ring) -> np.ndarray:
    """The ring as the library lays it out in memory: each record as three
    8-byte words (token, stamp), (position, stamp), (owner, stamp)."""
    dt = np.dtype([("token", "<i4"), ("stamp", "<u4"), ("position", "<i4"), ("stamp_pos", "<u4"),
                   ("owner", "<u4"), ("stamp_owner", "<u4")])
    return np.array([(t, st, p, st, o, st) for (t, p, o, st) in ring], dtype=dt)
