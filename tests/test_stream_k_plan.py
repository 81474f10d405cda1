"""The stream-K work plan's arithmetic, checked by enumeration on the host.

The tensor-core attention splits the sequence of (row tile, 64-key tile)
units, row tiles in lane-major order r = tile index * B + request, into
CTA-pair ranges [cW, (c+1)W) and cuts each range into pieces
at row-tile boundaries.  The plan kernel and the combine kernels give the
pieces of row tile r the partial slots base_r + (x / W - S_r / W), for a piece
starting at unit x, with base_r = r + floor(S_r / W) and a count per row tile
of 1 + (ceil((S_r + u_r) / W) - 1 - floor(S_r / W)).  The host sizes the
workspace for R + pairs + 1 slots and bounds the pieces of a row tile by 64
(W >= ceil(u_cap / 62)).  These tests enumerate the pieces directly and check
all of that on random ragged batches.
"""

import math

import numpy as np
import pytest


def plan(u_per_tile, pairs, wmin, wforce=0):
    S = np.concatenate([[0], np.cumsum(u_per_tile)[:-1]]).astype(np.int64)
    U = int(np.sum(u_per_tile))
    if wforce:
        W = max(wforce, wmin)
    else:
        W = max(-(-U // pairs), wmin)
    W = max(W, 1)
    base = np.arange(len(u_per_tile)) + S // W
    return S, U, W, base


def pieces(u_per_tile, S, U, W, pairs):
    """Every piece as (pair, row tile, first unit, end unit), by walking the ranges."""
    out = []
    for c in range(pairs):
        beg, end = c * W, min((c + 1) * W, U)
        x = beg
        while x < end:
            r = int(np.searchsorted(S, x, side="right") - 1)
            while u_per_tile[r] == 0 or S[r] + u_per_tile[r] <= x:
                r += 1
            stop = min(end, S[r] + u_per_tile[r])
            out.append((c, r, x, stop))
            x = stop
    return out


@pytest.mark.parametrize("seed", range(12))
def test_slots_are_distinct_bounded_and_counted(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    rt_count = int(rng.integers(1, 9))
    pairs = int(rng.integers(1, 80))
    t_cap = int(rng.integers(64, 20000))
    u_cap = -(-t_cap // 64)
    wmin = max(1, -(-u_cap // 62))
    u_req = rng.integers(0, u_cap + 1, size=B)
    u_req[rng.random(B) < 0.1] = 0                      # invalid requests hold no units
    u = np.tile(u_req, rt_count).astype(np.int64)     # lane-major: r = rt * B + b
    wforce = int(rng.integers(1, 40)) if seed % 3 == 0 else 0
    if wforce:   # the host launches enough pairs for a forced W
        pairs = max(pairs, -(-len(u) * u_cap // max(wforce, wmin)))
    S, U, W, base = plan(u, pairs, wmin, wforce)
    R = len(u)
    ps = pieces(u, S, U, W, pairs)
    # the pieces tile the whole unit sequence once
    assert sum(e - x for _, _, x, e in ps) == U
    slots = []
    per_tile = {}
    for c, r, x, e in ps:
        slot = int(base[r] + (x // W - S[r] // W))
        slots.append(slot)
        per_tile.setdefault(r, []).append(slot)
        # a piece starts at its row tile's first unit or at a multiple of W
        assert x == S[r] or x % W == 0
    assert len(set(slots)) == len(slots)
    assert 0 <= min(slots) and max(slots) < R + pairs + 1
    for r, sl in per_tile.items():
        count = 1 + (-(-(int(S[r]) + int(u[r])) // W) - 1 - int(S[r]) // W)
        assert sorted(sl) == list(range(int(base[r]), int(base[r]) + count))
        assert count <= 64
    # every pair's first unit lies in one non-empty row tile
    for c in range(pairs):
        if c * W < U:
            r = [r for r in range(R) if u[r] and S[r] <= c * W < S[r] + u[r]]
            assert len(r) == 1


def test_single_request_kimi_shape():
    """kimi_single: 32 row tiles of 65 units over 76 pairs: W = 28."""
    u = np.full(32, 65, dtype=np.int64)
    S, U, W, base = plan(u, 76, wmin=math.ceil(65 / 62))
    assert (U, W) == (2080, 28)
    ps = pieces(u, S, U, W, 76)
    assert max(c for c, *_ in ps) == 74                  # pairs 0..74 hold work
    assert sum(1 for *_, x, e in ps) == 32 + sum(1 for r in range(32)
                                                 for m in range(1, 200)
                                                 if S[r] < m * W < S[r] + 65)


def first_piece_from_record(rec, beg, end, W):
    """A pair's first piece as the attention kernel derives it from the pair's
    plan record {r, S_r, u_r, base_r} alone: (r, first unit, end unit, slot)."""
    r, S_r, u_r, base_r = rec
    return r, beg, min(end, S_r + u_r), base_r + (beg // W - S_r // W)


@pytest.mark.parametrize("seed", range(12))
def test_first_piece_records_match_enumeration(seed):
    """The per-pair plan record (the row tile holding unit cW with that tile's
    S, u and base) gives the same first piece and slot as walking the pair's
    range, for every pair with work; pairs without work have no record."""
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 30))
    rt_count = int(rng.integers(1, 9))
    pairs = int(rng.integers(1, 80))
    u_cap = int(rng.integers(1, 300))
    wmin = max(1, -(-u_cap // 62))
    u_req = rng.integers(0, u_cap + 1, size=B)
    u_req[rng.random(B) < 0.15] = 0
    u = np.tile(u_req, rt_count).astype(np.int64)
    S, U, W, base = plan(u, pairs, wmin)
    R = len(u)
    # the plan kernel's records: first[c] = the row tile holding unit cW
    first = [R] * pairs
    for r in range(R):
        c_beg, c_end = -(-int(S[r]) // W), -(-(int(S[r]) + int(u[r])) // W)
        for c in range(c_beg, min(c_end, pairs)):
            first[c] = r
    ps = pieces(u, S, U, W, pairs)
    for c in range(pairs):
        beg, end = c * W, min((c + 1) * W, U)
        mine = [p for p in ps if p[0] == c]
        if beg >= end:
            assert not mine
            continue
        r = first[c]
        assert r < R
        got = first_piece_from_record((r, int(S[r]), int(u[r]), int(base[r])), beg, end, W)
        _, r0, x0, e0 = mine[0]
        assert got == (r0, x0, e0, int(base[r0] + (x0 // W - S[r0] // W)))
