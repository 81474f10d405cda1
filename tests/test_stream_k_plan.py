"""The stream-K work plan's arithmetic, checked by enumeration on the host.

The tensor-core attention lays the (row tile, 64-key tile) units out in a
virtual sequence, row tiles in lane-major order r = tile index * B +
request, with a gap of `gap` units (0, or 6 for the boundary-aware plan)
before every non-empty row tile but the first: row tile r starts at vS_r =
S_r + gap * (non-empty tiles before r).  CTA pair c takes the virtual range
[cW, (c+1)W), so with a gap a pair whose range crosses into another row tile
takes fewer key tiles.  A row tile is cut where a multiple of W falls inside
(vS_r, vS_r + u_r); the plan kernel gives the pieces of row tile r the
partial slots base_r + (x / W - vS_r / W), for a piece starting at virtual
position x, with base_r the exclusive scan of the per-tile piece counts
1 + (ceil((vS_r + u_r) / W) - 1 - floor(vS_r / W)); the combine kernels use
the same count.  The host sizes the workspace for R + pairs + 1 slots and
bounds the pieces of a row tile by 64 (W >= ceil(u_cap / 62)).  These tests
walk every pair's range unit by unit and check all of that on random ragged
batches, with and without the gap.
"""

import math

import numpy as np
import pytest

GAP = 6          # kSkBoundary


def host_gap(R, pairs, u_cap, paged=False):
    """The host's choice: the boundary-aware plan when the cache capacity is
    under 128 key tiles per pair, or for a paged batch with more row tiles
    than pairs; the plain plan otherwise."""
    return GAP if (R * u_cap < 128 * pairs or (paged and R > pairs)) else 0


def plan(u_per_tile, pairs, wmin, wforce=0, gap=GAP):
    u = np.asarray(u_per_tile, dtype=np.int64)
    S = np.concatenate([[0], np.cumsum(u)[:-1]]).astype(np.int64)
    ne_before = np.concatenate([[0], np.cumsum(u > 0)[:-1]]).astype(np.int64)
    vS = S + gap * ne_before
    n_ne = int((u > 0).sum())
    V = int(u.sum()) + gap * max(n_ne - 1, 0)
    W = max(wforce, wmin) if wforce else max(-(-V // pairs), wmin)
    W = max(W, 1)
    count = np.where(u > 0, 1 + (-(-(vS + u) // W) - 1 - vS // W), 0)
    base = np.concatenate([[0], np.cumsum(count)[:-1]]).astype(np.int64)
    return dict(u=u, vS=vS, V=V, W=W, count=count, base=base, ne=ne_before, gap=gap)


def pieces(p, pairs):
    """Every piece as (pair, row tile, first key tile, end key tile, virtual
    start), by walking each pair's virtual range position by position."""
    u, vS, V, W = p["u"], p["vS"], p["V"], p["W"]
    owner = {}                                 # virtual position -> (row tile, key tile)
    for r in range(len(u)):
        for k in range(int(u[r])):
            owner[int(vS[r]) + k] = (r, k)
    out = []
    for c in range(pairs):
        cur = None
        for x in range(c * W, min((c + 1) * W, V)):
            if x not in owner:
                cur = None                     # a gap ends the piece
                continue
            r, k = owner[x]
            if cur is not None and cur[1] == r:
                cur[3] = k + 1
            else:
                cur = [c, r, k, k + 1, x]
                out.append(cur)
    return [tuple(x) for x in out]


def records(p, pairs):
    """The plan kernel's per-pair records: the row tile whose range, with the
    gap before it, holds cW (R when the pair's range holds no unit), and the
    pair's count of key tiles."""
    u, vS, W, gap = p["u"], p["vS"], p["W"], p["gap"]
    R = len(u)
    first = np.full(pairs, R, dtype=np.int64)
    tiles = np.zeros(pairs, dtype=np.int64)
    for r in range(R):
        if u[r] == 0:
            continue
        claim = vS[r] - gap if p["ne"][r] > 0 else 0
        for c in range(-(-int(claim) // W), min(-(-int(vS[r] + u[r]) // W), pairs)):
            first[c] = r if vS[r] < (c + 1) * W else R
        for c in range(int(vS[r]) // W, min(-(-int(vS[r] + u[r]) // W), pairs)):
            tiles[c] += min((c + 1) * W, vS[r] + u[r]) - max(c * W, vS[r])
    return first, tiles


def random_batch(rng):
    B = int(rng.integers(1, 40))
    rt_count = int(rng.integers(1, 9))
    pairs = int(rng.integers(1, 80))
    t_cap = int(rng.integers(64, 12000))
    u_cap = -(-t_cap // 64)
    wmin = max(1, -(-u_cap // 62))
    u_req = rng.integers(0, u_cap + 1, size=B)
    u_req[rng.random(B) < 0.1] = 0                    # invalid requests hold no units
    u = np.tile(u_req, rt_count).astype(np.int64)   # lane-major: r = rt * B + b
    return u, u_cap, pairs, wmin


@pytest.mark.parametrize("gap", [0, GAP])
@pytest.mark.parametrize("seed", range(10))
def test_slots_are_distinct_bounded_and_counted(seed, gap):
    rng = np.random.default_rng(seed)
    u, u_cap, pairs, wmin = random_batch(rng)
    R = len(u)
    wforce = int(rng.integers(1, 40)) if seed % 3 == 0 else 0
    if wforce:   # the host launches enough pairs for a forced W
        v_cap = R * u_cap + gap * (R - 1)
        pairs = max(pairs, -(-v_cap // max(wforce, wmin)))
    p = plan(u, pairs, wmin, wforce, gap)
    W, vS = p["W"], p["vS"]
    ps = pieces(p, pairs)
    # the pieces tile every unit once
    assert sum(e - k for _, _, k, e, _ in ps) == int(u.sum())
    seen = set()
    for _, r, k, e, _ in ps:
        for t in range(k, e):
            assert (r, t) not in seen
            seen.add((r, t))
    slots, per_tile = [], {}
    for c, r, k, e, x in ps:
        slot = int(p["base"][r] + (x // W - vS[r] // W))
        slots.append(slot)
        per_tile.setdefault(r, []).append(slot)
        # a piece starts at its row tile's first key tile or at a multiple of W
        assert k == 0 or x % W == 0
    assert len(set(slots)) == len(slots)
    assert 0 <= min(slots) and max(slots) < R + pairs + 1
    for r, sl in per_tile.items():
        assert sorted(sl) == list(range(int(p["base"][r]), int(p["base"][r]) + int(p["count"][r])))
        assert p["count"][r] <= 64
    # the records name each pair's first piece and its key tiles
    first, tiles = records(p, pairs)
    for c in range(pairs):
        mine = [q for q in ps if q[0] == c]
        assert tiles[c] == sum(e - k for _, _, k, e, _ in mine)
        assert first[c] == (mine[0][1] if mine else R)
        if gap == 0:   # without gaps a pair's key tiles are its whole range
            assert tiles[c] == max(0, min((c + 1) * W, p["V"]) - min(c * W, p["V"]))


@pytest.mark.parametrize("gap", [0, GAP])
@pytest.mark.parametrize("seed", range(10))
def test_pieces_from_records(seed, gap):
    """The attention kernel walks a pair's pieces from its record {r, vS_r,
    u_r, base_r} alone: the first piece is key tiles [max(cW, vS_r) - vS_r,
    min((c+1)W, vS_r + u_r) - vS_r) in slot base_r + (max(cW, vS_r) / W -
    vS_r / W); each next one starts at the next non-empty row tile, unless the
    range ends inside the current tile or in the gap before the next.  That
    equals the unit-by-unit walk, slots included.  Without gaps max(cW, vS_r)
    = cW, the plain plan's formula."""
    rng = np.random.default_rng(100 + seed)
    u, u_cap, pairs, wmin = random_batch(rng)
    p = plan(u, pairs, wmin, gap=gap)
    W, vS, V, base = p["W"], p["vS"], p["V"], p["base"]
    R = len(u)
    ps = pieces(p, pairs)
    first, _ = records(p, pairs)
    for c in range(pairs):
        beg, end = min(c * W, V), min(min(c * W, V) + W, V)
        mine = [(q, int(base[q[1]] + (q[4] // W - vS[q[1]] // W))) for q in ps if q[0] == c]
        got = []
        r = int(first[c])
        x = beg
        while r < R and x < end:
            x0 = max(x, int(vS[r]))
            if gap == 0 and not got:
                assert x0 == x
            if vS[r] >= end or x0 >= vS[r] + u[r]:
                break
            k0, k1 = x0 - int(vS[r]), min(end, int(vS[r] + u[r])) - int(vS[r])
            got.append(((c, r, k0, k1, x0), int(base[r] + (x0 // W - vS[r] // W))))
            x = int(vS[r]) + k1
            if x >= end:
                break
            r += 1
            while r < R and u[r] == 0:
                r += 1
        assert got == mine


@pytest.mark.parametrize("gap", [0, GAP])
def test_single_request_kimi_shape(gap):
    """kimi_single: 32 row tiles of 65 units over 76 pairs.  Without gaps W =
    28 and pairs 0..74 hold work; with them the sequence is 2080 + 6 * 31 =
    2266 units, W = 30, and a pair that crosses a row-tile boundary takes at
    most 24 key tiles, one that does not 30."""
    u = np.full(32, 65, dtype=np.int64)
    p = plan(u, 76, wmin=math.ceil(65 / 62), gap=gap)
    ps = pieces(p, 76)
    per_pair = {}
    for c, r, k, e, _ in ps:
        per_pair.setdefault(c, []).append(e - k)
    if gap == 0:
        assert (p["V"], p["W"]) == (2080, 28)
        assert max(per_pair) == 74
    else:
        assert (p["V"], p["W"]) == (2266, 30)
        crossing = [sum(v) for v in per_pair.values() if len(v) > 1]
        single = [sum(v) for v in per_pair.values() if len(v) == 1]
        assert crossing and max(crossing) <= 30 - GAP
        assert max(single) == 30


def test_host_gap_choice():
    """The workloads' plans: kimi_single (32 row tiles of 65 units, 27 per
    pair) and paged (256 row tiles over 76 pairs) take the boundary-aware
    plan; long (64 row tiles of 1026 units) and batched (128 row tiles of at
    most 129 units, a contiguous cache) keep the plain one."""
    assert host_gap(32, 76, -(-(4096 + 64) // 64)) == GAP
    assert host_gap(256, 76, 513, paged=True) == GAP
    assert host_gap(64, 76, -(-(65536 + 128) // 64)) == 0
    assert host_gap(128, 76, -(-(8192 + 32) // 64)) == 0
    assert host_gap(64, 76, 1026, paged=True) == 0
