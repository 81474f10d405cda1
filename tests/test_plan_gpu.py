"""The device-built stream-K plan and ancestor masks, bit for bit.

After a tensor-core call the workspace holds what `sk_plan_kernel` wrote:
* the plan table: the header {V, W, pairs, R}; {vS_r, u_r, base_r} per row
  tile (row tiles lane-major, r = tile index * B + request; vS_r the tile's
  start in the virtual sequence, which has a gap of 6 units before every
  non-empty row tile but the first when the host chose the boundary-aware
  plan, none otherwise); the row tile of each pair's first piece; one 8-int
  record per pair {r, vS_r, u_r, base_r, L_b, key tiles};
* the ancestor masks [B, N, 4] u32 (bit j of node i's mask set iff j lies on
  i's root path, i included).

Both are integer results with one correct value, so they are compared exactly
with a host model written from the same definitions (the enumeration in
tests/test_stream_k_plan.py checks that model against a walk of every pair's
range): units per row tile ceil((L_b + N) / 64) (0 for an invalid prefix),
the host's choice of gap, W = max(ceil(V / pairs), ceil(u_cap / 62)), base_r
the exclusive scan of the tiles' piece counts, and the root paths of
parent[].  The plan and the masks are the last two workspace regions of a
bf16 tensor-core call, each 256-byte aligned.  The cases cover both plans:
"long_plain" (one request, 64 row tiles of 1026 units), "paged_plain" (a
paged batch of 64 row tiles, capacity 175 units each) and "batched" take the
plain plan, the others the boundary-aware one; "many_tiles" (72 requests,
1152 row tiles) runs the plan kernel's scans over several 256-tile rounds.
"""

import numpy as np
import pytest
import torch

from speculative_decoding_tree_mla_gb300 import kdtv, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_mla_gb300 import build
    build.build()


def a256(x):
    return (x + 255) // 256 * 256


def host_plan(wl, pairs):
    from tests.test_stream_k_plan import host_gap, plan, records
    s = wl.spec
    B, N, H = s.B, s.N, s.H
    rt = -(-(N * H) // 128)
    R = B * rt
    t_cap = wl.max_pages * 64 if wl.page_size else wl.t_stride
    L = np.asarray(wl.f32["prefix_len"], dtype=np.int64)
    ok = (L >= 0) & (L + N <= t_cap)
    u_req = np.where(ok, -(-(L + N) // 64), 0)
    u = np.tile(u_req, rt)                      # r = tile index * B + request
    u_cap = -(-t_cap // 64)
    wmin = max(1, -(-u_cap // 62))
    p = plan(u, pairs, wmin, gap=host_gap(R, pairs, u_cap, paged=bool(wl.page_size)))
    first, tiles = records(p, pairs)
    rec = np.zeros((pairs, 8), dtype=np.int64)
    for c in range(pairs):
        r = int(first[c])
        rec[c, 0] = r
        if r < R:
            rec[c, 1:4] = p["vS"][r], u[r], p["base"][r]
            rec[c, 4] = L[r % B]
        rec[c, 5] = tiles[c]
    return dict(V=p["V"], W=p["W"], R=R, vS=p["vS"], u=u, base=p["base"], first=first, rec=rec)


def host_masks(parent):
    B, N = parent.shape
    m = np.zeros((B, N, 4), dtype=np.uint32)
    for b in range(B):
        for i in range(N):
            j = i
            while True:
                m[b, i, j >> 5] |= np.uint32(1 << (j & 31))
                if j == 0:
                    break
                j = int(parent[b, j])
    return m


CASES = {
    "ragged": lambda: W.make(W.small_spec("plan_r", B=3, N=16, prefix=("uniform", 30, 1500))),
    "paged": lambda: W.make(W.small_spec("plan_p", B=5, N=8, paged=True,
                                         prefix=("loguniform", 40, 900))),
    "batched": lambda: W.make("batched"),
    "kimi_single": lambda: W.make("kimi_single"),
    "long_plain": lambda: W.make(W.small_spec("plan_l", B=1, N=128, prefix=("fixed", 65536))),
    "paged_plain": lambda: W.make(W.small_spec("plan_pp", B=2, N=64, paged=True,
                                               prefix=("uniform", 9000, 12000))),
    # 72 requests x 16 row tiles = 1152 row tiles: five rounds of the scans
    "many_tiles": lambda: W.make(W.small_spec("plan_m", B=72, N=32, prefix=("uniform", 64, 256))),
}


@pytest.mark.parametrize("case", list(CASES) + ["bad_prefix"])
def test_device_plan_and_masks_match_host_model(case):
    wl = CASES["ragged"]() if case == "bad_prefix" else CASES[case]()
    if case == "bad_prefix":
        wl.t["prefix_len"][1] = wl.t_stride      # request 1 holds no units
        wl.f32["prefix_len"] = wl.t["prefix_len"].numpy().astype(np.int64)
    op = kdtv.for_workload(wl, "cuda")
    if kdtv.workspace_size(op.dims) == 0:
        pytest.skip("tensor-core path not compiled in")
    op.workspace.zero_()
    op()
    st = op.status()
    assert kdtv.STATUS[st] == ("KDTV_ERR_BAD_PREFIX" if case == "bad_prefix" else "KDTV_OK")
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    hp = host_plan(wl, pairs)
    B, N, R = wl.spec.B, wl.spec.N, hp["R"]
    ws = op.workspace.cpu().numpy()
    sk_ints = 4 + 3 * R + pairs + 3 + 8 * pairs
    off_anc = ws.size - a256(B * N * 16)
    off_sk = off_anc - a256(sk_ints * 4)
    sk = ws[off_sk: off_sk + sk_ints * 4].view(np.int32).astype(np.int64)
    assert sk[:4].tolist() == [hp["V"], hp["W"], pairs, R]
    e = sk[4: 4 + 3 * R].reshape(R, 3)
    assert np.array_equal(e[:, 0], hp["vS"]) and np.array_equal(e[:, 1], hp["u"])
    assert np.array_equal(e[:, 2], hp["base"])
    assert np.array_equal(sk[4 + 3 * R: 4 + 3 * R + pairs], hp["first"])
    rec_off = (4 + 3 * R + pairs + 3) & ~3
    rec = sk[rec_off: rec_off + 8 * pairs].reshape(pairs, 8)
    assert np.array_equal(rec, hp["rec"])
    anc = ws[off_anc: off_anc + B * N * 16].view(np.uint32).reshape(B, N, 4)
    assert np.array_equal(anc, host_masks(wl.f32["parent"]))
