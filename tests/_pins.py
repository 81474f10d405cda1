"""Independent checks that pin the fp64 oracle to what the pages and the
mathematics fix.  Each pin returns the largest deviation it saw; the tests
assert it is tiny, and the mutation test asserts that a planted mistake in
the oracle makes at least one pin fail.

None of these checks re-types the oracle's formulas: they go through a
library routine on the decompressed (non-absorbed) MLA form, a transitive
closure of the parent relation instead of a parent walk, pure-Python loops,
or a closed form.
"""

from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from speculative_decoding_tree_mla_gb300 import workloads as W

TOL = 1e-11


def tiny_inputs(parent=None, L=32, N=16, B=1, seed=None, paged=False, zero_q=False):
    spec = W.SPECS["tiny"]
    if B != spec.B or N != spec.N or paged:
        spec = W.Spec("tiny_var", 50, B=B, N=N, H=4, d_nope=32, d_rope=16, d_v=32,
                      d_c=64, dtype="f32", prefix=("fixed", L),
                      tree=("window", None, 8), paged=paged, vocab=512)
    if parent is not None:
        parent = np.broadcast_to(np.asarray(parent, np.int32), (B, N))
    wl = W.make(spec, parent=parent, prefix_len=np.full(B, L), seed=seed,
                zero_q=zero_q)
    return wl


def oracle_out(wl, nodes=None):
    f = wl.f32
    return oracle.verify_attn(f["q_nope"], f["q_rope"], f["W_UK"], f["W_UV"],
                              f["c_kv"], f["k_rope"], f["parent"],
                              f["prefix_len"], wl.spec.scale,
                              page_table=f.get("page_table"),
                              page_size=wl.page_size, nodes=nodes)


def closure_mask(parent_b):
    """Tree part of the visibility mask by transitive closure of the
    parent relation: R = I + A + A^2 + ... with A[i, parent[i]] = 1."""
    N = len(parent_b)
    A = np.zeros((N, N), dtype=np.int64)
    for i, p in enumerate(parent_b):
        if p >= 0:
            A[i, p] = 1
    reach = np.eye(N, dtype=bool)
    cur = np.eye(N, dtype=np.int64)
    for _ in range(N):
        cur = (cur @ A > 0).astype(np.int64)
        reach |= cur.astype(bool)
    return reach


def decompressed_sdpa(q_nope, q_rope, W_UK, W_UV, ckv_seq, krope_seq, mask, scale):
    """Ordinary multi-head attention on explicitly decompressed keys/values,
    through torch's scaled_dot_product_attention in float64.

    q_nope [N,H,dn], q_rope [N,H,dr], ckv_seq [T,dc], krope_seq [T,dr],
    mask [N,T] bool (True = visible) -> [N,H,dv].
    """
    t = lambda x: torch.as_tensor(np.asarray(x, dtype=np.float64))
    q_nope, q_rope, W_UK, W_UV = t(q_nope), t(q_rope), t(W_UK), t(W_UV)
    ckv, krope = t(ckv_seq), t(krope_seq)
    H = q_nope.shape[1]
    k_nope = torch.einsum("hed,td->hte", W_UK, ckv)            # K = W_UK[h] c
    k = torch.cat([k_nope, krope.unsqueeze(0).expand(H, -1, -1)], dim=-1)
    v = torch.einsum("hvd,td->htv", W_UV, ckv)                 # V = W_UV[h] c
    q = torch.cat([q_nope, q_rope], dim=-1).permute(1, 0, 2)   # [H, N, D]
    o = F.scaled_dot_product_attention(q[None], k[None], v[None],
                                       attn_mask=torch.as_tensor(mask)[None, None],
                                       scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def request_sequence(wl, b):
    """The logical latent sequence of request b (prefix + tree rows)."""
    f = wl.f32
    T = int(f["prefix_len"][b]) + wl.spec.N
    if wl.page_size:
        ps = wl.page_size
        pt = f["page_table"][b]
        ckv = np.concatenate([f["c_kv"][pt[k]] for k in range(-(-T // ps))])[:T]
        kr = np.concatenate([f["k_rope"][pt[k]] for k in range(-(-T // ps))])[:T]
        return ckv, kr
    return f["c_kv"][b, :T], f["k_rope"][b, :T]


def pin_sdpa(wl, tree_mask_fn=closure_mask):
    """Max |oracle - decompressed SDPA| over every request and node."""
    f = wl.f32
    out = oracle_out(wl)
    err = 0.0
    for b in range(wl.spec.B):
        L = int(f["prefix_len"][b])
        N = wl.spec.N
        ckv, kr = request_sequence(wl, b)
        mask = np.zeros((N, L + N), dtype=bool)
        mask[:, :L] = True
        mask[:, L:] = tree_mask_fn(f["parent"][b])
        ref = decompressed_sdpa(f["q_nope"][b], f["q_rope"][b], f["W_UK"], f["W_UV"],
                                ckv, kr, mask, wl.spec.scale)
        err = max(err, float(np.abs(out[b] - ref).max()))
    return err


def pin_causal_chain(seed=None, L=32, N=16):
    """Chain tree == causal attention over L + N tokens (query rows L..L+N-1)."""
    wl = tiny_inputs(parent=W.chain_tree(N), L=L, N=N, seed=seed)
    causal = lambda parent_b: np.tril(np.ones((len(parent_b),) * 2, dtype=bool))
    return pin_sdpa(wl, tree_mask_fn=causal)


def brute_force(q_nope, q_rope, W_UK, W_UV, ckv, krope, parent, L, scale):
    """Pure-Python loops for one request; ancestors found by walking each
    node's subtree downwards from the root (children lists)."""
    N, H, dn = len(q_nope), len(q_nope[0]), len(q_nope[0][0])
    dc, dr, dv = len(ckv[0]), len(krope[0]), len(W_UV[0])
    children = {j: [] for j in range(N)}
    for i in range(1, N):
        children[int(parent[i])].append(i)
    sees = [[False] * N for _ in range(N)]           # sees[i][j]: j on i's root path

    def mark(j, node):
        sees[node][j] = True
        for c in children[node]:
            mark(j, c)
    for j in range(N):
        mark(j, j)
    out = [[[0.0] * dv for _ in range(H)] for _ in range(N)]
    for i in range(N):
        keys = list(range(L)) + [L + j for j in range(N) if sees[i][j]]
        for h in range(H):
            ql = [sum(q_nope[i][h][e] * W_UK[h][e][d] for e in range(dn)) for d in range(dc)]
            s = []
            for t in keys:
                acc = sum(ql[d] * ckv[t][d] for d in range(dc))
                acc += sum(q_rope[i][h][r] * krope[t][r] for r in range(dr))
                s.append(scale * acc)
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = sum(e)
            ol = [sum(e[k] / z * ckv[t][d] for k, t in enumerate(keys)) for d in range(dc)]
            for v in range(dv):
                out[i][h][v] = sum(W_UV[h][v][d] * ol[d] for d in range(dc))
    return out


def pin_brute_force(seed=7):
    """Oracle vs pure-Python loops on a very small random tree."""
    rng = np.random.default_rng(seed)
    N, H, dn, dr, dc, dv, L = 6, 2, 3, 2, 4, 3, 3
    parent = W.random_tree(rng, N, None, 4)
    q_nope = rng.standard_normal((1, N, H, dn))
    q_rope = rng.standard_normal((1, N, H, dr))
    W_UK = rng.standard_normal((H, dn, dc)) / 2
    W_UV = rng.standard_normal((H, dv, dc)) / 2
    ckv = rng.standard_normal((1, L + N, dc))
    kr = rng.standard_normal((1, L + N, dr))
    scale = 1 / math.sqrt(dn + dr)
    got = oracle.verify_attn(q_nope, q_rope, W_UK, W_UV, ckv, kr, parent[None],
                             np.array([L]), scale)[0]
    ref = np.array(brute_force(q_nope[0].tolist(), q_rope[0].tolist(), W_UK.tolist(),
                               W_UV.tolist(), ckv[0].tolist(), kr[0].tolist(),
                               parent.tolist(), L, scale))
    return float(np.abs(got - ref).max())


def pin_row_sums(wl):
    """Softmax rows are non-negative, sum to 1 and cover L + depth(i) keys."""
    f = wl.f32
    depth = W.tree_depths(f["parent"][0])
    err = 0.0
    for i in range(wl.spec.N):
        r = oracle.verify_attn_node(f["q_nope"], f["q_rope"], f["W_UK"], f["W_UV"],
                                    f["c_kv"], f["k_rope"], f["parent"],
                                    f["prefix_len"], 0, i, wl.spec.scale)
        if r["p"].shape[1] != int(f["prefix_len"][0]) + depth[i] or r["p"].min() < 0:
            return float("inf")
        err = max(err, float(np.abs(r["p"].sum(axis=1) - 1).max()))
    return err


def pin_identical_rows(seed=3):
    """All visible latent rows equal r  =>  o_lat = r and out = W_UV[h] r."""
    wl = tiny_inputs(seed=seed)
    f = wl.f32
    r = np.random.default_rng(seed).standard_normal(wl.spec.d_c)
    f["c_kv"] = np.broadcast_to(r, f["c_kv"].shape).copy()
    out = oracle_out(wl)
    ref = np.einsum("hvd,d->hv", f["W_UV"], r)
    return float(np.abs(out[0] - ref[None]).max())


def pin_zero_query(seed=4):
    """q = 0  =>  uniform weights, o_lat = mean of the visible rows."""
    wl = tiny_inputs(seed=seed, zero_q=True)
    f = wl.f32
    L, N = int(f["prefix_len"][0]), wl.spec.N
    reach = closure_mask(f["parent"][0])
    err = 0.0
    for i in range(N):
        rows = np.concatenate([f["c_kv"][0, :L], f["c_kv"][0, L:L + N][reach[i]]])
        ref = np.einsum("hvd,d->hv", f["W_UV"], rows.astype(np.float64).mean(axis=0))
        got = oracle.verify_attn_node(f["q_nope"], f["q_rope"], f["W_UK"], f["W_UV"],
                                      f["c_kv"], f["k_rope"], f["parent"],
                                      f["prefix_len"], 0, i, wl.spec.scale)["out"]
        err = max(err, float(np.abs(got - ref).max()))
    return err


def pin_single_node(seed=5, L=40):
    """N = 1 is plain single-query decode attention over L + 1 keys."""
    wl = tiny_inputs(parent=[-1], L=L, N=1, seed=seed)
    return pin_sdpa(wl, tree_mask_fn=lambda p: np.ones((1, 1), dtype=bool))


def pin_star(seed=6, N=12):
    """Star tree: node i sees the prefix, the root and itself only."""
    wl = tiny_inputs(parent=W.star_tree(N), N=N, seed=seed)

    def star_mask(parent_b):
        m = np.eye(len(parent_b), dtype=bool)
        m[:, 0] = True
        return m
    return pin_sdpa(wl, tree_mask_fn=star_mask)


def pin_empty_prefix(seed=8, N=10):
    """L = 0: a node attends to its own root path only."""
    wl = tiny_inputs(L=0, N=N, seed=seed)
    return pin_sdpa(wl)


def pin_paged(seed=9, B=3, N=7, L=150):
    """Paged layout == the same logical sequence stored contiguously."""
    wl = tiny_inputs(B=B, N=N, L=L, seed=seed, paged=True)
    return pin_sdpa(wl)


def pin_ragged_batch(seed=10):
    """Requests with different prefix lengths (0, 17, 41) and shapes in which no
    two dimensions are equal: each request equals decompressed SDPA over its
    own rows.  Cache rows past each request's L_b + N hold NaN, so reading
    another request's rows or past a request's end shows up as a non-finite
    output."""
    rng = np.random.default_rng(seed)
    B, N, H, dn, dr, dv, dc = 3, 9, 3, 12, 6, 10, 20
    L = np.array([0, 17, 41])
    T = int(L.max()) + N + 5
    parents = np.stack([W.random_tree(rng, N, None, 5) for _ in range(B)])
    q_nope = rng.standard_normal((B, N, H, dn))
    q_rope = rng.standard_normal((B, N, H, dr))
    W_UK = rng.standard_normal((H, dn, dc)) / math.sqrt(dc)
    W_UV = rng.standard_normal((H, dv, dc)) / math.sqrt(dc)
    ckv = np.full((B, T, dc), np.nan)
    kr = np.full((B, T, dr), np.nan)
    for b in range(B):
        ckv[b, :L[b] + N] = rng.standard_normal((L[b] + N, dc))
        kr[b, :L[b] + N] = rng.standard_normal((L[b] + N, dr))
    scale = 1 / math.sqrt(dn + dr)
    out = oracle.verify_attn(q_nope, q_rope, W_UK, W_UV, ckv, kr, parents, L, scale)
    if not np.all(np.isfinite(out)):
        return float("inf")
    err = 0.0
    for b in range(B):
        Lb = int(L[b])
        mask = np.zeros((N, Lb + N), dtype=bool)
        mask[:, :Lb] = True
        mask[:, Lb:] = closure_mask(parents[b])
        ref = decompressed_sdpa(q_nope[b], q_rope[b], W_UK, W_UV, ckv[b, :Lb + N],
                                kr[b, :Lb + N], mask, scale)
        err = max(err, float(np.abs(out[b] - ref).max()))
    return err


def all_pins():
    wl = tiny_inputs()
    return {
        "causal_chain": lambda: pin_causal_chain(),
        "random_tree_sdpa": lambda: pin_sdpa(wl),
        "brute_force": lambda: pin_brute_force(),
        "row_sums": lambda: pin_row_sums(wl),
        "identical_rows": lambda: pin_identical_rows(),
        "zero_query": lambda: pin_zero_query(),
        "single_node": lambda: pin_single_node(),
        "star": lambda: pin_star(),
        "empty_prefix": lambda: pin_empty_prefix(),
        "paged": lambda: pin_paged(),
        "ragged_batch": lambda: pin_ragged_batch(),
    }
