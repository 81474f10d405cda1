"""GPU parity of the loop steps around the verify attention (tree accept,
in-place KV compaction, best-first tree build) against their CPU oracles,
through the C ABI.  Integer outputs and copies are compared bit for bit;
tree-build scores are float32 sums taken in the same order on both sides."""

import numpy as np
import pytest
import torch

from oracle import tree_steps as TS
from speculative_decoding_tree_mla_gb300 import kdtv, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_mla_gb300 import build
    build.build()


def _rand_accept_case(rng, B, N):
    parent = np.stack([W.random_tree(rng, N, 8, 12) for _ in range(B)]).astype(np.int32)
    tok = rng.integers(0, 4, size=(B, N)).astype(np.int32)
    am = rng.integers(0, 4, size=(B, N)).astype(np.int32)
    return parent, tok, am


@pytest.mark.parametrize("N", [1, 8, 33, 128])
def test_tree_accept_matches_oracle(N):
    rng = np.random.default_rng(N)
    B = 24
    parent, tok, am = _rand_accept_case(rng, B, N)
    t = lambda x: torch.from_numpy(x).cuda()
    path, plen, bonus = kdtv.tree_accept(t(parent), t(tok), t(am))
    torch.cuda.synchronize()
    path, plen, bonus = path.cpu().numpy(), plen.cpu().numpy(), bonus.cpu().numpy()
    for b in range(B):
        p, bo = TS.tree_accept(parent[b], tok[b], am[b])
        assert plen[b] == len(p)
        assert path[b, :len(p)].tolist() == p
        assert (path[b, len(p):] == -1).all()
        assert bonus[b] == bo


def test_tree_accept_full_chain():
    N, B = 8, 3
    parent = np.stack([W.chain_tree(N)] * B).astype(np.int32)
    tok = np.tile(np.arange(N, dtype=np.int32), (B, 1))
    am = tok + 1
    t = lambda x: torch.from_numpy(x).cuda()
    path, plen, bonus = kdtv.tree_accept(t(parent), t(tok), t(am))
    assert plen.cpu().tolist() == [N] * B
    assert bonus.cpu().tolist() == [N] * B


def _accepted_paths(rng, B, N):
    parent, tok, am = _rand_accept_case(rng, B, N)
    tok[:, 1:] = am[np.arange(B)[:, None], parent[:, 1:]]     # drafts tend to match
    paths = np.full((B, N), -1, np.int32)
    plen = np.zeros(B, np.int32)
    for b in range(B):
        p, _ = TS.tree_accept(parent[b], tok[b], am[b])
        paths[b, :len(p)] = p
        plen[b] = len(p)
    return paths, plen


@pytest.mark.parametrize("dtype", ["bf16", "f32", "fp8kv"])
@pytest.mark.parametrize("paged", [False, True])
def test_compact_kv_matches_oracle(dtype, paged):
    rng = np.random.default_rng(7)
    spec = W.small_spec("compact", B=6, N=40, dtype=dtype, paged=paged,
                        prefix=("uniform", 30, 300), d_c=512, d_rope=64)
    wl = W.make(spec)
    paths, plen = _accepted_paths(rng, spec.B, spec.N)
    d = kdtv.make_dims(spec, dtype=dtype, page_size=wl.page_size, t_stride=wl.t_stride,
                       max_pages=wl.max_pages, num_pages=wl.num_pages)
    c = wl.t["c_kv"].cuda().contiguous()
    k = wl.t["k_rope"].cuda().contiguous()
    pt = wl.t["page_table"].cuda() if paged else None
    st = kdtv.compact_kv(d, c, k, wl.t["prefix_len"].cuda(), torch.from_numpy(paths).cuda(),
                         torch.from_numpy(plen).cuda(), pt)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_c, ref_k = wl.f32["c_kv"], wl.f32["k_rope"]
    for b in range(spec.B):
        ref_c, ref_k = TS.compact_kv(ref_c, ref_k, b, int(wl.f32["prefix_len"][b]),
                                     paths[b, :plen[b]].tolist(),
                                     page_table=wl.f32.get("page_table"),
                                     page_size=wl.page_size)
    if dtype == "fp8kv":      # the cache holds E4M3 codes: compare the values they decode to
        got_c = W.fp8_e4m3_decode(c.cpu().numpy()) * np.float32(wl.kv_scale)
        got_k = W.fp8_e4m3_decode(k.cpu().numpy()) * np.float32(wl.kv_scale)
    else:
        got_c, got_k = c.float().cpu().numpy(), k.float().cpu().numpy()
    assert np.array_equal(got_c, ref_c)
    assert np.array_equal(got_k, ref_k)


def test_compact_kv_rejects_bad_path():
    spec = W.small_spec("compact_bad", B=2, N=8, prefix=("fixed", 40))
    wl = W.make(spec)
    d = kdtv.make_dims(spec, dtype="bf16", t_stride=wl.t_stride)
    paths = np.array([[0, 3, 2, -1, -1, -1, -1, -1], [0, 1, -1, -1, -1, -1, -1, -1]], np.int32)
    plen = np.array([3, 2], np.int32)
    c = wl.t["c_kv"].cuda()
    before = c.clone()
    st = kdtv.compact_kv(d, c, wl.t["k_rope"].cuda(), wl.t["prefix_len"].cuda(),
                         torch.from_numpy(paths).cuda(), torch.from_numpy(plen).cuda())
    torch.cuda.synchronize()
    assert kdtv.STATUS[int(st.item())] == "KDTV_ERR_BAD_TREE"
    assert torch.equal(c[0], before[0])            # the bad request is untouched


def _build_inputs(rng, B, D, K, ties=False):
    lp = np.sort(-rng.exponential(1.0, size=(B, D, K)).astype(np.float32), axis=2)[:, :, ::-1]
    if ties:
        lp = np.round(lp * 4) / 4
    lp = np.ascontiguousarray(lp.astype(np.float32))
    tok = rng.integers(0, 50000, size=(B, D, K)).astype(np.int32)
    root = rng.integers(0, 50000, size=B).astype(np.int32)
    return lp, tok, root


@pytest.mark.parametrize("B,D,K,N,ties", [(8, 16, 8, 64, False), (4, 3, 4, 128, False),
                                           (6, 12, 6, 100, True), (3, 1, 5, 10, False),
                                           (2, 0, 3, 5, False)])
def test_tree_build_matches_oracle(B, D, K, N, ties):
    rng = np.random.default_rng(B * 100 + D)
    lp, tok, root = _build_inputs(rng, B, D, K, ties)
    g = kdtv.tree_build(torch.from_numpy(lp).cuda(), torch.from_numpy(tok).cuda(),
                        torch.from_numpy(root).cuda(), N)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    for b in range(B):
        r = TS.tree_build(lp[b], tok[b], root[b], N)
        n = len(r["parent"])
        assert g["n_nodes"][b] == n
        for key in ("parent", "token", "depth"):
            assert np.array_equal(g[key][b, :n], r[key]), key
        assert np.array_equal(g["score"][b, :n], r["score"])
        assert (g["parent"][b, n:] == -1).all()
