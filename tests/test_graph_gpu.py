"""The verify call, and a whole speculative step around it, captured in a CUDA
graph and replayed.

The library's calls make no synchronous CUDA call, allocation or host read
of device data, so a serving loop can capture them.  A replay reads the live
input buffers and gives outputs bit-identical to the eager calls (the kernels
are deterministic); the status words the call zeroes and sets are part of the
graph too.
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


CASES = {
    "contiguous": dict(B=2, N=16, prefix=("uniform", 300, 900)),
    "paged": dict(B=5, N=8, paged=True, prefix=("loguniform", 40, 900), tree=("chain",)),
}


def _capture(fn):
    """Warm fn on a side stream, then capture it; returns (graph, fn's outputs)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = fn()
    return g, outs


@pytest.mark.parametrize("case", list(CASES))
def test_verify_attn_graph_replay(case):
    wl = W.make(W.small_spec("g_" + case, **CASES[case]))
    va = kdtv.for_workload(wl)
    t = va.t
    eager0 = va().clone()
    torch.cuda.synchronize()
    assert va.status() == 0
    # a second set of queries in the same buffers
    gen = torch.Generator().manual_seed(5)
    q2 = torch.randn(t["q_nope"].shape, generator=gen).to(t["q_nope"].dtype).cuda()
    r2 = torch.randn(t["q_rope"].shape, generator=gen).to(t["q_rope"].dtype).cuda()
    q1, r1 = t["q_nope"].clone(), t["q_rope"].clone()
    t["q_nope"].copy_(q2)
    t["q_rope"].copy_(r2)
    eager1 = va().clone()
    t["q_nope"].copy_(q1)
    t["q_rope"].copy_(r1)
    torch.cuda.synchronize()
    assert not torch.equal(eager0, eager1)

    g, _ = _capture(lambda: va())
    va.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(va.out, eager0)
    assert va.status() == 0
    t["q_nope"].copy_(q2)
    t["q_rope"].copy_(r2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(va.out, eager1)
    assert va.status() == 0


def test_speculative_step_graph_replay():
    """tree_build -> verify -> greedy tokens through a fixed LM head ->
    tree_accept -> compact_kv, as one graph: the replay's tree, output,
    accepted paths, bonus tokens and compacted cache equal the eager step's."""
    spec = W.small_spec("g_step", B=3, N=24, prefix=("uniform", 200, 700))
    wl = W.make(spec)
    va = kdtv.for_workload(wl)
    t = va.t
    B, N = spec.B, spec.N
    rng = np.random.default_rng(11)
    D, K, V = 16, 8, 32
    lp = np.sort(-rng.exponential(1.0, size=(B, D, K)).astype(np.float32), axis=2)[:, :, ::-1]
    lp = torch.from_numpy(np.ascontiguousarray(lp)).cuda()
    tok = torch.from_numpy(rng.integers(0, V, size=(B, D, K)).astype(np.int32)).cuda()
    root = torch.from_numpy(rng.integers(0, V, size=B).astype(np.int32)).cuda()
    Wlm = torch.from_numpy(rng.standard_normal((spec.H * spec.d_v, V))).cuda()
    cst = torch.zeros(1, dtype=torch.int32, device="cuda")
    c0, k0 = t["c_kv"].clone(), t["k_rope"].clone()

    def step():
        tb = kdtv.tree_build(lp, tok, root, N)
        t["parent"].copy_(tb["parent"])
        o = va()
        am = (o.reshape(B * N, -1).double() @ Wlm).argmax(-1).to(torch.int32).reshape(B, N)
        path, plen, bonus = kdtv.tree_accept(tb["parent"], tb["token"], am)
        cst.zero_()
        kdtv.compact_kv(va.dims, t["c_kv"], t["k_rope"], t["prefix_len"], path, plen,
                        status=cst)
        return tb["parent"], tb["token"], o, am, path, plen, bonus

    eager = [x.clone() for x in step()]
    torch.cuda.synchronize()
    assert va.status() == 0 and int(cst.item()) == 0
    cache_eager = (t["c_kv"].clone(), t["k_rope"].clone())
    assert int(eager[5].max().item()) >= 1            # every request accepts the root

    t["c_kv"].copy_(c0)
    t["k_rope"].copy_(k0)
    g, outs = _capture(step)
    for _ in range(2):                                 # replay from the same state twice
        t["c_kv"].copy_(c0)
        t["k_rope"].copy_(k0)
        g.replay()
        torch.cuda.synchronize()
        for got, ref in zip(outs, eager):
            assert torch.equal(got, ref)
        assert torch.equal(t["c_kv"], cache_eager[0]) and torch.equal(t["k_rope"], cache_eager[1])
        assert va.status() == 0 and int(cst.item()) == 0
