"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances: fp32 inputs max |err| <= 1e-5 (the pages' fp32 logit agreement
8.106e-6, "The Moment of Truth: Validating a Custom CUDA Inference Engine for
Kimi K2.6", opening section); bf16 inputs relative L2 <= 5e-3 and max |err|
<= 2e-2.  The greedy token through a fixed random LM head must equal the
oracle's wherever the oracle's top-1 margin exceeds what the relative-L2
tolerance can move (see ``argmax_mismatches``); near-ties must still pick a
token within that margin.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_mla_gb300 import kdtv, workloads as W

pytestmark = pytest.mark.gpu

F32_ABS = 1e-5
BF16_REL = 5e-3
BF16_ABS = 2e-2

TC, SIMT = 0, kdtv.KDTV_FLAG_SIMT


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_mla_gb300 import build
    build.build()


def tc_available(spec):
    d = kdtv.make_dims(spec, dtype="bf16", t_stride=4096)
    return kdtv.workspace_size(d) > 0


def run(wl, flags=0, kv_chunk=0, stream=None):
    op = kdtv.for_workload(wl, "cuda", flags=flags, kv_chunk=kv_chunk)
    out = op(stream=stream)
    st = op.status(stream=stream)
    return out.cpu().double().numpy(), st, op


def oracle_nodes(wl, nodes):
    f = wl.f32
    ref = {}
    for b, i in nodes:
        r = oracle.verify_attn_node(f["q_nope"], f["q_rope"], f["W_UK"], f["W_UV"],
                                    f["c_kv"], f["k_rope"], f["parent"],
                                    f["prefix_len"], b, i, wl.spec.scale,
                                    page_table=f.get("page_table"),
                                    page_size=wl.page_size)
        ref[(b, i)] = r["out"]
    return ref


def all_nodes(wl):
    return [(b, i) for b in range(wl.spec.B) for i in range(wl.spec.N)]


def sample_nodes(wl, k_req=4, seed=0):
    rng = np.random.default_rng(seed)
    B, N = wl.spec.B, wl.spec.N
    reqs = sorted(set([0, B - 1] + list(rng.choice(B, size=min(B, k_req), replace=False))))
    nodes = []
    for b in reqs:
        for i in sorted(set([0, N - 1, int(rng.integers(N))])):
            nodes.append((int(b), int(i)))
    return nodes


def argmax_mismatches(wl, got, ref, nodes, rel_tol):
    """(#exact, #near-tie flips, #bad flips) of the greedy token per node."""
    rng = np.random.default_rng(wl.spec.seed + 77)
    Wlm = rng.standard_normal((wl.spec.H * wl.spec.d_v, wl.spec.vocab)) / np.sqrt(
        wl.spec.H * wl.spec.d_v)
    exact = near = bad = 0
    for (b, i) in nodes:
        tg, _ = oracle.lm_head_argmax(got[b, i], Wlm)
        tr, lr = oracle.lm_head_argmax(ref[(b, i)], Wlm)
        if tg == tr:
            exact += 1
            continue
        margin = lr[tr] - lr[tg]
        bound = rel_tol * np.linalg.norm(ref[(b, i)]) * np.linalg.norm(Wlm[:, tr] - Wlm[:, tg])
        if margin <= bound:
            near += 1
        else:
            bad += 1
    return exact, near, bad


def check(wl, got, nodes, *, f32=False):
    ref = oracle_nodes(wl, nodes)
    g = np.stack([got[b, i] for b, i in nodes])
    r = np.stack([ref[n] for n in nodes])
    assert np.isfinite(g).all()
    err = np.abs(g - r)
    rel = float(np.linalg.norm(g - r) / np.linalg.norm(r))
    if f32:
        assert err.max() <= F32_ABS, f"max_abs {err.max():.3e}"
        exact, near, bad = argmax_mismatches(wl, got, ref, nodes, 1e-5)
        assert bad == 0 and near == 0
    else:
        assert rel <= BF16_REL and err.max() <= BF16_ABS, f"rel {rel:.3e} max {err.max():.3e}"
        exact, near, bad = argmax_mismatches(wl, got, ref, nodes, BF16_REL)
        assert bad == 0, f"{bad} greedy tokens differ beyond the tolerance margin"
    return float(err.max()), rel


# -- fp32 (tiny) ----------------------------------------------------------------
def test_tiny_fp32_full():
    wl = W.make("tiny")
    got, st, _ = run(wl)
    assert st == 0
    check(wl, got, all_nodes(wl), f32=True)


@pytest.mark.parametrize("chunk", [16, 32, 48])
def test_tiny_fp32_splits(chunk):
    wl = W.make("tiny")
    got, st, _ = run(wl, kv_chunk=chunk)
    assert st == 0
    check(wl, got, all_nodes(wl), f32=True)


# -- bf16, reduced sizes (several tiles, ragged tails) ---------------------------
def small(name, **kw):
    return W.make(W.small_spec(name, **kw))


PATH_IDS = {"tc": TC, "simt": SIMT}


def _skip_tc(flags, wl):
    if flags == TC and not tc_available(wl.spec):
        pytest.skip("tensor-core path not compiled in")


@pytest.mark.parametrize("path", list(PATH_IDS))
def test_bf16_small_contiguous(path):
    wl = small("s_contig", B=3, N=24, prefix=("uniform", 100, 700))
    _skip_tc(PATH_IDS[path], wl)
    got, st, _ = run(wl, flags=PATH_IDS[path])
    assert st == 0
    check(wl, got, all_nodes(wl))


@pytest.mark.parametrize("path", list(PATH_IDS))
def test_bf16_small_paged(path):
    wl = small("s_paged", B=5, N=8, paged=True, prefix=("loguniform", 40, 900),
               tree=("chain",))
    _skip_tc(PATH_IDS[path], wl)
    got, st, _ = run(wl, flags=PATH_IDS[path])
    assert st == 0
    check(wl, got, all_nodes(wl))


@pytest.mark.parametrize("path", list(PATH_IDS))
@pytest.mark.parametrize("chunk", [64, 192, 320])
def test_bf16_forced_splits(path, chunk):
    wl = small("s_split", B=2, N=16, prefix=("uniform", 300, 900))
    _skip_tc(PATH_IDS[path], wl)
    got, st, _ = run(wl, flags=PATH_IDS[path], kv_chunk=chunk)
    assert st == 0
    check(wl, got, all_nodes(wl))


@pytest.mark.parametrize("chunk", [0, 64 * 3, 64 * 7, 64 * 11])
def test_tc_piece_boundaries_match_simt(chunk):
    """Work units per CTA pair forced to 3, 7 or 11 key tiles (or the plan's own
    choice) on rows of 16 nodes x 64 heads = 8 row tiles per request: pairs
    cross row-tile boundaries, some pieces are a single key tile, and one pair
    may hold three pieces.  The whole tensor-core output matches the SIMT path,
    and sampled nodes match the oracle."""
    wl = small("s_pieces", B=3, N=16, prefix=("uniform", 200, 1300))
    _skip_tc(TC, wl)
    a, st1, _ = run(wl, flags=TC, kv_chunk=chunk)
    b, st2, _ = run(wl, flags=SIMT)
    assert st1 == st2 == 0
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel <= BF16_REL
    rows_bad = (np.abs(a - b).reshape(-1, a.shape[-1]).max(axis=1) >
                0.05 * (np.abs(b).reshape(-1, b.shape[-1]).max(axis=1) + 1e-3))
    assert int(rows_bad.sum()) == 0
    check(wl, a, [(bi, i) for bi in range(wl.spec.B) for i in (0, wl.spec.N // 2, wl.spec.N - 1)])


@pytest.mark.parametrize("path", list(PATH_IDS))
@pytest.mark.parametrize("case", ["single_node", "empty_prefix", "star", "max_nodes_chain",
                                  "few_heads"])
def test_bf16_edge_cases(path, case):
    if case == "single_node":
        wl = small("e1", B=2, N=1, prefix=("uniform", 1, 200))
    elif case == "empty_prefix":
        wl = small("e2", B=2, N=20, prefix=("fixed", 0))
    elif case == "star":
        spec = W.small_spec("e3", B=1, N=32, prefix=("fixed", 257))
        wl = W.make(spec, parent=W.star_tree(32)[None])
    elif case == "max_nodes_chain":
        wl = small("e4", B=1, N=128, prefix=("fixed", 130), tree=("chain",))
    else:
        wl = small("e5", B=2, N=40, H=4, prefix=("uniform", 10, 300))
    _skip_tc(PATH_IDS[path], wl)
    got, st, _ = run(wl, flags=PATH_IDS[path])
    assert st == 0
    check(wl, got, all_nodes(wl))


@pytest.mark.parametrize("path", list(PATH_IDS))
@pytest.mark.parametrize("H,d_nope,d_v", [(128, 128, 128), (16, 192, 128), (32, 64, 64),
                                          (8, 96, 192)])
def test_bf16_head_layouts(path, H, d_nope, d_v):
    """Head counts and head dims other than the Kimi layout, on the 512 + 64
    latent cache: 128 heads (row tiles of one node), a 192-wide nope dim, and
    head dims that the tensor-core absorb (d_nope % 64 != 0) or up-projection
    (d_v != 128) kernels do not take, so the call mixes tensor-core attention
    with CUDA-core projections."""
    wl = small(f"heads_{H}_{d_nope}_{d_v}", B=2, N=12, H=H, d_nope=d_nope, d_v=d_v,
               prefix=("uniform", 40, 400))
    _skip_tc(PATH_IDS[path], wl)
    got, st, _ = run(wl, flags=PATH_IDS[path])
    assert st == 0
    check(wl, got, all_nodes(wl))


@pytest.mark.parametrize("paged", [False, True])
def test_tc_attention_with_simt_projections(paged):
    """KDTV_FLAG_SIMT_PROJ: tensor-core attention between the CUDA-core absorb
    (bf16 q_lat) and the CUDA-core combine + up-projection reading the
    stream-K piece partials."""
    wl = small("s_proj", B=3, N=16, paged=paged, prefix=("uniform", 50, 900))
    _skip_tc(TC, wl)
    a, st1, op = run(wl, flags=kdtv.KDTV_FLAG_SIMT_PROJ)
    assert st1 == 0 and kdtv.launches_per_call(op.dims) == 5
    check(wl, a, all_nodes(wl))
    b, st2, _ = run(wl, flags=TC)
    assert st2 == 0 and np.linalg.norm(a - b) / np.linalg.norm(b) <= BF16_REL


# -- full-size workloads, sampled nodes -------------------------------------------
@pytest.mark.parametrize("path", list(PATH_IDS))
@pytest.mark.parametrize("name", ["kimi_single", "batched", "long", "paged"])
def test_full_size_sampled(path, name):
    wl = W.make(name)
    _skip_tc(PATH_IDS[path], wl)
    got, st, _ = run(wl, flags=PATH_IDS[path])
    assert st == 0
    nodes = sample_nodes(wl)
    check(wl, got, nodes)


# -- device-side error reporting ----------------------------------------------------
@pytest.mark.parametrize("path", list(PATH_IDS))
def test_bad_tree_reported(path):
    wl = small("bad_tree", B=2, N=8, prefix=("fixed", 64))
    _skip_tc(PATH_IDS[path], wl)
    wl.t["parent"][1, 5] = 7            # parent after child
    _, st, _ = run(wl, flags=PATH_IDS[path])
    assert kdtv.STATUS[st] == "KDTV_ERR_BAD_TREE"
    wl.t["parent"][1, 5] = 0
    wl.t["parent"][0, 0] = 3            # root not -1
    _, st, _ = run(wl, flags=PATH_IDS[path])
    assert kdtv.STATUS[st] == "KDTV_ERR_BAD_TREE"


@pytest.mark.parametrize("path", list(PATH_IDS))
def test_bad_prefix_reported(path):
    wl = small("bad_prefix", B=2, N=8, prefix=("fixed", 64))
    _skip_tc(PATH_IDS[path], wl)
    wl.t["prefix_len"][1] = wl.t_stride       # L + N > t_stride
    _, st, _ = run(wl, flags=PATH_IDS[path])
    assert kdtv.STATUS[st] == "KDTV_ERR_BAD_PREFIX"


@pytest.mark.parametrize("path", list(PATH_IDS))
def test_bad_page_reported(path):
    wl = small("bad_page", B=2, N=8, paged=True, prefix=("fixed", 100), tree=("chain",))
    _skip_tc(PATH_IDS[path], wl)
    wl.t["page_table"][0, 1] = wl.num_pages + 5
    _, st, _ = run(wl, flags=PATH_IDS[path])
    assert kdtv.STATUS[st] == "KDTV_ERR_BAD_PAGE"


@pytest.mark.parametrize("path", list(PATH_IDS))
def test_status_clears_on_next_call(path):
    wl = small("clear", B=1, N=8, prefix=("fixed", 64))
    _skip_tc(PATH_IDS[path], wl)
    wl.t["parent"][0, 3] = 5
    _, st, _ = run(wl, flags=PATH_IDS[path])
    assert st != 0
    wl.t["parent"][0, 3] = 0
    _, st, _ = run(wl, flags=PATH_IDS[path])
    assert st == 0


@pytest.mark.parametrize("path", list(PATH_IDS))
def test_deterministic_and_side_stream(path):
    wl = small("det", B=2, N=16, prefix=("uniform", 200, 500))
    _skip_tc(PATH_IDS[path], wl)
    s = torch.cuda.Stream()
    a, st1, _ = run(wl, flags=PATH_IDS[path], stream=s)
    b, st2, _ = run(wl, flags=PATH_IDS[path])
    assert st1 == st2 == 0
    assert np.array_equal(a, b)


def test_device_timeout_reported_and_context_usable():
    """A wait that nothing satisfies ends with KDTV_ERR_DEVICE_TIMEOUT after its
    limit (no trap, no hang), and the next call on the same context is correct."""
    wl = small("stall", B=1, N=8, prefix=("fixed", 256))
    _skip_tc(TC, wl)
    _, st, _ = run(wl, flags=kdtv.KDTV_FLAG_TEST_STALL)
    assert kdtv.STATUS[st] == "KDTV_ERR_DEVICE_TIMEOUT"
    got, st, _ = run(wl)
    assert st == 0
    check(wl, got, all_nodes(wl))


@pytest.mark.parametrize("name", ["kimi_single", "long"])
def test_tc_matches_simt_closely(name):
    """The two CUDA paths agree with each other on full-size inputs (sampled
    rows are also checked against the oracle in test_full_size_sampled)."""
    wl = W.make(name)
    _skip_tc(TC, wl)
    a, st1, _ = run(wl, flags=TC)
    b, st2, _ = run(wl, flags=SIMT)
    assert st1 == st2 == 0
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel <= BF16_REL
