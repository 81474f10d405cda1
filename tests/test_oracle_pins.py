"""The fp64 oracle against what the pages and the mathematics fix (CPU only).

Pins: (1) a chain tree equals causal attention (the pages' invariant that
tree-verify greedy output equals autoregressive output, "The Moment of Proof:
Validating a Native CUDA Speculative Decoding Engine", section "The Context:
Building a Native DDTree Engine from Scratch"); (2) the absorbed form equals
the decompressed form (section "Input Knowledge Required", absorb w_kc/w_vc);
(3) brute force per node; (4) softmax rows sum to 1; plus closed-form special
cases.  The mutation test plants plausible mistakes in the oracle and checks
that some pin catches each one.
"""

import importlib
import json
import os

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_mla_gb300 import workloads as W

from . import _pins as P

ORACLE_MOD = importlib.import_module("oracle.mla_tree_attn")


@pytest.mark.parametrize("name", list(P.all_pins().keys()))
def test_pin(name):
    err = P.all_pins()[name]()
    assert err < P.TOL, f"pin {name}: deviation {err:.3e}"


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_causal_chain_more_seeds(seed):
    assert P.pin_causal_chain(seed=seed, L=17, N=9) < P.TOL


@pytest.mark.parametrize("seed", [21, 22])
def test_random_trees_batched(seed):
    wl = P.tiny_inputs(B=2, N=13, L=5, seed=seed)
    assert P.pin_sdpa(wl) < P.TOL


def test_tree_validation():
    with pytest.raises(ValueError):
        oracle.ancestor_path([0, 0, 1], 2)          # root must be -1
    with pytest.raises(ValueError):
        oracle.ancestor_path([-1, 2, 0], 1)         # parent must precede child
    with pytest.raises(ValueError):
        oracle.ancestor_path([-1, 0, 2], 2)         # self-parent


def test_visible_positions_shape():
    pos = oracle.visible_positions(5, [3, 1, 0])
    assert pos.tolist() == [0, 1, 2, 3, 4, 5, 6, 8]


def test_lm_head_ties_break_low():
    W_lm = np.zeros((2, 4))
    W_lm[0, 1] = W_lm[0, 3] = 1.0
    tok, _ = oracle.lm_head_argmax(np.array([1.0, 0.0]), W_lm)
    assert tok == 1


def test_tiny_workload_matches_printed_model():
    """The tiny workload uses the toy model's printed head count, kv_lora and
    vocab ("The Moment of Proof: Running the Native DDTree Speculative
    Decoding Engine", section "The Message Itself")."""
    facts = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                        "pages_facts.json")))
    tm = facts["tiny_model"]
    s = W.SPECS["tiny"]
    assert (s.H, s.d_c, s.vocab) == (tm["heads"], tm["kv_lora"], tm["vocab"])


def test_workload_trees_follow_recipe():
    for name in ("tiny", "kimi_single", "batched", "long", "paged"):
        s = W.SPECS[name]
        rng = np.random.default_rng(0)
        if s.tree[0] == "chain":
            p = W.chain_tree(s.N)
            cap = s.N
        else:
            _, win, cap = s.tree
            p = W.random_tree(rng, s.N, win, cap)
        d = W.tree_depths(p)
        assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, s.N))
        assert d.max() <= cap


# -- mutations planted in the oracle (CPU only) -------------------------------
def _m_absorb_head0(q, Wk):
    return np.einsum("bnhe,ed->bnhd", np.asarray(q, np.float64), np.asarray(Wk, np.float64)[0])


def _m_no_rope(ql, qr, ck, kr, scale):
    return float(scale) * (np.asarray(ql, np.float64) @ np.asarray(ck, np.float64).T)


def _m_no_scale(ql, qr, ck, kr, scale):
    return (np.asarray(ql, np.float64) @ np.asarray(ck, np.float64).T
            + np.asarray(qr, np.float64) @ np.asarray(kr, np.float64).T)


def _m_exclude_self(L, path):
    return ORIG["visible_positions"](L, list(path)[1:])


def _m_causal_not_tree(L, path):
    return ORIG["visible_positions"](L, list(range(path[0] + 1)))


def _m_root_missing(parent_b, i):
    return [j for j in ORIG["ancestor_path"](parent_b, i) if j != 0] or [i]


def _m_softmax_heads(s):
    s = np.asarray(s, np.float64)
    e = np.exp(s - s.max(axis=0, keepdims=True))
    return e / e.sum(axis=0, keepdims=True)


def _m_up_sum_heads(o, Wv):
    return np.einsum("hvd,gd->hv", np.asarray(Wv, np.float64), np.asarray(o, np.float64))


def _m_paged_ignores_table(c_kv, k_rope, b, positions, page_table=None, page_size=0):
    if page_size:
        positions = np.asarray(positions, np.int64)
        pages = b * (np.asarray(page_table).shape[1]) + positions // page_size
        pages = np.minimum(pages, c_kv.shape[0] - 1)
        slots = positions % page_size
        return np.asarray(c_kv[pages, slots], np.float64), np.asarray(k_rope[pages, slots], np.float64)
    return ORIG["gather_cache"](c_kv, k_rope, b, positions, page_table, page_size)


def _m_first_request_prefix(q_nope, q_rope, W_UK, W_UV, c_kv, k_rope, parent, prefix_len,
                            b, i, scale, page_table=None, page_size=0, q_lat=None):
    same = np.full_like(np.asarray(prefix_len), np.asarray(prefix_len)[0])
    return ORIG["verify_attn_node"](q_nope, q_rope, W_UK, W_UV, c_kv, k_rope, parent, same,
                                    b, i, scale, page_table, page_size, q_lat)


def _m_gather_first_request(c_kv, k_rope, b, positions, page_table=None, page_size=0):
    return ORIG["gather_cache"](c_kv, k_rope, 0 if not page_size else b, positions,
                                page_table, page_size)


ORIG = {n: getattr(ORACLE_MOD, n) for n in
        ("absorb", "node_scores", "visible_positions", "ancestor_path", "softmax_rows",
         "up_project", "gather_cache", "verify_attn_node")}

MUTATIONS = {
    "absorb_uses_head0": ("absorb", _m_absorb_head0),
    "scores_drop_rope": ("node_scores", _m_no_rope),
    "scores_drop_scale": ("node_scores", _m_no_scale),
    "mask_excludes_self": ("visible_positions", _m_exclude_self),
    "mask_causal_not_tree": ("visible_positions", _m_causal_not_tree),
    "mask_drops_root": ("ancestor_path", _m_root_missing),
    "softmax_over_heads": ("softmax_rows", _m_softmax_heads),
    "up_project_sums_heads": ("up_project", _m_up_sum_heads),
    "paged_ignores_page_table": ("gather_cache", _m_paged_ignores_table),
    "prefix_of_first_request_for_all": ("verify_attn_node", _m_first_request_prefix),
    "contiguous_gather_ignores_request": ("gather_cache", _m_gather_first_request),
}


@pytest.mark.parametrize("mutation", list(MUTATIONS))
def test_pins_catch_planted_mistake(mutation, monkeypatch):
    attr, fn = MUTATIONS[mutation]
    monkeypatch.setattr(ORACLE_MOD, attr, fn)
    worst = 0.0
    for name, pin in P.all_pins().items():
        try:
            worst = max(worst, pin())
        except AssertionError:
            worst = float("inf")
        if worst > 1e-6:
            break
    assert worst > 1e-6, f"no pin caught mutation {mutation}"
