"""Pins for the oracles of the loop steps around the verify attention
(tree accept, KV compaction, best-first tree build); CPU only."""

import heapq
import itertools
import json
import os

import numpy as np
import pytest

from oracle import tree_steps as TS
from speculative_decoding_tree_mla_gb300 import workloads as W

FACTS = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")))


# -- tree accept -------------------------------------------------------------------------
def test_accept_reproduces_printed_run():
    """The printed demo: greedy AR tokens, block size 8, an oracle drafter that
    proposes the golden continuation as a chain => 3 verify steps of 8 tokens
    reproduce the 24 AR tokens ("The Moment of Proof: Running the Native DDTree
    Speculative Decoding Engine", section "The Message Itself"; 8.00 tokens per
    step, "The Build That Proved It: ...", section "The Output Knowledge
    Created")."""
    g = FACTS["greedy_tokens"]
    blk = FACTS["loop_counts"]["block_size"]
    seq = list(g["prompt"]) + list(g["ar_tokens"])
    committed = list(g["prompt"])
    steps, per_step = 0, []
    while len(committed) < len(seq):
        pos = len(committed)                 # index of the next token to produce
        root = committed[-1]
        drafts = [seq[pos + k] if pos + k < len(seq) else -1 for k in range(blk - 1)]
        tok = np.array([root] + drafts)
        parent = W.chain_tree(blk)
        # the target's greedy token after node i is the golden token at pos + i
        argmax = np.array([seq[pos + i] if pos + i < len(seq) else -2 for i in range(blk)])
        path, bonus = TS.tree_accept(parent, tok, argmax)
        new = [int(tok[p]) for p in path[1:]] + [bonus]
        committed += new
        per_step.append(len(new))
        steps += 1
    assert committed[len(g["prompt"]):] == g["ar_tokens"]
    assert steps == FACTS["loop_counts"]["ddtree_target_forwards"]
    assert np.mean(per_step) == FACTS["loop_counts"]["avg_accept_tokens_per_step"]
    assert committed[len(g["prompt"]):len(g["prompt"]) + 16] == g["ddtree_prefix_printed"]


def test_accept_stops_at_sentinel():
    parent = W.chain_tree(8)
    tok = np.array([5, 10, 11, 12, 99, 14, 15, 16])
    argmax = np.array([10, 11, 12, 13, 14, 15, 16, 17])
    path, bonus = TS.tree_accept(parent, tok, argmax)
    assert path == [0, 1, 2, 3] and bonus == 13


def _all_valid_paths(parent, tok, argmax):
    n = len(parent)
    best = [0]
    for i in range(n):
        path = []
        j = i
        while j != -1:
            path.append(j)
            j = parent[j]
        path = path[::-1]
        if all(tok[path[k + 1]] == argmax[path[k]] for k in range(len(path) - 1)):
            if len(path) > len(best):
                best = path
    return best


@pytest.mark.parametrize("seed", range(12))
def test_accept_is_longest_valid_path(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 40))
    parent = W.random_tree(rng, n, None, 10)
    # distinct tokens among siblings so the longest valid path is unique
    tok = np.zeros(n, dtype=np.int64)
    for u in range(n):
        kids = [c for c in range(n) if parent[c] == u]
        vals = rng.choice(6, size=len(kids), replace=False) if len(kids) <= 6 else np.arange(len(kids))
        for c, v in zip(kids, vals):
            tok[c] = v
    argmax = rng.integers(0, 6, size=n)
    path, bonus = TS.tree_accept(parent, tok, argmax)
    assert path == _all_valid_paths(parent, tok, argmax)
    assert bonus == argmax[path[-1]]


def test_accept_duplicate_siblings_take_lowest_index():
    parent = np.array([-1, 0, 0, 1, 2])
    tok = np.array([0, 7, 7, 3, 3])
    argmax = np.array([7, 3, 3, 0, 0])
    path, _ = TS.tree_accept(parent, tok, argmax)
    assert path == [0, 1, 3]


# -- KV compaction ------------------------------------------------------------------------
def test_compact_identity_on_chain_prefix():
    rng = np.random.default_rng(0)
    c = rng.standard_normal((2, 40, 8)); k = rng.standard_normal((2, 40, 4))
    c2, k2 = TS.compact_kv(c, k, 1, 10, [0, 1, 2, 3])
    assert np.array_equal(c2, c) and np.array_equal(k2, k)


@pytest.mark.parametrize("seed", range(6))
def test_compact_moves_rows_and_nothing_else(seed):
    rng = np.random.default_rng(seed)
    B, T, L, N = 3, 96, 40, 30
    c = rng.standard_normal((B, T, 8)); k = rng.standard_normal((B, T, 4))
    parent = W.random_tree(rng, N, 8, 12)
    leaf = int(rng.integers(N))
    path = []
    j = leaf
    while j != -1:
        path.append(j)
        j = parent[j]
    path = path[::-1]
    b = int(rng.integers(B))
    c2, k2 = TS.compact_kv(c, k, b, L, path)
    expect_c = c.copy()
    for kk, node in enumerate(path):
        expect_c[b, L + kk] = c[b, L + node]
    assert np.array_equal(c2, expect_c)
    mask = np.ones(c.shape[:2], dtype=bool)
    mask[b, L:L + len(path)] = False
    assert np.array_equal(k2[mask], k[mask])


def test_compact_paged_equals_contiguous():
    rng = np.random.default_rng(3)
    T, L, ps = 200, 90, 64
    c = rng.standard_normal((1, T, 8)); k = rng.standard_normal((1, T, 4))
    npg = -(-T // ps)
    perm = rng.permutation(npg)
    pc = np.zeros((npg, ps, 8)); pk = np.zeros((npg, ps, 4))
    for p in range(npg):
        seg = c[0, p * ps:(p + 1) * ps]
        pc[perm[p], :len(seg)] = seg
        pk[perm[p], :len(seg)] = k[0, p * ps:(p + 1) * ps]
    path = [0, 2, 5, 9, 30, 41]
    c2, _ = TS.compact_kv(c, k, 0, L, path)
    pc2, _ = TS.compact_kv(pc, pk, 0, L, path, page_table=perm[None], page_size=ps)
    for t in range(T):
        assert np.array_equal(pc2[perm[t // ps], t % ps], c2[0, t])


# -- best-first tree build ------------------------------------------------------------------
def _sorted_logp(rng, D, K):
    x = np.sort(-rng.exponential(1.0, size=(D, K)).astype(np.float32), axis=1)[:, ::-1]
    return np.ascontiguousarray(x)


def test_build_k1_is_chain():
    lp = np.full((6, 1), -0.5, np.float32)
    tok = np.arange(6)[:, None] + 100
    t = TS.tree_build(lp, tok, 7, 20)
    assert t["parent"].tolist() == list(range(-1, 6))
    assert t["token"].tolist() == [7] + list(range(100, 106))


def test_build_depth1_is_star_in_rank_order():
    rng = np.random.default_rng(1)
    lp = _sorted_logp(rng, 1, 6)
    tok = np.arange(6)[None] + 10
    t = TS.tree_build(lp, tok, 0, 5)
    assert t["parent"].tolist() == [-1, 0, 0, 0, 0]
    assert t["token"].tolist() == [0, 10, 11, 12, 13]


@pytest.mark.parametrize("seed", range(8))
def test_build_matches_brute_force_top_n(seed):
    rng = np.random.default_rng(seed)
    D, K, N = 4, 3, int(rng.integers(2, 30))
    lp = _sorted_logp(rng, D, K)
    tok = rng.integers(0, 1000, size=(D, K))
    t = TS.tree_build(lp, tok, 1, N)
    # every node of the complete K-ary tree, scored in float32 along its path
    cand = []
    for d in range(1, D + 1):
        for ks in itertools.product(range(K), repeat=d):
            s = np.float32(0.0)
            for depth, k in enumerate(ks):
                s = np.float32(s + lp[depth, k])
            cand.append((float(s), ks))
    cand.sort(key=lambda x: -x[0])
    want = {ks for _, ks in cand[:N - 1]}
    # recover each oracle node's rank path
    ranks = {0: ()}
    got = set()
    for i in range(1, len(t["parent"])):
        p = int(t["parent"][i])
        d = int(t["depth"][p])
        k = int(np.where(tok[d] == t["token"][i])[0][0]) if len(set(tok[d])) == K else None
        if k is None:
            pytest.skip("duplicate drafter tokens at a depth")
        ranks[i] = ranks[p] + (k,)
        got.add(ranks[i])
    assert got == want
    assert np.all(np.diff(t["score"]) <= 0)          # best-first order
    for i in range(1, len(t["parent"])):
        p = t["parent"][i]
        assert p < i and t["depth"][i] == t["depth"][p] + 1
        assert t["score"][i] == np.float32(t["score"][p] + lp[t["depth"][p], ranks[i][-1]])


def test_build_equal_scores_is_level_order_in_rank_order():
    """All proposals equally likely: every candidate at depth d scores d times
    the same value, so best-first with the stated tie rule (lower parent, then
    lower k) lays the complete K-ary tree out level by level, each node's
    children in rank order."""
    D, K = 3, 3
    lp = np.full((D, K), -0.25, np.float32)
    tok = np.arange(D * K).reshape(D, K) + 50
    n = 1 + K + K * K + K ** 3
    t = TS.tree_build(lp, tok, 9, n)
    want_parent, want_tok, frontier = [-1], [9], [0]
    for d in range(D):
        nxt = []
        for u in frontier:
            for k in range(K):
                want_parent.append(u)
                want_tok.append(int(tok[d, k]))
                nxt.append(len(want_parent) - 1)
        frontier = nxt
    assert t["parent"].tolist() == want_parent
    assert t["token"].tolist() == want_tok
    # one fewer node cuts the last level short at its highest parent / rank
    t2 = TS.tree_build(lp, tok, 9, n - 1)
    assert t2["parent"].tolist() == want_parent[:-1]


# -- planted mistakes: each must be caught by one of the pins above ------------------------
def _accept_highest_child(parent_b, draft_tok_b, target_argmax_b):
    parent_b = [int(p) for p in parent_b]
    path, u = [0], 0
    while True:
        kids = [c for c in range(1, len(parent_b)) if parent_b[c] == u
                and int(draft_tok_b[c]) == int(target_argmax_b[u])]
        if not kids:
            break
        u = kids[-1]
        path.append(u)
    return path, int(target_argmax_b[u])


def _accept_child_own_argmax(parent_b, draft_tok_b, target_argmax_b):
    parent_b = [int(p) for p in parent_b]
    path, u = [0], 0
    while True:
        kids = [c for c in range(1, len(parent_b)) if parent_b[c] == u
                and int(draft_tok_b[c]) == int(target_argmax_b[c])]
        if not kids:
            break
        u = kids[0]
        path.append(u)
    return path, int(target_argmax_b[u])


def _accept_bonus_from_root(parent_b, draft_tok_b, target_argmax_b):
    path, _ = ORIG_TS["tree_accept"](parent_b, draft_tok_b, target_argmax_b)
    return path, int(target_argmax_b[0])


def _accept_first_child_only(parent_b, draft_tok_b, target_argmax_b):
    parent_b = [int(p) for p in parent_b]
    path, u = [0], 0
    while True:
        kids = [c for c in range(1, len(parent_b)) if parent_b[c] == u]
        if not kids or int(draft_tok_b[kids[0]]) != int(target_argmax_b[u]):
            break
        u = kids[0]
        path.append(u)
    return path, int(target_argmax_b[u])


def _compact_dst_shifted(c_kv, k_rope, b, L, path, page_table=None, page_size=0):
    return ORIG_TS["compact_kv"](c_kv, k_rope, b, L + 1, [p - 1 if p else 0 for p in path],
                                 page_table, page_size)


def _compact_paged_ignores_table(c_kv, k_rope, b, L, path, page_table=None, page_size=0):
    if not page_size:
        return ORIG_TS["compact_kv"](c_kv, k_rope, b, L, path)
    c_new, k_new = np.array(c_kv, copy=True), np.array(k_rope, copy=True)
    for k, a in enumerate(path):
        s, d = L + int(a), L + k
        c_new[d // page_size, d % page_size] = c_kv[s // page_size, s % page_size]
        k_new[d // page_size, d % page_size] = k_rope[s // page_size, s % page_size]
    return c_new, k_new


def _build_worst_first(logp, tokens, root_token, n_nodes):
    return ORIG_TS["tree_build"](-np.asarray(logp, np.float32), tokens, root_token, n_nodes)


def _build_ties_high_parent(logp, tokens, root_token, n_nodes):
    logp = np.asarray(logp, np.float32)
    D, K = logp.shape
    parent, token, depth, score = [-1], [int(root_token)], [0], [np.float32(0.0)]
    heap = []

    def push(u):
        if depth[u] < D:
            for k in range(K):
                s = np.float32(score[u] + logp[depth[u], k])
                heapq.heappush(heap, (-float(s), -u, k, s))
    push(0)
    while heap and len(parent) < n_nodes:
        _, mu, k, s = heapq.heappop(heap)
        u = -mu
        parent.append(u)
        token.append(int(tokens[depth[u], k]))
        depth.append(depth[u] + 1)
        score.append(s)
        push(len(parent) - 1)
    return {"parent": np.asarray(parent, np.int32), "token": np.asarray(token, np.int32),
            "depth": np.asarray(depth, np.int32), "score": np.asarray(score, np.float32)}


def _build_depth_short(logp, tokens, root_token, n_nodes):
    return ORIG_TS["tree_build"](np.asarray(logp)[:-1], np.asarray(tokens)[:-1], root_token,
                                 n_nodes)


ORIG_TS = {n: getattr(TS, n) for n in ("tree_accept", "compact_kv", "tree_build")}

_ACCEPT_PINS = [test_accept_reproduces_printed_run, test_accept_stops_at_sentinel,
                test_accept_duplicate_siblings_take_lowest_index] + \
    [lambda s=s: test_accept_is_longest_valid_path(s) for s in range(12)]
_COMPACT_PINS = [test_compact_identity_on_chain_prefix, test_compact_paged_equals_contiguous] + \
    [lambda s=s: test_compact_moves_rows_and_nothing_else(s) for s in range(6)]
_BUILD_PINS = [test_build_k1_is_chain, test_build_depth1_is_star_in_rank_order,
               test_build_equal_scores_is_level_order_in_rank_order] + \
    [lambda s=s: test_build_matches_brute_force_top_n(s) for s in range(8)]

TREE_STEP_MUTATIONS = {
    "accept_takes_highest_matching_child": ("tree_accept", _accept_highest_child, _ACCEPT_PINS),
    "accept_compares_child_own_argmax": ("tree_accept", _accept_child_own_argmax, _ACCEPT_PINS),
    "accept_bonus_from_root": ("tree_accept", _accept_bonus_from_root, _ACCEPT_PINS),
    "accept_first_child_only": ("tree_accept", _accept_first_child_only, _ACCEPT_PINS),
    "compact_destination_shifted": ("compact_kv", _compact_dst_shifted, _COMPACT_PINS),
    "compact_paged_ignores_page_table": ("compact_kv", _compact_paged_ignores_table, _COMPACT_PINS),
    "build_worst_first": ("tree_build", _build_worst_first, _BUILD_PINS),
    "build_ties_to_higher_parent": ("tree_build", _build_ties_high_parent, _BUILD_PINS),
    "build_one_depth_short": ("tree_build", _build_depth_short, _BUILD_PINS),
}


@pytest.mark.parametrize("mutation", list(TREE_STEP_MUTATIONS))
def test_tree_step_pins_catch_planted_mistake(mutation, monkeypatch):
    attr, fn, pins = TREE_STEP_MUTATIONS[mutation]
    monkeypatch.setattr(TS, attr, fn)
    caught = False
    for pin in pins:
        try:
            pin()
        except pytest.skip.Exception:
            continue
        except AssertionError:
            caught = True
            break
    assert caught, f"no pin caught mutation {mutation}"
