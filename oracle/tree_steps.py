"""CPU oracles for the steps around the verify attention in the DDTree loop.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The loop itself is narrated on "The Moment of Proof: Validating a Native CUDA
Speculative Decoding Engine" (sections "The Context: Building a Native DDTree
Engine from Scratch" and "Input Knowledge Required"): a drafter proposes a
tree of candidate tokens, a GPU best-first builder lays it out, the target
verifies all nodes in one forward, a greedy tree-accept kernel keeps the
longest matching path, and the KV cache is compacted.  None of these steps
is given as a formula; each function states the plain reading it takes.
"""

from __future__ import annotations

import heapq

import numpy as np


def tree_accept(parent_b, draft_tok_b, target_argmax_b):
    """Greedy acceptance of one request's draft tree.

    Reading ("The Build That Proved It: Compiling the Native DDTree
    Speculative Decoding Engine", section "The Output Knowledge Created": the
    tree-accept kernel identifies the longest prefix match): node 0 is the
    root (the last committed token).  From the current node u, the walk moves
    to the child c of u whose draft token equals the target's greedy token at
    u, the lowest-indexed such child if several match, and stops when none
    does.  Returns (path, bonus): the accepted node indices starting with 0,
    and the target's greedy token at the last accepted node, which is
    committed after the path's draft tokens.
    """
    parent_b = [int(p) for p in parent_b]
    n = len(parent_b)
    children = [[] for _ in range(n)]
    for i in range(1, n):
        children[parent_b[i]].append(i)
    path = [0]
    u = 0
    while True:
        want = int(target_argmax_b[u])
        nxt = None
        for c in children[u]:            # ascending index
            if int(draft_tok_b[c]) == want:
                nxt = c
                break
        if nxt is None:
            break
        path.append(nxt)
        u = nxt
    return path, int(target_argmax_b[u])


def compact_kv(c_kv, k_rope, b, L, path, page_table=None, page_size=0):
    """Post-verify KV compaction of request b, returning new arrays.

    Reading ("The Moment of Truth: Validating a Custom CUDA Inference Engine
    for Kimi K2.6", section "What the Output Tells Us": the kept rows are
    gathered into a compact cache, via scratch to avoid an in-place race):
    the latent rows of the accepted nodes, at positions L + path[k], move to
    positions L + k for k = 0 .. len(path)-1; every other row is unchanged.
    Copy semantics: all sources are read before any destination is written.
    """
    c_new, k_new = np.array(c_kv, copy=True), np.array(k_rope, copy=True)
    src = [L + int(a) for a in path]
    dst = [L + k for k in range(len(path))]

    def loc(t):
        if page_size:
            return int(page_table[b, t // page_size]), t % page_size
        return b, t
    rows_c = [np.array(c_kv[loc(t)], copy=True) for t in src]
    rows_k = [np.array(k_rope[loc(t)], copy=True) for t in src]
    for t, rc, rk in zip(dst, rows_c, rows_k):
        c_new[loc(t)] = rc
        k_new[loc(t)] = rk
    return c_new, k_new


def tree_build(logp, tokens, root_token, n_nodes):
    """Best-first draft tree from per-depth top-K proposals.

    Reading ("The Moment of Proof: Validating a Native CUDA Speculative
    Decoding Engine", section "The Context: Building a Native DDTree Engine
    from Scratch": a GPU best-first tree builder replacing a per-request CPU
    heap): the drafter proposes, for every depth d = 1..D, K candidate tokens
    ``tokens[d-1, k]`` with log-probabilities ``logp[d-1, k]``.  Node 0 is the
    root (``root_token``, depth 0, score 0).  A node at depth d < D offers K
    candidate children with score ``score(node) + logp[d, k]`` (float32
    addition).  Repeatedly the best candidate is taken, highest score first,
    ties broken by lower parent index, then lower k, and becomes the next
    node; its own candidates join the frontier.  Stops at ``n_nodes`` nodes or
    an empty frontier.

    Returns dict(parent, token, depth, score) as arrays in node order (a
    topological order: parents precede children).
    """
    logp = np.asarray(logp, dtype=np.float32)
    tokens = np.asarray(tokens)
    D, K = logp.shape
    parent, token, depth, score = [-1], [int(root_token)], [0], [np.float32(0.0)]
    heap = []

    def push(u):
        if depth[u] >= D:
            return
        for k in range(K):
            s = np.float32(score[u] + logp[depth[u], k])
            heapq.heappush(heap, (-float(s), u, k, s))

    push(0)
    while heap and len(parent) < n_nodes:
        _, u, k, s = heapq.heappop(heap)
        parent.append(u)
        token.append(int(tokens[depth[u], k]))
        depth.append(depth[u] + 1)
        score.append(s)
        push(len(parent) - 1)
    return {"parent": np.asarray(parent, np.int32), "token": np.asarray(token, np.int32),
            "depth": np.asarray(depth, np.int32), "score": np.asarray(score, np.float32)}
