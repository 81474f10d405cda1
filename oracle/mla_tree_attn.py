"""fp64 oracle: tree-verify attention over an MLA latent cache, absorbed form.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

What it computes is stated on "The Moment of Proof: Validating a Native CUDA
Speculative Decoding Engine", section "Input Knowledge Required": the target
model scores every node of a draft token tree in ONE forward pass under a
custom attention mask, and MLA's absorbed form folds the key/value
up-projections (w_kc / w_vc) into the attention.  Section "The Context:
Building a Native DDTree Engine from Scratch" of the same page names the
kernel this oracle stands behind ("tree-verify MLA-absorb attention kernel
with visibility masking") and the invariant it must keep: the tree-verify
greedy output equals the autoregressive greedy output.

The pages give no formulas; the steps below are the plain definition, in the
order a reader would check them:

  1. absorb        q_lat[b,i,h,:] = W_UK[h]^T q_nope[b,i,h,:]
  2. visibility    node i sees the committed prefix 0..L_b-1 and the rows
                   L_b + a for every a on its own root path (itself included)
  3. scores        s_t = scale * (q_lat . c_kv[t] + q_rope . k_rope[t])
  4. softmax       over the visible keys only
  5. latent mix    o_lat = sum_t p_t c_kv[t]
  6. up-project    out[b,i,h,:] = W_UV[h] o_lat

Readings where the pages are silent:
  * a node sees itself (forced by the chain == causal invariant);
  * W_UK is [H, d_nope, d_c] with k_nope = W_UK[h] c; W_UV is [H, d_v, d_c];
  * k_rope is one shared head [T, d_rope]; q_rope / k_rope arrive rotated;
  * tree-node latents sit at positions L_b .. L_b+N-1 of request b;
  * paged caches resolve position t through page_table[b, t // page_size].

Every floating-point step runs in float64; inputs given as bf16-valued
float32 arrays widen exactly.  Library primitives used as steps: numpy
``einsum`` / ``@`` (dot products) and ``exp``.
"""

from __future__ import annotations

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


# -- step 1 -------------------------------------------------------------------
def absorb(q_nope, W_UK):
    """Step 1, the absorb of q_nope into the kv_lora latent space.

    "The Moment of Proof: Validating a Native CUDA Speculative Decoding
    Engine", section "Input Knowledge Required" (absorb form w_kc).
    q_nope [B, N, H, d_nope], W_UK [H, d_nope, d_c] -> q_lat [B, N, H, d_c],
    q_lat[b,i,h,d] = sum_e q_nope[b,i,h,e] * W_UK[h,e,d].
    """
    return np.einsum("bnhe,hed->bnhd", _f64(q_nope), _f64(W_UK))


# -- step 2 -------------------------------------------------------------------
def ancestor_path(parent_b, i):
    """Step 2a: the root path of node i: [i, parent[i], parent[parent[i]], ..., 0].

    Tree convention (same page, section "Input Knowledge Required": a tree of
    draft tokens): parent[0] == -1 and 0 <= parent[j] < j for j > 0, i.e. the
    nodes are in topological order.  Raises ValueError otherwise.
    """
    parent_b = [int(p) for p in parent_b]
    n = len(parent_b)
    if n == 0 or parent_b[0] != -1:
        raise ValueError("parent[0] must be -1 (the root)")
    if not (0 <= i < n):
        raise ValueError("node index out of range")
    path = []
    j = i
    while j != -1:
        p = parent_b[j]
        if j > 0 and not (0 <= p < j):
            raise ValueError(f"parent[{j}]={p} is not in [0, {j})")
        path.append(j)
        j = p
    return path


def visible_positions(L_b, path):
    """Step 2b: the positions node i may attend to: prefix rows 0..L_b-1 plus
    L_b + a for each a on its root path, ascending."""
    tree_rows = sorted(int(L_b) + int(a) for a in path)
    return np.concatenate([np.arange(int(L_b), dtype=np.int64),
                           np.asarray(tree_rows, dtype=np.int64)])


def gather_cache(c_kv, k_rope, b, positions, page_table=None, page_size=0):
    """Rows of request b's latent cache at the given logical positions.

    Contiguous mode: c_kv [B, T_stride, d_c], k_rope [B, T_stride, d_rope].
    Paged mode (page_size > 0): c_kv [P, page_size, d_c], k_rope
    [P, page_size, d_rope], and position t of request b lives in physical page
    page_table[b, t // page_size] at slot t % page_size.
    """
    positions = np.asarray(positions, dtype=np.int64)
    if page_size:
        pages = np.asarray(page_table)[b, positions // page_size].astype(np.int64)
        slots = positions % page_size
        return _f64(c_kv[pages, slots]), _f64(k_rope[pages, slots])
    return _f64(c_kv[b, positions]), _f64(k_rope[b, positions])


# -- step 3 -------------------------------------------------------------------
def node_scores(q_lat_bi, q_rope_bi, ckv_vis, krope_vis, scale):
    """Step 3: s[h, t] = scale * (q_lat[h] . c_kv[t] + q_rope[h] . k_rope[t]).

    q_lat_bi [H, d_c], q_rope_bi [H, d_rope], ckv_vis [V, d_c],
    krope_vis [V, d_rope] -> [H, V].
    """
    return float(scale) * (_f64(q_lat_bi) @ _f64(ckv_vis).T
                           + _f64(q_rope_bi) @ _f64(krope_vis).T)


# -- step 4 -------------------------------------------------------------------
def softmax_rows(s):
    """Step 4: p[h, t] = exp(s[h, t] - max_u s[h, u]) / sum_u exp(s[h, u] - max_u s[h, u])."""
    s = _f64(s)
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


# -- step 5 -------------------------------------------------------------------
def attend_latent(p, ckv_vis):
    """Step 5: o_lat[h, d] = sum_t p[h, t] * c_kv[t, d] (the value side of
    the absorbed form is the latent row itself)."""
    return _f64(p) @ _f64(ckv_vis)


# -- step 6 -------------------------------------------------------------------
def up_project(o_lat, W_UV):
    """Step 6, the w_vc half of the absorb ("The Moment of Proof: Validating
    a Native CUDA Speculative Decoding Engine", section "Input Knowledge
    Required"): out[h, v] = sum_d W_UV[h, v, d] * o_lat[h, d]."""
    return np.einsum("hvd,hd->hv", _f64(W_UV), _f64(o_lat))


def verify_attn_node(q_nope, q_rope, W_UK, W_UV, c_kv, k_rope, parent,
                     prefix_len, b, i, scale, page_table=None, page_size=0,
                     q_lat=None):
    """All six steps for one (request b, node i), every head at once.

    Returns a dict with ``out`` [H, d_v], ``o_lat`` [H, d_c], ``p`` [H, V],
    ``s`` [H, V] and ``positions`` [V].  ``q_lat`` may pass a precomputed
    step-1 result for request b / node i ([H, d_c]).
    """
    if q_lat is None:
        q_lat = absorb(q_nope[b:b + 1, i:i + 1], W_UK)[0, 0]
    path = ancestor_path(parent[b], i)
    positions = visible_positions(int(prefix_len[b]), path)
    ckv_vis, krope_vis = gather_cache(c_kv, k_rope, b, positions,
                                      page_table, page_size)
    s = node_scores(q_lat, q_rope[b, i], ckv_vis, krope_vis, scale)
    p = softmax_rows(s)
    o_lat = attend_latent(p, ckv_vis)
    out = up_project(o_lat, W_UV)
    return {"out": out, "o_lat": o_lat, "p": p, "s": s, "positions": positions}


def verify_attn(q_nope, q_rope, W_UK, W_UV, c_kv, k_rope, parent, prefix_len,
                scale, page_table=None, page_size=0, nodes=None):
    """The whole path: out [B, N, H, d_v] in float64.

    ``nodes`` optionally restricts the work to a list of (b, i) pairs (the
    other outputs stay NaN) so that full-size workloads can be checked on a
    sample.
    """
    B, N, H, _ = q_nope.shape
    d_v = W_UV.shape[1]
    out = np.full((B, N, H, d_v), np.nan)
    if nodes is None:
        nodes = [(b, i) for b in range(B) for i in range(N)]
    for b, i in nodes:
        r = verify_attn_node(q_nope, q_rope, W_UK, W_UV, c_kv, k_rope, parent,
                             prefix_len, b, i, scale, page_table, page_size)
        out[b, i] = r["out"]
    return out


def lm_head_argmax(out_bi, W_lm):
    """Greedy token of one node through a fixed LM head (test fixture).

    logits = flatten(out[b, i]) @ W_lm in float64; ties break to the lowest
    index (numpy argmax).  Returns (argmax, logits).
    """
    logits = _f64(out_bi).reshape(-1) @ _f64(W_lm)
    return int(np.argmax(logits)), logits
