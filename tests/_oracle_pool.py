"""The fp64 oracle over EVERY node of a named workload, in a process pool.

Each worker regenerates the seeded workload from its name (so no large array
crosses a process boundary) and runs ``oracle.verify_attn_node`` for the
(request, node) pairs it is handed.  The pool uses the ``spawn`` start
method: the calling test process has already initialised CUDA, and a worker
forked after that could hang.  BLAS runs single-threaded in each worker;
the pool supplies the parallelism.
"""

from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

_WL = None


def _init(name):
    global _WL
    from speculative_decoding_tree_mla_gb300 import workloads as W
    _WL = W.make(name)


def _nodes(pairs):
    import oracle
    f = _WL.f32
    out = []
    for b, i in pairs:
        r = oracle.verify_attn_node(f["q_nope"], f["q_rope"], f["W_UK"], f["W_UV"],
                                    f["c_kv"], f["k_rope"], f["parent"], f["prefix_len"],
                                    b, i, _WL.spec.scale, page_table=f.get("page_table"),
                                    page_size=_WL.page_size)
        out.append((b, i, r["out"]))
    return out


_THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def all_nodes(name, procs=None):
    """Oracle output [B, N, H, d_v] (float64) of every node of workload `name`."""
    from speculative_decoding_tree_mla_gb300 import workloads as W
    spec = W.SPECS[name]
    pairs = [(b, i) for b in range(spec.B) for i in range(spec.N)]
    procs = procs or max(1, min(16, os.cpu_count() or 1, len(pairs)))
    # round-robin chunks keep long and short requests spread over the workers
    chunks = [pairs[k::procs * 4] for k in range(procs * 4)]
    chunks = [c for c in chunks if c]
    saved = {v: os.environ.get(v) for v in _THREAD_VARS}
    for v in _THREAD_VARS:
        os.environ[v] = "1"
    try:
        # A worker that dies breaks the executor (BrokenProcessPool) instead
        # of being replaced in a loop.
        with cf.ProcessPoolExecutor(procs, mp_context=mp.get_context("spawn"),
                                    initializer=_init, initargs=(name,)) as ex:
            results = list(ex.map(_nodes, chunks))
    finally:
        for v, x in saved.items():
            if x is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = x
    out = np.full((spec.B, spec.N, spec.H, spec.d_v), np.nan)
    for chunk in results:
        for b, i, r in chunk:
            out[b, i] = r
    assert np.isfinite(out).all()
    return out
