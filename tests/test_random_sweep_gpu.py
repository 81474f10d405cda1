"""Randomised shapes against the oracle: a fixed list of configurations drawn
from a seeded generator (batch, tree size and shape, head count, prefix
lengths, contiguous or paged cache), each run on the tensor-core path (bf16
bar) and the CUDA-core path (fp32 bar), every node of every request compared
with the fp64 oracle; each with a bf16 cache and with an FP8 E4M3 cache (the
oracle then reads the exactly dequantised values).

The list spans what the hand-written cases pick one at a time: ragged
batches of one to ten requests, 1 to 128 tree nodes, 4 to 64 heads (so the
absorb kernel's row-block groups and the stream-K plan's piece counts vary),
prefixes from empty to about 6k keys, window and chain trees.
"""

import numpy as np
import pytest
import torch

from speculative_decoding_tree_mla_gb300 import workloads as W
from tests.test_parity_gpu import BF16_ABS, BF16_REL, F32_ABS, SIMT, TC, _skip_tc, all_nodes, \
    oracle_nodes, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_mla_gb300 import build
    build.build()


def _configs(n=24, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        B = int(rng.integers(1, 11))
        N = int(rng.choice([1, 3, 8, 17, 33, 64, 100, 128]))
        H = int(rng.choice([4, 8, 16, 32, 64]))
        hi = int(rng.integers(1, 6000))
        lo = int(rng.integers(0, hi))
        paged = bool(rng.random() < 0.4)
        tree = ("chain",) if rng.random() < 0.25 else \
            ("window", int(rng.integers(1, 17)), int(rng.integers(2, 17)))
        # keep the oracle's fp64 work to a few seconds per configuration
        if B * N * H * (hi + N) > 1.5e8:
            continue
        out.append(dict(B=B, N=N, H=H, prefix=("uniform", lo, hi), paged=paged, tree=tree))
    return out


CONFIGS = _configs()


@pytest.mark.parametrize("dtype", ["bf16", "fp8kv"])
@pytest.mark.parametrize("path", ["tc", "simt"])
@pytest.mark.parametrize("k", range(len(CONFIGS)))
def test_random_config_every_node(k, path, dtype):
    cfg = CONFIGS[k]
    wl = W.make(W.small_spec(f"sweep_{k}", dtype=dtype, **cfg))
    flags = TC if path == "tc" else SIMT
    _skip_tc(flags, wl)
    got, st, _ = run(wl, flags=flags)
    assert st == 0, cfg
    nodes = all_nodes(wl)
    ref = oracle_nodes(wl, nodes)
    g = np.stack([got[b, i] for b, i in nodes])
    r = np.stack([ref[n] for n in nodes])
    assert np.isfinite(g).all(), cfg
    err = np.abs(g - r)
    if path == "simt":
        assert err.max() <= F32_ABS, (cfg, float(err.max()))
    else:
        node_rel = np.linalg.norm((g - r).reshape(len(nodes), -1), axis=1) / \
            np.linalg.norm(r.reshape(len(nodes), -1), axis=1)
        assert node_rel.max() <= BF16_REL and err.max() <= BF16_ABS, \
            (cfg, float(node_rel.max()), float(err.max()))
