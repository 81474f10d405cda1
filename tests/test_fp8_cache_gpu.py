"""The FP8 E4M3 latent-cache variant (dtype KDTV_BF16_FP8KV) through the C ABI.

Queries and weights are bf16; c_kv and k_rope are stored one byte per element
and read as fp8 * kv_scale.  The oracle receives the exactly dequantised cache
(decoded from the E4M3 definition by the shared input generator, pinned in
tests/test_fp8_codec.py), so the only differences left are the CUDA path's own
rounding.  The CUDA-core path computes in fp32 on exactly dequantised values
(scale 2^-3): relative L2 <= 1e-5 against the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_mla_gb300 import kdtv, workloads as W

pytestmark = pytest.mark.gpu

FP32_REL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_mla_gb300 import build
    build.build()


def _oracle(wl, nodes):
    f = wl.f32
    return np.stack([
        oracle.verify_attn_node(f["q_nope"], f["q_rope"], f["W_UK"], f["W_UV"], f["c_kv"],
                                f["k_rope"], f["parent"], f["prefix_len"], b, i, wl.spec.scale,
                                page_table=f.get("page_table"), page_size=wl.page_size)["out"]
        for b, i in nodes])


def _run(wl, **kw):
    op = kdtv.for_workload(wl, "cuda", **kw)
    out = op().cpu().double().numpy()
    return out, op.status()


def _rel(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


@pytest.mark.parametrize("paged", [False, True])
def test_fp8_cache_small_matches_oracle(paged):
    spec = W.small_spec("s_fp8", B=3, N=12, dtype="fp8kv", paged=paged,
                        prefix=("uniform", 60, 500))
    wl = W.make(spec)
    assert wl.t["c_kv"].dtype == torch.uint8 and wl.kv_scale == W.FP8_KV_SCALE
    got, st = _run(wl)
    assert st == 0
    nodes = [(b, i) for b in range(spec.B) for i in range(spec.N)]
    ref = _oracle(wl, nodes)
    g = np.stack([got[b, i] for b, i in nodes])
    assert np.isfinite(g).all()
    assert _rel(g, ref) <= FP32_REL


def test_fp8_cache_full_kimi_shape_sampled():
    spec = W.Spec("kimi_fp8", 1, B=1, N=64, dtype="fp8kv", prefix=("fixed", 4096),
                  tree=("window", 8, 8), **W.KIMI)
    wl = W.make(spec)
    got, st = _run(wl)
    assert st == 0
    nodes = [(0, 0), (0, 17), (0, 63)]
    ref = _oracle(wl, nodes)
    g = np.stack([got[b, i] for b, i in nodes])
    assert _rel(g, ref) <= FP32_REL


def test_fp8_cache_scale_is_applied():
    """Doubling kv_scale equals the same call on a cache whose every value doubled."""
    spec = W.small_spec("s_fp8_scale", B=1, N=8, dtype="fp8kv", prefix=("fixed", 200))
    wl = W.make(spec)
    a, st1 = _run(wl, kv_scale=2 * W.FP8_KV_SCALE)
    f = dict(wl.f32)
    f["c_kv"] = f["c_kv"] * 2
    f["k_rope"] = f["k_rope"] * 2
    wl2 = W.Workload(spec=spec, t=wl.t, f32=f, t_stride=wl.t_stride)
    ref = _oracle(wl2, [(0, 0), (0, 7)])
    assert st1 == 0
    assert _rel(np.stack([a[0, 0], a[0, 7]]), ref) <= FP32_REL


def test_unknown_dtype_rejected():
    """A dtype code outside the enum is refused on the host."""
    spec = W.small_spec("s_fp8_bad", B=1, N=4, dtype="fp8kv", prefix=("fixed", 64))
    d = kdtv.make_dims(spec, dtype=7, t_stride=128)
    assert kdtv.workspace_size(d) == 0
