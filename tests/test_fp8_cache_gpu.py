"""The FP8 E4M3 latent-cache variant (dtype KDTV_BF16_FP8KV) through the C ABI.

Queries and weights are bf16; c_kv and k_rope are stored one byte per element
and read as fp8 * kv_scale.  The oracle receives the exactly dequantised cache
(decoded from the E4M3 definition by the shared input generator, pinned in
tests/test_fp8_codec.py), so the only differences left are the CUDA path's own
rounding.

* Tensor-core path (the default for the 512 / 64 latent layout): the cache rows
  a call reads are widened exactly to bf16 and the bf16 kernels run on them,
  with kv_scale moved onto the scores and o_lat.  Bar: the bf16 path's
  relative L2 <= 5e-3, max |err| <= 2e-2.  For a power-of-two kv_scale every
  moved factor is exact, so the output must equal, bit for bit, the bf16 call
  on a bf16 cache holding the dequantised values.
* CUDA-core path (KDTV_FLAG_SIMT): fp32 on exactly dequantised values,
  relative L2 <= 1e-5.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_mla_gb300 import kdtv, workloads as W

pytestmark = pytest.mark.gpu

FP32_REL = 1e-5
BF16_REL = 5e-3
BF16_ABS = 2e-2
TC, SIMT = 0, kdtv.KDTV_FLAG_SIMT


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


def _check(g, ref, flags):
    assert np.isfinite(g).all()
    if flags & SIMT:
        assert _rel(g, ref) <= FP32_REL
    else:
        err = np.abs(g - ref)
        assert _rel(g, ref) <= BF16_REL and err.max() <= BF16_ABS, \
            f"rel {_rel(g, ref):.3e} max {err.max():.3e}"


def _bf16_twin(wl):
    """The same problem with a bf16 cache holding the dequantised fp8 values
    (exact: an E4M3 value times a power of two is a bf16 value)."""
    spec = W.Spec(wl.spec.name + "_bf16", wl.spec.index, B=wl.spec.B, N=wl.spec.N, H=wl.spec.H,
                  d_nope=wl.spec.d_nope, d_rope=wl.spec.d_rope, d_v=wl.spec.d_v,
                  d_c=wl.spec.d_c, dtype="bf16", prefix=wl.spec.prefix, tree=wl.spec.tree,
                  paged=wl.spec.paged)
    t = dict(wl.t)
    for n in ("c_kv", "k_rope"):
        t[n] = torch.from_numpy(wl.f32[n]).to(torch.bfloat16)
        assert torch.equal(t[n].float(), torch.from_numpy(wl.f32[n]))
    return W.Workload(spec=spec, t=t, f32=wl.f32, t_stride=wl.t_stride,
                      max_pages=wl.max_pages, num_pages=wl.num_pages)


@pytest.mark.parametrize("flags", [TC, SIMT], ids=["tc", "simt"])
@pytest.mark.parametrize("paged", [False, True])
def test_fp8_cache_small_matches_oracle(paged, flags):
    spec = W.small_spec("s_fp8", B=3, N=12, dtype="fp8kv", paged=paged,
                        prefix=("uniform", 60, 500))
    wl = W.make(spec)
    assert wl.t["c_kv"].dtype == torch.uint8 and wl.kv_scale == W.FP8_KV_SCALE
    got, st = _run(wl, flags=flags)
    assert st == 0
    nodes = [(b, i) for b in range(spec.B) for i in range(spec.N)]
    ref = _oracle(wl, nodes)
    _check(np.stack([got[b, i] for b, i in nodes]), ref, flags)


@pytest.mark.parametrize("flags", [TC, SIMT], ids=["tc", "simt"])
def test_fp8_cache_full_kimi_shape_sampled(flags):
    spec = W.Spec("kimi_fp8", 1, B=1, N=64, dtype="fp8kv", prefix=("fixed", 4096),
                  tree=("window", 8, 8), **W.KIMI)
    wl = W.make(spec)
    got, st = _run(wl, flags=flags)
    assert st == 0
    nodes = [(0, 0), (0, 17), (0, 63)]
    _check(np.stack([got[b, i] for b, i in nodes]), _oracle(wl, nodes), flags)


@pytest.mark.parametrize("paged", [False, True])
def test_fp8_tc_equals_bf16_on_dequantised_cache(paged):
    spec = W.small_spec("s_fp8_twin", B=4, N=24, dtype="fp8kv", paged=paged,
                        prefix=("uniform", 100, 900))
    wl = W.make(spec)
    a, st_a = _run(wl)
    b, st_b = _run(_bf16_twin(wl))
    assert st_a == 0 and st_b == 0
    assert np.array_equal(a, b)


def test_fp8_tc_ragged_stride_and_garbage_rows():
    """t_stride not a multiple of 64 (request 0's last key tile runs into
    request 1's rows) and NaN codes in every row past L_b + N: the rows the
    attention loads but masks are zeroed, so the output is finite, equals the
    call on a clean cache bit for bit, and matches the oracle."""
    N = 12
    prefix = np.array([260, 10, 100])
    wl = W.make(W.small_spec("s_fp8_ragged", B=3, N=N, dtype="fp8kv", prefix=("fixed", 0)),
                 prefix_len=prefix)
    T = prefix + N
    ts = int(T.max()) + 5
    assert ts % 64 and ts <= wl.t_stride and -(-int(T[0]) // 64) * 64 > ts

    def with_stride(t):
        t = dict(t)
        for n in ("c_kv", "k_rope"):
            t[n] = t[n][:, :ts].contiguous()
        return t

    clean = W.Workload(spec=wl.spec, t=with_stride(wl.t),
                       f32={k: (v[:, :ts] if k in ("c_kv", "k_rope") else v)
                            for k, v in wl.f32.items()},
                       t_stride=ts, kv_scale=wl.kv_scale)
    dirty_t = with_stride(wl.t)
    for n in ("c_kv", "k_rope"):
        for b in range(3):
            dirty_t[n][b, int(T[b]):] = 0x7F          # E4M3 NaN
    dirty = W.Workload(spec=wl.spec, t=dirty_t, f32=clean.f32, t_stride=ts,
                       kv_scale=wl.kv_scale)
    a, st_a = _run(clean)
    b, st_b = _run(dirty)
    assert st_a == 0 and st_b == 0
    assert np.isfinite(b).all() and np.array_equal(a, b)
    nodes = [(b_, i) for b_ in range(3) for i in (0, 5, N - 1)]
    _check(np.stack([b[x, y] for x, y in nodes]), _oracle(clean, nodes), TC)


@pytest.mark.parametrize("flags", [TC, SIMT], ids=["tc", "simt"])
@pytest.mark.parametrize("factor", [2.0, 2.4])
def test_fp8_cache_scale_is_applied(flags, factor):
    """kv_scale = factor * the stored scale equals the same call on a cache
    whose every value is factor times larger (a power of two and not)."""
    spec = W.small_spec("s_fp8_scale", B=1, N=8, dtype="fp8kv", prefix=("fixed", 200))
    wl = W.make(spec)
    a, st1 = _run(wl, kv_scale=factor * W.FP8_KV_SCALE, flags=flags)
    f = dict(wl.f32)
    f["c_kv"] = f["c_kv"].astype(np.float64) * factor
    f["k_rope"] = f["k_rope"].astype(np.float64) * factor
    wl2 = W.Workload(spec=spec, t=wl.t, f32=f, t_stride=wl.t_stride)
    ref = _oracle(wl2, [(0, 0), (0, 7)])
    assert st1 == 0
    _check(np.stack([a[0, 0], a[0, 7]]), ref, flags)


@pytest.mark.parametrize("case", ["tree", "prefix", "page"])
def test_fp8_tc_errors_reported_then_clean_call(case):
    """A bad tree, prefix or page id in an fp8 call is reported through the
    status word (the widening kernel skips what it cannot read), and the next
    good call returns the same output as before."""
    spec = W.small_spec("s_fp8_err", B=2, N=8, dtype="fp8kv", paged=case == "page",
                        prefix=("fixed", 100), tree=("chain",))
    wl = W.make(spec)
    good, st = _run(wl)
    assert st == 0
    saved = {k: v.clone() for k, v in wl.t.items()}
    if case == "tree":
        wl.t["parent"][1, 5] = 7                    # parent after child
        want = "KDTV_ERR_BAD_TREE"
    elif case == "prefix":
        wl.t["prefix_len"][1] = wl.t_stride         # L + N > t_stride
        want = "KDTV_ERR_BAD_PREFIX"
    else:
        wl.t["page_table"][0, 1] = wl.num_pages + 5
        want = "KDTV_ERR_BAD_PAGE"
    _, st = _run(wl)
    assert kdtv.STATUS[st] == want
    wl.t.update(saved)
    again, st = _run(wl)
    assert st == 0 and np.array_equal(again, good)


def test_unknown_dtype_rejected():
    """A dtype code outside the enum is refused on the host."""
    spec = W.small_spec("s_fp8_bad", B=1, N=4, dtype="fp8kv", prefix=("fixed", 64))
    d = kdtv.make_dims(spec, dtype=7, t_stride=128)
    assert kdtv.workspace_size(d) == 0
