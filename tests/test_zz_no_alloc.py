"""The allocation-free entry point, kdtv_verify_attn_noalloc, through the C ABI.

Some callers of this library cannot call cudaMalloc where they run the
attention (code inside an arena or pool allocator that owns all device
memory, server plugins limited to pre-registered buffers, processes that
forbid device allocation after start-up).  For them the library offers a
variant whose scratch is a fixed array in its own device image.  These tests
check that variant against the regular workspace entry point, on two calls in
a row (the array is shared and keeps the previous call's contents): both run
the same kernels on the same plan, so the outputs must be identical bit for
bit.  They also check that a device-side error reaches the caller through
status_out and clears on the next good call, and that a call needing more
scratch than the array holds is refused.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process.
"""

import ctypes

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


def _noalloc(op, out, status, stream=None):
    t = op.t
    pt = t.get("page_table")
    s = stream if stream is not None else torch.cuda.current_stream()
    return kdtv.lib().kdtv_verify_attn_noalloc(
        ctypes.byref(op.dims), t["q_nope"].data_ptr(), t["q_rope"].data_ptr(),
        t["W_UK"].data_ptr(), t["W_UV"].data_ptr(), t["c_kv"].data_ptr(),
        t["k_rope"].data_ptr(), t["parent"].data_ptr(), t["prefix_len"].data_ptr(),
        pt.data_ptr() if pt is not None else None, out.data_ptr(), status.data_ptr(),
        s.cuda_stream or None)


def _workload(kind):
    if kind == "tiny_fp32":
        return W.make("tiny")
    if kind == "bf16_contiguous":
        return W.make(W.small_spec("na_c", B=2, N=16, prefix=("uniform", 100, 600)))
    if kind == "fp8_cache":
        # the widened cache copies are the largest regions carved from the array
        return W.make(W.small_spec("na_8", B=2, N=16, dtype="fp8kv", prefix=("uniform", 100, 600)))
    return W.make(W.small_spec("na_p", B=3, N=8, paged=True, prefix=("loguniform", 40, 700),
                               tree=("chain",)))


@pytest.mark.parametrize("kind", ["tiny_fp32", "bf16_contiguous", "bf16_paged", "fp8_cache"])
def test_noalloc_matches_workspace_entry_point(kind):
    wl = _workload(kind)
    op = kdtv.for_workload(wl, "cuda")
    ref = op().clone()
    assert op.status() == 0
    ref = ref.double().cpu().numpy()
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for _ in range(2):                        # the shared scratch keeps the last call's data
        out = torch.full(op.out.shape, float("nan"), dtype=torch.float32, device="cuda")
        status.fill_(12345)
        rc = _noalloc(op, out, status)
        assert kdtv.STATUS[rc] == "KDTV_OK"
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.double().cpu().numpy()
        assert np.isfinite(got).all()
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("fault", ["bad_tree", "bad_page"])
def test_noalloc_reports_device_errors(fault):
    """A malformed tree or an out-of-range page id, made on the host, reaches the
    caller through status_out; the next good call reports KDTV_OK again."""
    wl = W.make(W.small_spec("na_err", B=2, N=8, paged=True, prefix=("fixed", 100),
                             tree=("chain",)))
    op = kdtv.for_workload(wl, "cuda")
    good = op().clone()
    assert op.status() == 0
    bad = {k: v.clone() for k, v in op.t.items()}
    if fault == "bad_tree":
        bad["parent"][1, 5] = 7                     # a parent after its child
        want = "KDTV_ERR_BAD_TREE"
    else:
        bad["page_table"][0, 1] = wl.num_pages + 5   # a page id past the pool
        want = "KDTV_ERR_BAD_PAGE"
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(op.out)
    saved, op.t = op.t, bad
    rc = _noalloc(op, out, status)
    op.t = saved
    assert kdtv.STATUS[rc] == "KDTV_OK"
    torch.cuda.synchronize()
    assert kdtv.STATUS[int(status.item())] == want
    status.fill_(12345)
    rc = _noalloc(op, out, status)
    assert kdtv.STATUS[rc] == "KDTV_OK"
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out, good)


def test_noalloc_refuses_oversized_call():
    spec = W.small_spec("na_big", B=8, N=128, prefix=("fixed", 8192))
    d = kdtv.make_dims(spec, dtype="bf16", t_stride=8320)
    assert kdtv.workspace_size(d) > 64 << 20
    fake = 256
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = kdtv.lib().kdtv_verify_attn_noalloc(ctypes.byref(d), fake, fake, fake, fake, fake,
                                             fake, fake, fake, None, fake, status.data_ptr(),
                                             None)
    assert kdtv.STATUS[rc] == "KDTV_ERR_UNSUPPORTED"
