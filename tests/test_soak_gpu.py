"""Back-to-back calls on the full-size workloads: thousands of launches of the
persistent attention kernel and its neighbours, with every mbarrier phase,
the programmatic-launch overlap between calls' kernels and the status words
exercised many times.  The status stays OK and the output stays bit-identical
to the first call's.
"""

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


@pytest.mark.parametrize("name,calls", [("kimi_single", 3000), ("batched", 600),
                                        ("paged", 300), ("long", 120)])
def test_back_to_back_calls(name, calls):
    wl = W.make(name)
    op = kdtv.for_workload(wl, "cuda")
    if kdtv.workspace_size(op.dims) == 0:
        pytest.skip("tensor-core path not compiled in")
    first = op().clone()
    torch.cuda.synchronize()
    assert op.status() == 0
    for k in range(calls):
        op()
        if k % 500 == 499:            # a status check now and then: it synchronises
            assert op.status() == 0, k
    torch.cuda.synchronize()
    assert op.status() == 0
    assert torch.equal(op.out, first)
