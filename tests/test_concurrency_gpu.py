"""Calls from several host threads at once, each on its own stream and
workspace, in a fresh process (so that the library's first-use lookups — the
tensor-map encoder, the SM count — happen concurrently too).  Every thread's
outputs must equal, bit for bit, the same calls made one after another.

The calls go through ctypes, which releases the interpreter lock, so the
threads really do enter the library together.
"""

import os
import subprocess
import sys
import textwrap

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_mla_gb300 import build
    build.build()


CHILD = textwrap.dedent("""
    import sys, threading
    sys.path.insert(0, sys.argv[1])
    import torch
    from speculative_decoding_tree_mla_gb300 import kdtv, workloads as W
    specs = [W.small_spec("thr0", B=2, N=16, prefix=("uniform", 300, 900)),
             W.small_spec("thr1", B=3, N=8, paged=True, prefix=("loguniform", 40, 900), tree=("chain",)),
             W.small_spec("thr2", B=1, N=64, prefix=("fixed", 1500)),
             W.small_spec("thr3", B=4, N=12, H=16, prefix=("uniform", 10, 600))]
    wls = [W.make(s) for s in specs]
    torch.cuda.init()
    ops = [kdtv.for_workload(wl, "cuda") for wl in wls]
    streams = [torch.cuda.Stream() for _ in ops]
    outs = [None] * len(ops)
    errs = []
    barrier = threading.Barrier(len(ops))
    def work(j):
        try:
            barrier.wait()
            for _ in range(6):
                ops[j](stream=streams[j])
            streams[j].synchronize()
            outs[j] = (ops[j].out.clone(), ops[j].status(stream=streams[j]))
        except Exception as e:
            errs.append(repr(e))
    ts = [threading.Thread(target=work, args=(j,)) for j in range(len(ops))]
    for t in ts: t.start()
    for t in ts: t.join()
    assert not errs, errs
    for j, op in enumerate(ops):        # the same calls, one after another
        op.out.zero_()
        op()
        torch.cuda.synchronize()
        got, st = outs[j]
        assert st == 0 and op.status() == 0, (j, st)
        assert torch.equal(got, op.out), j
    print("CONCURRENT_OK")
""")


def test_concurrent_calls_from_threads():
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0 and "CONCURRENT_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
