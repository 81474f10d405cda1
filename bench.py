#!/usr/bin/env python3
"""Benchmark of kdtv_verify_attn (tree-verify MLA-absorb attention).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl ours|reference] [--path tc|simt]

One step = one kdtv_verify_attn call (absorb, tree-masked attention,
split-KV combine, W_UV up-projection) on a seeded synthetic workload whose
inputs are already resident in HBM; L2 is flushed (a 256 MiB write) before
every timed call, outside the timed interval.  Prints ONE JSON line.

The headline workload is the largest single-GPU one: the Kimi-K2-shaped
long-context request (64 heads, kv_lora 512, rope 64, prefix 65536,
128-node tree).  The other Kimi-shaped workloads (single request, batched,
paged) are timed in the same run and reported under "workloads", each with
its own roofline.  ``--impl reference`` times the fp64 CPU oracle on the
headline workload instead (one sampled node per step, scaled to the whole
call).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-verify MLA attn µs/call; HBM TB/s + TC TFLOP/s as % of roofline"
UNIT = "us/call"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM bytes (read + write) of one attention-kernel launch, from an ncu
# capture of that workload, keyed by the SHA-256 of the kernel source the
# capture was taken on: a changed kernel reports null until it is captured
# again.
ATTN_TRAFFIC = {
    "long": ("b5d5562c0f989a7f2c3e99e4c95f34af435c9a3f864d73e4408a0c563882066b", 939578880 + 10908928),
    "kimi_single": ("b5d5562c0f989a7f2c3e99e4c95f34af435c9a3f864d73e4408a0c563882066b", 9601024 + 0),
    "batched": ("b5d5562c0f989a7f2c3e99e4c95f34af435c9a3f864d73e4408a0c563882066b", 109379328 + 12590080),
    "paged": ("b5d5562c0f989a7f2c3e99e4c95f34af435c9a3f864d73e4408a0c563882066b", 710946048 + 33332224),
}


def attn_traffic(workload):
    rec = ATTN_TRAFFIC.get(workload)
    if rec is None:
        return None
    import hashlib
    src = os.path.join(ROOT, "speculative_decoding_tree_mla_gb300", "csrc", "kdtv_tc.cu")
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()
    return rec[1] if digest == rec[0] else None


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="long")
    ap.add_argument("--extra", default="kimi_single,batched,paged",
                    help="other workloads timed in the same run ('' for none)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="tc", choices=["tc", "simt"])
    ap.add_argument("--cache", default="native", choices=["native", "fp8"],
                    help="fp8: the same workload with an FP8 E4M3 latent cache")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-only", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def work(wl):
    """Algorithmic work of one call: visible-key FLOPs, latent-cache bytes,
    all compulsory bytes."""
    import numpy as np
    from speculative_decoding_tree_mla_gb300 import workloads as W
    s = wl.spec
    f = wl.f32
    attn = 0
    for b in range(s.B):
        depth = W.tree_depths(f["parent"][b])
        attn += s.H * int((f["prefix_len"][b] + depth).sum()) * (
            2 * (s.d_c + s.d_rope) + 2 * s.d_c)
    absorb = 2 * s.B * s.N * s.H * s.d_nope * s.d_c
    uproj = 2 * s.B * s.N * s.H * s.d_c * s.d_v
    esz = 2 if s.dtype in ("bf16", "fp8kv") else 4
    T = (np.asarray(f["prefix_len"]) + s.N).sum()
    cache_bytes = int(T) * (s.d_c + s.d_rope) * (1 if s.dtype == "fp8kv" else esz)
    weights = s.H * s.d_c * (s.d_nope + s.d_v) * esz
    q = s.B * s.N * s.H * (s.d_nope + s.d_rope) * esz
    out = s.B * s.N * s.H * s.d_v * 4
    return {"attn_flops": attn, "total_flops": attn + absorb + uproj,
            "cache_bytes": cache_bytes, "all_bytes": cache_bytes + weights + q + out}


class Clocks:
    """nvidia-smi sampler run around the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}",
                                       f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        time.sleep(0.3)

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        mx = max(num(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(num(r[3]) for r in rows)}


def dist_init(args):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def allmax(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# -- the oracle on the host (reference arm and cpu_baseline leg) ---------------
def oracle_time(wl, seconds, max_nodes=None, seed=0):
    """Times the oracle on a bounded node sample (nodes in a random order drawn
    from `seed`); returns (us per whole call, sample description, threads,
    seconds per node)."""
    import numpy as np
    import oracle
    f = wl.f32
    s = wl.spec
    nodes = [(b, i) for b in range(s.B) for i in range(s.N)]
    rng = np.random.default_rng(seed)
    order = rng.permutation(len(nodes))
    done = 0
    t0 = time.perf_counter()
    while (time.perf_counter() - t0 < seconds and done < len(nodes)
           and (max_nodes is None or done < max_nodes)):
        b, i = nodes[order[done]]
        oracle.verify_attn_node(f["q_nope"], f["q_rope"], f["W_UK"], f["W_UV"], f["c_kv"],
                                f["k_rope"], f["parent"], f["prefix_len"], b, i, s.scale,
                                page_table=f.get("page_table"), page_size=wl.page_size)
        done += 1
    dt = time.perf_counter() - t0
    us_call = dt / done * len(nodes) * 1e6
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS") or os.cpu_count() or 1)
    return (us_call, f"{done} of {len(nodes)} (request, node) pairs in a random order, "
            f"timed and scaled to all {len(nodes)}", threads, dt / done)


def cpu_baseline_single_thread(args):
    """The same oracle timing with one BLAS thread, in a child process (the
    thread count is fixed when numpy loads)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-only", "--config", args.config,
           "--cpu-seconds", str(args.cpu_seconds)]
    if args.cache == "fp8":
        cmd += ["--cache", "fp8"]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:   # the GPU numbers stand without it
        return {"error": f"single-thread oracle timing failed: {e}"}


def run_reference(args, wl, rank, ws):
    """The reference arm: the oracle as it stands, on the host cores.  A step
    is one (request, node) pair drawn at random for that step; `value` scales
    its time to the whole call, `ms_per_step` is the measured step."""
    if rank != 0:
        return
    per_step, step_s = [], []
    threads = 1
    for k in range(args.warmup + args.steps):
        us, sample, threads, node_s = oracle_time(wl, seconds=1e9, max_nodes=1, seed=k)
        if k >= args.warmup:
            per_step.append(us)
            step_s.append(node_s)
    v = statistics.mean(per_step)
    cfg = config_dict(wl)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(step_s) * 1000.0,
        "step": "one (request, node) pair of the workload; value = its time x the pairs of a call",
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "each step: one (request, node) pair of the workload, "
                                   "drawn at random per step, scaled to all pairs"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def loop_steps(wl, dev, reps=200):
    """Device time of the loop steps around the verify attention on this
    workload's shapes: best-first tree build (K=8 proposals per depth), greedy
    tree accept, in-place KV compaction of the accepted path."""
    import numpy as np
    import torch
    from speculative_decoding_tree_mla_gb300 import kdtv
    s = wl.spec
    rng = np.random.default_rng(s.seed)
    D, K = 16, 8
    lp = np.sort(-rng.exponential(1.0, size=(s.B, D, K)).astype(np.float32), axis=2)[:, :, ::-1]
    lp = torch.from_numpy(np.ascontiguousarray(lp)).to(dev)
    tok = torch.from_numpy(rng.integers(0, 50000, size=(s.B, D, K)).astype(np.int32)).to(dev)
    root = torch.zeros(s.B, dtype=torch.int32, device=dev)
    parent = wl.t["parent"].to(dev)
    draft = torch.from_numpy(rng.integers(0, 4, size=(s.B, s.N)).astype(np.int32)).to(dev)
    argmax = torch.from_numpy(rng.integers(0, 4, size=(s.B, s.N)).astype(np.int32)).to(dev)
    path, plen, _ = kdtv.tree_accept(parent, draft, argmax)
    d = kdtv.make_dims(s, dtype=s.dtype, page_size=wl.page_size, t_stride=wl.t_stride,
                       max_pages=wl.max_pages, num_pages=wl.num_pages)
    c = wl.t["c_kv"].to(dev)
    k = wl.t["k_rope"].to(dev)
    pl = wl.t["prefix_len"].to(dev)
    pt = wl.t["page_table"].to(dev) if wl.page_size else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    fns = {
        "tree_build_us": lambda: kdtv.tree_build(lp, tok, root, s.N),
        "tree_accept_us": lambda: kdtv.tree_accept(parent, draft, argmax),
        "compact_kv_us": lambda: kdtv.compact_kv(d, c, k, pl, path, plen, pt, status),
    }
    res = {}
    inner = 20
    graphs = True
    for name, fn in fns.items():
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        # Replay a CUDA graph of `inner` calls, so that the host-side cost of a
        # Python call (output allocation, ctypes) is not what gets timed.
        g = None
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                fn()
            torch.cuda.current_stream().wait_stream(side)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(inner):
                    fn()
            g.replay()
            torch.cuda.synchronize()
        except Exception:
            g = None
            graphs = False
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        outer = max(1, reps // inner)
        e0.record()
        if g is not None:
            for _ in range(outer):
                g.replay()
            calls = outer * inner
        else:
            for _ in range(reps):
                fn()
            calls = reps
        e1.record()
        e1.synchronize()
        res[name] = e0.elapsed_time(e1) * 1000.0 / calls
    res["shapes"] = f"B={s.B} N={s.N} tree_build D={D} K={K}"
    res["timing"] = ("CUDA graph of 20 calls, replayed" if graphs
                     else "back-to-back Python calls")
    return res


def config_dict(wl):
    s = wl.spec
    f = wl.f32
    return {"workload": s.name + ("+fp8cache" if s.dtype == "fp8kv" else ""),
            "batch": s.B, "tree_nodes": s.N, "heads": s.H,
            "d_nope": s.d_nope, "d_rope": s.d_rope, "d_v": s.d_v, "kv_lora": s.d_c,
            "prefix_len_mean": float(sum(int(x) for x in f["prefix_len"]) / s.B),
            "paged": s.paged, "seed": s.seed, "l2": "flushed (256 MiB write) before every call"}


def make_spec(name, cache):
    from speculative_decoding_tree_mla_gb300 import workloads as W
    spec = W.SPECS[name]
    if cache == "fp8":
        import dataclasses
        spec = dataclasses.replace(spec, dtype="fp8kv")
    return spec


def measure(wl, dev, flags, K, Wm, ws, flush, traffic_key=None, clocks=None):
    """Device-timed calls of one workload with inputs resident in HBM: K calls
    each bracketed by events on the call's stream (L2 flushed before each,
    outside the events), then a pass with the library's phase events for the
    attention kernel's own duration, then K back-to-back calls without the
    flush.  Returns the workload's numbers and the op."""
    import torch
    from speculative_decoding_tree_mla_gb300 import kdtv
    op = kdtv.for_workload(wl, dev, flags=flags)
    stream = torch.cuda.current_stream(dev)
    for _ in range(Wm):
        flush.zero_()
        op()
    torch.cuda.synchronize()
    if op.status() != 0:
        raise SystemExit(f"{wl.spec.name}: device status {kdtv.STATUS[op.status()]}")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    if clocks:
        clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        op()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop() if clocks else None
    st = op.status()
    if st != 0:
        raise SystemExit(f"{wl.spec.name}: device status {kdtv.STATUS[st]}")
    call_ms = [a.elapsed_time(b) for a, b in ev]

    # Phase pass: events recorded by the library between its kernels give the
    # attention kernel's own duration (the roofline's denominator).
    K_ph = min(K, 200)
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K_ph)]
    for k in range(K_ph):
        flush.zero_()
        op.set_phase_events(pev[k])
        op()
    torch.cuda.synchronize()
    op.set_phase_events(None)
    phase_ms = [[e[j].elapsed_time(e[j + 1]) for e in pev] for j in range(4)]

    # Warm L2: the same call back to back with no flush between calls.
    K_w = min(K, 500)
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K_w)]
    for k in range(K_w):
        wev[k][0].record(stream)
        op()
        wev[k][1].record(stream)
    torch.cuda.synchronize()

    mean_ms = allmax(statistics.mean(call_ms), ws)
    wk = work(wl)
    pk, pk_kind = peaks()
    attn_ms = statistics.mean(phase_ms[1])
    tflops = wk["attn_flops"] / (attn_ms * 1e-3) / 1e12
    peak_tc = pk["bf16_tflops"]
    us_replica = mean_ms * 1000.0
    roof_us = max(wk["cache_bytes"] / (pk["hbm_gbs"] * 1e9),
                  wk["total_flops"] / (peak_tc * 1e12)) * 1e6
    res = {
        "us_per_call_per_replica": us_replica,
        "us_call": us_replica / ws,       # whole job: ws replicas run side by side
        "mean_ms": mean_ms,
        "p50_us": statistics.median(call_ms) * 1000.0,
        "warm_l2_us": allmax(statistics.mean(a.elapsed_time(b) for a, b in wev), ws) * 1000.0,
        "phases": {n: statistics.mean(x) * 1000.0 for n, x in
                   zip(["absorb_us", "attention_us", "combine_us", "up_proj_us"], phase_ms)},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak_tc, "unit": "TFLOP/s",
                     "frac": tflops / peak_tc,
                     "traffic": attn_traffic(traffic_key) if traffic_key else None,
                     "kernel": "attention (tree-masked scores, online softmax, P.c_kv)",
                     "attention_us": attn_ms * 1000.0,
                     "algorithmic_flops": wk["attn_flops"],
                     "peak_source": f"{pk_kind} bf16_tflops (burst)"},
        "call_roofline": {"t_roof_us": roof_us, "frac": roof_us / us_replica,
                          "tflops": wk["total_flops"] / (us_replica * 1e-6) / 1e12,
                          "cache_tbs": wk["cache_bytes"] / (us_replica * 1e-6) / 1e12,
                          "flops": wk["total_flops"], "cache_bytes": wk["cache_bytes"],
                          "all_bytes": wk["all_bytes"]},
        "steps": K,
        "wall_s_timed_region": t_wall,
        "clocks": clk,
    }
    return res, op


def e2e_time(wl, op, dev, K, Wm, ws, flush):
    """End to end through the public call: every step copies the call's inputs
    from pinned host memory and reads the output back, inside the events.

    Every input of the call lives in one pinned host block, mirrored by one
    device block with the same 256-byte aligned layout (the kernels read views
    of it), so a step moves its inputs with a single DMA."""
    import torch
    stream = torch.cuda.current_stream(dev)
    names = ["q_nope", "q_rope", "W_UK", "W_UV", "c_kv", "k_rope", "parent", "prefix_len"]
    if wl.page_size:
        names.append("page_table")
    src = {n: wl.t[n].contiguous() for n in names}
    offs, total = {}, 0
    for n in names:
        total = (total + 255) // 256 * 256
        offs[n] = total
        total += src[n].numel() * src[n].element_size()
    host_blk = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_blk = torch.empty(total, dtype=torch.uint8, device=dev)
    saved = dict(op.t)
    for n in names:
        nb = src[n].numel() * src[n].element_size()
        host_blk[offs[n]:offs[n] + nb].copy_(src[n].view(-1).view(torch.uint8))
        op.t[n] = dev_blk[offs[n]:offs[n] + nb].view(src[n].dtype).view(src[n].shape)
    out_before = op.out.clone()
    out_host = torch.empty(op.out.shape, dtype=op.out.dtype).pin_memory()
    e2e_ms = []
    for k in range(Wm + K):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dev_blk.copy_(host_blk, non_blocking=True)
        op()
        out_host.copy_(op.out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if k >= Wm:
            e2e_ms.append(e0.elapsed_time(e1))
    # the block-backed calls compute the same output as the resident inputs did
    assert op.status() == 0 and torch.equal(op.out, out_before)
    op.t.update(saved)
    us = allmax(statistics.mean(e2e_ms), ws) * 1000.0 / ws
    return {"value": us, "unit": UNIT, "h2d_bytes_per_step": total,
            "d2h_bytes_per_step": out_host.numel() * out_host.element_size()}


def main():
    args = parse()
    if args.impl == "reference":
        os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))
    import numpy as np  # noqa: F401
    from speculative_decoding_tree_mla_gb300 import workloads as W
    spec = make_spec(args.config, args.cache)
    if args.cpu_only:
        v, sample, threads, _ = oracle_time(W.make(spec), args.cpu_seconds)
        print(json.dumps({"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                          "sample": sample}), flush=True)
        return
    if args.impl == "reference":
        # host-only: no process group; ranks other than 0 exit without work
        rank = int(os.environ.get("RANK", "0"))
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        if rank == 0:
            run_reference(args, W.make(spec), rank, ws)
        return
    import torch
    rank, ws, local = dist_init(args)
    wl = W.make(spec)

    from speculative_decoding_tree_mla_gb300 import build, kdtv
    if rank == 0:
        build.build()
    barrier(ws)
    dev = torch.device("cuda", local)
    flags = kdtv.KDTV_FLAG_SIMT if args.path == "simt" else 0
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    K, Wm = args.steps, max(3, args.warmup)
    native = not flags and args.cache == "native"

    head, op = measure(wl, dev, flags, K, Wm, ws, flush,
                       traffic_key=args.config if native else None, clocks=Clocks(local))
    e2e = e2e_time(wl, op, dev, min(K, 200), Wm, ws, flush)
    launches = op.launches()
    del op

    extras = {}
    for name in [x for x in args.extra.split(",") if x and x != args.config]:
        wlx = W.make(make_spec(name, args.cache))
        r, opx = measure(wlx, dev, flags, min(K, 300), Wm, ws, flush,
                         traffic_key=name if native else None)
        r.pop("clocks", None)
        r["config"] = config_dict(wlx)
        extras[name] = r
        del opx, wlx
        torch.cuda.empty_cache()

    steps_us = loop_steps(W.make(make_spec("kimi_single", "native")), dev) if rank == 0 else None

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, sample, threads, _ = oracle_time(wl, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
               "single_thread": cpu_baseline_single_thread(args)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["us_call"], "unit": UNIT, "n_gpus": ws, "steps": K,
            "warmup": Wm, "ms_per_step": head["mean_ms"], "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if (wl.spec.dtype == "f32" or flags) else "bf16",
            "data": "synthetic", "config": config_dict(wl),
            "roofline": head["roofline"],
            "call_roofline": head["call_roofline"],
            "phases": head["phases"],
            "p50_us": head["p50_us"],
            "warm_l2_us": head["warm_l2_us"],
            "us_per_call_per_replica": head["us_per_call_per_replica"],
            "value_note": ("value = mean device time of one call on one GPU divided by the "
                           "number of GPUs (each GPU runs its own replica of the call)"),
            "e2e": e2e,
            "gpu_launches": launches * K,
            "path": args.path,
            "clocks": head["clocks"],
            "wall_s_timed_region": head["wall_s_timed_region"],
            "workloads": extras,
            "loop_steps": steps_us,
        }
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
