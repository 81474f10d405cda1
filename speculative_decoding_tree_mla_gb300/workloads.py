"""Seeded synthetic inputs for tree-verify MLA attention.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can consume its
output.  Every tensor comes from its own numpy PCG64 stream, spawned from the
workload seed in a fixed order, so any one tensor can be regenerated alone.

Workloads (shapes from the Kimi-K2 MLA layout and the toy model printed on
"The Moment of Proof: Running the Native DDTree Speculative Decoding
Engine", section "The Message Itself": 4 heads, kv_lora 64, vocab 512):

  tiny         fp32, B=1, H=4,  d_nope=32,  d_rope=16, d_v=32,  d_c=64,
               prefix 32, 16 nodes, parent window [0, i-1], depth <= 8
  kimi_single  bf16, B=1, H=64, d_nope=128, d_rope=64, d_v=128, d_c=512,
               prefix 4096, 64 nodes, window [i-8, i-1], depth <= 8
  batched      bf16, B=8, Kimi heads, prefix ~ U{2048..8192}, 32 nodes,
               window [i-8, i-1], depth <= 8
  long         bf16, B=1, Kimi heads, prefix 65536, 128 nodes,
               window [i-16, i-1], depth <= 12
  paged        bf16, B=64, Kimi heads, prefix log-uniform in [1024, 32768],
               chain of 8 nodes, 64-token pages placed by a seeded permutation

Value distributions: q_nope, q_rope, c_kv, k_rope ~ N(0, 1); W_UK, W_UV ~
N(0, std = 1/sqrt(d_c)); rounded to bf16 for the bf16 workloads.  The tree
nodes' own latent rows are appended at positions L_b .. L_b+N-1.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BASE_SEED = 20261202
PAGE_SIZE = 64

# Order of the per-tensor streams (never reorder: stored seeds depend on it).
_STREAMS = ("q_nope", "q_rope", "W_UK", "W_UV", "c_kv", "k_rope", "tree",
            "prefix_len", "pages", "W_lm")


@dataclass(frozen=True)
class Spec:
    name: str
    index: int                 # position in the workload list; seed = BASE_SEED + index
    B: int
    N: int
    H: int
    d_nope: int
    d_rope: int
    d_v: int
    d_c: int
    dtype: str                 # "f32", "bf16" or "fp8kv" (bf16 q / weights, FP8 E4M3 cache)
    prefix: tuple              # ("fixed", L) | ("uniform", lo, hi) | ("loguniform", lo, hi)
    tree: tuple                # ("window", w or None, depth_cap) | ("chain",)
    paged: bool = False
    vocab: int = 4096

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_nope + self.d_rope)

    @property
    def seed(self) -> int:
        return BASE_SEED + self.index


KIMI = dict(H=64, d_nope=128, d_rope=64, d_v=128, d_c=512)

SPECS = {
    "tiny": Spec("tiny", 0, B=1, N=16, H=4, d_nope=32, d_rope=16, d_v=32, d_c=64,
                 dtype="f32", prefix=("fixed", 32), tree=("window", None, 8),
                 vocab=512),
    "kimi_single": Spec("kimi_single", 1, B=1, N=64, dtype="bf16",
                        prefix=("fixed", 4096), tree=("window", 8, 8), **KIMI),
    "batched": Spec("batched", 2, B=8, N=32, dtype="bf16",
                    prefix=("uniform", 2048, 8192), tree=("window", 8, 8), **KIMI),
    "long": Spec("long", 3, B=1, N=128, dtype="bf16",
                 prefix=("fixed", 65536), tree=("window", 16, 12), **KIMI),
    "paged": Spec("paged", 4, B=64, N=8, dtype="bf16",
                  prefix=("loguniform", 1024, 32768), tree=("chain",),
                  paged=True, **KIMI),
}


def _streams(seed):
    children = np.random.SeedSequence(seed).spawn(len(_STREAMS))
    return {name: np.random.Generator(np.random.PCG64(c))
            for name, c in zip(_STREAMS, children)}


def random_tree(rng, N, window=None, depth_cap=None):
    """parent[] of a random draft tree in topological order.

    parent[0] = -1; node i > 0 draws its parent uniformly among the window
    candidates j in [max(0, i - window), i - 1] (all j < i when window is None)
    whose depth is below the cap (the root has depth 1).  If no window
    candidate qualifies it draws among all earlier nodes below the cap; the
    root always qualifies.
    """
    parent = np.full(N, -1, dtype=np.int32)
    depth = np.zeros(N, dtype=np.int64)
    if N == 0:
        return parent
    depth[0] = 1
    for i in range(1, N):
        lo = 0 if window is None else max(0, i - window)
        cand = [j for j in range(lo, i) if depth_cap is None or depth[j] < depth_cap]
        if not cand:
            cand = [j for j in range(i) if depth_cap is None or depth[j] < depth_cap]
        j = int(cand[int(rng.integers(len(cand)))])
        parent[i] = j
        depth[i] = depth[j] + 1
    return parent


def chain_tree(N):
    return np.arange(-1, N - 1, dtype=np.int32)


def star_tree(N):
    p = np.zeros(N, dtype=np.int32)
    if N:
        p[0] = -1
    return p


def tree_depths(parent):
    d = np.zeros(len(parent), dtype=np.int64)
    for i, p in enumerate(parent):
        d[i] = 1 if p < 0 else d[p] + 1
    return d


@dataclass
class Workload:
    """One seeded problem instance.

    ``t`` holds the tensors in the CUDA path's storage dtypes (CPU; move them
    with ``to(device)``); ``f32`` holds the same values widened exactly to
    float32 numpy arrays for the oracle.
    """
    spec: Spec
    t: dict = field(default_factory=dict)
    f32: dict = field(default_factory=dict)
    t_stride: int = 0
    max_pages: int = 0
    num_pages: int = 0
    kv_scale: float = 0.0        # fp8kv: cache value = fp8 * kv_scale (0: not used)

    @property
    def page_size(self) -> int:
        return PAGE_SIZE if self.spec.paged else 0


def _normal(rng, shape, std=1.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def _as_dtype(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype in ("bf16", "fp8kv"):
        t = t.to(torch.bfloat16)
        return t, t.float().numpy()
    return t, x


# ---- OCP FP8 E4M3 (storage format of the fp8kv cache) -------------------------------------
# Byte S.EEEE.MMM: exponent bias 7; E = 0 holds subnormals M * 2^-9; E = 15 with
# M = 7 is NaN; there are no infinities, so the largest value is 1.75 * 2^8 = 448.
FP8_KV_SCALE = 0.125           # the fp8kv workloads store x / 0.125 and read fp8 * 0.125


def fp8_e4m3_decode(codes):
    """float32 values of E4M3 byte codes (uint8 array)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return (sign * mag).astype(np.float32)


_E4M3_POS = fp8_e4m3_decode(np.arange(0x7F, dtype=np.uint8))   # codes 0x00 .. 0x7E, increasing


def fp8_e4m3_encode(x):
    """Nearest E4M3 byte code of each float32 (ties to the even code, saturating at
    448), by search over the 127 non-negative finite values."""
    x = np.asarray(x, dtype=np.float32)
    a = np.minimum(np.abs(x), np.float32(448.0))
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    dl, dh = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
    pick_hi = (dh < dl) | ((dh == dl) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)   # -0 for tiny negatives


def _as_fp8_cache(x):
    codes = fp8_e4m3_encode(x / np.float32(FP8_KV_SCALE))
    return torch.from_numpy(codes), fp8_e4m3_decode(codes) * np.float32(FP8_KV_SCALE)


def make(spec, *, parent=None, prefix_len=None, with_lm_head=False,
         seed=None, zero_q=False):
    """Build the workload of ``spec`` (a Spec or a name from SPECS).

    ``parent`` ([B, N]) and ``prefix_len`` ([B]) override the drawn tree /
    prefix lengths; ``seed`` overrides the spec's seed.
    """
    if isinstance(spec, str):
        spec = SPECS[spec]
    rs = _streams(spec.seed if seed is None else seed)
    B, N, H = spec.B, spec.N, spec.H
    wl = Workload(spec=spec)

    # Tree and prefix lengths first: they fix the cache extents.
    if parent is None:
        if spec.tree[0] == "chain":
            parent = np.stack([chain_tree(N) for _ in range(B)])
        else:
            _, window, cap = spec.tree
            parent = np.stack([random_tree(rs["tree"], N, window, cap)
                               for _ in range(B)])
    parent = np.asarray(parent, dtype=np.int32).reshape(B, N)
    if prefix_len is None:
        kind = spec.prefix[0]
        if kind == "fixed":
            prefix_len = np.full(B, spec.prefix[1], dtype=np.int64)
        elif kind == "uniform":
            prefix_len = rs["prefix_len"].integers(spec.prefix[1], spec.prefix[2] + 1,
                                                   size=B)
        else:
            lo, hi = math.log(spec.prefix[1]), math.log(spec.prefix[2])
            prefix_len = np.rint(np.exp(rs["prefix_len"].uniform(lo, hi, size=B)))
    prefix_len = np.asarray(prefix_len, dtype=np.int64).reshape(B)
    T = prefix_len + N                       # rows per request incl. tree nodes

    q_nope = _normal(rs["q_nope"], (B, N, H, spec.d_nope))
    q_rope = _normal(rs["q_rope"], (B, N, H, spec.d_rope))
    if zero_q:
        q_nope[:] = 0
        q_rope[:] = 0
    w_std = 1.0 / math.sqrt(spec.d_c)
    W_UK = _normal(rs["W_UK"], (H, spec.d_nope, spec.d_c), w_std)
    W_UV = _normal(rs["W_UV"], (H, spec.d_v, spec.d_c), w_std)

    if spec.paged:
        pages_per_req = -(-T // PAGE_SIZE)
        num_pages = int(pages_per_req.sum())
        perm = rs["pages"].permutation(num_pages).astype(np.int32)
        max_pages = int(pages_per_req.max()) if B else 0
        page_table = np.full((B, max(max_pages, 1)), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            k = int(pages_per_req[b])
            page_table[b, :k] = perm[off:off + k]
            off += k
        c_kv = _normal(rs["c_kv"], (num_pages, PAGE_SIZE, spec.d_c))
        k_rope = _normal(rs["k_rope"], (num_pages, PAGE_SIZE, spec.d_rope))
        wl.max_pages, wl.num_pages = page_table.shape[1], num_pages
    else:
        t_stride = int(-(-int(T.max()) // 64) * 64) if B else 64
        c_kv = _normal(rs["c_kv"], (B, t_stride, spec.d_c))
        k_rope = _normal(rs["k_rope"], (B, t_stride, spec.d_rope))
        page_table = None
        wl.t_stride = t_stride

    for name, arr in (("q_nope", q_nope), ("q_rope", q_rope), ("W_UK", W_UK),
                      ("W_UV", W_UV), ("c_kv", c_kv), ("k_rope", k_rope)):
        if spec.dtype == "fp8kv" and name in ("c_kv", "k_rope"):
            wl.t[name], wl.f32[name] = _as_fp8_cache(arr)
        else:
            wl.t[name], wl.f32[name] = _as_dtype(arr, spec.dtype)
    if spec.dtype == "fp8kv":
        wl.kv_scale = FP8_KV_SCALE
    wl.t["parent"] = torch.from_numpy(parent.copy())
    wl.t["prefix_len"] = torch.from_numpy(prefix_len.astype(np.int32))
    wl.f32["parent"], wl.f32["prefix_len"] = parent, prefix_len
    if page_table is not None:
        wl.t["page_table"] = torch.from_numpy(page_table)
        wl.f32["page_table"] = page_table
    if with_lm_head:
        wl.f32["W_lm"] = rs["W_lm"].standard_normal(
            (H * spec.d_v, spec.vocab)) / math.sqrt(H * spec.d_v)
    return wl


def small_spec(name, *, B, N, H=64, dtype="bf16", paged=False, prefix=("fixed", 256),
               tree=("window", 8, 8), index=100, d_nope=128, d_rope=64, d_v=128,
               d_c=512):
    """A reduced-size spec with the Kimi head layout, for parity sweeps."""
    return Spec(name, index, B=B, N=N, H=H, d_nope=d_nope, d_rope=d_rope, d_v=d_v,
                d_c=d_c, dtype=dtype, prefix=prefix, tree=tree, paged=paged)
