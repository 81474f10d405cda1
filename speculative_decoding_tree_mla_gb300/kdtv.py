"""ctypes binding of libkdtv.so (include/kdtv.h), plus a torch-side caller.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  ``torch`` supplies device memory and the stream.  There is no CPU
fallback: if the library was not built, every call raises.
"""

from __future__ import annotations

import ctypes
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkdtv.so")

KDTV_F32, KDTV_BF16, KDTV_BF16_FP8KV = 0, 1, 2
KDTV_FLAG_SIMT = 0x1
KDTV_FLAG_SIMT_PROJ = 0x2
KDTV_FLAG_TEST_STALL = 0x100
STATUS = {0: "KDTV_OK", 1: "KDTV_ERR_INVALID_ARG", 2: "KDTV_ERR_UNSUPPORTED",
          3: "KDTV_ERR_CUDA", 4: "KDTV_ERR_BAD_TREE", 5: "KDTV_ERR_DEVICE_TIMEOUT",
          6: "KDTV_ERR_BAD_PREFIX", 7: "KDTV_ERR_BAD_PAGE"}
STATUS_CODE = {v: k for k, v in STATUS.items()}

# Every symbol include/kdtv.h declares (checked by the CPU tests).
EXPORTS = ("kdtv_workspace_size", "kdtv_verify_attn", "kdtv_get_device_status",
           "kdtv_strerror", "kdtv_launches_per_call", "kdtv_tree_accept", "kdtv_compact_kv",
           "kdtv_tree_build", "kdtv_verify_attn_noalloc")


class KdtvDims(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("N", ctypes.c_int32), ("H", ctypes.c_int32),
        ("d_nope", ctypes.c_int32), ("d_rope", ctypes.c_int32),
        ("d_v", ctypes.c_int32), ("d_c", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("t_stride", ctypes.c_int32), ("max_pages", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("scale", ctypes.c_float),
        ("flags", ctypes.c_uint32), ("kv_chunk", ctypes.c_int32),
        ("kv_scale", ctypes.c_float), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t), ("phase_events", ctypes.c_void_p),
    ]


class KdtvError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


_lib = None


def lib():
    """Loads libkdtv.so once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m speculative_decoding_tree_mla_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(KdtvDims)
        vp = ctypes.c_void_p
        L.kdtv_workspace_size.argtypes = [P]
        L.kdtv_workspace_size.restype = ctypes.c_size_t
        L.kdtv_verify_attn.argtypes = [P] + [vp] * 10 + [vp]
        L.kdtv_verify_attn.restype = ctypes.c_int
        L.kdtv_get_device_status.argtypes = [P, vp]
        L.kdtv_get_device_status.restype = ctypes.c_int
        L.kdtv_strerror.argtypes = [ctypes.c_int]
        L.kdtv_strerror.restype = ctypes.c_char_p
        L.kdtv_launches_per_call.argtypes = [P]
        L.kdtv_launches_per_call.restype = ctypes.c_int
        i32 = ctypes.c_int
        L.kdtv_tree_accept.argtypes = [i32, i32] + [vp] * 6 + [vp]
        L.kdtv_tree_accept.restype = ctypes.c_int
        L.kdtv_compact_kv.argtypes = [P] + [vp] * 7 + [vp]
        L.kdtv_compact_kv.restype = ctypes.c_int
        L.kdtv_tree_build.argtypes = [i32, i32, i32, i32] + [vp] * 8 + [vp]
        L.kdtv_tree_build.restype = ctypes.c_int
        L.kdtv_verify_attn_noalloc.argtypes = [P] + [vp] * 11 + [vp]
        L.kdtv_verify_attn_noalloc.restype = ctypes.c_int
        _lib = L
    return _lib


def strerror(code):
    return lib().kdtv_strerror(int(code)).decode()


DTYPE_CODE = {"f32": KDTV_F32, "bf16": KDTV_BF16, "fp8kv": KDTV_BF16_FP8KV}


def make_dims(spec_or_shape, *, dtype, page_size=0, t_stride=0, max_pages=0,
              num_pages=0, scale=0.0, flags=0, kv_chunk=0, kv_scale=0.0):
    s = spec_or_shape
    d = KdtvDims()
    d.B, d.N, d.H = s.B, s.N, s.H
    d.d_nope, d.d_rope, d.d_v, d.d_c = s.d_nope, s.d_rope, s.d_v, s.d_c
    d.dtype = DTYPE_CODE.get(dtype, dtype if isinstance(dtype, int) else KDTV_F32)
    d.kv_scale = kv_scale
    d.page_size, d.t_stride = page_size, t_stride
    d.max_pages, d.num_pages = max_pages, num_pages
    d.scale, d.flags, d.kv_chunk = scale, flags, kv_chunk
    return d


def workspace_size(dims):
    return int(lib().kdtv_workspace_size(ctypes.byref(dims)))


def launches_per_call(dims):
    return int(lib().kdtv_launches_per_call(ctypes.byref(dims)))


def verify_attn_raw(dims, q_nope, q_rope, W_UK, W_UV, c_kv, k_rope, parent,
                    prefix_len, page_table, out, stream):
    """Direct C-ABI call with integer device pointers; returns the status."""
    return int(lib().kdtv_verify_attn(ctypes.byref(dims), q_nope, q_rope, W_UK, W_UV,
                                      c_kv, k_rope, parent, prefix_len,
                                      page_table or None, out, stream or None))


def get_device_status(dims, stream=0):
    return int(lib().kdtv_get_device_status(ctypes.byref(dims), stream or None))


class VerifyAttn:
    """Torch-side caller: holds the dims, the workspace and the output buffer.

    ``tensors`` maps q_nope, q_rope, W_UK, W_UV, c_kv, k_rope, parent,
    prefix_len and (paged) page_table to contiguous CUDA tensors.
    """

    def __init__(self, spec, tensors, *, t_stride=0, max_pages=0, num_pages=0,
                 page_size=0, flags=0, kv_chunk=0, scale=0.0, kv_scale=0.0):
        import torch
        self.torch = torch
        self.t = tensors
        dev = tensors["c_kv"].device
        self.dims = make_dims(spec, dtype=spec.dtype, page_size=page_size,
                              t_stride=t_stride, max_pages=max_pages,
                              num_pages=num_pages, scale=scale or spec.scale,
                              flags=flags, kv_chunk=kv_chunk, kv_scale=kv_scale)
        nbytes = workspace_size(self.dims)
        if nbytes == 0:
            raise KdtvError(STATUS_CODE["KDTV_ERR_UNSUPPORTED"], "workspace size")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.dims.workspace = self.workspace.data_ptr()
        self.dims.workspace_bytes = nbytes
        self.out = torch.empty((spec.B, spec.N, spec.H, spec.d_v), dtype=torch.float32,
                               device=dev)
        self._ev = None

    def set_phase_events(self, events):
        """events: list of 5 torch.cuda.Event (created with enable_timing)."""
        if events is None:
            self.dims.phase_events = None
            self._ev = None
            return
        for e in events:             # torch creates the CUDA event lazily
            if not e.cuda_event:
                e.record()
        handles = (ctypes.c_void_p * 5)(*[e.cuda_event for e in events])
        if not all(handles):
            raise RuntimeError("phase events could not be created")
        self._ev = handles
        self.dims.phase_events = ctypes.cast(handles, ctypes.c_void_p)

    def __call__(self, stream=None, out=None):
        t = self.t
        s = stream if stream is not None else self.torch.cuda.current_stream()
        o = self.out if out is None else out
        pt = t.get("page_table")
        code = verify_attn_raw(self.dims, t["q_nope"].data_ptr(), t["q_rope"].data_ptr(),
                               t["W_UK"].data_ptr(), t["W_UV"].data_ptr(),
                               t["c_kv"].data_ptr(), t["k_rope"].data_ptr(),
                               t["parent"].data_ptr(), t["prefix_len"].data_ptr(),
                               pt.data_ptr() if pt is not None else 0, o.data_ptr(),
                               s.cuda_stream)
        if code != 0:
            raise KdtvError(code, "kdtv_verify_attn")
        return o

    def status(self, stream=None):
        s = stream if stream is not None else self.torch.cuda.current_stream()
        return get_device_status(self.dims, s.cuda_stream)

    def launches(self):
        return launches_per_call(self.dims)


def for_workload(wl, device="cuda", **kw):
    """VerifyAttn over a ``workloads.Workload`` moved to ``device``."""
    names = ["q_nope", "q_rope", "W_UK", "W_UV", "c_kv", "k_rope", "parent", "prefix_len"]
    if wl.page_size:
        names.append("page_table")
    tens = {n: wl.t[n].to(device).contiguous() for n in names}
    kw.setdefault("kv_scale", wl.kv_scale)
    return VerifyAttn(wl.spec, tens, t_stride=wl.t_stride, max_pages=wl.max_pages,
                      num_pages=wl.num_pages, page_size=wl.page_size, **kw)


def default_scale(d_nope, d_rope):
    return 1.0 / math.sqrt(d_nope + d_rope)


def _p(t):
    return t.data_ptr() if t is not None else None


def _s(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def tree_accept(parent, draft_tok, target_argmax, stream=None):
    """Torch caller of kdtv_tree_accept; returns (path, path_len, bonus)."""
    import torch
    B, N = parent.shape
    dev = parent.device
    path = torch.empty((B, N), dtype=torch.int32, device=dev)
    plen = torch.empty(B, dtype=torch.int32, device=dev)
    bonus = torch.empty(B, dtype=torch.int32, device=dev)
    code = lib().kdtv_tree_accept(B, N, _p(parent), _p(draft_tok), _p(target_argmax),
                                  _p(path), _p(plen), _p(bonus), _s(stream))
    if code:
        raise KdtvError(code, "kdtv_tree_accept")
    return path, plen, bonus


def compact_kv(dims, c_kv, k_rope, prefix_len, path, path_len, page_table=None,
               status=None, stream=None):
    """Torch caller of kdtv_compact_kv (in place); returns the status tensor."""
    import torch
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=c_kv.device)
    code = lib().kdtv_compact_kv(ctypes.byref(dims), _p(c_kv), _p(k_rope), _p(prefix_len),
                                 _p(path), _p(path_len), _p(page_table), _p(status),
                                 _s(stream))
    if code:
        raise KdtvError(code, "kdtv_compact_kv")
    return status


def tree_build(logp, tokens, root_token, n_nodes, stream=None):
    """Torch caller of kdtv_tree_build; returns dict(parent, token, depth,
    score, n_nodes)."""
    import torch
    B, D, K = logp.shape
    dev = logp.device
    N = n_nodes
    out = {k: torch.empty((B, N), dtype=torch.int32, device=dev)
           for k in ("parent", "token", "depth")}
    out["score"] = torch.empty((B, N), dtype=torch.float32, device=dev)
    out["n_nodes"] = torch.empty(B, dtype=torch.int32, device=dev)
    code = lib().kdtv_tree_build(B, D, K, N, _p(logp), _p(tokens), _p(root_token),
                                 _p(out["parent"]), _p(out["token"]), _p(out["depth"]),
                                 _p(out["score"]), _p(out["n_nodes"]), _s(stream))
    if code:
        raise KdtvError(code, "kdtv_tree_build")
    return out
