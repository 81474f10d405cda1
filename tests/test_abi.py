"""C-ABI boundary checks that need no GPU: the library builds, loads, exports
every symbol include/kdtv.h declares, and rejects bad arguments on the host
before any CUDA work."""

import ctypes
import os
import re

import pytest

from speculative_decoding_tree_mla_gb300 import kdtv, workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_tree_mla_gb300 import build
    build.build()
    return kdtv.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "kdtv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kdtv_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = header_functions()
    assert names, "no functions parsed from kdtv.h"
    assert set(names) == set(kdtv.EXPORTS)
    for n in names:
        assert hasattr(L, n), f"{n} not exported"


def _dims(name="kimi_single", **kw):
    wl_spec = W.SPECS[name]
    kw.setdefault("flags", kdtv.KDTV_FLAG_SIMT)
    d = kdtv.make_dims(wl_spec, dtype=wl_spec.dtype, t_stride=kw.pop("t_stride", 8192),
                       **kw)
    return d


@pytest.mark.parametrize("flags", [0, kdtv.KDTV_FLAG_SIMT])
def test_workspace_sizes(L, flags):
    if flags == 0 and kdtv.workspace_size(_dims(flags=0)) == 0:
        pytest.skip("tensor-core path not compiled in")
    for name, spec in W.SPECS.items():
        if spec.paged:
            d = kdtv.make_dims(spec, dtype=spec.dtype, page_size=64, max_pages=520,
                               num_pages=10000, flags=flags)
        else:
            d = kdtv.make_dims(spec, dtype=spec.dtype, t_stride=65664, flags=flags)
        n = kdtv.workspace_size(d)
        assert n > 0 and n % 256 == 0
        assert kdtv.launches_per_call(d) > 0


@pytest.mark.parametrize("paged", [False, True])
def test_fp8_cache_plan(L, paged):
    """The tensor-core fp8 call is the bf16 call plus one launch that widens the
    cache into the workspace (one bf16 copy of c_kv and k_rope in the input's
    layout); the CUDA-core fp8 call keeps the bf16 CUDA-core plan."""
    spec = W.SPECS["kimi_single"]
    if paged:
        kw = dict(page_size=64, max_pages=70, num_pages=300)
        kv_rows = 300 * 64
    else:
        kw = dict(t_stride=4165)
        kv_rows = spec.B * 4165
    d16 = kdtv.make_dims(spec, dtype="bf16", **kw)
    d8 = kdtv.make_dims(spec, dtype="fp8kv", kv_scale=0.125, **kw)
    if kdtv.workspace_size(d16) == 0:
        pytest.skip("tensor-core path not compiled in")
    copies = kv_rows * (spec.d_c + spec.d_rope) * 2
    assert kdtv.workspace_size(d16) + copies <= kdtv.workspace_size(d8) \
        <= kdtv.workspace_size(d16) + copies + 512
    assert kdtv.launches_per_call(d8) == kdtv.launches_per_call(d16) + 1
    s16 = kdtv.make_dims(spec, dtype="bf16", flags=kdtv.KDTV_FLAG_SIMT, **kw)
    s8 = kdtv.make_dims(spec, dtype="fp8kv", flags=kdtv.KDTV_FLAG_SIMT, **kw)
    assert kdtv.workspace_size(s8) == kdtv.workspace_size(s16) > 0
    assert kdtv.launches_per_call(s8) == kdtv.launches_per_call(s16) == 4


@pytest.mark.parametrize("field,value,code", [
    ("N", 0, "KDTV_ERR_INVALID_ARG"),
    ("H", -1, "KDTV_ERR_INVALID_ARG"),
    ("N", 129, "KDTV_ERR_UNSUPPORTED"),
    ("dtype", 7, "KDTV_ERR_INVALID_ARG"),
    ("t_stride", 3, "KDTV_ERR_INVALID_ARG"),
    ("d_c", 1024, "KDTV_ERR_UNSUPPORTED"),
])
def test_bad_dims_rejected_on_host(L, field, value, code):
    d = _dims()
    setattr(d, field, value)
    assert kdtv.workspace_size(d) == 0
    fake = 256
    rc = kdtv.verify_attn_raw(d, fake, fake, fake, fake, fake, fake, fake, fake, 0, fake, 0)
    assert kdtv.STATUS[rc] == code
    # the allocation-free entry point returns the same host-side code
    rc2 = L.kdtv_verify_attn_noalloc(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake,
                                     fake, None, fake, fake, None)
    assert kdtv.STATUS[rc2] == code


def test_null_pointers_and_workspace_rejected(L):
    d = _dims()
    fake = 256
    # no workspace set
    rc = kdtv.verify_attn_raw(d, fake, fake, fake, fake, fake, fake, fake, fake, 0, fake, 0)
    assert kdtv.STATUS[rc] == "KDTV_ERR_INVALID_ARG"
    d.workspace = 4096
    d.workspace_bytes = kdtv.workspace_size(d)
    rc = kdtv.verify_attn_raw(d, 0, fake, fake, fake, fake, fake, fake, fake, 0, fake, 0)
    assert kdtv.STATUS[rc] == "KDTV_ERR_INVALID_ARG"
    # page_table given for a contiguous cache
    rc = kdtv.verify_attn_raw(d, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 0)
    assert kdtv.STATUS[rc] == "KDTV_ERR_INVALID_ARG"
    # workspace too small / misaligned
    d.workspace_bytes = 1024
    rc = kdtv.verify_attn_raw(d, fake, fake, fake, fake, fake, fake, fake, fake, 0, fake, 0)
    assert kdtv.STATUS[rc] == "KDTV_ERR_INVALID_ARG"
    d.workspace = 4096 + 16
    d.workspace_bytes = 1 << 40
    rc = kdtv.verify_attn_raw(d, fake, fake, fake, fake, fake, fake, fake, fake, 0, fake, 0)
    assert kdtv.STATUS[rc] == "KDTV_ERR_INVALID_ARG"


def test_strerror(L):
    for code, name in kdtv.STATUS.items():
        assert kdtv.strerror(code) == name


def test_workloads_deterministic():
    a = W.make("tiny")
    b = W.make("tiny")
    for k in a.t:
        assert (a.t[k] == b.t[k]).all()
    c = W.make("tiny", seed=123)
    assert not (a.t["c_kv"] == c.t["c_kv"]).all()


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "speculative_decoding_tree_mla_gb300")
    for dp, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dp, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", txt, re.M), f
                assert "mla_tree_attn" not in txt, f


def test_next_steps_reject_bad_args_on_host(L):
    fake = 256
    assert kdtv.STATUS[L.kdtv_tree_accept(0, 8, fake, fake, fake, fake, fake, fake, None)] == "KDTV_ERR_INVALID_ARG"
    assert kdtv.STATUS[L.kdtv_tree_accept(2, 129, fake, fake, fake, fake, fake, fake, None)] == "KDTV_ERR_UNSUPPORTED"
    assert kdtv.STATUS[L.kdtv_tree_accept(2, 8, None, fake, fake, fake, fake, fake, None)] == "KDTV_ERR_INVALID_ARG"
    assert kdtv.STATUS[L.kdtv_tree_build(2, 4, 65, 8, fake, fake, fake, fake, fake, fake, fake, fake, None)] == "KDTV_ERR_UNSUPPORTED"
    assert kdtv.STATUS[L.kdtv_tree_build(2, 4, 4, 0, fake, fake, fake, fake, fake, fake, fake, fake, None)] == "KDTV_ERR_INVALID_ARG"
    d = _dims()
    assert kdtv.STATUS[L.kdtv_compact_kv(ctypes.byref(d), fake, fake, fake, fake, fake, None, None, None)] == "KDTV_ERR_INVALID_ARG"
    assert kdtv.STATUS[L.kdtv_compact_kv(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, None)] == "KDTV_ERR_INVALID_ARG"


def test_header_is_plain_c_and_links(L, tmp_path):
    """A C11 program (gcc, -pedantic -Werror) includes kdtv.h, takes the address
    of every declared entry point, links against the library and calls the
    host-only parts: the boundary needs no C++ or Python on the caller's side."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = None
    for root in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if root and os.path.exists(os.path.join(root, "include", "cuda_runtime_api.h")):
            cuda_inc = os.path.join(root, "include")
            break
    if not cc or not cuda_inc:
        pytest.skip("no C compiler or CUDA headers")
    names = header_functions()
    lib_dir = os.path.dirname(kdtv.lib()._name)
    src = tmp_path / "caller.c"
    src.write_text("\n".join([
        '#include "kdtv.h"',
        "#include <stdio.h>",
        "#include <string.h>",
        "typedef void (*entry_fn)(void);",
        "static const entry_fn entries[] = {" + ", ".join(f"(entry_fn){n}" for n in names) + "};",
        "int main(void) {",
        "  kdtv_dims d;",
        "  memset(&d, 0, sizeof d);",
        "  d.B = 1; d.N = 16; d.H = 4; d.d_nope = 32; d.d_rope = 16; d.d_v = 32; d.d_c = 64;",
        "  d.dtype = KDTV_F32; d.t_stride = 64; d.scale = 0.125f;",
        "  int st = kdtv_verify_attn(&d, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,",
        "                            NULL, 0);",
        '  printf("%d %zu %d %s\\n", (int)(sizeof entries / sizeof entries[0]),',
        "         kdtv_workspace_size(&d), st, kdtv_strerror(st));",
        "  return 0;",
        "}",
        ""]))
    exe = tmp_path / "caller"
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src),
                        "-L", lib_dir, "-lkdtv", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    count, ws, st, name = r.stdout.split()
    assert int(count) == len(names)
    spec = W.small_spec("c_caller", B=1, N=16, H=4, d_nope=32, d_rope=16, d_v=32, d_c=64,
                        dtype="f32", prefix=("fixed", 0))
    d = kdtv.make_dims(spec, dtype="f32", t_stride=64, scale=0.125)
    assert int(ws) == kdtv.workspace_size(d) > 0
    assert name == "KDTV_ERR_INVALID_ARG" and kdtv.STATUS[int(st)] == name


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library every call raises: there is no CPU fallback."""
    monkeypatch.setattr(kdtv, "LIB_PATH", str(tmp_path / "libkdtv.so"))
    monkeypatch.setattr(kdtv, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        kdtv.workspace_size(_dims())
    with pytest.raises(RuntimeError, match="missing"):
        kdtv.strerror(0)


@pytest.mark.parametrize("flags", [0, kdtv.KDTV_FLAG_SIMT])
def test_size_limits_on_host(L, flags):
    """At the largest accepted batch (B N H = 2^28 query rows) the workspace size
    is computed without overflow; one more request is refused, and so is a
    paged cache of more than 2^30 positions per request."""
    spec = W.small_spec("max_rows", B=(1 << 28) // (128 * 64), N=128, H=64)
    d = kdtv.make_dims(spec, dtype="bf16", t_stride=128, flags=flags)
    if flags == 0 and kdtv.workspace_size(_dims(flags=0)) == 0:
        pytest.skip("tensor-core path not compiled in")
    rows = spec.B * spec.N * spec.H
    assert rows == 1 << 28
    assert kdtv.workspace_size(d) >= 2 * rows * spec.d_c * 2     # q_lat + o_lat, >= bf16 each
    d.B += 1
    assert kdtv.workspace_size(d) == 0
    fake = 256
    rc = kdtv.verify_attn_raw(d, fake, fake, fake, fake, fake, fake, fake, fake, 0, fake, 0)
    assert kdtv.STATUS[rc] == "KDTV_ERR_UNSUPPORTED"
    paged = kdtv.make_dims(W.SPECS["kimi_single"], dtype="bf16", page_size=64,
                           max_pages=(1 << 24) + 1, num_pages=1 << 20, flags=flags)
    assert kdtv.workspace_size(paged) == 0
    rc = kdtv.verify_attn_raw(paged, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 0)
    assert kdtv.STATUS[rc] == "KDTV_ERR_INVALID_ARG"
