"""The C ABI: library loads, exports every declared symbol, struct layouts match the
header, and host-side validation rejects bad arguments before anything is enqueued.
CPU only: no call here reaches a CUDA kernel."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from block_top_sparse_centroid_b300 import _lib as L
from block_top_sparse_centroid_b300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kin.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kin_\w+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("kin_centroids_build", "kin_centroids_append", "kin_blocktopk_decode",
              "kin_dense_decode", "kin_workspace_size", "kin_status_str"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(L.SIGNATURES), "binding signatures out of sync with the header"


def test_only_the_abi_is_exported():
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True,
                         text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert {s for s in syms if s.startswith("kin_")} == set(declared_functions())


def test_struct_layout_matches_header(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text("""
#include <stdio.h>
#include <stddef.h>
#include "kin.h"
#define F(T, f) printf("%s.%s %zu\\n", #T, #f, offsetof(T, f));
int main(void) {
  printf("kin_kv_cache %zu\\n", sizeof(kin_kv_cache));
  printf("kin_decode_args %zu\\n", sizeof(kin_decode_args));
  F(kin_kv_cache, num_pages) F(kin_kv_cache, k_pages) F(kin_kv_cache, v_pages)
  F(kin_decode_args, sm_scale) F(kin_decode_args, q) F(kin_decode_args, centroids)
  F(kin_decode_args, scores) F(kin_decode_args, workspace) F(kin_decode_args, workspace_bytes)
  F(kin_decode_args, err_flag) F(kin_decode_args, flags)
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)],
                   check=True)
    got = dict(line.rsplit(" ", 1) for line in subprocess.run(
        [str(exe)], capture_output=True, text=True, check=True).stdout.splitlines())
    assert int(got["kin_kv_cache"]) == ctypes.sizeof(L.KvCache)
    assert int(got["kin_decode_args"]) == ctypes.sizeof(L.DecodeArgs)
    for key, val in got.items():
        if "." in key:
            sname, field = key.split(".")
            cls = L.KvCache if sname == "kin_kv_cache" else L.DecodeArgs
            assert getattr(cls, field).offset == int(val), key


def _cache(**kw):
    c = L.KvCache(L.KIN_BF16, 8, 128, 16, 1024, 0x1000, 0x2000)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _args(**kw):
    a = L.DecodeArgs()
    a.batch, a.num_q_heads, a.max_blocks, a.top_k, a.sm_scale = 2, 16, 64, 8, 0.1
    a.q, a.block_table, a.seq_lens, a.centroids, a.out = 0x3000, 0x4000, 0x5000, 0x6000, 0x7000
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _decode(lib, c, a, dense=False):
    fn = lib.kin_dense_decode if dense else lib.kin_blocktopk_decode
    return fn(ctypes.byref(c) if c is not None else None,
              ctypes.byref(a) if a is not None else None, None)


def test_status_names(lib):
    for code, name in ((0, "KIN_OK"), (1, "KIN_ERR_INVALID_ARG"), (2, "KIN_ERR_UNSUPPORTED"),
                       (3, "KIN_ERR_WORKSPACE"), (4, "KIN_ERR_CUDA")):
        assert lib.kin_status_str(code).decode() == name


@pytest.mark.parametrize("case,status", [
    (dict(cache=None), L.KIN_ERR_INVALID_ARG),
    (dict(args=None), L.KIN_ERR_INVALID_ARG),
    (dict(cache_kw=dict(head_dim=96)), L.KIN_ERR_UNSUPPORTED),
    (dict(cache_kw=dict(page_size=8)), L.KIN_ERR_UNSUPPORTED),
    (dict(cache_kw=dict(dtype=7)), L.KIN_ERR_UNSUPPORTED),
    (dict(cache_kw=dict(num_kv_heads=0)), L.KIN_ERR_INVALID_ARG),
    (dict(cache_kw=dict(num_pages=0)), L.KIN_ERR_INVALID_ARG),
    (dict(cache_kw=dict(num_pages=1 << 28)), L.KIN_ERR_UNSUPPORTED),
    (dict(cache_kw=dict(k_pages=None)), L.KIN_ERR_INVALID_ARG),
    (dict(cache_kw=dict(v_pages=0x2008)), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(num_q_heads=12)), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(num_q_heads=8 * 17)), L.KIN_ERR_UNSUPPORTED),
    (dict(args_kw=dict(batch=0)), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(max_blocks=0)), L.KIN_ERR_UNSUPPORTED),
    (dict(args_kw=dict(max_blocks=16385)), L.KIN_ERR_UNSUPPORTED),
    (dict(args_kw=dict(top_k=0)), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(sm_scale=0.0)), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(sm_scale=float("nan"))), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(q=None)), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(q=0x3004)), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(centroids=None)), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(seq_lens=None)), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(flags=2)), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(shared_prefix_blocks=-1)), L.KIN_ERR_INVALID_ARG),
    (dict(args_kw=dict(shared_prefix_blocks=65)), L.KIN_ERR_INVALID_ARG),
    (dict(), L.KIN_ERR_WORKSPACE),                                   # no workspace
    (dict(args_kw=dict(workspace=0x10000, workspace_bytes=16)), L.KIN_ERR_WORKSPACE),
    (dict(args_kw=dict(workspace=0x10010, workspace_bytes=1 << 30)), L.KIN_ERR_WORKSPACE),
])
def test_host_validation_rejects(lib, case, status):
    c = None if case.get("cache", 1) is None else _cache(**case.get("cache_kw", {}))
    a = None if case.get("args", 1) is None else _args(**case.get("args_kw", {}))
    assert _decode(lib, c, a) == status
    assert lib.kin_last_error().decode() != ""


def test_dense_ignores_topk_and_centroids(lib):
    c, a = _cache(), _args(top_k=0, centroids=None)
    assert _decode(lib, c, a, dense=True) == L.KIN_ERR_WORKSPACE   # got past the arguments
    a.flags = L.KIN_DECODE_APPEND_FINAL                               # appending needs them
    assert _decode(lib, c, a, dense=True) == L.KIN_ERR_INVALID_ARG


def test_workspace_size(lib):
    c = _cache()
    sizes = {}
    for mode in (0, 1, 2):
        for maxb in (1, 64, 2048):
            for k in (1, 64, 128):
                n = ctypes.c_size_t(0)
                a = _args(max_blocks=maxb, top_k=k)
                assert lib.kin_workspace_size(ctypes.byref(c), ctypes.byref(a), mode,
                                              ctypes.byref(n)) == 0
                assert n.value % 256 == 0 and n.value > 0
                sizes[mode, maxb, k] = n.value
    assert sizes[0, 2048, 128] >= sizes[0, 64, 128]
    # token top-k: scores for every token position of every row at least
    assert sizes[2, 2048, 128] >= 2 * 8 * 16 * 2048 * 4
    n = ctypes.c_size_t(0)
    assert lib.kin_workspace_size(ctypes.byref(c), ctypes.byref(_args()), 3,
                                  ctypes.byref(n)) == L.KIN_ERR_INVALID_ARG
    assert lib.kin_workspace_size(ctypes.byref(c), ctypes.byref(_args(top_k=0)), 2,
                                  ctypes.byref(n)) == L.KIN_ERR_INVALID_ARG
    assert lib.kin_workspace_size(ctypes.byref(c), ctypes.byref(_args()), 0,
                                  None) == L.KIN_ERR_INVALID_ARG


@pytest.mark.parametrize("case,status", [
    ("f32_cache", L.KIN_ERR_UNSUPPORTED),
    ("append_flag", L.KIN_ERR_INVALID_ARG),
    ("zero_budget", L.KIN_ERR_INVALID_ARG),
    ("no_workspace", L.KIN_ERR_WORKSPACE),
    ("no_args", L.KIN_ERR_INVALID_ARG),
])
def test_token_topk_validation(lib, case, status):
    """kin_token_topk_decode's host checks, all before any device pointer is used."""
    c = _cache(dtype=L.KIN_F32) if case == "f32_cache" else _cache()
    a = _args(centroids=None)
    if case == "append_flag":
        a.flags = L.KIN_DECODE_APPEND_FINAL
    if case == "zero_budget":
        a.top_k = 0
    ap = None if case == "no_args" else ctypes.byref(a)
    assert lib.kin_token_topk_decode(ctypes.byref(c), ap, None) == status


def test_centroid_validation(lib):
    c = _cache()
    assert lib.kin_centroids_build(ctypes.byref(c), None, 5, 0x8000, None, None) == L.KIN_ERR_INVALID_ARG
    assert lib.kin_centroids_build(ctypes.byref(c), 0x9000, -1, 0x8000, None, None) == L.KIN_ERR_INVALID_ARG
    assert lib.kin_centroids_build(ctypes.byref(c), 0x9000, 4, None, None, None) == L.KIN_ERR_INVALID_ARG
    assert lib.kin_centroids_append(ctypes.byref(c), None, 3, 0x8000, None, None) == L.KIN_ERR_INVALID_ARG
    assert lib.kin_centroids_append(ctypes.byref(c), 0x9000, 0, 0x8000, None, None) == L.KIN_OK
    bad = _cache(head_dim=32)
    assert lib.kin_centroids_build(ctypes.byref(bad), 0x9000, 4, 0x8000, None, None) == L.KIN_ERR_UNSUPPORTED
