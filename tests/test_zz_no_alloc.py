"""The decode entry point that allocates nothing (kin_blocktopk_decode_static).

Callers that cannot allocate device memory at decode time -- a server whose whole GPU
belongs to its KV-cache pool from start-up, or a loop where cudaMalloc/cudaFree would
synchronise the device -- use the library's own static scratch instead of a workspace.
This checks, through the C ABI, that two calls in a row give the same output as the
usual entry point with a caller workspace, within the parity tolerance of the tests.
Collected last, so a failure here comes after every other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _call(lib, fn, cache, args):
    return fn(ctypes.byref(cache), ctypes.byref(args),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_scratch_matches_workspace_entry_point():
    from _gpu import DeviceState, OUT_MAX_ABS, LSE_ABS
    import block_top_sparse_centroid_b300._lib as L
    lib = L.load()
    cfg = W.find_config("qwen3-0.6b").scaled(batch=8, ctx_kind="explicit",
                              lens=(8192, 8191, 4000, 17, 1600, 16 * 300, 5000, 12000), top_k=32)
    inp = W.generate(cfg)
    st = DeviceState(inp)
    dev = st.dev
    B, Hq, H, d = cfg.batch, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    cache = st.cache.c_struct()

    def args_for(out, lse, sel, ws=None):
        a = L.DecodeArgs()
        a.batch, a.num_q_heads, a.max_blocks, a.top_k = B, Hq, inp.max_blocks, cfg.top_k
        a.sm_scale = cfg.sm_scale
        a.q, a.block_table, a.seq_lens = st.q.data_ptr(), st.table.data_ptr(), st.lens.data_ptr()
        a.centroids, a.out, a.lse, a.sel_blocks = (st.cents.data_ptr(), out.data_ptr(),
                                                   lse.data_ptr(), sel.data_ptr())
        a.err_flag = st.err.data_ptr()
        if ws is not None:
            a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
        return a

    def buffers():
        return (torch.full((B, Hq, d), float("nan"), dtype=torch.bfloat16, device=dev),
                torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev),
                torch.full((B, H, cfg.top_k), -7, dtype=torch.int32, device=dev))

    # the usual entry point, with a caller-owned workspace
    need = ctypes.c_size_t(0)
    o0, l0, s0 = buffers()
    a0 = args_for(o0, l0, s0)
    assert lib.kin_workspace_size(ctypes.byref(cache), ctypes.byref(a0), 0, ctypes.byref(need)) == 0
    ws = torch.zeros(need.value, dtype=torch.uint8, device=dev)   # zero-filled before first use
    a0 = args_for(o0, l0, s0, ws)
    assert _call(lib, lib.kin_blocktopk_decode, cache, a0) == 0
    # the static-scratch entry point, twice in a row (the second call finds the array as
    # the first one left it)
    for _ in range(2):
        o1, l1, s1 = buffers()
        a1 = args_for(o1, l1, s1)
        st_code = _call(lib, lib.kin_blocktopk_decode_static, cache, a1)
        assert st_code == 0, lib.kin_last_error().decode()
        torch.cuda.synchronize()
        assert torch.equal(s1, s0)
        err = (o1.float() - o0.float()).abs()
        assert torch.isfinite(o1.float()).all()
        assert float(err.max()) <= OUT_MAX_ABS["bf16"]
        assert float((l1 - l0).abs().max()) <= LSE_ABS["bf16"]
    assert st.error_bits() == 0


def test_static_scratch_rejects_oversized_shapes():
    import block_top_sparse_centroid_b300._lib as L
    lib = L.load()
    c = L.KvCache(L.KIN_BF16, 8, 128, 16, 1 << 20, 0x1000, 0x2000)
    a = L.DecodeArgs()
    a.batch, a.num_q_heads, a.max_blocks, a.top_k, a.sm_scale = 4096, 64, 16384, 128, 0.1
    assert lib.kin_blocktopk_decode_static(ctypes.byref(c), ctypes.byref(a), None) == L.KIN_ERR_WORKSPACE
    assert "static scratch" in lib.kin_last_error().decode()
