"""The device-side timeout path: a bounded wait that can never complete gives up, the
kernel returns with KIN_DEVERR_TIMEOUT set, and the next call on the same workspace is
complete and correct.

It runs on a test build of the library whose waits give up after 4096 tries
(libkin_shortwait.so, same sources; the product library allows about four million), so the
timeout comes after about a millisecond.  The wait is made impossible without any fault:
the score-arrival counter of sequence 0 (workspace word 2: the words are the work-queue
head, the CTA exit count, then one score-arrival counter per (sequence, head range)) is
set far below zero, so the sequence's score items can never bring it to the count its
selection waits for.  Nothing traps and nothing reads or writes out of bounds: the
selection gives up, keeps a valid list for the row, and the kernel winds down.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def test_wait_that_cannot_complete_times_out():
    from _gpu import DeviceState, all_rows, compare_rows
    from block_top_sparse_centroid_b300 import _lib as L
    from block_top_sparse_centroid_b300 import build as B
    lib = L.open_library(B.build(variant="shortwait"))
    cfg = W.find_config("qwen3-0.6b").scaled(batch=4, num_q_heads=4, num_kv_heads=2,
                                             ctx_kind="explicit", lens=(2000, 1500, 3001, 777),
                                             top_k=16)
    inp = W.generate(cfg)
    st = DeviceState(inp)
    B_, Hq, H, d = cfg.batch, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    cache = st.cache.c_struct()
    out = torch.full((B_, Hq, d), float("nan"), dtype=torch.bfloat16, device=st.dev)
    lse = torch.full((B_, Hq), float("nan"), dtype=torch.float32, device=st.dev)
    sel = torch.full((B_, H, cfg.top_k), -7, dtype=torch.int32, device=st.dev)
    a = L.DecodeArgs()
    a.batch, a.num_q_heads, a.max_blocks, a.top_k = B_, Hq, inp.max_blocks, cfg.top_k
    a.sm_scale = cfg.sm_scale
    a.q, a.block_table, a.seq_lens = st.q.data_ptr(), st.table.data_ptr(), st.lens.data_ptr()
    a.centroids, a.out, a.lse, a.sel_blocks = (st.cents.data_ptr(), out.data_ptr(),
                                               lse.data_ptr(), sel.data_ptr())
    a.err_flag = st.err.data_ptr()
    need = ctypes.c_size_t(0)
    assert lib.kin_workspace_size(ctypes.byref(cache), ctypes.byref(a), 0, ctypes.byref(need)) == 0
    ws = torch.zeros(need.value, dtype=torch.uint8, device=st.dev)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    ws.view(torch.int32)[2] = -(1 << 30)      # sequence 0's scores can never all arrive
    assert lib.kin_blocktopk_decode(ctypes.byref(cache), ctypes.byref(a), stream) == 0
    torch.cuda.synchronize()                  # the kernel returned
    assert int(st.err.item()) & L.KIN_DEVERR_TIMEOUT
    kept = sel.cpu().numpy()
    assert np.all((kept >= -1) & (kept < inp.max_blocks))   # in range, whatever the rows hold
    # the last CTA to finish left every counter zero: the workspace is ready for reuse
    assert int(ws[:65536].count_nonzero()) == 0

    st.err.zero_()
    out.fill_(float("nan"))
    sel.fill_(-7)
    scores = torch.full((B_, H, inp.max_blocks), float("nan"), dtype=torch.float32,
                        device=st.dev)
    a.scores = scores.data_ptr()
    assert lib.kin_blocktopk_decode(ctypes.byref(cache), ctypes.byref(a), stream) == 0
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    res = dict(out=out.float().cpu().numpy(), lse=lse.cpu().numpy(), sel=sel.cpu().numpy(),
               scores=scores.cpu().numpy())
    stats = compare_rows(inp, res, all_rows(cfg))
    assert stats["rows"] == B_ * H
