"""Python binding of libkin: argument marshalling over torch tensors, nothing else.

Every step of the path runs in the CUDA library; this module only checks tensor
shapes / dtypes / devices, allocates outputs and the workspace through torch when the
caller does not pass them, and forwards raw pointers and the current stream to the C ABI.

The method (block top-k decode attention over a paged KV cache, blocks of 16 tokens
scored by their mean key vectors, summed over the GQA group) follows the Pith review of
"Kinetics: Rethinking Test-Time Scaling Laws", section "What carries the argument", and
the Kinetics README, section "Benchmark Block TopK Attention throughput".
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional

import torch

from . import _lib as L

BLOCK = 16
_DTYPES = {torch.float32: L.KIN_F32, torch.bfloat16: L.KIN_BF16}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, shape, dtype, device) -> None:
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


@dataclasses.dataclass
class PagedKVCache:
    """K and V pages of one attention layer: [num_pages, num_kv_heads, 16, head_dim]."""

    k_pages: torch.Tensor
    v_pages: torch.Tensor

    def __post_init__(self):
        k, v = self.k_pages, self.v_pages
        if k.dim() != 4 or k.shape[2] != BLOCK:
            raise ValueError("k_pages must be [num_pages, num_kv_heads, 16, head_dim]")
        if v.shape != k.shape or v.dtype != k.dtype or v.device != k.device:
            raise ValueError("v_pages must match k_pages in shape, dtype and device")
        if k.dtype not in _DTYPES:
            raise ValueError(f"unsupported dtype {k.dtype}")
        if not (k.is_contiguous() and v.is_contiguous()):
            raise ValueError("pages must be contiguous")

    @property
    def device(self):
        return self.k_pages.device

    @property
    def dtype(self):
        return self.k_pages.dtype

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k_pages.shape[1])

    @property
    def head_dim(self) -> int:
        return int(self.k_pages.shape[3])

    @property
    def centroid_shape(self) -> tuple:
        """Shape of the centroid table: [P, H, d] for fp32 caches; [2, P, H, d] for bf16
        caches (plane 0: the fp32 mean rounded to bf16, plane 1: its rounding residual
        rounded to bf16)."""
        shape = (self.num_pages, self.num_kv_heads, self.head_dim)
        return (2,) + shape if self.dtype == torch.bfloat16 else shape

    def c_struct(self) -> L.KvCache:
        return L.KvCache(_DTYPES[self.dtype], self.num_kv_heads, self.head_dim, BLOCK,
                         self.num_pages, self.k_pages.data_ptr(), self.v_pages.data_ptr())


def _shape_args(cache: PagedKVCache, batch: int, num_q_heads: int, max_blocks: int,
                top_k: int) -> L.DecodeArgs:
    a = L.DecodeArgs()
    a.batch, a.num_q_heads, a.max_blocks, a.top_k = batch, num_q_heads, max_blocks, top_k
    a.sm_scale = 1.0
    return a


def workspace_size(cache: PagedKVCache, batch: int, num_q_heads: int, max_blocks: int,
                   top_k: int = 1, dense: bool = False, tokens: bool = False) -> int:
    """Bytes of workspace one decode call needs (kin_workspace_size): block top-k, dense
    (dense=True) or token top-k (tokens=True, top_k in tokens)."""
    lib = L.load()
    c = cache.c_struct()
    a = _shape_args(cache, batch, num_q_heads, max_blocks, top_k)
    n = ctypes.c_size_t(0)
    mode = L.MODE_TOKENTOPK if tokens else (L.MODE_DENSE if dense else L.MODE_BLOCKTOPK)
    L.check(lib.kin_workspace_size(ctypes.byref(c), ctypes.byref(a), mode, ctypes.byref(n)),
            "kin_workspace_size")
    return int(n.value)


class Workspace:
    """A device scratch buffer that grows on demand (one per stream of decode calls)."""

    def __init__(self, device):
        self.device = torch.device(device)
        self.buf = torch.zeros(0, dtype=torch.uint8, device=self.device)

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws = {}


def _workspace(device, nbytes: int, workspace: Optional[Workspace]) -> torch.Tensor:
    if workspace is None:
        key = (device.type, device.index)
        workspace = _default_ws.get(key)
        if workspace is None:
            workspace = _default_ws[key] = Workspace(device)
    return workspace.get(nbytes)


def _err_ptr(err_flag: Optional[torch.Tensor], device):
    if err_flag is None:
        return None
    _need(err_flag, "err_flag", (1,), torch.int32, device)
    return _ptr(err_flag)


def centroids_build(cache: PagedKVCache, centroids: Optional[torch.Tensor] = None,
                    page_ids: Optional[torch.Tensor] = None,
                    err_flag: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Mean key of every listed page (all pages when page_ids is None): kin_centroids_build."""
    lib = L.load()
    dev = cache.device
    shape = cache.centroid_shape
    if centroids is None:
        centroids = torch.empty(shape, dtype=cache.dtype, device=dev)
    _need(centroids, "centroids", shape, cache.dtype, dev)
    n = cache.num_pages
    if page_ids is not None:
        if page_ids.dim() != 1:
            raise ValueError("page_ids must be 1-D")
        _need(page_ids, "page_ids", (page_ids.numel(),), torch.int32, dev)
        n = page_ids.numel()
    c = cache.c_struct()
    L.check(lib.kin_centroids_build(ctypes.byref(c), _ptr(page_ids), n, _ptr(centroids),
                                    _err_ptr(err_flag, dev), _stream(stream, dev)),
            "kin_centroids_build")
    return centroids


def centroids_append(cache: PagedKVCache, page_ids: torch.Tensor, centroids: torch.Tensor,
                     err_flag: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Mean key of pages a decode step just completed: kin_centroids_append."""
    lib = L.load()
    dev = cache.device
    _need(centroids, "centroids", cache.centroid_shape, cache.dtype, dev)
    if page_ids.dim() != 1:
        raise ValueError("page_ids must be 1-D")
    _need(page_ids, "page_ids", (page_ids.numel(),), torch.int32, dev)
    c = cache.c_struct()
    L.check(lib.kin_centroids_append(ctypes.byref(c), _ptr(page_ids), page_ids.numel(),
                                     _ptr(centroids), _err_ptr(err_flag, dev),
                                     _stream(stream, dev)),
            "kin_centroids_append")
    return centroids


class PreparedDecode:
    """A decode call whose tensors are fixed: shapes, dtypes and devices are checked and the
    C structs built once, so that each call only enqueues the kernels (kin_blocktopk_decode,
    kin_dense_decode or kin_token_topk_decode).  It keeps every tensor it was given alive.  For a decode loop whose
    buffers stay the same from step to step (q, out, the cache, the block table and
    seq_lens updated in place), this is the low-overhead way to call the library.

    stream: a torch stream baked into the call, or None for the current stream of the
    cache's device at each call.  shared_prefix_blocks: the leading logical blocks every
    sequence shares (a Best-of-N prompt), kept in L2 for the step; a hint that changes no
    result."""

    def __init__(self, mode: int, cache: PagedKVCache, q, block_table, seq_lens, sm_scale,
                 top_k, centroids=None, out=None, lse=None, sel_blocks=None, scores=None,
                 workspace: Optional[Workspace] = None, err_flag=None, append_final=False,
                 stream=None, shared_prefix_blocks: int = 0):
        lib = L.load()
        dev = cache.device
        if q.dim() != 3:
            raise ValueError("q must be [batch, num_q_heads, head_dim]")
        B, Hq, d = (int(x) for x in q.shape)
        H = cache.num_kv_heads
        _need(q, "q", (B, Hq, cache.head_dim), cache.dtype, dev)
        if block_table.dim() != 2:
            raise ValueError("block_table must be [batch, max_blocks]")
        maxb = int(block_table.shape[1])
        _need(block_table, "block_table", (B, maxb), torch.int32, dev)
        _need(seq_lens, "seq_lens", (B,), torch.int32, dev)
        if out is None:
            out = torch.empty_like(q)
        _need(out, "out", (B, Hq, d), cache.dtype, dev)
        if lse is not None:
            _need(lse, "lse", (B, Hq), torch.float32, dev)
        if mode == L.MODE_BLOCKTOPK or append_final:
            if centroids is None:
                raise ValueError("centroids are required")
            _need(centroids, "centroids", cache.centroid_shape, cache.dtype, dev)
        if mode == L.MODE_BLOCKTOPK:
            if sel_blocks is not None:
                _need(sel_blocks, "sel_blocks", (B, H, top_k), torch.int32, dev)
            if scores is not None:
                _need(scores, "scores", (B, H, maxb), torch.float32, dev)
        if mode == L.MODE_TOKENTOPK:
            if sel_blocks is not None:
                _need(sel_blocks, "sel_tokens", (B, H, top_k), torch.int32, dev)
            if scores is not None:
                _need(scores, "scores", (B, H, 16 * maxb), torch.float32, dev)
        a = L.DecodeArgs()
        a.batch, a.num_q_heads, a.max_blocks, a.top_k = B, Hq, maxb, int(top_k)
        a.sm_scale = float(sm_scale)
        a.q, a.block_table, a.seq_lens = q.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr()
        a.centroids = centroids.data_ptr() if (centroids is not None and
                                               (mode == L.MODE_BLOCKTOPK or append_final)) else None
        a.flags = L.KIN_DECODE_APPEND_FINAL if append_final else 0
        a.shared_prefix_blocks = int(shared_prefix_blocks)
        a.out = out.data_ptr()
        a.lse = None if lse is None else lse.data_ptr()
        a.sel_blocks = None if (sel_blocks is None or mode == L.MODE_DENSE) else sel_blocks.data_ptr()
        a.scores = None if (scores is None or mode == L.MODE_DENSE) else scores.data_ptr()
        c = cache.c_struct()
        need = ctypes.c_size_t(0)
        L.check(lib.kin_workspace_size(ctypes.byref(c), ctypes.byref(a), mode, ctypes.byref(need)),
                "kin_workspace_size")
        ws = _workspace(dev, int(need.value), workspace)
        a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
        a.err_flag = None if err_flag is None else _err_ptr(err_flag, dev).value
        self._keep = (cache, q, block_table, seq_lens, centroids, out, lse, sel_blocks, scores,
                      ws, err_flag)
        self._lib, self._c, self._a, self._mode, self._dev = lib, c, a, mode, dev
        self._cref, self._aref = ctypes.byref(c), ctypes.byref(a)
        self._name = {L.MODE_BLOCKTOPK: "kin_blocktopk_decode", L.MODE_DENSE: "kin_dense_decode",
                      L.MODE_TOKENTOPK: "kin_token_topk_decode"}[mode]
        self._fn = getattr(lib, self._name)
        self._stream = None if stream is None else ctypes.c_void_p(stream.cuda_stream)
        self.out = out

    def __call__(self, stream=None) -> torch.Tensor:
        st = self._stream if stream is None and self._stream is not None else _stream(stream, self._dev)
        L.check(self._fn(self._cref, self._aref, st), self._name)
        return self.out

    def timed(self, events, stream=None) -> torch.Tensor:
        """The same call through kin_decode_timed, recording 4 torch.cuda.Events."""
        st = self._stream if stream is None and self._stream is not None else _stream(stream, self._dev)
        handles = (ctypes.c_void_p * 4)(*[_event_handle(e, stream, self._dev) for e in events])
        L.check(self._lib.kin_decode_timed(self._cref, self._aref, self._mode, handles, st),
                "kin_decode_timed")
        return self.out


def _decode(mode: int, cache: PagedKVCache, q, block_table, seq_lens, sm_scale, top_k,
            centroids, out, lse, sel_blocks, scores, workspace, err_flag, stream, events=None,
            append_final=False, shared_prefix_blocks=0):
    call = PreparedDecode(mode, cache, q, block_table, seq_lens, sm_scale, top_k, centroids,
                          out, lse, sel_blocks, scores, workspace, err_flag, append_final,
                          shared_prefix_blocks=shared_prefix_blocks)
    if events is not None:
        return call.timed(list(events), stream)
    return call(stream)


def prepare_blocktopk_decode(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                             seq_lens: torch.Tensor, centroids: torch.Tensor, top_k: int,
                             sm_scale: float, out: Optional[torch.Tensor] = None,
                             lse: Optional[torch.Tensor] = None,
                             sel_blocks: Optional[torch.Tensor] = None,
                             scores: Optional[torch.Tensor] = None,
                             workspace: Optional[Workspace] = None,
                             err_flag: Optional[torch.Tensor] = None,
                             append_final: bool = False, stream=None,
                             shared_prefix_blocks: int = 0) -> PreparedDecode:
    """A block top-k decode call (kin_blocktopk_decode) prepared once, run by calling it."""
    return PreparedDecode(L.MODE_BLOCKTOPK, cache, q, block_table, seq_lens, sm_scale, top_k,
                          centroids, out, lse, sel_blocks, scores, workspace, err_flag,
                          append_final, stream, shared_prefix_blocks)


def prepare_dense_decode(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                         seq_lens: torch.Tensor, sm_scale: float,
                         out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                         workspace: Optional[Workspace] = None,
                         err_flag: Optional[torch.Tensor] = None, stream=None,
                         shared_prefix_blocks: int = 0) -> PreparedDecode:
    """A dense decode call (kin_dense_decode) prepared once, run by calling it."""
    return PreparedDecode(L.MODE_DENSE, cache, q, block_table, seq_lens, sm_scale, 1, None,
                          out, lse, None, None, workspace, err_flag, False, stream,
                          shared_prefix_blocks)


def prepare_token_topk_decode(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                              seq_lens: torch.Tensor, top_tokens: int, sm_scale: float,
                              out: Optional[torch.Tensor] = None,
                              lse: Optional[torch.Tensor] = None,
                              sel_tokens: Optional[torch.Tensor] = None,
                              scores: Optional[torch.Tensor] = None,
                              workspace: Optional[Workspace] = None,
                              err_flag: Optional[torch.Tensor] = None,
                              stream=None) -> PreparedDecode:
    """A token top-k decode call (kin_token_topk_decode) prepared once, run by calling it."""
    return PreparedDecode(L.MODE_TOKENTOPK, cache, q, block_table, seq_lens, sm_scale,
                          top_tokens, None, out, lse, sel_tokens, scores, workspace, err_flag,
                          False, stream)


def token_topk_decode(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                      seq_lens: torch.Tensor, top_tokens: int, sm_scale: float,
                      out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                      sel_tokens: Optional[torch.Tensor] = None,
                      scores: Optional[torch.Tensor] = None,
                      workspace: Optional[Workspace] = None,
                      err_flag: Optional[torch.Tensor] = None, stream=None,
                      events=None) -> torch.Tensor:
    """One token-level (oracle) top-k decode step: every token scored by the group-summed
    q.k, the top_tokens best of each (sequence, KV head) kept, attention over them
    (kin_token_topk_decode; with events, kin_decode_timed mode 2).  sel_tokens: optional
    [B, H, top_tokens] int32 kept positions; scores: optional [B, H, 16 max_blocks] fp32."""
    call = PreparedDecode(L.MODE_TOKENTOPK, cache, q, block_table, seq_lens, sm_scale,
                          top_tokens, None, out, lse, sel_tokens, scores, workspace, err_flag,
                          False)
    if events is not None:
        return call.timed(list(events), stream)
    return call(stream)


def _event_handle(ev: "torch.cuda.Event", stream, dev) -> int:
    """Raw cudaEvent_t of a torch event (torch creates the event on its first record)."""
    if ev.cuda_event == 0:
        ev.record(stream if stream is not None else torch.cuda.current_stream(dev))
    return ev.cuda_event


def blocktopk_decode(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                     seq_lens: torch.Tensor, centroids: torch.Tensor, top_k: int,
                     sm_scale: float, out: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None,
                     sel_blocks: Optional[torch.Tensor] = None,
                     scores: Optional[torch.Tensor] = None,
                     workspace: Optional[Workspace] = None,
                     err_flag: Optional[torch.Tensor] = None, stream=None,
                     append_final: bool = False, shared_prefix_blocks: int = 0) -> torch.Tensor:
    """One block top-k decode step (score, select, sparse attention): kin_blocktopk_decode.

    append_final: also write the centroid of each sequence's final block when that block
    is complete (KIN_DECODE_APPEND_FINAL), i.e. the append the next steps need.
    shared_prefix_blocks: the leading logical blocks all sequences share (their pages are
    kept in L2 for the step; results do not depend on it)."""
    return _decode(L.MODE_BLOCKTOPK, cache, q, block_table, seq_lens, sm_scale, top_k,
                   centroids, out, lse, sel_blocks, scores, workspace, err_flag, stream,
                   append_final=append_final, shared_prefix_blocks=shared_prefix_blocks)


def decode_timed(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                 seq_lens: torch.Tensor, sm_scale: float, events, dense: bool = False,
                 centroids: Optional[torch.Tensor] = None, top_k: int = 1,
                 out: Optional[torch.Tensor] = None, workspace: Optional[Workspace] = None,
                 err_flag: Optional[torch.Tensor] = None, stream=None,
                 append_final: bool = False, shared_prefix_blocks: int = 0) -> torch.Tensor:
    """One decode step that also records 4 torch.cuda.Events around its kernels
    (before scoring, after scoring, after selection, after attention): kin_decode_timed."""
    mode = L.MODE_DENSE if dense else L.MODE_BLOCKTOPK
    return _decode(mode, cache, q, block_table, seq_lens, sm_scale, top_k, centroids, out,
                   None, None, None, workspace, err_flag, stream, events=list(events),
                   append_final=append_final, shared_prefix_blocks=shared_prefix_blocks)


def dense_decode(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                 seq_lens: torch.Tensor, sm_scale: float, out: Optional[torch.Tensor] = None,
                 lse: Optional[torch.Tensor] = None, workspace: Optional[Workspace] = None,
                 err_flag: Optional[torch.Tensor] = None, stream=None,
                 centroids: Optional[torch.Tensor] = None,
                 append_final: bool = False, shared_prefix_blocks: int = 0) -> torch.Tensor:
    """Dense paged decode over every block (the comparison baseline): kin_dense_decode."""
    return _decode(L.MODE_DENSE, cache, q, block_table, seq_lens, sm_scale, 1, centroids,
                   out, lse, None, None, workspace, err_flag, stream,
                   append_final=append_final, shared_prefix_blocks=shared_prefix_blocks)
