"""Seeded synthetic inputs for block top-k decode attention.

This module is shared by the CUDA path's tests, the benchmark and the CPU oracle, and
for that reason it holds random draws and shapes only: no centroid, score, selection or
attention arithmetic lives here.

The shapes follow the per-layer decode benchmark of the Kinetics README (GitLite mirror,
section "Benchmark Block TopK Attention throughput"): a paged KV cache whose page is
one 16-token block, a top-k counted in pages, Qwen3-family GQA layouts and contexts up
to 32K tokens.  The value recipe is:

* K = N(0, 1) per element, plus a per-(page, KV head) offset vector whose elements are
  N(0, 0.5^2); the offset is shared by the 16 keys of the page, which makes the blocks'
  mean keys distinct.
* V ~ N(0, 1);  Q ~ N(0, 1) * q_std  (q_std = 1/sqrt(128) for the Qwen3-shaped cases).
* Everything is drawn in fp32 on the CPU with torch generators seeded from
  (seed, purpose, chunk), then rounded once to the storage dtype (bf16 round-to-nearest-
  even via torch).  The same bits are copied to the GPU and handed to the oracle.
* Slots of a page past a sequence's length hold a large "poison" value, so that an
  attention kernel which forgets to mask them produces an obviously wrong result.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import hashlib
import math
import os
from typing import List, Optional

import torch

BLOCK = 16            # tokens per block == tokens per KV page
POISON_K = 512.0      # stale-slot marker in K (exact in bf16)
POISON_V = -512.0     # stale-slot marker in V (exact in bf16)


def _seed(*keys) -> int:
    """A 63-bit generator seed derived from a tuple of keys (stable across runs)."""
    h = hashlib.sha256(repr(keys).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(*keys) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(_seed(*keys))
    return g


@dataclasses.dataclass(frozen=True)
class Config:
    """One synthetic decode workload (one attention layer, one or more decode steps)."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    top_k: int
    dtype: str                  # "f32" or "bf16": storage of Q, K, V, centroids and O
    ctx_kind: str               # "uniform" | "ragged" | "best_of_n" | "explicit"
    ctx_lo: int                 # uniform: the context; ragged / best_of_n: lower bound
    ctx_hi: int = 0             # ragged / best_of_n: upper bound (inclusive)
    prefix: int = 0             # best_of_n: shared prompt tokens (a multiple of 16)
    q_std: float = 1.0
    sm_scale: float = 1.0
    shuffled: bool = True       # page table is a random permutation of the page pool
    steps: int = 1              # decode steps (best_of_n: tokens appended per sample)
    seed: int = 1234
    lens: tuple = ()            # "explicit": the context of every sequence

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def scaled(self, **kw) -> "Config":
        """A copy with some fields replaced (smaller batch or contexts for quick tests)."""
        return dataclasses.replace(self, **kw)


_S128 = 1.0 / math.sqrt(128.0)

CONFIGS: List[Config] = [
    # 0: tiny fp32 case the oracle finishes instantly.
    Config("tiny", 1, 2, 1, 64, 8, "f32", "uniform", 1024,
           q_std=1.0, sm_scale=1.0 / 8.0, shuffled=False, seed=1234),
    # 1: Qwen3-0.6B-shaped layer, uniform 8K context, top-64 pages.
    Config("qwen3-0.6b", 64, 16, 8, 128, 64, "bf16", "uniform", 8192,
           q_std=_S128, sm_scale=_S128, seed=1235),
    # 2: Qwen3-8B-shaped layer, 32K context, top-128 pages, final block just completed.
    Config("qwen3-8b", 32, 32, 8, 128, 128, "bf16", "uniform", 32768,
           q_std=_S128, sm_scale=_S128, seed=1236),
    # 3: Qwen3-32B-shaped ragged paged decode, contexts U[8192, 32768], shuffled pool.
    Config("qwen3-32b-ragged", 16, 64, 8, 128, 128, "bf16", "ragged", 8192, 32768,
           q_std=_S128, sm_scale=_S128, seed=1237),
    # 4: Best-of-N Qwen3-14B-shaped decode, 256 samples sharing a 1024-token prompt,
    #    generated lengths U[2048, 16384], 64 consecutive decode steps.
    Config("best-of-n-qwen3-14b", 256, 40, 8, 128, 128, "bf16", "best_of_n", 2048, 16384,
           prefix=1024, q_std=_S128, sm_scale=_S128, shuffled=False, steps=64, seed=1238),
]


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


@dataclasses.dataclass
class Inputs:
    """Host (CPU) tensors of one workload.  Shapes:

    k_pages, v_pages : [num_pages, num_kv_heads, 16, head_dim]   storage dtype
    k_offset         : [num_pages, num_kv_heads, head_dim]       fp32 (generator state)
    q                : [batch, num_q_heads, head_dim]            storage dtype
    block_table      : [batch, max_blocks] int32, physical page ids, -1 where unused
    seq_lens         : [batch] int32, tokens including the current one
    """

    cfg: Config
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    k_offset: torch.Tensor
    q: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    def complete_pages(self) -> torch.Tensor:
        """Physical ids of pages that hold 16 valid tokens (each listed once)."""
        ids = []
        for b in range(self.cfg.batch):
            nfull = int(self.seq_lens[b]) // BLOCK
            ids.append(self.block_table[b, :nfull])
        return torch.unique(torch.cat(ids)).to(torch.int32)

    def last_pages(self) -> torch.Tensor:
        """Physical page of each sequence's final (current) block, in batch order."""
        nb = (self.seq_lens.to(torch.int64) + BLOCK - 1) // BLOCK
        return self.block_table[torch.arange(self.cfg.batch), nb - 1].to(torch.int32)


def _draw_lengths(cfg: Config) -> torch.Tensor:
    g = _gen(cfg.seed, "lengths")
    if cfg.ctx_kind == "uniform":
        return torch.full((cfg.batch,), cfg.ctx_lo, dtype=torch.int64)
    if cfg.ctx_kind == "ragged":
        return torch.randint(cfg.ctx_lo, cfg.ctx_hi + 1, (cfg.batch,), generator=g)
    if cfg.ctx_kind == "best_of_n":
        gen = torch.randint(cfg.ctx_lo, cfg.ctx_hi + 1, (cfg.batch,), generator=g)
        return gen + cfg.prefix
    if cfg.ctx_kind == "explicit":
        assert len(cfg.lens) == cfg.batch
        return torch.tensor(cfg.lens, dtype=torch.int64)
    raise ValueError(cfg.ctx_kind)


def _fill_pages(num_pages: int, cfg: Config, purpose: str, with_offset: bool,
                chunk: int = 1024):
    """Draw [num_pages, H, 16, d] values chunk by chunk (fp32), plus the K offsets.

    Every chunk has its own generator (seeded from its first page), so the chunks are
    drawn on several threads with the same values as one after the other."""
    H, d = cfg.num_kv_heads, cfg.head_dim
    out = torch.empty((num_pages, H, BLOCK, d), dtype=torch_dtype(cfg.dtype))
    offs = torch.zeros((num_pages, H, d), dtype=torch.float32) if with_offset else None

    def fill(c0):
        c1 = min(num_pages, c0 + chunk)
        g = _gen(cfg.seed, purpose, c0)
        x = torch.randn((c1 - c0, H, BLOCK, d), generator=g, dtype=torch.float32)
        if with_offset:
            o = torch.randn((c1 - c0, H, d), generator=g, dtype=torch.float32) * 0.5
            offs[c0:c1] = o
            x += o[:, :, None, :]
        out[c0:c1] = x.to(out.dtype)

    starts = list(range(0, num_pages, chunk))
    workers = min(len(starts), os.cpu_count() or 1, 32)
    if workers <= 1:
        for c0 in starts:
            fill(c0)
    else:
        with concurrent.futures.ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, starts))
    return out, offs


def generate(cfg: Config, poison: bool = True) -> Inputs:
    """Materialise the workload's initial decode state on the host.

    Page allocation: every sequence owns ceil((L_b + steps - 1) / 16) blocks (room for the
    tokens later decode steps append); best-of-N samples share the prompt's pages.
    """
    lens = _draw_lengths(cfg)
    B = cfg.batch
    extra = cfg.steps - 1 if cfg.ctx_kind == "best_of_n" else 0
    need = (lens + extra + BLOCK - 1) // BLOCK           # blocks each sequence may touch
    max_blocks = int(need.max())
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    if cfg.ctx_kind == "best_of_n":
        assert cfg.prefix % BLOCK == 0
        npre = cfg.prefix // BLOCK
        own = need - npre
        num_pages = npre + int(own.sum())
        nxt = npre
        for b in range(B):
            table[b, :npre] = torch.arange(npre, dtype=torch.int32)
            n = int(own[b])
            table[b, npre:npre + n] = torch.arange(nxt, nxt + n, dtype=torch.int32)
            nxt += n
    else:
        num_pages = int(need.sum())
        ids = torch.arange(num_pages, dtype=torch.int32)
        if cfg.shuffled:
            ids = ids[torch.randperm(num_pages, generator=_gen(cfg.seed, "pages"))]
        pos = 0
        for b in range(B):
            n = int(need[b])
            table[b, :n] = ids[pos:pos + n]
            pos += n

    k_pages, k_off = _fill_pages(num_pages, cfg, "k", with_offset=True)
    v_pages, _ = _fill_pages(num_pages, cfg, "v", with_offset=False)
    q = (torch.randn((B, cfg.num_q_heads, cfg.head_dim), generator=_gen(cfg.seed, "q", 0),
                     dtype=torch.float32) * cfg.q_std).to(torch_dtype(cfg.dtype))
    inp = Inputs(cfg, k_pages, v_pages, k_off, q, table, lens.to(torch.int32))
    if poison:
        mark_stale_slots(inp)
    return inp


def mark_stale_slots(inp: Inputs) -> None:
    """Write the poison markers into every slot at or past each sequence's length."""
    used = set()
    for b in range(inp.cfg.batch):
        L = int(inp.seq_lens[b])
        row = inp.block_table[b]
        for j in range(inp.max_blocks):
            p = int(row[j])
            if p < 0:
                break
            t0 = L - j * BLOCK
            if t0 >= BLOCK:
                continue
            if p in used:
                continue
            used.add(p)
            t0 = max(t0, 0)
            inp.k_pages[p, :, t0:, :] = POISON_K
            inp.v_pages[p, :, t0:, :] = POISON_V


@dataclasses.dataclass
class StepTokens:
    """One decode step of the best-of-N workload: the new token's q, k and v per sample,
    and where its k and v go (position L_b of each sequence before the step)."""

    q: torch.Tensor        # [batch, num_q_heads, head_dim]
    k_new: torch.Tensor    # [batch, num_kv_heads, head_dim]
    v_new: torch.Tensor    # [batch, num_kv_heads, head_dim]
    pages: torch.Tensor    # [batch] int64 physical page of position L_b
    slots: torch.Tensor    # [batch] int64 slot of position L_b in that page


def step_tokens(inp: Inputs, step: int) -> StepTokens:
    """Draw the q / k / v of decode step `step` (k carries its page's offset vector)."""
    cfg = inp.cfg
    g = _gen(cfg.seed, "step", step)
    B, H, Hq, d = cfg.batch, cfg.num_kv_heads, cfg.num_q_heads, cfg.head_dim
    q = torch.randn((B, Hq, d), generator=g, dtype=torch.float32) * cfg.q_std
    k = torch.randn((B, H, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, d), generator=g, dtype=torch.float32)
    L = inp.seq_lens.to(torch.int64)
    pages = inp.block_table[torch.arange(B), L // BLOCK].to(torch.int64)
    k += inp.k_offset[pages]
    dt = torch_dtype(cfg.dtype)
    return StepTokens(q.to(dt), k.to(dt), v.to(dt), pages, L % BLOCK)


def write_step_tokens(inp: Inputs, tok: StepTokens) -> torch.Tensor:
    """Append one token per sequence into the host cache (the caller's job in decode).

    Writes k_new / v_new at position L_b, advances seq_lens, replaces q, and returns the
    physical ids of the pages that this write completed (16 valid tokens now).
    """
    pages, slots = tok.pages, tok.slots
    inp.k_pages[pages, :, slots, :] = tok.k_new
    inp.v_pages[pages, :, slots, :] = tok.v_new
    inp.seq_lens += 1
    inp.q = tok.q
    done = (slots == BLOCK - 1)
    return pages[done].to(torch.int32)


def decode_plan(inp: Inputs) -> List[Optional[StepTokens]]:
    """The tokens of the workload's decode steps 0 .. steps-1, advancing the host state.

    Step 0 decodes the initial state (its current token is already in the cache: entry
    None); step t >= 1 first appends the token it draws at position L_b of every sequence.
    The host cache ends in the state of the last step.  Pages were allocated for every
    step's token by ``generate``.
    """
    plan: List[Optional[StepTokens]] = [None]
    for t in range(1, inp.cfg.steps):
        tok = step_tokens(inp, t)
        write_step_tokens(inp, tok)
        plan.append(tok)
    return plan


def qwen3_sizes(cfg: Config) -> dict:
    """Shape summary used in reports (no arithmetic of the method)."""
    return dict(batch=cfg.batch, num_q_heads=cfg.num_q_heads, num_kv_heads=cfg.num_kv_heads,
                head_dim=cfg.head_dim, top_k=cfg.top_k, dtype=cfg.dtype, block=BLOCK)


def sample_rows(cfg: Config, n: int, seed: int = 7) -> List[tuple]:
    """A seeded sample of (sequence, KV head) rows for sampled parity checks."""
    g = _gen(cfg.seed, "sample", seed)
    total = cfg.batch * cfg.num_kv_heads
    n = min(n, total)
    idx = torch.randperm(total, generator=g)[:n].tolist()
    return sorted((i // cfg.num_kv_heads, i % cfg.num_kv_heads) for i in idx)


def host_arrays(inp: Inputs) -> dict:
    """The whole workload as numpy arrays (float32 values of the stored dtype)."""
    return dict(q=inp.q.float().numpy(), k_pages=inp.k_pages.float().numpy(),
                v_pages=inp.v_pages.float().numpy(),
                block_table=inp.block_table.numpy().astype("int64"),
                seq_lens=inp.seq_lens.numpy().astype("int64"))


def row_problem(inp: Inputs, b: int, h: int) -> dict:
    """The inputs one (sequence b, KV head h) row reads, as a one-row numpy problem.

    The row's pages are gathered in logical block order (page j of the result is the
    row's logical block j), so the problem has batch 1, one KV head and an identity
    page table.  Used to check sampled rows of full-size workloads one by one.
    """
    G = inp.cfg.group
    L = int(inp.seq_lens[b])
    nb = (L + BLOCK - 1) // BLOCK
    pages = inp.block_table[b, :nb].to(torch.int64)
    return dict(q=inp.q[b:b + 1, h * G:(h + 1) * G].float().numpy(),
                k_pages=inp.k_pages[pages, h:h + 1].float().numpy(),
                v_pages=inp.v_pages[pages, h:h + 1].float().numpy(),
                block_table=torch.arange(nb, dtype=torch.int64)[None, :].numpy(),
                seq_lens=torch.tensor([L], dtype=torch.int64).numpy())


def find_config(name_or_index) -> Config:
    if isinstance(name_or_index, int):
        return CONFIGS[name_or_index]
    for c in CONFIGS:
        if c.name == name_or_index:
            return c
    raise KeyError(name_or_index)


__all__ = ["BLOCK", "POISON_K", "POISON_V", "Config", "CONFIGS", "Inputs", "StepTokens",
           "generate", "step_tokens", "write_step_tokens", "decode_plan", "mark_stale_slots",
           "sample_rows", "find_config", "host_arrays", "row_problem", "torch_dtype", "qwen3_sizes"]
