#!/usr/bin/env python3
"""Benchmark of block top-k decode attention (one attention layer).

Default workload: best-of-N decode, Qwen3-14B-shaped (256 samples, 40 query / 8 KV heads,
head_dim 128, bf16, a shared 1024-token prompt plus generated lengths U[2048, 16384],
top-128 pages of 16 tokens), 64 consecutive decode steps, synthetic seeded inputs.  One
timed step = one decode step of that loop: the block top-k decode (score, select, sparse
attention with its split merge, and the centroid append of the pages the step's token
completed).  Each step's K/V token write and seq_lens advance (the caller's part) run
before it, outside its timed events, and are reported separately.  The Qwen3-0.6B, -8B and
-32B-shaped single-step workloads are measured in the same run and reported under
"configs".

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle instead (the
reference arm): rank 0 only, a bounded sample of rows per step on all host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-top-k decode: seq-steps/s, achieved HBM GB/s vs peak, speedup vs dense"
UNIT = "seq-steps/s"
L2_FLUSH_BYTES = 256 << 20       # > 126 MB of L2
# every source the fused decode kernel is compiled from (its launch plan included)
KERNEL_SOURCES = [os.path.join(ROOT, "block_top_sparse_centroid_b300", "csrc", f)
                  for f in ("decode_fused.cu", "attn_common.cuh", "kin_common.cuh",
                            "kin_internal.h", "kin_api.cu")]


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--config", type=int, default=4, help="workload index (0..4)")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (small profiling cases)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-shared-prefix", action="store_true",
                    help="best-of-N loop: do not pass the prompt's blocks as the shared-prefix hint")
    ap.add_argument("--no-hint-compare", action="store_true",
                    help="best-of-N loop: skip the comparison run without the shared-prefix hint")
    ap.add_argument("--no-token", action="store_true",
                    help="skip the token-level (oracle) top-k decode of the same step")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-others", action="store_true",
                    help="skip the single-step Qwen3 workloads reported under \"configs\"")
    ap.add_argument("--other-steps", type=int, default=30)
    return ap.parse_args(argv)


def max_over_ranks(x: float, world: int, device) -> float:
    """A per-rank time reduced to the job's: its slowest rank (identity on one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_config(cfg, rank: int):
    """Replicas decode batches of the same shapes with their own seeds (rank 0: the
    workload itself), so the job processes world x batch sequences per step."""
    return cfg.scaled(seed=cfg.seed + 1000 * rank) if rank else cfg


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units all ranks processed per second of the slowest rank."""
    return units_per_rank * world / seconds


def workload(args):
    import workloads as W
    cfg = W.CONFIGS[args.config]
    if args.batch:
        cfg = cfg.scaled(batch=args.batch)
    return W, cfg


def describe(cfg) -> str:
    ctx = {"uniform": f"context {cfg.ctx_lo}",
           "ragged": f"contexts U[{cfg.ctx_lo}, {cfg.ctx_hi}]",
           "best_of_n": f"prefix {cfg.prefix} + U[{cfg.ctx_lo}, {cfg.ctx_hi}]",
           "explicit": "explicit contexts"}[cfg.ctx_kind]
    return (f"{cfg.name}-shaped layer decode: batch {cfg.batch}, {cfg.num_q_heads} q / "
            f"{cfg.num_kv_heads} KV heads, head_dim {cfg.head_dim}, {cfg.dtype}, {ctx}, "
            f"block 16, top-{cfg.top_k} blocks")


def kv_bytes(cfg, lens) -> dict:
    """Algorithmic bytes of one step: kept K/V tokens, scored centroids, Q read + O write."""
    es = 2 if cfg.dtype == "bf16" else 4
    H, d, k = cfg.num_kv_heads, cfg.head_dim, cfg.top_k
    kv = cent = 0
    for L in lens:
        nb = (L + 15) // 16
        toks = L if nb <= k else (k - 1) * 16 + (L - 16 * (nb - 1))
        kv += 2 * toks * H * d * es
        if nb > k:
            cent += (nb - 1) * H * d * es
    qo = 2 * len(lens) * cfg.num_q_heads * d * es
    dense_kv = sum(2 * L * H * d * es for L in lens)
    return dict(kv=kv, centroids=cent, qo=qo, dense_kv=dense_kv)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank space, so that only code changes (not
    comment or layout edits) change the fingerprint of the kernel sources."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":                                   # string / char literal, kept whole
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            while i < n and src[i] != "\n":
                i += 1
        elif src.startswith("/*", i):
            k = src.find("*/", i + 2)
            i = n if k < 0 else k + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_sha(read=None) -> str:
    """Fingerprint of the code the fused kernel is compiled from (comments excluded)."""
    read = read or (lambda f: open(f, encoding="utf-8").read())
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(strip_comments(read(f)).encode())
    return h.hexdigest()


def traffic_record(workload_name: str):
    """DRAM bytes per fused-kernel launch from the committed ncu summary, if it was taken
    on this workload and on the kernel sources as they are now (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p))
    if rec.get("source_sha256") != kernel_source_sha():
        return None
    return rec.get("workloads", {}).get(workload_name)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}




# ------------------------------------------------------------------------------- oracle
_POOL_STATE = {}


def _bf16_to_f32(x):
    import numpy as np
    return (x.astype(np.uint16).astype(np.uint32) << 16).view(np.float32)


def _pool_state(inp) -> dict:
    """Numpy views of a workload's host inputs (no copy), for the oracle's workers."""
    import torch
    bf = inp.k_pages.dtype == torch.bfloat16
    view = (lambda t: t.view(torch.int16).numpy()) if bf else (lambda t: t.numpy())
    return dict(bf16=bf, k=view(inp.k_pages), v=view(inp.v_pages), q=view(inp.q),
                table=inp.block_table.numpy(), lens=inp.seq_lens.numpy(), cfg=inp.cfg)


def _oracle_row(bh) -> int:
    """One (sequence, KV head) row of the CPU oracle, on the inputs in _POOL_STATE: the
    row's pages gathered in block order (numpy only), then the oracle as it stands."""
    import numpy as np
    import oracle as O
    st = _POOL_STATE
    cfg = st["cfg"]
    b, h = bh
    G = cfg.group
    L = int(st["lens"][b])
    nb = (L + 15) // 16
    pages = st["table"][b, :nb].astype(np.int64)
    conv = _bf16_to_f32 if st["bf16"] else (lambda x: np.asarray(x, np.float32))
    q = conv(st["q"][b:b + 1, h * G:(h + 1) * G])
    kp = conv(st["k"][pages, h:h + 1])
    vp = conv(st["v"][pages, h:h + 1])
    O.blocktopk_decode(q, kp, vp, np.arange(nb, dtype=np.int64)[None, :],
                       np.array([L], dtype=np.int64), cfg.sm_scale, cfg.top_k)
    return 1


def _pool_init():
    try:
        from threadpoolctl import threadpool_limits
        threadpool_limits(limits=1)
    except Exception:  # pragma: no cover
        pass
    try:
        # keep freed temporaries in the worker's heap: no page faults per oracle row
        import ctypes
        libc = ctypes.CDLL("libc.so.6")
        libc.mallopt(-1, 1 << 30)   # M_TRIM_THRESHOLD
        libc.mallopt(-3, 1 << 30)   # M_MMAP_THRESHOLD
    except Exception:  # pragma: no cover
        pass


class OraclePool:
    """Worker processes for timing the CPU oracle on all host cores.  They are forked
    from this process, so create the pool before the process's first CUDA call: the
    workers share the host inputs (copy on write, as numpy views) and use no torch."""

    def __init__(self, inp, workers: int):
        import multiprocessing as mp
        global _POOL_STATE
        _POOL_STATE = _pool_state(inp)
        self.cfg = inp.cfg
        self.workers = workers
        self.pool = mp.get_context("fork").Pool(workers, initializer=_pool_init)

    def close(self):
        self.pool.terminate()
        self.pool.join()

    def rate(self, seconds: float, seed: int = 11) -> dict:
        """Rows done in about `seconds`, cycling over a seeded sample of rows."""
        import workloads as W
        rows = W.sample_rows(self.cfg, 4096, seed=seed)
        self.pool.map(_oracle_row, rows[:self.workers])        # start-up, untimed
        nxt = 0
        done = 0
        t0 = time.perf_counter()
        pending = []
        for _ in range(2 * self.workers):
            pending.append(self.pool.apply_async(_oracle_row, (rows[nxt % len(rows)],)))
            nxt += 1
        while pending:
            pending[0].wait()
            r = pending.pop(0)
            done += r.get()
            if time.perf_counter() - t0 < seconds:
                pending.append(self.pool.apply_async(_oracle_row, (rows[nxt % len(rows)],)))
                nxt += 1
        return dict(rows=done, seconds=time.perf_counter() - t0)


def oracle_rate_single(inp, seconds: float, seed: int = 11) -> dict:
    """The same oracle rows in this process, one thread (BLAS limited to one)."""
    import contextlib
    import workloads as W
    global _POOL_STATE
    _POOL_STATE = _pool_state(inp)
    rows = W.sample_rows(inp.cfg, 4096, seed=seed)
    try:
        from threadpoolctl import threadpool_limits
        limit = threadpool_limits(limits=1)
    except Exception:  # pragma: no cover
        limit = contextlib.nullcontext()
    done = 0
    with limit:
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            done += _oracle_row(rows[done % len(rows)])
    return dict(rows=done, seconds=time.perf_counter() - t0)


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def worker_counts(cores: int) -> list:
    """Process counts the CPU baseline tries: all host cores, then halves down to 4."""
    out, n = [], cores
    while n >= 4 or not out:
        out.append(n)
        n //= 2
    return out


def best_pool_rate(inp, seconds: float, cores: int):
    """The oracle's row rate on `cores` processes and on fewer (halving): on some hosts
    the memory system saturates before the cores do, and fewer processes then finish
    more rows.  Returns (best rate, its process count, every measured rate)."""
    rates = {}
    for n in worker_counts(cores):
        pool = OraclePool(inp, n)
        try:
            r = pool.rate(seconds)
        finally:
            pool.close()
        rates[n] = (r["rows"], r["seconds"])
    best = max(rates, key=lambda n: rates[n][0] / rates[n][1])
    return rates[best], best, rates


def cpu_baseline(inp, seconds: float) -> dict:
    """The CPU oracle on the host cores (one process per core, on the workload's first
    decode step: the best rate over all cores and halvings of them) and on one thread, on
    a bounded sample of the workload's rows.  Call it before the process's first CUDA call
    (its workers are forked)."""
    cfg = inp.cfg
    H = cfg.num_kv_heads
    one = oracle_rate_single(inp, seconds / 3)
    counts = worker_counts(host_cores())
    (rows, secs), n, rates = best_pool_rate(inp, seconds / len(counts), host_cores())
    tried = ", ".join(f"{k} processes {v[0] / H / v[1]:.1f}" for k, v in rates.items())
    return {"value": rows / H / secs, "unit": UNIT, "cores": n, "kind": "oracle",
            "host_cores": host_cores(),
            "single_thread_value": one["rows"] / H / one["seconds"],
            "sample": f"{rows} (sequence, KV head) rows of the workload's first decode step = "
                      f"{rows / H:.1f} sequence-steps in {secs:.1f} s on {n} processes (one "
                      f"thread each, numpy; seq-steps/s tried: {tried}); one thread alone: "
                      f"{one['rows']} rows in {one['seconds']:.1f} s"}


def run_reference(args) -> int:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    W, cfg = workload(args)
    inp = W.generate(cfg)
    _, n, _ = best_pool_rate(inp, 1.0, host_cores())   # process count with the best rate
    pool = OraclePool(inp, n)
    H = cfg.num_kv_heads
    per_step_s = 1.0                     # a bounded sample of rows per step
    times, rows = [], []
    try:
        for i in range(args.warmup + args.steps):
            r = pool.rate(per_step_s, seed=100 + i)
            if i >= args.warmup:
                times.append(r["seconds"])
                rows.append(r["rows"])
    finally:
        pool.close()
    t = sum(times) / len(times)
    seq_steps = sum(rows) / len(rows) / H
    value = seq_steps / t
    sample = (f"about {seq_steps:.1f} sequence-steps ({sum(rows) // len(rows)} (sequence, KV "
              f"head) rows) per step, cycling over a seeded row sample of the workload's "
              f"first decode step, on {pool.workers} processes (one thread each)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(cfg), "batch": cfg.batch, "sample_per_step": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.workers, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------------- GPU
class Ctx:
    """Process-wide state of one benchmark run."""

    def __init__(self):
        import torch
        import torch.distributed as dist
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        local = int(os.environ.get("LOCAL_RANK", "0"))
        if self.world > 1:
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        self.dev = torch.device("cuda", local)
        torch.cuda.set_device(self.dev)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=self.dev)
        self.peak, self.peak_kind = peaks()

    def barrier(self):
        import torch
        import torch.distributed as dist
        torch.cuda.synchronize()
        if self.world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def job_seconds(self, ms_list) -> float:
        return max_over_ranks(sum(ms_list) / len(ms_list) / 1e3, self.world, self.dev)


class DeviceWorkload:
    """A workload's decode state on the device: cache, centroids of the complete pages
    (those the current token just completed excepted: the decode appends them)."""

    def __init__(self, cx, cfg, inp=None):
        import torch
        import workloads as W
        import block_top_sparse_centroid_b300 as K
        self.cfg = cfg
        self.inp = inp = inp if inp is not None else W.generate(cfg)
        dev = cx.dev
        self.lens0 = [int(x) for x in inp.seq_lens]
        self.cache = K.PagedKVCache(inp.k_pages.to(dev), inp.v_pages.to(dev))
        self.q = inp.q.to(dev)
        self.table = inp.block_table.to(dev)
        self.seq0 = inp.seq_lens.to(dev)
        self.seq = self.seq0.clone()
        self.cents = torch.zeros(self.cache.centroid_shape, dtype=self.q.dtype, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        last = inp.last_pages().tolist()
        self.just = [int(p) for b, p in enumerate(last) if self.lens0[b] % 16 == 0]
        before = sorted(set(inp.complete_pages().tolist()) - set(self.just))
        K.centroids_build(self.cache, self.cents,
                          page_ids=torch.tensor(before, dtype=torch.int32, device=dev),
                          err_flag=self.err)
        self.out = torch.empty_like(self.q)
        self.ws = K.Workspace(dev)
        self.wsd = K.Workspace(dev)

    def step_bytes(self, lens, appended: int) -> dict:
        cfg = self.cfg
        byt = kv_bytes(cfg, lens)
        es = 2 if cfg.dtype == "bf16" else 4
        # the appended centroids: two bf16 codes (or one fp32 value) per element
        byt["append"] = appended * cfg.num_kv_heads * cfg.head_dim * es * (2 if es == 2 else 1)
        byt["step"] = byt["kv"] + byt["centroids"] + byt["qo"] + byt["append"]
        return byt


def timed_graphs(cx, step_fns, n_warm: int, n_steps: int):
    """Capture each decode step into its own CUDA graph (with external event-record nodes
    around its kernels), then replay: n_warm untimed steps, then exactly n_steps timed
    ones, cycling over the graphs in order (graph 0 restores the initial state).  The L2 is
    flushed (a write larger than it) before every step, outside the events.  Returns the
    per-step event times (ms) and, per step, the index of its graph."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(6)]
           for _ in step_fns]
    for i, fn in enumerate(step_fns):          # eager warm-up of every step
        cx.flush.zero_()
        fn(evs[i])
    torch.cuda.synchronize()
    graphs = []
    for i, fn in enumerate(step_fns):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            fn(evs[i])
        graphs.append(g)
    n = len(graphs)
    for i in range(max(n_warm, 1)):
        cx.flush.zero_()
        graphs[i % n].replay()
    cx.barrier()
    res = dict(step_ms=[], kern_ms=[], write_ms=[], phase_ms=[], idx=[])
    for i in range(n_steps):
        j = i % n
        cx.flush.zero_()                         # L2 flush, outside the timed events
        graphs[j].replay()
        e = evs[j]
        e[3].synchronize()
        res["step_ms"].append(e[0].elapsed_time(e[3]))
        res["kern_ms"].append(e[2].elapsed_time(e[3]))
        res["write_ms"].append(e[4].elapsed_time(e[5]))
        res["phase_ms"].append([e[k].elapsed_time(e[k + 1]) for k in range(3)])
        res["idx"].append(j)
    cx.barrier()
    return res


def run_single(cx, cfg, n_warm, n_steps, want_dense=True, want_e2e=True, inp=None):
    """One decode step of a single-step workload, timed as a graph replay."""
    import torch
    import block_top_sparse_centroid_b300 as K
    dw = DeviceWorkload(cx, cfg, inp)

    def step(evs, dense):
        evs[4].record()
        evs[5].record()
        if dense:
            K.decode_timed(dw.cache, dw.q, dw.table, dw.seq, cfg.sm_scale, evs[:4], dense=True,
                           out=dw.out, workspace=dw.wsd, err_flag=dw.err)
        else:
            K.decode_timed(dw.cache, dw.q, dw.table, dw.seq, cfg.sm_scale, evs[:4],
                           centroids=dw.cents, top_k=cfg.top_k, out=dw.out, workspace=dw.ws,
                           err_flag=dw.err, append_final=True)

    clocks = ClockSampler(cx.dev.index)
    sp = timed_graphs(cx, [lambda e: step(e, False)], n_warm, n_steps)
    clk = clocks.stop()
    de = timed_graphs(cx, [lambda e: step(e, True)], n_warm, n_steps) if want_dense else None
    torch.cuda.synchronize()
    if int(dw.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(dw.err.item())}")
    byt = dw.step_bytes(dw.lens0, len(dw.just))
    r = summarize(cx, cfg, sp, [byt["step"]], de, [byt["dense_kv"] + byt["qo"]])
    r["clocks"] = clk
    if want_e2e:
        r["e2e"] = e2e_single(cx, dw, n_warm, n_steps)
    return r, dw


def token_bytes(cfg, lens, budget: int) -> dict:
    """Algorithmic bytes of one token top-k step (every key read once to score it, the kept
    tokens' keys and values read again to attend, q and out) and of its score kernel alone
    (the keys, q, and one fp32 score written per token)."""
    H, d, G = cfg.num_kv_heads, cfg.head_dim, cfg.group
    es = 2 if cfg.dtype == "bf16" else 4
    ntok = sum(lens)
    all_k = ntok * H * d * es
    kept = sum(min(L, budget) for L in lens) * H * 2 * d * es
    qo = 2 * len(lens) * H * G * d * es
    return {"step": all_k + kept + qo, "score_kernel": all_k + len(lens) * H * G * d * es + ntok * H * 4,
            "all_k": all_k, "kept_kv": kept, "qo": qo}


def run_token(cx, cfg, dw, n_warm, n_steps) -> dict:
    """The token-level (oracle) top-k decode of the same step (budget: 16 tokens per kept
    block, the equal-KV budget), timed like the block decode: score, select and attend
    kernel times, the step rate, and the score kernel's roofline (it streams every key)."""
    import torch
    import block_top_sparse_centroid_b300 as K
    budget = 16 * cfg.top_k
    ws = K.Workspace(cx.dev)

    def step(evs):
        evs[4].record()
        evs[5].record()
        K.token_topk_decode(dw.cache, dw.q, dw.table, dw.seq0, budget, cfg.sm_scale, out=dw.out,
                            workspace=ws, err_flag=dw.err, events=evs[:4])

    sp = timed_graphs(cx, [step], n_warm, n_steps)
    torch.cuda.synchronize()
    if int(dw.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(dw.err.item())}")
    byt = token_bytes(cfg, dw.lens0, budget)
    step_s = cx.job_seconds(sp["step_ms"])
    ph = [sum(x[k] for x in sp["phase_ms"]) / len(sp["phase_ms"]) for k in range(3)]
    score_gbs = byt["score_kernel"] / (ph[0] / 1e3) / 1e9
    return {"budget_tokens": budget, "value": whole_job_rate(cfg.batch, cx.world, step_s),
            "unit": UNIT, "ms_per_step": step_s * 1e3,
            "score_us": ph[0] * 1e3, "select_us": ph[1] * 1e3, "attend_us": ph[2] * 1e3,
            "bytes_per_step": byt["step"],
            "step_gbs": byt["step"] / step_s / 1e9,
            "roofline": {"bound": "hbm", "kernel": "token_score_kernel", "achieved": score_gbs,
                         "peak": cx.peak, "unit": "GB/s", "frac": score_gbs / cx.peak,
                         "bytes_per_launch": byt["score_kernel"], "launch_us": ph[0] * 1e3},
            "launches": 3 * len(sp["idx"])}


def summarize(cx, cfg, sp, step_bytes, de, dense_bytes) -> dict:
    """Rates, roofline and dense comparison from per-step event times."""
    B = cfg.batch
    step_s = cx.job_seconds(sp["step_ms"])
    kern_s = sum(sp["kern_ms"]) / len(sp["kern_ms"]) / 1e3
    tot_bytes = sum(step_bytes[j] for j in sp["idx"])
    achieved = tot_bytes / (sum(sp["kern_ms"]) / 1e3) / 1e9
    r = {"value": whole_job_rate(B, cx.world, step_s), "ms_per_step": step_s * 1e3,
         "kernel_us": kern_s * 1e6, "bytes_per_step": tot_bytes / len(sp["idx"]),
         "achieved_gbs": achieved, "frac": achieved / cx.peak,
         "token_write_us": sum(sp["write_ms"]) / len(sp["write_ms"]) * 1e3,
         "launches": len(sp["idx"])}
    if de is not None:
        dense_s = cx.job_seconds(de["step_ms"])
        dbytes = sum(dense_bytes[j] for j in de["idx"])
        r["dense"] = {"ms_per_step": dense_s * 1e3,
                      "seq_steps_per_s": whole_job_rate(B, cx.world, dense_s),
                      "hbm_gbs": dbytes / (sum(de["kern_ms"]) / 1e3) / 1e9,
                      "speedup_blocktopk_over_dense": dense_s / step_s}
        r["launches"] += len(de["idx"])
    return r


def e2e_single(cx, dw, n_warm, n_steps) -> dict:
    """The same step through the public API with host buffers: pinned q in, out back."""
    import torch
    import block_top_sparse_centroid_b300 as K
    cfg = dw.cfg
    stream = torch.cuda.current_stream(cx.dev)
    q_host = dw.inp.q.clone().pin_memory()
    out_host = torch.empty_like(dw.inp.q).pin_memory()
    e_ms = []
    for i in range(n_warm + n_steps):
        cx.flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dw.q.copy_(q_host, non_blocking=True)
        K.blocktopk_decode(dw.cache, dw.q, dw.table, dw.seq, dw.cents, cfg.top_k, cfg.sm_scale,
                           out=dw.out, workspace=dw.ws, err_flag=dw.err, append_final=True)
        out_host.copy_(dw.out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= n_warm:
            e_ms.append(e0.elapsed_time(e1))
    e_s = cx.job_seconds(e_ms)
    return {"value": whole_job_rate(cfg.batch, cx.world, e_s), "unit": UNIT,
            "h2d_bytes_per_step": q_host.numel() * q_host.element_size(),
            "d2h_bytes_per_step": out_host.numel() * out_host.element_size(),
            "ms_per_step": e_s * 1e3,
            "path": "public Python API over the C ABI; pinned host q in, host out back, per "
                    "step; L2 flushed between steps outside the timed region"}


class LoopPlan:
    """The best-of-N decode loop on the device: every step's tokens, where they go, and
    the sequence lengths and appended pages of every step (known on the host)."""

    def __init__(self, cx, dw):
        import torch
        import workloads as W
        inp = dw.inp
        self.q0_host = inp.q.clone()            # step 0's queries (the plan replaces inp.q)
        plan = W.decode_plan(inp)               # advances the host state to the last step
        self.n = len(plan)
        dev = cx.dev
        cfg = dw.cfg
        self.q = [dw.q] + [t.q.to(dev) for t in plan[1:]]
        self.k_new = [None] + [t.k_new.to(dev) for t in plan[1:]]
        self.v_new = [None] + [t.v_new.to(dev) for t in plan[1:]]
        self.pages = [None] + [t.pages.to(dev) for t in plan[1:]]
        self.slots = [None] + [t.slots.to(dev) for t in plan[1:]]
        self.lens = [list(dw.lens0)]
        for t in range(1, self.n):
            self.lens.append([x + 1 for x in self.lens[-1]])
        self.appended = [sum(1 for L in lens if L % 16 == 0) for lens in self.lens]
        self.host_tokens = plan
        self.bytes = [dw.step_bytes(lens, a) for lens, a in zip(self.lens, self.appended)]


def run_loop(cx, cfg, n_warm, n_steps, want_dense=True, want_e2e=True, inp=None, shared=0):
    """The best-of-N loop: step t (t >= 1) writes each sample's new token into its page
    (torch indexing: the caller's part) and advances seq_lens, then decodes; step 0 decodes
    the initial state and restores it first, so the steps replay in a cycle.  shared: the
    prompt's blocks, passed as the decode's shared-prefix hint (block top-k and dense)."""
    import torch
    import block_top_sparse_centroid_b300 as K
    dw = DeviceWorkload(cx, cfg, inp)
    lp = LoopPlan(cx, dw)

    def step(t, evs, dense):
        evs[4].record()
        if t == 0:
            dw.seq.copy_(dw.seq0)
        else:
            dw.cache.k_pages[lp.pages[t], :, lp.slots[t], :] = lp.k_new[t]
            dw.cache.v_pages[lp.pages[t], :, lp.slots[t], :] = lp.v_new[t]
            dw.seq.add_(1)
        evs[5].record()
        if dense:
            K.decode_timed(dw.cache, lp.q[t], dw.table, dw.seq, cfg.sm_scale, evs[:4], dense=True,
                           out=dw.out, workspace=dw.wsd, err_flag=dw.err,
                           shared_prefix_blocks=shared)
        else:
            K.decode_timed(dw.cache, lp.q[t], dw.table, dw.seq, cfg.sm_scale, evs[:4],
                           centroids=dw.cents, top_k=cfg.top_k, out=dw.out, workspace=dw.ws,
                           err_flag=dw.err, append_final=True, shared_prefix_blocks=shared)

    clocks = ClockSampler(cx.dev.index)
    sp = timed_graphs(cx, [lambda e, t=t: step(t, e, False) for t in range(lp.n)], n_warm, n_steps)
    clk = clocks.stop()
    de = (timed_graphs(cx, [lambda e, t=t: step(t, e, True) for t in range(lp.n)], n_warm, n_steps)
          if want_dense else None)
    torch.cuda.synchronize()
    if int(dw.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(dw.err.item())}")
    r = summarize(cx, cfg, sp, [b["step"] for b in lp.bytes], de,
                  [b["dense_kv"] + b["qo"] for b in lp.bytes])
    r["clocks"] = clk
    r["unique"] = unique_bytes_step0(cx, dw, lp)
    if want_e2e:
        r["e2e"] = e2e_loop(cx, dw, lp, n_warm, n_steps, shared)
    return r, dw


def unique_bytes_step0(cx, dw, lp) -> dict:
    """Logical and unique (each physical page read once) bytes of the loop's first step,
    from the kept lists of an untimed decode of the initial state."""
    import torch
    import numpy as np
    import block_top_sparse_centroid_b300 as K
    cfg = dw.cfg
    B, H, k = cfg.batch, cfg.num_kv_heads, cfg.top_k
    dw.seq.copy_(dw.seq0)
    sel = torch.full((B, H, k), -1, dtype=torch.int32, device=cx.dev)
    K.blocktopk_decode(dw.cache, lp.q[0], dw.table, dw.seq, dw.cents, k, cfg.sm_scale,
                       out=dw.out, sel_blocks=sel, workspace=dw.ws, err_flag=dw.err,
                       append_final=True)
    sel = sel.cpu().numpy()
    table = dw.inp.block_table.numpy()
    es = 2
    kv_pairs, cent_pairs = {}, set()
    for b in range(B):
        L = dw.lens0[b]
        nb = (L + 15) // 16
        for h in range(H):
            for j in sel[b, h]:
                if j < 0:
                    continue
                key = (int(table[b, j]), h)
                kv_pairs[key] = max(kv_pairs.get(key, 0), min(16, L - 16 * int(j)))
            if nb > k:
                for j in range(nb - 1):
                    cent_pairs.add((int(table[b, j]), h))
    d = cfg.head_dim
    uniq = 2 * sum(kv_pairs.values()) * d * es + len(cent_pairs) * d * es + lp.bytes[0]["qo"]
    return {"logical_bytes": lp.bytes[0]["step"] - lp.bytes[0]["append"],
            "unique_bytes": uniq,
            "note": "first decode step without its centroid appends; unique counts each "
                    "(physical page, KV head) once although several samples read it"}


def e2e_loop(cx, dw, lp, n_warm, n_steps, shared=0) -> dict:
    """The loop through the public API with host buffers: per step the token's q, k, v and
    its positions go host -> device from pinned memory, the caller writes k, v into the
    cache and advances seq_lens, one block top-k decode runs, and out comes back."""
    import torch
    import block_top_sparse_centroid_b300 as K
    cfg = dw.cfg
    stream = torch.cuda.current_stream(cx.dev)
    pin = lambda t: t.clone().pin_memory()  # noqa: E731
    hq = [pin(lp.q0_host if t == 0 else lp.host_tokens[t].q) for t in range(lp.n)]
    hk = [None] + [pin(lp.host_tokens[t].k_new) for t in range(1, lp.n)]
    hv = [None] + [pin(lp.host_tokens[t].v_new) for t in range(1, lp.n)]
    hp = [None] + [pin(lp.host_tokens[t].pages) for t in range(1, lp.n)]
    hs = [None] + [pin(lp.host_tokens[t].slots) for t in range(1, lp.n)]
    out_host = torch.empty_like(hq[0]).pin_memory()
    q_dev = torch.empty_like(dw.q)
    k_dev = torch.empty_like(lp.k_new[1])
    v_dev = torch.empty_like(lp.v_new[1])
    p_dev = torch.empty_like(lp.pages[1])
    s_dev = torch.empty_like(lp.slots[1])
    h2d = d2h = 0
    e_ms = []
    for i in range(n_warm + n_steps):
        t = i % lp.n
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        q_dev.copy_(hq[t], non_blocking=True)
        nb_in = hq[t].numel() * hq[t].element_size()
        if t == 0:
            dw.seq.copy_(dw.seq0)
        else:
            for dst, src in ((k_dev, hk[t]), (v_dev, hv[t]), (p_dev, hp[t]), (s_dev, hs[t])):
                dst.copy_(src, non_blocking=True)
                nb_in += src.numel() * src.element_size()
            dw.cache.k_pages[p_dev, :, s_dev, :] = k_dev
            dw.cache.v_pages[p_dev, :, s_dev, :] = v_dev
            dw.seq.add_(1)
        K.blocktopk_decode(dw.cache, q_dev, dw.table, dw.seq, dw.cents, cfg.top_k, cfg.sm_scale,
                           out=dw.out, workspace=dw.ws, err_flag=dw.err, append_final=True,
                           shared_prefix_blocks=shared)
        out_host.copy_(dw.out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= n_warm:
            e_ms.append(e0.elapsed_time(e1))
            h2d += nb_in
            d2h += out_host.numel() * out_host.element_size()
    e_s = cx.job_seconds(e_ms)
    return {"value": whole_job_rate(cfg.batch, cx.world, e_s), "unit": UNIT,
            "h2d_bytes_per_step": h2d // n_steps, "d2h_bytes_per_step": d2h // n_steps,
            "ms_per_step": e_s * 1e3,
            "path": "public Python API over the C ABI, per decode step of the loop: pinned host "
                    "q, k, v and token positions in, the K/V token write and seq_lens advance "
                    "(torch indexing), one block top-k decode, out back to pinned host memory"}


def main() -> int:
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    W, cfg = workload(args)
    cfg = replica_config(cfg, int(os.environ.get("RANK", "0")))
    inp = W.generate(cfg)
    cpu = None
    if int(os.environ.get("RANK", "0")) == 0 and not args.no_cpu_baseline:
        # The oracle on the host cores, before this process touches the GPU: its workers
        # are forked before the first CUDA call and run while nothing else does.
        cpu = cpu_baseline(inp, args.cpu_seconds)
    cx = Ctx()
    loop = cfg.ctx_kind == "best_of_n" and cfg.steps > 1
    shared = cfg.prefix // 16 if loop and not args.no_shared_prefix else 0
    no_hint = None
    if shared and not args.no_hint_compare:
        # the same loop without the hint, for the comparison (kernel time only), on inputs of
        # its own (a loop advances its host inputs to its last step)
        r0, dw0 = run_loop(cx, cfg, 5, min(args.steps, args.other_steps), False, False,
                           W.generate(cfg), 0)
        no_hint = {"kernel_us": r0["kernel_us"], "achieved_gbs": r0["achieved_gbs"],
                   "frac": r0["frac"], "steps": min(args.steps, args.other_steps),
                   "launches": r0["launches"]}
        del dw0
        torch.cuda.empty_cache()
    if loop:
        r, dw = run_loop(cx, cfg, args.warmup, args.steps, not args.no_dense, not args.no_e2e,
                         inp, shared)
    else:
        r, dw = run_single(cx, cfg, args.warmup, args.steps, not args.no_dense, not args.no_e2e,
                           inp)
    trec = traffic_record(describe(cfg))
    if no_hint:
        r["launches"] += no_hint["launches"]
    tok = None
    if cfg.dtype == "bf16" and not args.no_token:
        # the decode's initial state (positions below the initial lengths are untouched by
        # the loop's token writes)
        tok = run_token(cx, cfg, dw, 5, min(args.steps, args.other_steps))
        r["launches"] += tok["launches"]
    del dw
    torch.cuda.empty_cache()

    others = {}
    if not args.no_others and args.config == 4 and not args.batch:
        for i in (1, 2, 3):
            oc = replica_config(W.CONFIGS[i], cx.rank)
            o, odw = run_single(cx, oc, 5, args.other_steps, not args.no_dense, False)
            otok = None if args.no_token else run_token(cx, oc, odw, 5, args.other_steps)
            if otok is not None:
                r["launches"] += otok["launches"]
            del odw
            torch.cuda.empty_cache()
            orec = traffic_record(describe(oc))
            others[oc.name] = {
                "workload": describe(oc), "value": o["value"], "unit": UNIT,
                "ms_per_step": o["ms_per_step"], "steps": args.other_steps,
                "roofline": {"bound": "hbm", "achieved": o["achieved_gbs"], "peak": cx.peak,
                             "unit": "GB/s", "frac": o["frac"],
                             "traffic": orec["dram_bytes_per_launch"] if orec else None,
                             "bytes_per_launch": o["bytes_per_step"],
                             "launch_us": o["kernel_us"]},
                "dense": o.get("dense"), "clocks": o["clocks"], "token_topk": otok}
            r["launches"] += o["launches"]

    per_launch_kernel = "fused_decode_kernel" if cfg.dtype == "bf16" else "attn_f32_kernel"
    line = {
        "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": cx.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic",
        "config": {"workload": describe(cfg), "batch": cfg.batch,
                   "num_q_heads": cfg.num_q_heads, "num_kv_heads": cfg.num_kv_heads,
                   "head_dim": cfg.head_dim, "top_k": cfg.top_k,
                   "decode_steps_per_loop": cfg.steps if loop else 1,
                   "parallelism": f"replicas x{cx.world}" if cx.world > 1 else "single GPU",
                   "l2": "flushed (256 MB write) before every timed step, outside the timed "
                         "events",
                   "step": ("one decode step of the best-of-N loop: block top-k decode (score, "
                            "select, split-KV attention with merge) and the centroid append of "
                            "the pages the step's token completed, one fused kernel; the "
                            "caller's K/V token write and seq_lens advance run before it, "
                            "outside its events" if loop else
                            "one block top-k decode call: score, select, split-KV attention "
                            "with merge, and the centroid append of the pages the current token "
                            "completed (fused, one kernel for bf16)")},
        "roofline": {"bound": "hbm", "kernel": per_launch_kernel, "achieved": r["achieved_gbs"],
                     "peak": cx.peak, "unit": "GB/s", "frac": r["frac"],
                     "peak_source": f"{cx.peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "bytes_per_launch": r["bytes_per_step"], "launch_us": r["kernel_us"],
                     "traffic": trec["dram_bytes_per_launch"] if trec else None},
        "token_write_us": r["token_write_us"] if loop else None,
        "gpu_launches": r["launches"] + (args.steps if r.get("e2e") else 0),
        "clocks": r["clocks"],
        "e2e": r.get("e2e"),
        "dense": r.get("dense"),
        "token_topk": tok,
    }
    if loop:
        line["roofline"]["unique_step0"] = r["unique"]
        line["shared_prefix"] = {
            "blocks": shared,
            "what": "the prompt's blocks passed as kin_decode_args.shared_prefix_blocks: their "
                    "pages' K, V and centroid copies use the L2 evict-last policy, every other "
                    "copy evict-first (block top-k and dense decode alike)",
            "without_hint": no_hint}
    if others:
        line["configs"] = others
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if cx.rank == 0:
        print(json.dumps(line))
    if cx.world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
