#!/usr/bin/env python3
"""Benchmark of block top-k decode attention (one attention layer, one decode step).

Default workload: the Qwen3-0.6B-shaped layer decode (batch 64, 16 query / 8 KV heads,
head_dim 128, bf16, uniform context 8192, top-64 pages of 16 tokens), synthetic seeded
inputs.  One timed step = the centroid append of the pages the current token completed
+ one block top-k decode (score, select, sparse attention with its split merge).

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle instead (the
reference arm): rank 0 only, a bounded sample of rows per step.

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
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=1, help="workload index (0..4)")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (small profiling cases)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
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


def cpu_baseline(inp, cfg, seconds: float, rows_cap: int = 100000) -> dict:
    """The CPU oracle as it stands, on a bounded sample of the workload's rows."""
    import numpy as np  # noqa: F401
    import oracle as O
    import workloads as W
    import contextlib
    try:
        from threadpoolctl import threadpool_limits
        limit = threadpool_limits(limits=1)
    except Exception:  # pragma: no cover
        limit = contextlib.nullcontext()
    rows = W.sample_rows(cfg, rows_cap, seed=11)
    done = 0
    with limit:
        t0 = time.perf_counter()
        while True:                      # cycle over the sampled rows until the budget ends
            for b, h in rows:
                rp = W.row_problem(inp, b, h)
                O.blocktopk_decode(rp["q"], rp["k_pages"], rp["v_pages"], rp["block_table"],
                                   rp["seq_lens"], cfg.sm_scale, cfg.top_k,
                                   store="bf16" if cfg.dtype == "bf16" else "f32")
                done += 1
                if time.perf_counter() - t0 >= seconds:
                    break
            if time.perf_counter() - t0 >= seconds:
                break
        el = time.perf_counter() - t0
    seq_steps = done / cfg.num_kv_heads
    return {"value": seq_steps / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} (sequence, KV head) rows of the workload = {seq_steps:.2f} "
                      f"sequence-steps in {el:.1f} s, one thread (numpy, BLAS limited to 1)"}


def run_reference(args) -> int:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    W, cfg = workload(args)
    inp = W.generate(cfg)
    rows_per_step = max(8, min(cfg.batch * cfg.num_kv_heads, 64))
    per_step = []
    for i in range(args.warmup + args.steps):
        import oracle as O
        rows = W.sample_rows(cfg, rows_per_step, seed=100 + i)
        t0 = time.perf_counter()
        for b, h in rows:
            rp = W.row_problem(inp, b, h)
            O.blocktopk_decode(rp["q"], rp["k_pages"], rp["v_pages"], rp["block_table"],
                               rp["seq_lens"], cfg.sm_scale, cfg.top_k,
                               store="bf16" if cfg.dtype == "bf16" else "f32")
        if i >= args.warmup:
            per_step.append(time.perf_counter() - t0)
    t = sum(per_step) / len(per_step)
    seq_steps = rows_per_step / cfg.num_kv_heads
    value = seq_steps / t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(cfg), "batch": cfg.batch,
                       "sample_per_step": f"{rows_per_step} (sequence, KV head) rows"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{rows_per_step} rows per step = {seq_steps:.2f} "
                                       f"sequence-steps, one thread"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main() -> int:
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import block_top_sparse_centroid_b300 as K
    W, cfg = workload(args)
    cfg = replica_config(cfg, rank)
    inp = W.generate(cfg)
    B, H, Hq, d = cfg.batch, cfg.num_kv_heads, cfg.num_q_heads, cfg.head_dim
    lens = [int(x) for x in inp.seq_lens]

    cache = K.PagedKVCache(inp.k_pages.to(dev), inp.v_pages.to(dev))
    q = inp.q.to(dev)
    table = inp.block_table.to(dev)
    seq = inp.seq_lens.to(dev)
    cents = torch.zeros((inp.num_pages, H, d), dtype=q.dtype, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    last = inp.last_pages()
    just = [int(p) for b, p in enumerate(last.tolist()) if lens[b] % 16 == 0]
    full = set(inp.complete_pages().tolist())
    before = sorted(full - set(just))
    K.centroids_build(cache, cents, page_ids=torch.tensor(before, dtype=torch.int32, device=dev),
                      err_flag=err)
    just_dev = torch.tensor(just, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    ws = K.Workspace(dev)
    wsd = K.Workspace(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def sparse_step(evs):
        K.decode_timed(cache, q, table, seq, cfg.sm_scale, evs, centroids=cents,
                       top_k=cfg.top_k, out=out, workspace=ws, err_flag=err, append_final=True)

    def dense_step(evs):
        K.decode_timed(cache, q, table, seq, cfg.sm_scale, evs, dense=True, out=out,
                       workspace=wsd, err_flag=err)

    def timed(step_fn, n_warm, n_steps, launches_per_step):
        """Warm up eagerly, capture one step into a CUDA graph, then time n_steps replays.

        The graph holds the step's kernel(s) (and any counter memsets) with external event-record
        nodes around them, so every replay timestamps its own kernels on the device and
        no host-side marshalling or launch latency falls inside the timed region."""
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
        for _ in range(n_warm):
            flush.zero_()
            step_fn(evs)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            step_fn(evs)
        for _ in range(n_warm):
            flush.zero_()
            graph.replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        step_ms, attn_ms, score_ms, sel_ms = [], [], [], []
        for i in range(n_steps):
            flush.zero_()                       # L2 flush, outside the timed events
            graph.replay()
            evs[3].synchronize()
            step_ms.append(evs[0].elapsed_time(evs[3]))
            score_ms.append(evs[0].elapsed_time(evs[1]))
            sel_ms.append(evs[1].elapsed_time(evs[2]))
            attn_ms.append(evs[2].elapsed_time(evs[3]))
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        return dict(step_ms=step_ms, attn_ms=attn_ms, score_ms=score_ms, sel_ms=sel_ms,
                    launches=launches_per_step * n_steps)

    per_step = 1 if cfg.dtype == "bf16" else 3   # fused kernel, or score + select + attention
    clocks = ClockSampler(dev.index)
    sp = timed(sparse_step, args.warmup, args.steps, per_step)
    clk = clocks.stop()
    de = None if args.no_dense else timed(dense_step, args.warmup, args.steps, 1)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flag {int(err.item())}")

    step_s = max_over_ranks(sum(sp["step_ms"]) / len(sp["step_ms"]) / 1e3, world, dev)
    value = whole_job_rate(B, world, step_s)

    byt = kv_bytes(cfg, lens)
    es = 2 if cfg.dtype == "bf16" else 4
    append_bytes = len(just) * H * d * es      # centroid writes; the keys are already on chip
    step_bytes = byt["kv"] + byt["centroids"] + byt["qo"] + append_bytes
    # bf16: one fused kernel does the whole step; fp32: the attention kernel dominates
    attn_bytes = step_bytes if cfg.dtype == "bf16" else byt["kv"] + byt["qo"]
    attn_s = statistics.mean(sp["attn_ms"]) / 1e3
    peak, peak_kind = peaks()
    achieved = attn_bytes / attn_s / 1e9
    trec = traffic_record(describe(cfg))

    e2e = None
    if not args.no_e2e:
        q_host = inp.q.clone().pin_memory()
        out_host = torch.empty_like(inp.q).pin_memory()
        e_ms = []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            q.copy_(q_host, non_blocking=True)
            K.blocktopk_decode(cache, q, table, seq, cents, cfg.top_k, cfg.sm_scale, out=out,
                               workspace=ws, err_flag=err, append_final=True)
            out_host.copy_(out, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            if i >= args.warmup:
                e_ms.append(e0.elapsed_time(e1))
        e_s = max_over_ranks(sum(e_ms) / len(e_ms) / 1e3, world, dev)
        e2e = {"value": whole_job_rate(B, world, e_s), "unit": UNIT,
               "h2d_bytes_per_step": q_host.numel() * q_host.element_size(),
               "d2h_bytes_per_step": out_host.numel() * out_host.element_size(),
               "ms_per_step": e_s * 1e3,
               "path": "public Python API over the C ABI; pinned host q in, host out back, "
                       "per step; L2 flushed between steps outside the timed region"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
        "config": {"workload": describe(cfg), "batch": B, "num_q_heads": Hq,
                   "num_kv_heads": H, "head_dim": d, "top_k": cfg.top_k,
                   "context": lens[0] if cfg.ctx_kind == "uniform" else "per-sequence",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed (256 MB write) between timed steps, outside the timed events",
                   "step": "one block top-k decode call: score, select, split-KV attention with "
                           "merge, and the centroid append of the pages the current token "
                           "completed (fused, one kernel for bf16)"},
        "roofline": {"bound": "hbm", "kernel": "fused_decode_kernel" if cfg.dtype == "bf16" else "attn_f32_kernel",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "bytes_per_launch": attn_bytes,
                     "launch_us": attn_s * 1e6,
                     "traffic": (trec["dram_bytes_per_launch"] if trec else None)},
        "step_hbm": {"bytes": step_bytes, "gbs": step_bytes / step_s / 1e9,
                     "frac": step_bytes / step_s / 1e9 / peak},
        "kernels_us": ({"before_kernel": statistics.mean(sp["score_ms"]) * 1e3,
                        "fused_decode_kernel": attn_s * 1e6} if cfg.dtype == "bf16" else
                       {"score": statistics.mean(sp["score_ms"]) * 1e3,
                        "select": statistics.mean(sp["sel_ms"]) * 1e3,
                        "attention": attn_s * 1e6}),
        "gpu_launches": sp["launches"] + (e2e is not None) * per_step * args.steps,
        "clocks": clk,
        "e2e": e2e,
    }
    if de is not None:
        dense_s = max_over_ranks(sum(de["step_ms"]) / len(de["step_ms"]) / 1e3, world, dev)
        line["dense"] = {"ms_per_step": dense_s * 1e3, "seq_steps_per_s": whole_job_rate(B, world, dense_s),
                         "hbm_gbs": (byt["dense_kv"] + byt["qo"]) / dense_s / 1e9,
                         "speedup_blocktopk_over_dense": dense_s / step_s}
        line["gpu_launches"] += de["launches"]
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, cfg, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
