"""The benchmark's multi-process path on CPU: two ranks over gloo, as `torchrun` launches
them with N > 1.  The path shards without any exchange (each replica decodes its own batch;
every (sequence, KV head) row is independent), so the only cross-rank steps are the
reduction of each timing to the slowest rank and the whole-job rate; the reference arm runs
on rank 0 alone."""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        per_rank_s = 0.010 * (rank + 1)                    # rank 1 is the slower one
        job_s = bench.max_over_ranks(per_rank_s, world, "cpu")
        rate = bench.whole_job_rate(64, world, job_s)
        base = W.find_config("qwen3-0.6b")
        mine = bench.replica_config(base, rank)
        same_shapes = mine.scaled(seed=0) == base.scaled(seed=0)
        # the reference arm: every rank but 0 returns at once, without work
        ref_rc = bench.run_reference(bench.parse(["--impl", "reference", "--steps", "1",
                                                  "--warmup", "0"])) if rank else None
        out.put((rank, job_s, rate, mine.seed, same_shapes, ref_rc))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_over_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, job_s, rate, seed, same_shapes, ref_rc = out.get(timeout=120)
        res[rank] = (job_s, rate, seed, same_shapes, ref_rc)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks report the slowest rank's time and the same whole-job rate
    assert res[0][0] == res[1][0] == 0.020
    assert res[0][1] == res[1][1] == 64 * 2 / 0.020
    # replicas: same shapes, different seeds (each decodes its own batch)
    assert res[0][2] != res[1][2]
    assert res[0][3] and res[1][3]
    # the reference arm ran on rank 0 only
    assert res[1][4] == 0
