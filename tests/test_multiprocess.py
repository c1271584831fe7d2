"""The multi-rank plumbing of bench.py on CPU: world size 2 over gloo.

The hot path shards into independent problems (one per rank, no data-path
collective); the only cross-rank steps are the timing barrier and the max over
ranks of the measured times, and only rank 0 prints.  These run as two spawned
processes with a gloo process group on 127.0.0.1."""
import os
import socket
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from selective_state_space_115_b300 import workloads as W
        w, r, local = bench.dist_env()
        bench.barrier(w)
        # each rank reports a different time; everyone must see the slowest
        slowest = bench.max_over_ranks(1.5 * (rank + 1), w)
        # each rank draws its own independent problem (seed = rank)
        x = W.make_scan_inputs(W.SCAN_CONFIGS["tiny"], seed=rank)
        q.put({"rank": r, "world": w, "local": local, "slowest": slowest,
               "u0": float(np.asarray(x["u"]).ravel()[0])})
        bench.barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_ranks_barrier_and_max_over_ranks():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort(key=lambda d: d["rank"])
    assert [d["rank"] for d in out] == [0, 1]
    assert all(d["world"] == 2 and d["local"] == d["rank"] for d in out)
    assert all(d["slowest"] == 3.0 for d in out)
    assert out[0]["u0"] != out[1]["u0"]  # independent problems per rank


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm's other ranks exit 0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""

