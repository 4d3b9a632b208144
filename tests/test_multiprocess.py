"""Host logic of `bench.py --gpus N` on CPU: N replicas (one process per GPU,
no collective on the data path) combine their timings with a max over ranks,
and only rank 0 prints the JSON line.  world_size 2 over gloo, rendezvous on
127.0.0.1."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [12.5, 20.0][rank]
    total = bench.max_over_ranks(mine, world)
    q.put((rank, total, bench.job_gbs(world, 1_000_000_000, 10, total)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    # Both ranks see the slowest rank's 20 ms; 2 ranks x 10 steps x 1 GB / 20 ms.
    assert [r[1] for r in res] == [20.0, 20.0]
    assert all(abs(r[2] - 1000.0) < 1e-9 for r in res)


def test_bench_single_process_value():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert abs(bench.job_gbs(1, 2e9, 5, 10.0) - 1000.0) < 1e-9


def test_reference_arm_under_torchrun_prints_one_line():
    """`--impl reference --gpus 2` under torchrun: rank 0 alone runs the CPU
    oracle and prints; the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
