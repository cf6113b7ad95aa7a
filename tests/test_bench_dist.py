"""The multi-process plumbing of bench.py, on CPU.

bench.py runs one process per GPU (torchrun, NCCL). Its rank-side helpers are:
- the barrier around the timed region;
- the maximum of the per-rank times;
- the reference arm's rank-0-only output.
Here they run as world-size-2 gloo process groups and as a 2-process torchrun on the host.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    got = bench.max_over_ranks(10.0 * rank + 3.0, world)      # rank times 3 and 13 ms
    bench.barrier(world)
    dist.destroy_process_group()
    with open(os.path.join(out, "rank%d.json" % rank), "w") as f:
        json.dump({"max": got}, f)


def test_barrier_and_max_over_ranks_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [json.load(open(tmp_path / ("rank%d.json" % r)))["max"] for r in range(world)]
    assert got == [13.0, 13.0]          # every rank sees the slowest rank's time


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    bench.barrier(1)                     # no process group: a no-op


def test_reference_arm_prints_once_under_torchrun(ref):
    # two ranks, as the driver launches the reference arm for N > 1: rank 0
    # runs the bounded oracle sample and prints the line, rank 1 exits quietly
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "prefill_32k",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-rows", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["config"]["workload"] == "prefill_32k"
