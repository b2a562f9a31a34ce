"""The benchmark's multi-process path on CPU (gloo, world size 2).

With N GPUs every rank runs its own replica of the workload; the only
cross-rank steps are the barrier around the timed region and the maximum of
the elapsed times.  Those run here on gloo ranks, without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    elapsed = 10.0 + 5.0 * rank           # rank 1 is the slower one
    worst = d.max(elapsed)
    d.barrier()
    d.finish()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": rank, "max": worst, "world": d.world}, f)


def test_max_over_ranks_with_gloo(tmp_path):
    import torch.multiprocessing as mp
    port = free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert all(g["max"] == 15.0 and g["world"] == 2 for g in got)


def test_single_process_dist_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    if d.world == 1:
        d.init("gloo")
        d.barrier()
        assert d.max(3.5) == 3.5


def test_reference_arm_under_torchrun_prints_once():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "0", "--steps", "2", "--warmup", "3",
           "--reference-seconds", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0
    assert res["cpu_baseline"]["kind"] == "oracle"
    assert res["e2e"]["h2d_bytes_per_step"] == 0
