"""The multi-rank path of bench.py on CPU: world_size-2 gloo process groups
(the step shards by sequence with no exchange; the only collectives are the
timing barrier and the max/sum reductions of the result)."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        res = {"max": d.max(float(rank) * 2.5), "sum": d.sum(float(rank + 1)),
               "world": d.world, "rank": d.rank}
        d.barrier()
    finally:
        d.close()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump(res, f)


def test_gloo_reductions_world2(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        res = json.load(open(tmp_path / f"r{r}.json"))
        assert res["world"] == 2 and res["rank"] == r
        assert res["max"] == 2.5          # max over ranks: the slowest rank's time
        assert res["sum"] == 3.0          # sum over ranks: every replica's bytes


def test_reference_arm_prints_once_under_torchrun():
    """Launched as the driver launches it for N = 2, the reference arm (the
    CPU oracle) runs on rank 0 alone and prints one JSON line."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--workload", "tiny_qwen3_decode"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
