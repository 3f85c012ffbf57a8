"""bench.py's multi-rank path on CPU (two gloo ranks): the ranks rendezvous, the step time is
the maximum over ranks, and under torchrun only rank 0 prints (the reference arm's other ranks
exit without work). Attention has no exchange step, so N GPUs run N independent replicas."""
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


def _worker(rank, world, port, outdir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    torch.cuda.is_available = lambda: False  # CPU ranks: gloo
    import bench
    w, r, local = bench.dist_setup()
    got = bench.max_over_ranks(float(r + 1) * 1.5, w)
    bench.barrier(w)
    with open(os.path.join(outdir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "local": local, "max": got}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max(tmp_path):
    mp.start_processes(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [x["rank"] for x in res] == [0, 1] and all(x["world"] == 2 for x in res)
    assert all(x["max"] == 3.0 for x in res)  # max(1.5, 3.0) on both ranks


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
