"""The N > 1 host path of bench.py on CPU: world-size-2 process groups over
gloo (the bench runs one independent replica per GPU and meets the other ranks
only at barriers and at the max-over-ranks of the timed region)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import workloads
    w_, r_, l_ = bench.dist_setup()
    bench.dist_barrier(w_)
    # every rank times its own replica; the job's time is the slowest rank's
    slowest = bench.dist_max(w_, 10.0 + 5.0 * rank)
    # each rank's replica: the bench offsets the seed by 1000 per rank
    w = workloads.WORKLOADS["gemm256"]
    wr = workloads.Workload(**{**w.__dict__, "seed": w.seed + 1000 * rank})
    A, _, _ = wr.make()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"world": w_, "rank": r_, "slowest": slowest,
                   "a_sum": float(np.asarray(A, dtype=np.float64).sum())}, f)
    bench.dist_barrier(w_)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_world2(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    port = free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [r["world"] for r in res] == [2, 2] and [r["rank"] for r in res] == [0, 1]
    assert res[0]["slowest"] == res[1]["slowest"] == 15.0
    assert res[0]["a_sum"] != res[1]["a_sum"]          # independent replicas


def test_replica_inputs_are_deterministic_per_rank():
    sys.path.insert(0, ROOT)
    import numpy as np
    import workloads
    w = workloads.WORKLOADS["gemm256"]
    a = workloads.Workload(**{**w.__dict__, "seed": w.seed + 1000}).make()[0]
    b = workloads.Workload(**{**w.__dict__, "seed": w.seed + 1000}).make()[0]
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


@pytest.mark.parametrize("workload", ["gemm256", "attn_small"])
def test_reference_arm_under_torchrun_world2(workload):
    # rank 0 alone prints the JSON line; the other rank exits 0 without work
    pytest.importorskip("torch")
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", workload, "--steps", "1", "--warmup", "0"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
