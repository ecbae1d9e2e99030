"""The N > 1 host path of bench.py on CPU with the gloo backend (world size 2).

Each rank runs an independent replica of the workload (the path partitions into
independent layers, batches and heads: no collective on the data path).  What the ranks
share is the bookkeeping: a barrier around the timed region, the slowest rank's time
(max over ranks) and the tokens of all ranks (sum), and rank 0 alone prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    ws, r, local = bench._dist()
    bench._barrier(ws)
    step_ms = bench._max_over_ranks(1.0 + rank, ws, "cpu")      # rank 1 is the slower one
    tokens = bench._sum_over_ranks(8192.0 * (rank + 1), ws, "cpu")
    bench._barrier(ws)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ws": ws, "rank": r, "local": local, "backend": dist.get_backend(), "step_ms": step_ms,
                   "tokens": tokens, "value": tokens / (step_ms * 1e-3)}, f)
    dist.destroy_process_group()


def test_rank_bookkeeping_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert (d["ws"], d["rank"], d["local"], d["backend"]) == (2, r, r, "gloo")
        assert d["step_ms"] == 2.0                 # the slowest rank's time
        assert d["tokens"] == 3 * 8192.0           # every rank's tokens
        assert d["value"] == pytest.approx(3 * 8192.0 / 2e-3)


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_once(tmp_path):
    """`--impl reference` launched like the multi-GPU bench: rank 0 alone runs the oracle and
    prints one JSON line; rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=580)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
