"""The multi-rank host logic of bench.py on the CPU: two gloo ranks.

Attention does not shard across GPUs (every rank is an independent replica), so the only
cross-rank steps are the barriers around the timed region, the max-reduction of its length and
the whole-job throughput; the reference arm runs on rank 0 alone.  These tests run those steps
as two processes over gloo on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench

    w, r, lr = bench.rank_layout()
    dist = bench.init_ranks(w)
    assert dist is not None and dist.get_backend() == "gloo"
    dist.barrier()
    # rank r "took" (r + 1) * 1.5 ms; the job took the slowest rank's time
    ms = bench.max_over_ranks((r + 1) * 1.5, dist, "cpu")
    value = bench.job_throughput(1000, 10, w, ms)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"layout": [w, r, lr], "ms": ms, "value": value}, f)


def test_single_rank_layout(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    assert bench.rank_layout() == (1, 0, 0)
    assert bench.init_ranks(1) is None
    assert bench.max_over_ranks(2.5, None, "cpu") == 2.5
    # 1000 tokens x 10 steps in 2 ms of one rank
    assert bench.job_throughput(1000, 10, 1, 2.0) == pytest.approx(5.0e6)


def test_two_gloo_ranks_max_and_throughput(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert d["layout"] == [2, r, r]
        assert d["ms"] == pytest.approx(3.0)  # max of 1.5 and 3.0, seen by both ranks
        # both ranks' 10 x 1000 tokens over the slowest rank's 3 ms
        assert d["value"] == pytest.approx(2 * 10 * 1000 / 3.0e-3)


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny", "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=240)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
