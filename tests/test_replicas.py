"""Multi-GPU path = independent replicas (the forward shards over batch and head
with no exchange step). Its host logic is tested here on CPU: two gloo ranks take
the max of their timed milliseconds, the whole-job rate counts every replica's
work over the slowest rank's time, and the reference arm launched by
torch.distributed.run prints exactly one line, from rank 0."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from exact_tiled_attention_forward_gb300 import replicas as R  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    slowest = R.slowest_rank_ms(ms, world)
    dist.barrier()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"slowest": slowest, "rate": R.whole_job_rate(2.0, 4, slowest, world)}, f)
    dist.destroy_process_group()


def test_slowest_rank_and_whole_job_rate_gloo(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    mp.start_processes(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert [g["slowest"] for g in got] == [15.0, 15.0]
    # 2 replicas x 4 steps x 2.0 units in 15 ms
    assert got[0]["rate"] == pytest.approx(2 * 4 * 2.0 / 15e-3)


def test_single_process_is_its_own_slowest_rank():
    assert R.slowest_rank_ms(7.5, 1) == 7.5
    assert R.whole_job_rate(3.0, 10, 30.0, 1) == pytest.approx(3.0 * 10 / 30e-3)


def test_reference_arm_under_torchrun_prints_one_line():
    pytest.importorskip("torch")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--workload", "tiny_n256_d64"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env={**os.environ, "OPENBLAS_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
