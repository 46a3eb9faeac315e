"""Host logic of bench.py that runs without a GPU: the replica timing rule (max over ranks,
whole-job throughput) on two gloo ranks, and the oracle arm's JSON line."""
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


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r took (r + 1) s for the timed steps and (5 - r) s end to end
    got = bench.replica_max([rank + 1.0, 5.0 - rank], dist, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as fh:
        json.dump(got, fh)


def test_replica_max_over_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        with open(tmp_path / ("rank%d.json" % r)) as fh:
            assert json.load(fh) == [2.0, 5.0]      # every rank sees the slowest rank's times


def test_replica_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_max([1.5, 2.0], None, "cpu") == [1.5, 2.0]
    # 2 replicas x 16 sequences x 10 steps in 2 s (the slowest replica's time)
    assert bench.replica_throughput(2, 16, 10, 2.0) == 160.0
    assert bench.replica_throughput(1, 16, 10, 2.0) == 80.0


def _bench(args, rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True,
                          text=True, env=env, timeout=600, cwd=ROOT)


def test_reference_arm_other_ranks_exit_without_output():
    r = _bench(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"], rank=1)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


@pytest.mark.timeout(600)
def test_reference_arm_prints_one_oracle_line():
    r = _bench(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"], rank=0)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["unit"] == "tok/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tok/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
