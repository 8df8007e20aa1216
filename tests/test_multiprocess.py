"""The multi-process paths of bench.py, on CPU with the gloo backend (two
ranks on 127.0.0.1): each rank times its own replica and the job reports the
work of all ranks over the slowest rank's time; the reference arm runs on
rank 0 only and the other ranks exit cleanly without output."""
import json
import os
import socket
import subprocess
import sys
import tempfile

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    ms_local = 100.0 + 25.0 * rank           # rank 1 is the slower replica
    ms_max = bench.max_over_ranks(ms_local, world, torch.device("cpu"))
    value = bench.whole_job_value(4.0e12, world, ms_max)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
        json.dump({"ms_max": ms_max, "value": value}, fh)


def test_replicas_report_all_work_over_the_slowest_rank():
    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank, args=(world, _free_port(), d), nprocs=world, join=True,
                           start_method="spawn")
        res = [json.load(open(os.path.join(d, f"rank{r}.json"))) for r in range(world)]
    for r in res:
        assert r["ms_max"] == 125.0
        assert abs(r["value"] - 4.0e12 * world / 0.125 / 1e12) < 1e-9


def test_single_rank_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.whole_job_value(2.0e12, 1, 500.0) == 4.0


def test_reference_arm_on_a_non_zero_rank_prints_nothing():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""
