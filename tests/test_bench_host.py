"""Host logic of bench.py without a GPU: replica aggregation across ranks
(gloo, world size 2) and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import bench

    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    # rank r took (10 + r) ms and moved (1 + r) GB
    ms, total = bench.aggregate(dist, torch.device("cpu"), 10.0 + rank, 1e9 * (1 + rank))
    out[rank] = (ms, total)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_aggregation_max_time_sum_bytes():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r] == (11.0, 3e9)          # slowest rank's time, all ranks' bytes


def test_aggregate_single_process_is_identity():
    import bench

    assert bench.aggregate(None, torch.device("cpu"), 5.0, 7.0) == (5.0, 7.0)


def _run_bench(args, env_extra=None):
    env = dict(os.environ, **(env_extra or {}))
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True,
                       text=True, env=env, timeout=600, cwd=ROOT)
    return p


def test_reference_arm_prints_one_line():
    p = _run_bench(["--impl", "reference", "--workload", "tiny_f32_split_half", "--steps", "2",
                    "--warmup", "1"])
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "tiny_f32_split_half"


def test_reference_arm_other_ranks_exit_quietly():
    p = _run_bench(["--impl", "reference", "--workload", "tiny_f32_split_half", "--steps", "1",
                    "--warmup", "1"], {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0 and p.stdout.strip() == ""


def test_attention_reference_arm_prints_one_line():
    p = _run_bench(["--impl", "reference", "--op", "attention", "--steps", "1", "--warmup", "0"])
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["op"] == "attention" and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "llama3_8b_prefill_attention_bf16"


def test_attention_reference_arm_other_ranks_exit_quietly():
    p = _run_bench(["--impl", "reference", "--op", "attention", "--steps", "1", "--warmup", "0"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0 and p.stdout.strip() == ""
