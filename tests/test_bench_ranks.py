"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

bench.py runs one replica per GPU; its only cross-rank steps are the barrier
around the timed region, the maximum of the per-rank times, and the
whole-job aggregate.  Here two processes stand in for two GPUs."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        mine = 1.5 if rank == 0 else 2.5            # per-rank seconds of the timed region
        bench.barrier(world)
        t = bench.reduce_max(mine, world)
        # 10 units per rank over the slowest rank's time
        out[rank] = (t, bench.aggregate(10.0, t, world))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        t, agg = out[r]
        assert t == 2.5                              # every rank sees the slowest rank's time
        assert agg == pytest.approx(20.0 / 2.5)      # all ranks' units over that time


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    """Under torchrun the reference arm runs on rank 0 alone; other ranks exit 0 silently."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tile_d64", "--steps", "1", "--warmup", "1", "--ref-budget", "0.2"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert not [line for line in r.stdout.splitlines() if line.startswith("{")]
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tile_d64", "--steps", "1", "--warmup", "1", "--ref-budget", "0.2"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.parametrize("workload", ["gemm_qkv_proj", "layer_gqa_d128", "causal_d64_bigq"])
def test_reference_arm_line_contract(workload):
    """The reference arm's JSON line carries the keys the benchmark contract
    names, for the attention, GEMM and layer workloads."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", workload,
                        "--steps", "1", "--warmup", "1", "--ref-budget", "0.3"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["config"]["workload"] == workload
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
