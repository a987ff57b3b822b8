"""bench.py's host logic on CPU: two gloo ranks, barrier and the
max-over-ranks reduction of the timed duration (the only collectives the
benchmark uses; the data path has none), and the reference arm (the fp64
oracle timed on the host cores, printed by rank 0 alone)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch
    import bench
    w, r, _ = bench.dist_setup(torch)
    bench.barrier(torch, w)
    m = bench.max_over_ranks(torch, w, 10.0 + 5.0 * r)
    out[r] = m
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 15.0, 1: 15.0}


def _run_reference_arm(env_extra):
    import json
    import subprocess
    import sys
    env = dict(os.environ, **env_extra)
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    return [json.loads(ln) for ln in lines]


@pytest.mark.timeout(300)
def test_reference_arm_prints_one_line_with_the_decode_metric():
    """The reference arm (the fp64 oracle on the host cores) keeps the
    GPU arm's metric, unit and config, and reports itself as its own CPU
    baseline and end-to-end value with no host-device bytes."""
    import bench
    (line,) = _run_reference_arm({"RANK": "0", "WORLD_SIZE": "1"})
    assert line["impl"] == "reference" and line["metric"] == bench.DECODE_METRIC
    assert line["unit"] == "rows/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["steps"] == 2 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["config"] == bench.decode_config(2 * bench.DECODE_ROWS, 1)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


@pytest.mark.timeout(120)
def test_reference_arm_other_ranks_exit_without_work():
    assert _run_reference_arm({"RANK": "1", "WORLD_SIZE": "2"}) == []
