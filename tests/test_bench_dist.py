"""bench.py's multi-process plumbing on CPU (gloo, world size 2).

Batch rows are independent, so N GPUs run N disjoint shards of one global
batch with no collective on the data path; the only collectives are the
timing reductions (max of the per-rank times, sum of the per-rank rows).
These tests run that plumbing as two gloo ranks on the host, and check the
reference arm's rank handling under torchrun-style environments.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shards_partition_the_global_batch():
    for world in (1, 2, 3, 8):
        B = 5
        rows = [r for rank in range(world) for r in bench.shard_rows(rank, world, B)]
        assert rows == list(range(world * B))  # disjoint, contiguous, complete


def test_single_rank_reductions_are_identity():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.reduce_sum(7.0, 1) == 7.0


def _rank_main(rank: int, world: int, port: int, q) -> None:
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        ms = 10.0 + 5.0 * r                      # per-rank step times
        rows = float(len(bench.shard_rows(r, w, 4)) * 9)
        q.put((r, w, local, bench.reduce_max(ms, w), bench.reduce_sum(rows, w)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_rows():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[:3] for o in out] == [(0, 2, 0), (1, 2, 1)]
    for o in out:
        assert o[3] == 15.0          # max over ranks of the step time
        assert o[4] == 2 * 4 * 9.0   # rows of both shards


def _run_reference(env_extra: dict) -> subprocess.CompletedProcess:
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "cfg1", "--steps", "1", "--warmup", "3"],
                          env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_line_on_rank0():
    p = _run_reference({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "rows/s"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    # the threads it reports are the ones that had a batch row to work on
    assert line["cpu_baseline"]["cores"] <= max(1, line["config"]["sample_rows_per_step"])
    assert line["e2e"] == {"value": line["value"], "unit": "rows/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_is_silent_on_other_ranks():
    p = _run_reference({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""


def test_gpus_flag_spawns_ranks_dry_run():
    """`bench.py --gpus 2` outside torchrun starts two ranks itself; in the
    host-only dry mode (gloo, no kernels) rank 0 prints one line with the
    world size and the rows of both shards."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--dry-run",
                        "--workload", "cfg3", "--steps", "3", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["dry_run"] is True and line["value"] is None
    assert line["n_gpus"] == 2 and line["scaling"] == "weak"
    assert line["rows_per_step_all_ranks"] == 2 * 64 * 5  # two shards of B=64 rows, K+1 = 5


def test_gpus_flag_without_enough_gpus_fails():
    """Asking for more GPUs than the node has is an error, not a silent
    one-GPU run."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--steps", "3", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode != 0
    assert "error" in json.loads(p.stdout.strip().splitlines()[-1])


def test_pinned_page_placement_is_read_from_numa_maps():
    """The host placement recorded beside the end-to-end figure: the NUMA
    node(s) holding a buffer's pages, from /proc/self/numa_maps."""
    import numpy as np
    a = np.ones(1 << 22, np.uint8)  # 4 MiB, touched
    nodes = bench.numa_nodes()
    placed = bench.pages_node(a.ctypes.data)
    if not os.path.exists("/proc/self/numa_maps") or not nodes:
        pytest.skip("no NUMA information on this host")
    assert placed and all(k.startswith("N") and int(k[1:]) in nodes for k in placed)
    assert sum(placed.values()) >= 1
