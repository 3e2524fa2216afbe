"""The bench's multi-rank host logic on CPU with gloo, world size 2: the
timing reduction takes the max over ranks, a leg runs on every rank or on
none, and the reference arm runs on rank 0 only."""
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


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.5], torch.device("cpu"))
        # a leg runs on every rank or on none: rank 1 alone cannot, so none does
        agree = (bench.all_ranks_agree(True, torch.device("cpu")),
                 bench.all_ranks_agree(rank != 1, torch.device("cpu")))
        out.put((rank, (got, agree)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == ([2.0, 10.0, 3.5], (True, False))


def test_reference_arm_prints_on_rank0_only(tmp_path):
    env = dict(os.environ, WORLD_SIZE="2", MASTER_ADDR="127.0.0.1")
    outs = {}
    for rank in (0, 1):
        env.update(RANK=str(rank), LOCAL_RANK=str(rank))
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                            "--config", "tiny", "--steps", "3", "--warmup", "3"],
                           env=env, capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr
        outs[rank] = r.stdout.strip()
    assert outs[1] == ""
    line = json.loads(outs[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["value"] > 0


def test_recorded_traffic_matches_current_kernel_source():
    # the committed ncu summary of the fused kernel carries the hash of the
    # kernel sources it was measured on; bench.py reports its traffic only
    # while that hash matches
    import bench
    t = bench.recorded_traffic("llama70b_block_unit_n8")
    assert t is not None, "profiles/ summary missing or taken on another version of the kernel"
    assert 0.99 * 42 * 855654400 <= t <= 1.01 * 42 * 855654400
