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
    # while that hash matches. The 70B and 13B units take it from two small
    # captures of the same kernel build, read off the line through them;
    # it must stay within 1 % of the algorithmic 42 B per element
    import bench
    for workload, P in (("llama70b_block_unit_n8", 855654400), ("gpt3_13b_block_unit_n8", 314639360)):
        t = bench.recorded_traffic(workload, P)
        assert t is not None, "profiles/ summary missing or taken on another version of the kernel"
        assert 0.99 * 42 * P <= t <= 1.01 * 42 * P, (workload, t / (42 * P))
    # the --numel cases of the 70B workload take the same line, which passes
    # through the captured points
    vals = bench.read_summary(os.path.join(ROOT, "profiles", bench.TRAFFIC_SUMMARY["llama70b_block_unit_n8"]))
    n2 = int(vals["captured_numel"].split(",")[1])
    t2 = float(vals["traffic_bytes"].split(",")[1])
    assert bench.recorded_traffic(f"llama70b_block_unit_n8_numel{n2}", n2) == t2


def test_recorded_traffic_line_through_two_captures(tmp_path, monkeypatch):
    # the line through two captures, and the refusals: a changed kernel, a
    # one-point summary asked for another size, an unknown workload
    import bench
    (tmp_path / "profiles").mkdir()
    f = tmp_path / "profiles" / "rsa_n8_bf16_numel33m_67m_ncu.md"
    h = bench.kernel_source_hash()
    f.write_text(f"- captured_numel: 100, 200\n- traffic_bytes: 1000, 1900\n- kernel_source_sha256: `{h}`\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: h)
    assert bench.recorded_traffic("llama70b_block_unit_n8", 1200) == 1900 + 9 * 1000
    f.write_text("- captured_numel: 100, 200\n- traffic_bytes: 1000, 1900\n- kernel_source_sha256: `0`\n")
    assert bench.recorded_traffic("llama70b_block_unit_n8", 1200) is None
    g = tmp_path / "profiles" / "rsa_gpt2_small_block_unit_n8_ncu.md"
    g.write_text(f"- captured_numel: 7087872\n- traffic_bytes: 297000000\n- kernel_source_sha256: `{h}`\n")
    assert bench.recorded_traffic("gpt2_small_block_unit_n8", 7087872) == 297000000
    assert bench.recorded_traffic("gpt2_small_block_unit_n8", 50000) is None
    assert bench.recorded_traffic("tiny_unit_4099_n2", 4100) is None
