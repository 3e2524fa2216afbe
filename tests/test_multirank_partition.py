"""The method's own partition across ranks, on CPU with gloo (world sizes 2
and 3): each process is one data-parallel rank that holds its own flat
gradient and only its 1/N shard of the fp32 master, m and v.

Per step, as "Fully Sharded Data Parallel: faster AI training with fewer
GPUs", "From all-reduce to sharded parameters" and "FSDP (Fully Sharded Data
Parallel)", "The Per-Layer Communication" lay it out:

1. reduce-scatter: block k of every rank's gradient goes to rank k (a gloo
   all_to_all_single moves the blocks); rank r sums the N blocks it received
   in rank order 0..N-1 in fp32 and scales by 1/(N * loss scale) with the
   oracle's own reduce-scatter (the reading that fixes the order, so that
   the result is deterministic);
2. rank r updates its own shard with the oracle's AdamW and casts it to the
   compute dtype;
3. all-gather: every rank receives every shard (gloo all_gather) and
   concatenates them in rank order into the full compute-dtype parameters.

Every rank's gathered parameters after every step, and the shards of the
state concatenated in rank order after the last step, must equal a
single-process full-replica DDP step of the oracle bit for bit (the pages:
FSDP's results are identical to DDP's). This pins, on the CPU, the split a
real cross-GPU version of the kernels would make, with padding
(P not a multiple of N), fp32, bf16 and loss-scaled fp16 gradients.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (P, gradient dtype, compute dtype, loss scale)
CASES = [(4099, "bf16", "bf16", 1.0), (1001, "f16", "f16", 1024.0), (777, "f32", "bf16", 1.0)]
STEPS = 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(P, gfmt, scale, world, rank, t):
    """Rank `rank`'s flat gradient at step t (padded, in its storage dtype)
    and the initial master weights (the same on every rank)."""
    import fsdp_inputs as fi
    import oracle as orc
    cfg = fi.CONFIGS["tiny"]
    x = fi.gen_grad(cfg, rank, t, numel=P, seed_base=77).float() * scale
    if gfmt == "f32":
        g = x.numpy()
    else:
        import torch
        dt = torch.bfloat16 if gfmt == "bf16" else torch.float16
        g = x.to(dt).view(torch.int16).numpy().view(np.uint16)
    return orc.flatten_pad([g], world)


def _master(P, world):
    import fsdp_inputs as fi
    import oracle as orc
    return orc.flatten_pad([fi.gen_master(fi.CONFIGS["tiny"], numel=P, seed_base=77).numpy()], world)


def _hp(orc, t, scale):
    return orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, t, scale)


def _as_wire(a):
    """A gloo tensor carrying an array exactly (16-bit patterns widened to int32)."""
    import torch
    if a.dtype == np.float32:
        return torch.from_numpy(a.copy())
    return torch.from_numpy(a.astype(np.int32))


def _from_wire(t, like):
    a = t.numpy()
    return a.astype(like) if like != np.float32 else a.astype(np.float32)


def _rank(rank, world, port, case, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import oracle as orc
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        orc.set_threads(1)
        P, gfmt, ofmt, scale = case
        P_pad = orc.padded_numel(P, world)
        S = P_pad // world
        lo, hi = rank * S, (rank + 1) * S
        master = _master(P, world)
        p, m, v = master[lo:hi].copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)
        gathered = []
        for t in range(1, STEPS + 1):
            g_own = _inputs(P, gfmt, scale, world, rank, t)
            # 1. reduce-scatter: rank k receives block k of every rank's gradient
            recv = torch.empty(P_pad, dtype=torch.float32 if gfmt == "f32" else torch.int32)
            dist.all_to_all_single(recv, _as_wire(g_own))
            blocks = _from_wire(recv, g_own.dtype).reshape(world, S)  # row q: rank q's block `rank`
            placed = []
            for q in range(world):  # each block at its own offset, as the oracle's reduce-scatter reads it
                full_q = np.zeros(P_pad, dtype=g_own.dtype)
                full_q[lo:hi] = blocks[q]
                placed.append(full_q)
            hp = _hp(orc, t, scale)
            g = orc.reduce_scatter(placed, gfmt, world, rank, orc.scalars(hp, world).c)
            # 2. the shard's AdamW step and cast
            orc.adamw(p, m, v, g, orc.scalars(hp, world))
            shard = orc.cast_out(p, ofmt)
            # 3. all-gather of the compute-dtype shards, in rank order
            parts = [torch.empty(S, dtype=torch.int32) for _ in range(world)]
            dist.all_gather(parts, _as_wire(shard))
            gathered.append(np.concatenate([_from_wire(x, shard.dtype) for x in parts]))
        out.put((rank, gathered, p, m, v))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}_{c[1]}" for c in CASES])
def test_sharded_ranks_equal_one_ddp_replica(orc, world, case):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, case, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = dict((r, rest) for r, *rest in (q.get(timeout=240) for _ in procs))
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    # the single-process DDP replica on the same bytes
    P, gfmt, ofmt, scale = case
    master = _master(P, world)
    P_pad = master.size
    dm, dv = np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)
    for t in range(1, STEPS + 1):
        grads = [_inputs(P, gfmt, scale, world, r, t) for r in range(world)]
        full = orc.ddp_step(grads, gfmt, world, master, dm, dv, ofmt, _hp(orc, t, scale))
        for r in range(world):
            np.testing.assert_array_equal(res[r][0][t - 1], full)  # every rank gathered the replica's parameters
        assert not full[P:].any()                                  # and the pad stays zero
    for k, ref in enumerate((master, dm, dv)):
        shards = np.concatenate([res[r][1 + k] for r in range(world)])
        np.testing.assert_array_equal(shards.view(np.uint32), ref.view(np.uint32))
