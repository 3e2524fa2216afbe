"""The multi-unit step (fsdp_step_units through UnitSequence): a model's FSDP
units stepped in order by one native call. Each unit must end bit-identical
to stepping it on its own with the single-unit entry points, and to the
oracle; units of different N, dtypes and sizes, offloaded and HBM-resident,
share one call.
"""
import numpy as np
import pytest
import torch

import fsdp_inputs as fi
from gpu_util import host

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sharded_fsdp_reduce_gb300 as F
    return F


# (params, world, grad dtype, out dtype): a tiny odd unit, a GPT-2 small
# block, an fp16 unit at N=2, and fp32 gradients at N=3 with a ragged pad
MODEL = [
    ((("w", (64, 64)), ("b", (3,))), 2, torch.bfloat16, torch.bfloat16),
    (fi.CONFIGS["gpt2_small"].params, 8, torch.bfloat16, torch.bfloat16),
    ((("w", (1280, 777)), ("b", (5,))), 2, torch.float16, torch.float16),
    ((("w", (1001,)),), 3, torch.float32, torch.bfloat16),
]


def build_model(F, seed, state_on_host=()):
    units = []
    g = torch.Generator().manual_seed(seed)
    for k, (params, world, gdt, odt) in enumerate(MODEL):
        u = F.FlatParamUnit(params, world, gdt, odt, device=DEV, state_on_host=k in state_on_host)
        flat = (torch.rand(u.numel, generator=g) * 0.2 - 0.1)
        u.load_master([flat.to(DEV)])
        units.append(u)
    torch.cuda.synchronize()
    return units


def load_grads(units, t, seed):
    g = torch.Generator().manual_seed(seed * 1000 + t)
    for u in units:
        for r in range(u.world):
            x = torch.randn(u.numel, generator=g) * 1e-2
            if u.grads[r].dtype == torch.float16:
                x = x * 1024
            u.load_grad(r, [x.to(DEV).to(u.grads[r].dtype)])


def same(a, b):
    iv = torch.int32 if a.element_size() == 4 else torch.int16
    return torch.equal(a.detach().cpu().view(iv), b.detach().cpu().view(iv))


def hp_for(F, u, t):
    scale = 1024.0 if u.grads[0].dtype == torch.float16 else 1.0
    return F.AdamWHParams(1e-3, weight_decay=0.01, step=t, grad_scale=scale)


@pytest.mark.parametrize("gathers,fuse", [(1, False), (2, False), (1, True), (2, True), (0, False)])
def test_units_match_single_unit_steps(F, gathers, fuse):
    a = build_model(F, 1)
    b = build_model(F, 1)
    seq = F.UnitSequence(a)
    for t in (1, 2, 3):
        load_grads(a, t, 5)
        load_grads(b, t, 5)
        # one call for the whole model; the fp16 unit carries its loss scale
        # in its own hyperparameters, so it steps separately in both runs
        fp16 = [u for u in a if u.grads[0].dtype == torch.float16]
        F.UnitSequence([u for u in a if u not in fp16]).step(hp_for(F, a[0], t), gathers=gathers, fuse_gather=fuse)
        for u in fp16:
            F.UnitSequence([u]).step(hp_for(F, u, t), gathers=gathers, fuse_gather=fuse)
        for u in b:
            u.step(hp_for(F, u, t), gathers=gathers, fuse_gather=fuse)
    torch.cuda.synchronize()
    assert len(seq.units) == len(MODEL)
    for ua, ub in zip(a, b):
        for x, y in ((ua.master, ub.master), (ua.exp_avg, ub.exp_avg), (ua.exp_avg_sq, ub.exp_avg_sq),
                     (ua.shard_out, ub.shard_out)):
            assert same(x, y)
        for fa, fb in zip(ua.full, ub.full):
            assert same(fa, fb)
        if gathers:
            for f in ua.full:
                assert same(f, ua.shard_out)


def test_units_match_oracle(F, orc):
    units = build_model(F, 2)
    units = [u for u in units if u.grads[0].dtype != torch.float16]  # one loss scale per call
    seq = F.UnitSequence(units)
    fmt = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}
    st = [[host(u.master), np.zeros(u.padded_numel, np.float32), np.zeros(u.padded_numel, np.float32)]
          for u in units]
    for t in (1, 2):
        load_grads(units, t, 9)
        seq.step(hp_for(F, units[0], t), gathers=2)
        torch.cuda.synchronize()
        for u, (p, m, v) in zip(units, st):
            g_o = [host(g) for g in u.grads]
            shards_o, _ = orc.fsdp_step(g_o, fmt[u.grads[0].dtype], u.world, p, m, v, fmt[u.shard_out.dtype],
                                        orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, t, 1.0))
            np.testing.assert_array_equal(host(u.master).view(np.uint32), p.view(np.uint32))
            np.testing.assert_array_equal(host(u.exp_avg).view(np.uint32), m.view(np.uint32))
            np.testing.assert_array_equal(host(u.exp_avg_sq).view(np.uint32), v.view(np.uint32))
            np.testing.assert_array_equal(host(u.shard_out), shards_o)
            for f in u.full:
                assert torch.equal(f, u.shard_out)


def test_twelve_block_model_as_benched_matches_oracle(F, orc):
    # the driver's bench model: 12 GPT-2 small block units (N=8, one gather
    # each) on the two side streams, stepped twice by fsdp_step_units and
    # twice by one launch of the captured step, bit for bit against the oracle
    cfg = fi.CONFIGS["gpt2_small"]
    gdt, odt = fi.torch_dtype(cfg.grad_dtype), fi.torch_dtype(cfg.out_dtype)
    units = []
    for k in range(12):
        u = F.FlatParamUnit(cfg.params, cfg.world, gdt, odt, device=DEV)
        u.load_master([fi.gen_master(cfg, device=DEV, seed_base=7000 + k)])
        units.append(u)
    seq = F.UnitSequence(units)
    graph = seq.capture(gathers=cfg.gathers)
    st = [[host(u.master), np.zeros(u.padded_numel, np.float32), np.zeros(u.padded_numel, np.float32)]
          for u in units]
    for t in (1, 2, 3, 4):
        for k, u in enumerate(units):
            for r in range(cfg.world):
                u.load_grad(r, [fi.gen_grad(cfg, r, t, device=DEV, seed_base=7000 + k)])
        hp = F.AdamWHParams(cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, t, cfg.grad_scale)
        if t <= 2:
            seq.step(hp, gathers=cfg.gathers)
        else:
            graph.launch(hp)
        torch.cuda.synchronize()
        for u, (p, m, v) in zip(units, st):
            shards_o, _ = orc.fsdp_step([host(g) for g in u.grads], cfg.grad_dtype, cfg.world, p, m, v,
                                        cfg.out_dtype, orc.hparams(cfg.lr, cfg.beta1, cfg.beta2, cfg.eps,
                                                                   cfg.weight_decay, t, cfg.grad_scale))
            np.testing.assert_array_equal(host(u.master).view(np.uint32), p.view(np.uint32))
            np.testing.assert_array_equal(host(u.exp_avg).view(np.uint32), m.view(np.uint32))
            np.testing.assert_array_equal(host(u.exp_avg_sq).view(np.uint32), v.view(np.uint32))
            np.testing.assert_array_equal(host(u.shard_out), shards_o)
            for f in u.full:
                assert torch.equal(f, u.shard_out)
    graph.close()


def test_units_with_offloaded_state_and_a_shared_counter(F):
    a = [u for u in build_model(F, 3, state_on_host={0, 1}) if u.grads[0].dtype != torch.float16]
    b = [u for u in build_model(F, 3) if u.grads[0].dtype != torch.float16]
    nf_a = torch.zeros(1, dtype=torch.int32, device=DEV)
    nf_b = torch.zeros(1, dtype=torch.int32, device=DEV)
    load_grads(a, 1, 4)
    load_grads(b, 1, 4)
    for us in (a, b):  # two non-finite gradients in unit 0, one in unit 2
        us[0].grads[0][5] = float("inf")
        us[0].grads[1][7] = float("nan")
        us[2].grads[1][0] = float("-inf")
    F.UnitSequence(a).step(hp_for(F, a[0], 1), gathers=1, nonfinite_count=nf_a)
    for u in b:
        u.step(hp_for(F, u, 1), gathers=1, nonfinite_count=nf_b)
    torch.cuda.synchronize()
    assert int(nf_a.item()) == int(nf_b.item()) == 3
    for ua, ub in zip(a, b):
        for x, y in ((ua.master, ub.master), (ua.exp_avg, ub.exp_avg), (ua.shard_out, ub.shard_out)):
            assert same(x, y)


def test_units_rejects_shared_buffers_and_enqueues_nothing(F):
    a = build_model(F, 4)
    a[1].exp_avg = a[0].master  # two units writing one buffer (sizes differ: the binding catches it)
    with pytest.raises(ValueError):
        F.UnitSequence(a)
    b = build_model(F, 4)
    b[3].exp_avg = b[0].exp_avg.narrow(0, 0, b[3].padded_numel)  # same size: only the library sees it
    before = [u.master.clone() for u in b]
    with pytest.raises(F.FsdpError):
        F.UnitSequence(b).step(hp_for(F, b[0], 1), gathers=1)
    torch.cuda.synchronize()
    for u, p in zip(b, before):
        assert same(u.master, p)  # nothing ran, not even the units before the bad one


def test_units_empty(F):
    F.UnitSequence([]).step(F.AdamWHParams(1e-3, step=1), gathers=2)
    e = F.FlatParamUnit([("x", (0,))], 2, torch.bfloat16, torch.bfloat16, device=DEV)
    assert e.padded_numel == 0
    F.UnitSequence([e]).step(F.AdamWHParams(1e-3, step=1), gathers=1)
    torch.cuda.synchronize()


def test_units_order_with_the_callers_stream(F):
    # the units run on the library's side streams, forked from and joined
    # back into the caller's stream: gradients written on that stream just
    # before the call (behind a 0.1 s spin) must be the ones used, and work
    # queued on it just after must see every unit finished. Only the
    # caller's stream is synchronized.
    a = [u for u in build_model(F, 6) if u.grads[0].dtype != torch.float16]
    b = [u for u in build_model(F, 6) if u.grads[0].dtype != torch.float16]
    load_grads(b, 1, 8)
    for u in b:
        u.step(hp_for(F, u, 1), gathers=1)
    torch.cuda.synchronize()
    seq = F.UnitSequence(a)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(200_000_000)  # ~0.1 s of spinning before the gradients land
        load_grads(a, 1, 8)
        seq.step(hp_for(F, a[0], 1), gathers=1, stream=s)
        after = [(u.master.clone(), u.full[-1].clone()) for u in a]
    s.synchronize()
    for (m, f), ub in zip(after, b):
        assert same(m, ub.master)
        assert same(f, ub.full[-1])


def test_units_from_concurrent_host_threads(F):
    # two host threads step their own models through the native driver on
    # their own streams at once (side streams and their fork/join events are
    # per thread); every unit ends as in a sequential run
    import threading

    def make(seed):
        return [u for u in build_model(F, seed) if u.grads[0].dtype != torch.float16]

    def run(units, stream, seed, errors):
        try:
            with torch.cuda.stream(stream):
                seq = F.UnitSequence(units)
                for t in range(1, 5):
                    load_grads(units, t, seed)
                    seq.step(hp_for(F, units[0], t), gathers=2, stream=stream, fuse_gather=(t % 2 == 0))
            stream.synchronize()
        except Exception as e:  # surfaced below
            errors.append(e)

    ref = [make(10), make(11)]
    for units, seed in zip(ref, (20, 21)):
        run(units, torch.cuda.current_stream(), seed, [])
    torch.cuda.synchronize()
    par = [make(10), make(11)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    errors = []
    threads = [threading.Thread(target=run, args=(u, s, seed, errors))
               for u, s, seed in zip(par, streams, (20, 21))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for ma, mb in zip(ref, par):
        for ua, ub in zip(ma, mb):
            for x, y in ((ua.master, ub.master), (ua.exp_avg, ub.exp_avg), (ua.exp_avg_sq, ub.exp_avg_sq),
                         (ua.shard_out, ub.shard_out)):
                assert same(x, y)
            for fa, fb in zip(ua.full, ub.full):
                assert same(fa, fb)


def test_model_step_captured_in_a_cuda_graph(F):
    # the native driver's launches, side streams and fork/join events inside
    # a CUDA graph: replaying the captured step equals running it eagerly.
    # The step's scalars are the kernels' by-value arguments, so a graph
    # replays the step it captured (here step 2 from the same state).
    a = [u for u in build_model(F, 12) if u.grads[0].dtype != torch.float16]
    b = [u for u in build_model(F, 12) if u.grads[0].dtype != torch.float16]
    seq_a, seq_b = F.UnitSequence(a), F.UnitSequence(b)
    load_grads(a, 1, 13)
    load_grads(b, 1, 13)
    seq_a.step(hp_for(F, a[0], 1), gathers=2)  # eager step 1 (also warms every launch cache)
    seq_b.step(hp_for(F, b[0], 1), gathers=2)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        seq_a.step(hp_for(F, a[0], 2), gathers=2, fuse_gather=True)
    graph.replay()
    seq_b.step(hp_for(F, b[0], 2), gathers=2, fuse_gather=True)
    torch.cuda.synchronize()
    for ua, ub in zip(a, b):
        for x, y in ((ua.master, ub.master), (ua.exp_avg, ub.exp_avg), (ua.exp_avg_sq, ub.exp_avg_sq),
                     (ua.shard_out, ub.shard_out)):
            assert same(x, y)
        for fa, fb in zip(ua.full, ub.full):
            assert same(fa, fb)


@pytest.mark.parametrize("gathers,fuse", [(2, False), (2, True), (1, True), (0, False)])
def test_captured_step_matches_the_driver(F, gathers, fuse):
    # one graph, launched for steps 1..4 with each step's scalars, against
    # the native driver step by step; offloaded units included
    a = [u for u in build_model(F, 14, state_on_host={1}) if u.grads[0].dtype != torch.float16]
    b = [u for u in build_model(F, 14, state_on_host={1}) if u.grads[0].dtype != torch.float16]
    nf_a = torch.zeros(1, dtype=torch.int32, device=DEV)
    nf_b = torch.zeros(1, dtype=torch.int32, device=DEV)
    graph = F.UnitSequence(a).capture(gathers=gathers, fuse_gather=fuse, nonfinite_count=nf_a)
    seq_b = F.UnitSequence(b)
    s = torch.cuda.Stream()
    for t in (1, 2, 3, 4):
        load_grads(a, t, 15)
        load_grads(b, t, 15)
        torch.cuda.synchronize()
        graph.launch(hp_for(F, a[0], t), stream=s)
        seq_b.step(hp_for(F, b[0], t), gathers=gathers, fuse_gather=fuse, nonfinite_count=nf_b)
        s.synchronize()
        torch.cuda.synchronize()
    for ua, ub in zip(a, b):
        for x, y in ((ua.master, ub.master), (ua.exp_avg, ub.exp_avg), (ua.exp_avg_sq, ub.exp_avg_sq),
                     (ua.shard_out, ub.shard_out)):
            assert same(x, y)
        for fa, fb in zip(ua.full, ub.full):
            assert same(fa, fb)
    assert int(nf_a.item()) == int(nf_b.item()) == 0
    graph.close()
    with pytest.raises(RuntimeError):
        graph.launch(hp_for(F, a[0], 5))


def test_captured_step_refusals(F):
    a = [u for u in build_model(F, 16) if u.grads[0].dtype != torch.float16]
    graph = F.UnitSequence(a).capture(gathers=1)
    before = [u.master.clone() for u in a]
    with pytest.raises(F.FsdpError):
        graph.launch(F.AdamWHParams(1e-3, step=0))  # invalid step: nothing launched
    torch.cuda.synchronize()
    for u, p in zip(a, before):
        assert same(u.master, p)
    b = [u for u in build_model(F, 16) if u.grads[0].dtype != torch.float16]
    b[2].exp_avg = b[0].exp_avg.narrow(0, 0, b[2].padded_numel)  # two units writing one buffer
    with pytest.raises(F.FsdpError):
        F.UnitSequence(b).capture(gathers=1)
    v = F.FlatParamUnit([("w", (64,))], 2, torch.bfloat16, torch.bfloat16, device=DEV, optimizer="sgd")
    with pytest.raises(ValueError):  # the captured step is the fused AdamW step
        F.UnitSequence([v]).capture()


def test_resources_are_released(F):
    # captured steps created and destroyed, and short-lived host threads that
    # each create their side streams and events and exit: device memory
    # returns to where it started and every step still matches the driver
    import threading
    a = [u for u in build_model(F, 30) if u.grads[0].dtype != torch.float16]
    b = [u for u in build_model(F, 30) if u.grads[0].dtype != torch.float16]
    seq_b = F.UnitSequence(b)
    load_grads(a, 1, 31)
    load_grads(b, 1, 31)
    warm = F.UnitSequence(a).capture(gathers=1)  # first capture and launch of these builds
    warm.close()
    torch.cuda.Stream()  # torch's stream pool is set up on first use (not the library's memory)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    free0, _ = torch.cuda.mem_get_info()
    for t in range(1, 41):
        graph = F.UnitSequence(a).capture(gathers=1)
        graph.launch(hp_for(F, a[0], t))
        graph.close()
        seq_b.step(hp_for(F, b[0], t), gathers=1)
    torch.cuda.synchronize()
    errors = []

    def worker(t):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                F.UnitSequence(a).step(hp_for(F, a[0], t), gathers=1, stream=s)
            s.synchronize()
        except Exception as e:  # surfaced below
            errors.append(e)

    for t in range(41, 61):  # one thread per step, run one after another
        th = threading.Thread(target=worker, args=(t,))
        th.start()
        th.join()
        seq_b.step(hp_for(F, b[0], t), gathers=1)
    torch.cuda.synchronize()
    assert not errors, errors
    torch.cuda.empty_cache()
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free1 - free0) < 8 << 20, (free0, free1)
    for ua, ub in zip(a, b):
        assert same(ua.master, ub.master) and same(ua.full[0], ub.full[0])
