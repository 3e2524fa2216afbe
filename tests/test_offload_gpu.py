"""Offload mode: the optimizer state and the fp32 master in pinned host
memory, updated in place by the same kernels over the host link; gradients
optionally read from pinned host memory too. Compared with the oracle and,
bit for bit, with the same steps on device-resident state (the kernels
perform the same operations whatever memory the pointers name).
"""
import numpy as np
import pytest
import torch

import fsdp_inputs as fi
from gpu_util import assert_out_close, host

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sharded_fsdp_reduce_gb300 as F
    return F


def hp_for(F, cfg, t):
    return F.AdamWHParams(cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, t, cfg.grad_scale)


def ohp_for(orc, cfg, t):
    return orc.hparams(cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, t, cfg.grad_scale)


def new_unit(F, cfg, **kw):
    return F.FlatParamUnit(cfg.params, cfg.world, fi.torch_dtype(cfg.grad_dtype), fi.torch_dtype(cfg.out_dtype),
                           device=DEV, **kw)


def split_views(unit, flat):
    return [flat.narrow(0, v.offset, v.numel).contiguous() for v in unit.views]


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    iv = torch.int32 if a.element_size() == 4 else torch.int16
    return torch.equal(a.detach().cpu().view(iv), b.detach().cpu().view(iv))


@pytest.mark.parametrize("name", ["tiny", "gpt2_small", "gpt2_large"])
def test_offload_trajectory_matches_oracle(F, orc, name):
    cfg = fi.CONFIGS[name]
    N = cfg.world
    unit = new_unit(F, cfg, state_on_host=True)
    for t_ in (unit.master, unit.exp_avg, unit.exp_avg_sq):
        assert t_.device.type == "cpu" and t_.is_pinned()
    master = fi.gen_master(cfg)
    unit.load_master(split_views(unit, master.to(DEV)))
    torch.cuda.synchronize()
    p_o = orc.flatten_pad([master.numpy()], N)
    m_o = np.zeros_like(p_o)
    v_o = np.zeros_like(p_o)
    np.testing.assert_array_equal(host(unit.master), p_o)
    for t in range(1, cfg.steps + 1):
        grads = [fi.gen_grad(cfg, r, t) for r in range(N)]
        for r in range(N):
            unit.load_grad(r, split_views(unit, grads[r].to(DEV)))
        g_o = [orc.flatten_pad([host(g)], N) for g in grads]
        unit.step(hp_for(F, cfg, t), gathers=cfg.gathers)
        shards_o, _ = orc.fsdp_step(g_o, cfg.grad_dtype, N, p_o, m_o, v_o, cfg.out_dtype, ohp_for(orc, cfg, t))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(unit.master).view(np.uint32), p_o.view(np.uint32))
        np.testing.assert_array_equal(host(unit.exp_avg).view(np.uint32), m_o.view(np.uint32))
        np.testing.assert_array_equal(host(unit.exp_avg_sq).view(np.uint32), v_o.view(np.uint32))
        assert_out_close(host(unit.shard_out), shards_o, cfg.out_dtype, f"{name} shard_out t={t}")
        np.testing.assert_array_equal(host(unit.shard_out), shards_o)
        for k, f in enumerate(unit.full):
            assert torch.equal(f, unit.shard_out), f"{name} full[{k}] t={t}"
        assert not host(unit.master)[unit.numel:].any()  # the pad stays zero


@pytest.mark.parametrize("fuse_gather", [False, True])
def test_offload_equals_device_state(F, fuse_gather):
    cfg = fi.CONFIGS["gpt2_small"]
    N = cfg.world
    a, b = new_unit(F, cfg, state_on_host=True), new_unit(F, cfg)
    master = fi.gen_master(cfg, device=DEV)
    a.load_master([master])
    b.load_master([master])
    nf_a = torch.zeros(1, dtype=torch.int32, device=DEV)
    nf_b = torch.zeros(1, dtype=torch.int32, device=DEV)
    for t in (1, 2, 3):
        for r in range(N):
            g = fi.gen_grad(cfg, r, t, device=DEV)
            a.grads[r].copy_(g)
            b.grads[r].copy_(g)
        a.step(hp_for(F, cfg, t), gathers=2, fuse_gather=fuse_gather, nonfinite_count=nf_a)
        b.step(hp_for(F, cfg, t), gathers=2, fuse_gather=fuse_gather, nonfinite_count=nf_b)
    torch.cuda.synchronize()
    for x, y in ((a.master, b.master), (a.exp_avg, b.exp_avg), (a.exp_avg_sq, b.exp_avg_sq),
                 (a.shard_out, b.shard_out)):
        assert same_bits(x, y)
    for fa, fb in zip(a.full, b.full):
        assert same_bits(fa, fb)
    assert int(nf_a.item()) == int(nf_b.item()) == 0


@pytest.mark.parametrize("offset", [0, 1])
@pytest.mark.parametrize("world,P", [(2, 4099), (8, 8 * 1000 + 3)])
def test_offload_state_and_host_gradients(F, world, P, offset):
    # every buffer the update streams (gradients, master, m, v) in pinned host
    # memory, optionally one element off 16-byte alignment (the scalar path)
    P_pad = F.fsdp_padded_numel(P, world)
    rng = np.random.default_rng(world + P + offset)
    master0 = torch.from_numpy(rng.uniform(-0.1, 0.1, P_pad).astype(np.float32))
    master0[P:] = 0

    def pinned(n, dt):
        return torch.zeros(n + offset, dtype=dt, pin_memory=True)[offset:]

    def dev(n, dt):
        return torch.zeros(n + offset, dtype=dt, device=DEV)[offset:]

    hs = [pinned(P_pad, torch.float32) for _ in range(3)]
    ds = [dev(P_pad, torch.float32) for _ in range(3)]
    hs[0].copy_(master0)
    ds[0].copy_(master0)
    hg = [pinned(P_pad, torch.bfloat16) for _ in range(world)]
    dg = [dev(P_pad, torch.bfloat16) for _ in range(world)]
    ho, do = dev(P_pad, torch.bfloat16), dev(P_pad, torch.bfloat16)
    for t in (1, 2, 3):
        for q in range(world):
            g = torch.from_numpy((rng.standard_normal(P_pad) * 1e-2).astype(np.float32)).to(torch.bfloat16)
            g[P:] = 0
            hg[q].copy_(g)
            dg[q].copy_(g)
        hp = F.AdamWHParams(1e-3, weight_decay=0.01, step=t)
        F.fsdp_reduce_scatter_adam_cast(hg, *hs, ho, hp)
        F.fsdp_reduce_scatter_adam_cast(dg, *ds, do, hp)
    torch.cuda.synchronize()
    for x, y in zip(hs, ds):
        assert same_bits(x, y)
    assert same_bits(ho, do)
    assert not hs[0][P:].any()


@pytest.mark.parametrize("opt", ["adamw", "sgd", "adamax", "adadelta"])
@pytest.mark.parametrize("sdt", [torch.float32, torch.bfloat16])
def test_offload_variant_steps(F, opt, sdt):
    world, P = 8, 8 * 4096 + 3
    P_pad = F.fsdp_padded_numel(P, world)
    rng = np.random.default_rng(11)
    ns = 1 if opt == "sgd" else 2
    p0 = torch.from_numpy(rng.uniform(-0.1, 0.1, P_pad).astype(np.float32)).to(sdt)
    hp_ = [torch.zeros(P_pad, dtype=sdt, pin_memory=True) for _ in range(1 + ns)]
    dp_ = [torch.zeros(P_pad, dtype=sdt, device=DEV) for _ in range(1 + ns)]
    hp_[0].copy_(p0)
    dp_[0].copy_(p0)
    grads = [torch.zeros(P_pad, dtype=torch.bfloat16, device=DEV) for _ in range(world)]
    out_h = torch.zeros(P_pad, dtype=torch.bfloat16, device=DEV) if sdt == torch.float32 else None
    out_d = torch.zeros(P_pad, dtype=torch.bfloat16, device=DEV) if sdt == torch.float32 else None
    lr = 1.0 if opt == "adadelta" else 1e-3
    for t in (1, 2, 3):
        for g in grads:
            g.copy_(torch.from_numpy((rng.standard_normal(P_pad) * 1e-2).astype(np.float32)))
        cfg = F.StepConfig(opt, lr, weight_decay=0.01, step=t)
        F.fsdp_reduce_scatter_step(grads, hp_[0], hp_[1], hp_[2] if ns == 2 else None, out_h, cfg)
        F.fsdp_reduce_scatter_step(grads, dp_[0], dp_[1], dp_[2] if ns == 2 else None, out_d, cfg)
    torch.cuda.synchronize()
    for x, y in zip(hp_, dp_):
        assert same_bits(x, y), opt
    if out_h is not None:
        assert same_bits(out_h, out_d)


def test_offload_step_from_host(F):
    # the pipelined host-buffer step with the state in host memory as well
    cfg = fi.CONFIGS["gpt2_small"]
    N = cfg.world
    a, b = new_unit(F, cfg, state_on_host=True), new_unit(F, cfg)
    master = fi.gen_master(cfg, device=DEV)
    a.load_master([master])
    b.load_master([master])
    T = 3
    hg = [[fi.gen_grad(cfg, r, t).pin_memory() for r in range(N)] for t in range(1, T + 1)]
    for t in range(1, T + 1):
        a.step_from_host(hg[t - 1], None, hp_for(F, cfg, t), gathers=2)
    torch.cuda.synchronize()
    for t in range(1, T + 1):
        for r in range(N):
            b.grads[r].copy_(hg[t - 1][r])
        b.step(hp_for(F, cfg, t), gathers=2)
    torch.cuda.synchronize()
    for x, y in ((a.master, b.master), (a.exp_avg, b.exp_avg), (a.exp_avg_sq, b.exp_avg_sq)):
        assert same_bits(x, y)
    for f in a.full:
        assert same_bits(f, b.shard_out)


@pytest.mark.parametrize("name", ["gpt3_13b", "llama70b"])
def test_offload_full_size_sampled(F, orc, name):
    # the 13B and 70B units at full size with their state (3.8 and 10.3 GB)
    # in host memory, in the bench's launch configuration; sampled elements
    # against the oracle
    cfg = fi.CONFIGS[name]
    N = cfg.world
    unit = new_unit(F, cfg, state_on_host=True)
    unit.load_master([fi.gen_master(cfg, device=DEV)])
    torch.cuda.synchronize()
    P_pad = unit.padded_numel
    S = P_pad // N
    rng = np.random.default_rng(13)
    idx = np.unique(np.concatenate([rng.integers(0, P_pad, 1 << 18)] +
                                   [np.arange(r * S, r * S + 32) for r in range(N)] +
                                   [np.arange((r + 1) * S - 32, (r + 1) * S) for r in range(N)]))
    idx_c = torch.from_numpy(idx)
    idx_d = idx_c.to(DEV)
    p_s = unit.master[idx_c].numpy().copy()
    m_s = np.zeros_like(p_s)
    v_s = np.zeros_like(p_s)
    for t in (1, 2):
        for r in range(N):
            unit.load_grad(r, [fi.gen_grad(cfg, r, t, device=DEV)])
        g_s = [host(unit.grads[r][idx_d]) for r in range(N)]
        unit.step(hp_for(F, cfg, t), gathers=cfg.gathers)
        s = orc.scalars(ohp_for(orc, cfg, t), N)
        orc.adamw(p_s, m_s, v_s, orc.all_reduce_avg(g_s, cfg.grad_dtype, N, s.c), s)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(unit.master[idx_c].numpy().view(np.uint32), p_s.view(np.uint32))
        np.testing.assert_array_equal(unit.exp_avg[idx_c].numpy().view(np.uint32), m_s.view(np.uint32))
        np.testing.assert_array_equal(unit.exp_avg_sq[idx_c].numpy().view(np.uint32), v_s.view(np.uint32))
        assert_out_close(host(unit.shard_out[idx_d]), orc.cast_out(p_s, cfg.out_dtype), cfg.out_dtype, f"t={t}")
        for f in unit.full:
            assert torch.equal(f, unit.shard_out)
    del unit
    torch.cuda.empty_cache()


def test_binding_keeps_outputs_in_device_memory(F):
    # the compute-dtype shard, the gathered buffers and the counter must be
    # device memory; unpinned host memory is refused everywhere. Each refusal
    # is raised by the binding before the library is called.
    P, world = 64, 2
    grads = [torch.ones(P, dtype=torch.bfloat16, device=DEV) for _ in range(world)]
    st = [torch.zeros(P, pin_memory=True) for _ in range(3)]
    out_h = torch.zeros(P, dtype=torch.bfloat16, pin_memory=True)
    out_d = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    hp = F.AdamWHParams(1e-3, step=1)
    with pytest.raises(ValueError):
        F.fsdp_reduce_scatter_adam_cast(grads, *st, out_h, hp)
    with pytest.raises(ValueError):
        F.fsdp_all_gather(out_d, [out_h], world)
    with pytest.raises(ValueError):
        F.fsdp_all_gather(out_h, [out_d], world)
    with pytest.raises(ValueError):
        F.fsdp_reduce_scatter_adam_cast_gather(grads, *st, None, [out_h], hp)
    with pytest.raises(ValueError):
        F.fsdp_reduce_scatter_adam_cast(grads, torch.zeros(P), st[1], st[2], out_d, hp)
    with pytest.raises(ValueError):
        F.fsdp_reduce_scatter_adam_cast([torch.ones(P, dtype=torch.bfloat16)] * world, *st, out_d, hp)
    torch.cuda.synchronize()
    assert not out_d.any() and not st[0].any()


@pytest.mark.parametrize("world,P,rb,re", [(8, 8 * 1000 + 3, 3, 7), (2, 4099, 1, 2), (8, 8 * 40000, 0, 5),
                                           (4, 4 * 33, 1, 3)])
def test_offload_rank_subrange_and_ragged_blocks(F, world, P, rb, re):
    # host state over a rank subrange: the vector part starts off the
    # 256-element block grid of the host-state layout and ends on a ragged
    # tail; the blocks outside the range stay untouched
    P_pad = F.fsdp_padded_numel(P, world)
    S = P_pad // world
    g = torch.Generator().manual_seed(world + P)
    master0 = (torch.rand(P_pad, generator=g) * 0.2 - 0.1)
    master0[P:] = 0
    hs = [torch.zeros(P_pad, pin_memory=True) for _ in range(3)]
    ds = [torch.zeros(P_pad, device=DEV) for _ in range(3)]
    hs[0].copy_(master0)
    ds[0].copy_(master0)
    grads = [torch.zeros(P_pad, dtype=torch.bfloat16, device=DEV) for _ in range(world)]
    ho, do = (torch.zeros(P_pad, dtype=torch.bfloat16, device=DEV) for _ in range(2))
    for t in (1, 2):
        for q in range(world):
            x = (torch.randn(P_pad, generator=g) * 1e-2).to(torch.bfloat16)
            x[P:] = 0
            grads[q].copy_(x)
        hp = F.AdamWHParams(1e-3, weight_decay=0.01, step=t)
        F.fsdp_reduce_scatter_adam_cast(grads, *hs, ho, hp, rank_begin=rb, rank_end=re)
        F.fsdp_reduce_scatter_adam_cast(grads, *ds, do, hp, rank_begin=rb, rank_end=re)
    torch.cuda.synchronize()
    for x, y in zip(hs, ds):
        assert same_bits(x, y)
    assert same_bits(ho, do)
    assert torch.equal(hs[0][:rb * S], master0[:rb * S]) and torch.equal(hs[0][re * S:], master0[re * S:])
    assert not ho[:rb * S].any() and not ho[re * S:].any()


@pytest.mark.parametrize("opt,sdt", [("sgd", torch.float32), ("adamax", torch.float32), ("adamw", torch.bfloat16),
                                     ("adadelta", torch.float16)])
def test_offload_variant_rank_subrange(F, opt, sdt):
    # the variant kernels' host-state build (lane-interleaved chunks) over a
    # rank subrange that starts off the 256-element block grid
    world, P, rb, re = 8, 8 * 3000 + 5, 3, 7
    P_pad = F.fsdp_padded_numel(P, world)
    S = P_pad // world
    ns = 1 if opt == "sgd" else 2
    g = torch.Generator().manual_seed(P + ns)
    p0 = (torch.rand(P_pad, generator=g) * 0.2 - 0.1).to(sdt)
    p0[P:] = 0
    gdt = torch.float16 if sdt == torch.float16 else torch.bfloat16
    hs = [torch.zeros(P_pad, dtype=sdt, pin_memory=True) for _ in range(1 + ns)]
    ds = [torch.zeros(P_pad, dtype=sdt, device=DEV) for _ in range(1 + ns)]
    hs[0].copy_(p0)
    ds[0].copy_(p0)
    out_h = torch.zeros(P_pad, dtype=torch.bfloat16, device=DEV) if sdt == torch.float32 else None
    out_d = torch.zeros(P_pad, dtype=torch.bfloat16, device=DEV) if sdt == torch.float32 else None
    grads = [torch.zeros(P_pad, dtype=gdt, device=DEV) for _ in range(world)]
    lr = 1.0 if opt == "adadelta" else 1e-3
    for t in (1, 2):
        for q in range(world):
            x = (torch.randn(P_pad, generator=g) * 1e-2).to(gdt)
            x[P:] = 0
            grads[q].copy_(x)
        cfg = F.StepConfig(opt, lr, weight_decay=0.01, step=t)
        F.fsdp_reduce_scatter_step(grads, hs[0], hs[1], hs[2] if ns == 2 else None, out_h, cfg, rank_begin=rb,
                                   rank_end=re)
        F.fsdp_reduce_scatter_step(grads, ds[0], ds[1], ds[2] if ns == 2 else None, out_d, cfg, rank_begin=rb,
                                   rank_end=re)
    torch.cuda.synchronize()
    for x, y in zip(hs, ds):
        assert same_bits(x, y), opt
    if out_h is not None:
        assert same_bits(out_h, out_d)
    assert same_bits(hs[0][:rb * S], p0[:rb * S]) and same_bits(hs[0][re * S:], p0[re * S:])
