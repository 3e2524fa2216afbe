"""Units that take the variant step (SGD with momentum, Adamax, Adadelta,
AdamW with bf16/fp16 state or a gradient-dtype reduction) through
FlatParamUnit and the multi-unit step fsdp_step_units_ex: bit-identical to
calling fsdp_reduce_scatter_step on the same buffers, and to the oracle.
"""
import numpy as np
import pytest
import torch

from gpu_util import host

pytestmark = pytest.mark.gpu
DEV = "cuda"

LR = {"adamw": 1e-3, "sgd": 1e-2, "adamax": 2e-3, "adadelta": 1.0}
FMT = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sharded_fsdp_reduce_gb300 as F
    return F


def same(a, b):
    iv = torch.int32 if a.element_size() == 4 else torch.int16
    return torch.equal(a.detach().cpu().view(iv), b.detach().cpu().view(iv))


def make(F, opt, sdt, world=8, P=8 * 3000 + 5, gdt=torch.bfloat16, seed=0):
    odt = torch.bfloat16 if sdt == torch.float32 else sdt
    u = F.FlatParamUnit([("w", (P,))], world, gdt, odt, device=DEV, optimizer=opt, state_dtype=sdt)
    g = torch.Generator().manual_seed(seed)
    u.load_master([(torch.rand(P, generator=g) * 0.2 - 0.1).to(DEV)])
    torch.cuda.synchronize()
    return u


def set_grads(units, t, seed):
    g = torch.Generator().manual_seed(seed * 100 + t)
    for u in units:
        for r in range(u.world):
            u.grads[r].copy_((torch.randn(u.padded_numel, generator=g) * 1e-2).to(u.grads[r].dtype))
            u.grads[r][u.numel:] = 0


def cfg(F, opt, t, lowp_reduce, gdt=torch.bfloat16):
    return F.StepConfig(opt, LR[opt], 0.9, 0.999, 1e-8 if opt != "adadelta" else 1e-6, 0.01, t,
                        reduce_dtype=gdt if lowp_reduce else None)


@pytest.mark.parametrize("opt", ["adamw", "sgd", "adamax", "adadelta"])
@pytest.mark.parametrize("sdt", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("lowp_reduce", [False, True])
def test_variant_unit_matches_the_entry_point_and_the_oracle(F, orc, opt, sdt, lowp_reduce):
    gdt = torch.float16 if sdt == torch.float16 else torch.bfloat16
    u = make(F, opt, sdt, gdt=gdt, seed=1)
    # the same step through fsdp_reduce_scatter_step on separate buffers
    p, s0 = u.master.clone(), u.exp_avg.clone()
    s1 = u.exp_avg_sq.clone() if u.exp_avg_sq is not None else None
    out = torch.zeros_like(u.shard_out) if sdt == torch.float32 else None
    p_o = host(u.master)
    st_o = [np.zeros_like(p_o) for _ in range(1 if opt == "sgd" else 2)]
    for t in (1, 2, 3):
        set_grads([u], t, 3)
        c = cfg(F, opt, t, lowp_reduce, gdt)
        u.step(c, gathers=1)
        F.fsdp_reduce_scatter_step(u.grads, p, s0, s1, out, c)
        _, _ = orc.step_ex(opt, lowp_reduce, [host(g) for g in u.grads], FMT[gdt], u.world, p_o, st_o[0],
                           st_o[1] if len(st_o) > 1 else None, FMT[sdt], FMT[u.shard_out.dtype],
                           orc.hparams(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay, t, 1.0))
        torch.cuda.synchronize()
    assert same(u.master, p) and same(u.exp_avg, s0)
    if s1 is not None:
        assert same(u.exp_avg_sq, s1)
    if out is not None:
        assert same(u.shard_out, out)
    np.testing.assert_array_equal(host(u.master).view(np.uint8), p_o.view(np.uint8))
    np.testing.assert_array_equal(host(u.exp_avg).view(np.uint8), st_o[0].view(np.uint8))
    for f in u.full:
        assert same(f, u.shard_out)


@pytest.mark.parametrize("opt", ["sgd", "adamax", "adadelta", "adamw"])
@pytest.mark.parametrize("gathers", [0, 1, 2])
def test_variant_units_in_one_call(F, opt, gathers):
    # units of mixed N, sizes and state dtypes under one StepConfig, against
    # stepping each on its own
    shapes = [(8, 8 * 3000 + 5, torch.float32), (2, 4099, torch.bfloat16), (3, 1001, torch.float32),
              (8, 8 * 512, torch.bfloat16)]
    a = [make(F, opt, sdt, world=w, P=P, seed=k) for k, (w, P, sdt) in enumerate(shapes)]
    b = [make(F, opt, sdt, world=w, P=P, seed=k) for k, (w, P, sdt) in enumerate(shapes)]
    seq = F.UnitSequence(a)
    nf_a = torch.zeros(1, dtype=torch.int32, device=DEV)
    nf_b = torch.zeros(1, dtype=torch.int32, device=DEV)
    for t in (1, 2):
        set_grads(a, t, 7)
        set_grads(b, t, 7)
        seq.step(cfg(F, opt, t, False), gathers=gathers, nonfinite_count=nf_a)
        for u in b:
            u.step(cfg(F, opt, t, False), gathers=gathers, nonfinite_count=nf_b)
    torch.cuda.synchronize()
    for ua, ub in zip(a, b):
        for name in ("master", "exp_avg", "exp_avg_sq", "shard_out"):
            x, y = getattr(ua, name), getattr(ub, name)
            assert (x is None) == (y is None)
            if x is not None:
                assert same(x, y), name
        for fa, fb in zip(ua.full, ub.full):
            assert same(fa, fb)
    assert int(nf_a.item()) == int(nf_b.item()) == 0


def test_adamw_units_with_a_step_config_take_the_variant_kernel(F):
    # fp32 AdamW units stepped with a bf16-reduction StepConfig: the whole
    # model goes through fsdp_step_units_ex, each unit as its own variant step
    a = [make(F, "adamw", torch.float32, seed=k) for k in range(3)]
    b = [make(F, "adamw", torch.float32, seed=k) for k in range(3)]
    set_grads(a, 1, 9)
    set_grads(b, 1, 9)
    c = cfg(F, "adamw", 1, True)
    F.UnitSequence(a).step(c, gathers=2)
    for u in b:
        F.fsdp_reduce_scatter_step(u.grads, u.master, u.exp_avg, u.exp_avg_sq, u.shard_out, c)
        u.all_gather()
        u.all_gather()
    torch.cuda.synchronize()
    for ua, ub in zip(a, b):
        assert same(ua.master, ub.master) and same(ua.shard_out, ub.shard_out)
        for f in ua.full:
            assert same(f, ub.shard_out)
    with pytest.raises(ValueError):  # the fused gather needs the fused AdamW kernel
        F.UnitSequence(a).step(c, gathers=1, fuse_gather=True)


def test_variant_unit_host_pipeline_and_resume(F):
    # an SGD unit stepped from host gradients, and a bf16-state unit resumed
    # from per-rank snapshots
    a, b = make(F, "sgd", torch.float32, seed=2), make(F, "sgd", torch.float32, seed=2)
    hg = [[torch.zeros(a.padded_numel, dtype=torch.bfloat16).pin_memory() for _ in range(a.world)] for _ in range(3)]
    for t in range(3):
        set_grads([b], t + 1, 4)
        for r in range(a.world):
            hg[t][r].copy_(b.grads[r])
        b.step(cfg(F, "sgd", t + 1, False), gathers=1)
    for t in range(3):
        a.step_from_host(hg[t], None, cfg(F, "sgd", t + 1, False), gathers=1)
    torch.cuda.synchronize()
    assert same(a.master, b.master) and same(a.exp_avg, b.exp_avg) and same(a.full[0], b.full[0])

    c = make(F, "adamw", torch.bfloat16, seed=3)
    d = make(F, "adamw", torch.bfloat16, seed=3)
    for t in (1, 2):
        set_grads([c], t, 5)  # the same draw for each unit
        set_grads([d], t, 5)
        c.step(F.AdamWHParams(1e-3, weight_decay=0.01, step=t), gathers=1)
        d.step(F.AdamWHParams(1e-3, weight_decay=0.01, step=t), gathers=1)
    snap = [d.state_dict(rank=r) for r in range(d.world)]
    e = make(F, "adamw", torch.bfloat16, seed=99)
    for r, sd in enumerate(snap):
        e.load_state_dict(sd, rank=r)
    for u in (c, e):
        set_grads([u], 3, 5)
        u.step(F.AdamWHParams(1e-3, weight_decay=0.01, step=3), gathers=1)
    torch.cuda.synchronize()
    for name in ("master", "exp_avg", "exp_avg_sq"):
        assert same(getattr(c, name), getattr(e, name)), name
    assert same(c.full[0], e.full[0])


def test_variant_units_refuse_shared_buffers(F):
    a = [make(F, "adamax", torch.float32, seed=k) for k in range(2)]
    a[1].exp_avg = a[0].exp_avg.narrow(0, 0, a[1].padded_numel)  # two units write one buffer
    before = [u.master.clone() for u in a]
    with pytest.raises(F.FsdpError):
        F.UnitSequence(a).step(cfg(F, "adamax", 1, False), gathers=1)
    torch.cuda.synchronize()
    for u, p in zip(a, before):
        assert same(u.master, p)  # nothing ran


@pytest.mark.parametrize("opt", ["sgd", "adamax", "adadelta", "adamw"])
def test_captured_variant_step_matches_the_driver(F, opt):
    # one graph of the variant step, launched for steps 1..3 (with and
    # without a gradient-dtype reduction), against fsdp_step_units_ex
    shapes = [(8, 8 * 3000 + 5, torch.float32), (2, 4099, torch.bfloat16), (3, 1001, torch.float32)]
    a = [make(F, opt, sdt, world=w, P=P, seed=20 + k) for k, (w, P, sdt) in enumerate(shapes)]
    b = [make(F, opt, sdt, world=w, P=P, seed=20 + k) for k, (w, P, sdt) in enumerate(shapes)]
    graph = F.UnitSequence(a).capture(gathers=2, config=cfg(F, opt, 1, False))
    seq_b = F.UnitSequence(b)
    for t in (1, 2, 3):
        set_grads(a, t, 21)
        set_grads(b, t, 21)
        c = cfg(F, opt, t, t == 2)
        graph.launch(c)
        seq_b.step(c, gathers=2)
    torch.cuda.synchronize()
    for ua, ub in zip(a, b):
        for name in ("master", "exp_avg", "exp_avg_sq", "shard_out"):
            x, y = getattr(ua, name), getattr(ub, name)
            if x is not None:
                assert same(x, y), name
        for fa, fb in zip(ua.full, ub.full):
            assert same(fa, fb)
    other = "adamax" if opt != "adamax" else "sgd"
    with pytest.raises(F.FsdpError):  # the graph holds this optimizer's kernels
        graph.launch(F.StepConfig(other, 1e-3, step=4))
    with pytest.raises(F.FsdpError):  # a reduction in another dtype than the gradients'
        graph.launch(F.StepConfig(opt, 1e-3, step=4, reduce_dtype=torch.float16))
    with pytest.raises(ValueError):
        F.UnitSequence(a).capture(gathers=1)  # variant units need a StepConfig
    graph.close()
