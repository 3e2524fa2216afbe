"""Batched launches of small units: fsdp_step_units (and a captured step)
runs the fused update and the all-gathers of up to 256 small units of one
world size and dtype pair as one launch each. Every element sees the per-unit
kernel's operations, so the results must equal stepping each unit on its own
bit for bit, and the oracle.
"""
import types

import numpy as np
import pytest
import torch

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


def make_units(F, specs, seed, **kw):
    """Two identical sets of units (a, b) with random masters; specs are
    (numel, world, grad dtype, out dtype)."""
    g = torch.Generator().manual_seed(seed)
    a, b = [], []
    for numel, world, gdt, odt in specs:
        x = torch.rand(numel, generator=g) * 0.2 - 0.1
        for dst in (a, b):
            u = F.FlatParamUnit([("w", (numel,))], world, gdt, odt, device=DEV, **kw)
            u.load_master([x.to(DEV)])
            dst.append(u)
    torch.cuda.synchronize()
    return a, b


def load_grads(units_sets, t, seed):
    g = torch.Generator().manual_seed(seed * 7919 + t)
    for k in range(len(units_sets[0])):
        u0 = units_sets[0][k]
        for r in range(u0.world):
            x = (torch.randn(u0.numel, generator=g) * 1e-2).to(DEV)
            for units in units_sets:
                units[k].load_grad(r, [x.to(units[k].grads[r].dtype)])


def same(x, y):
    iv = torch.int32 if x.element_size() == 4 else torch.int16
    return torch.equal(x.view(iv), y.view(iv))


def assert_units_equal(a, b, gathers):
    for k, (ua, ub) in enumerate(zip(a, b)):
        for name in ("master", "exp_avg", "exp_avg_sq", "shard_out"):
            assert same(getattr(ua, name), getattr(ub, name)), (k, name)
        for fa, fb in zip(ua.full, ub.full):
            assert same(fa, fb), k
        if gathers:
            for f in ua.full:
                assert same(f, ua.shard_out), k


def hp(F, t):
    return F.AdamWHParams(1e-3 * t, 0.9, 0.999, 1e-8, 0.01, t)


@pytest.mark.parametrize("gathers", [0, 1, 2])
def test_small_units_batched_equal_their_own_steps(F, gathers):
    # 300 units: sizes from 1 element to 60 k (ragged tails, units smaller than
    # one chunk), N in {1, 2, 4, 8}, two dtype pairs; 280 of one kind, so that
    # kind fills one group of 256 and starts a second
    rng = np.random.default_rng(gathers)
    specs = [(int(rng.integers(1, 60000)), 8, torch.bfloat16, torch.bfloat16) for _ in range(280)]
    specs += [(int(n), int(w), torch.bfloat16, torch.float16)
              for n, w in zip(rng.integers(1, 20000, 20), rng.choice([1, 2, 4, 8], 20))]
    specs[3] = (1, 8, torch.bfloat16, torch.bfloat16)
    specs[4] = (7, 8, torch.bfloat16, torch.bfloat16)
    a, b = make_units(F, specs, 11 + gathers)
    seq = F.UnitSequence(a)
    for t in (1, 2, 3):
        load_grads([a, b], t, 3)
        seq.step(hp(F, t), gathers=gathers)
        for u in b:
            u.step(hp(F, t), gathers=gathers)
        torch.cuda.synchronize()
        assert_units_equal(a, b, gathers)


def test_units_with_different_gather_fanouts_batch_together(F):
    # one batch of units with 1 to 8 gathered buffers each (n_full); every
    # buffer receives the unit's shards, bit-equal to each unit's own step
    rng = np.random.default_rng(9)
    g = torch.Generator().manual_seed(19)
    a, b = [], []
    for k in range(30):
        numel, n_full = int(rng.integers(1, 20000)), int(rng.integers(1, 9))
        x = torch.rand(numel, generator=g) * 0.2 - 0.1
        for dst in (a, b):
            u = F.FlatParamUnit([("w", (numel,))], 8, torch.bfloat16, torch.bfloat16, device=DEV, n_full=n_full)
            u.load_master([x.to(DEV)])
            dst.append(u)
    seq = F.UnitSequence(a)
    for t in (1, 2):
        load_grads([a, b], t, 41)
        seq.step(hp(F, t), gathers=2)
        for u in b:
            u.step(hp(F, t), gathers=2)
        torch.cuda.synchronize()
        assert_units_equal(a, b, 2)


@pytest.mark.parametrize("gathers", [1, 2])
def test_fused_gather_units_batched_equal_their_own_steps(F, gathers):
    # units whose first gather is written by the update kernel batch too, up
    # to 128 per launch: 150 units, 140 of one kind (a full fused batch and a
    # second), sizes from 1 to 60 k elements, 1-8 gathered buffers each, two
    # dtype pairs; the planned step and the captured step, each bit-equal to
    # every unit's own fused step
    rng = np.random.default_rng(30 + gathers)
    g = torch.Generator().manual_seed(23)
    a, b, c = [], [], []
    for k in range(150):
        numel, n_full = int(rng.integers(1, 60000)), int(rng.integers(1, 9))
        world, odt = (8, torch.bfloat16) if k < 140 else (int(rng.choice([2, 4])), torch.float16)
        x = torch.rand(numel, generator=g) * 0.2 - 0.1
        for dst in (a, b, c):
            u = F.FlatParamUnit([("w", (numel,))], world, torch.bfloat16, odt, device=DEV, n_full=n_full)
            u.load_master([x.to(DEV)])
            dst.append(u)
    seq = F.UnitSequence(a)
    assert seq.launches(gathers=gathers, fuse_gather=True) < 10 * gathers
    graph = F.UnitSequence(c).capture(gathers=gathers, fuse_gather=True)
    for t in (1, 2, 3):
        load_grads([a, b, c], t, 47)
        seq.step(hp(F, t), gathers=gathers, fuse_gather=True)
        graph.launch(hp(F, t))
        for u in b:
            u.step(hp(F, t), gathers=gathers, fuse_gather=True)
        torch.cuda.synchronize()
        assert_units_equal(a, b, gathers)
        assert_units_equal(c, b, gathers)
    graph.close()


def test_launch_counts_of_batched_models(F):
    # the planning query on real buffers: 300 small units batch into 2
    # launches per kernel (groups of 256 and 44), N = 3 units keep their own,
    # the variant call too
    a, _ = make_units(F, [(20000, 8, torch.bfloat16, torch.bfloat16)] * 300, 3)
    seq = F.UnitSequence(a)
    assert seq.launches(gathers=1) == 4 and seq.launches(gathers=2) == 6 and seq.launches(gathers=0) == 2
    assert F.UnitSequence(a[:200]).launches(gathers=1) == 2
    assert seq.launches(gathers=1, fuse_gather=True) == 3  # fused batches of 128, 128 and 44
    assert seq.launches(gathers=2, fuse_gather=True) == 6  # each with its separate second gather
    c, _ = make_units(F, [(3000, 3, torch.bfloat16, torch.bfloat16)] * 4, 4)
    assert F.UnitSequence(a[:10] + c).launches(gathers=1) == 2 + 8
    v, _ = make_variant_units(F, [(20000, 4, torch.bfloat16, torch.bfloat16)] * 260, 5, "sgd", torch.float32)
    assert F.UnitSequence(v).launches(gathers=1) == 4
    assert F.UnitSequence(v).launches(gathers=1, config=vcfg(F, "sgd", 1)) == 4


def test_a_full_group_and_a_group_of_one(F):
    # 257 units of one kind: a full group of 256 and one unit left over,
    # which is launched on its own; both bit-equal to each unit's own step
    rng = np.random.default_rng(5)
    specs = [(int(n), 2, torch.bfloat16, torch.bfloat16) for n in rng.integers(1, 3000, 257)]
    a, b = make_units(F, specs, 13)
    seq = F.UnitSequence(a)
    for t in (1, 2):
        load_grads([a, b], t, 37)
        seq.step(hp(F, t), gathers=1)
        for u in b:
            u.step(hp(F, t), gathers=1)
        torch.cuda.synchronize()
        assert_units_equal(a, b, 1)


def _odd_unit(F, numel, world, offset, seed, host_grads=False):
    """A unit whose buffers start `offset` elements into their allocations
    (offset 1: not 16-byte aligned, so it keeps its own launches); with
    host_grads its gradients are pinned host memory the kernel reads over
    the host link (the unit still batches when aligned)."""
    g = torch.Generator().manual_seed(seed)
    P = F.fsdp_padded_numel(numel, world)

    def alloc(dt, pinned=False):
        if pinned:
            return torch.zeros(P + offset, dtype=dt, pin_memory=True)[offset:]
        return torch.zeros(P + offset, dtype=dt, device=DEV)[offset:]

    u = types.SimpleNamespace(world=world, numel=numel, padded_numel=P)
    u.grads = [alloc(torch.bfloat16, host_grads) for _ in range(world)]
    u.master, u.exp_avg, u.exp_avg_sq = alloc(torch.float32), alloc(torch.float32), alloc(torch.float32)
    u.shard_out = alloc(torch.bfloat16)
    u.full = [alloc(torch.bfloat16) for _ in range(world)]
    u.master[:numel].copy_((torch.rand(numel, generator=g) * 0.2 - 0.1).to(DEV))
    return u


def test_batched_and_own_launches_in_one_call(F):
    # small aligned units batch (one of them reading its gradients from
    # pinned host memory); an unaligned unit, a unit of N = 3, a unit with
    # host-resident state and a unit above the batching size keep their own
    # kernels, all in one call, all equal to stepping each unit alone
    specs = [(int(n), 4, torch.bfloat16, torch.bfloat16) for n in (5000, 333, 70000, 12, 4099, 65536)]
    a, b = make_units(F, specs, 21)
    for dst in (a, b):
        dst.append(F.FlatParamUnit([("w", (3001,))], 3, torch.bfloat16, torch.bfloat16, device=DEV))
        dst.append(F.FlatParamUnit([("w", (9000,))], 4, torch.bfloat16, torch.bfloat16, device=DEV,
                                   state_on_host=True))
        dst.append(F.FlatParamUnit([("w", ((1 << 24) + 8,))], 4, torch.bfloat16, torch.bfloat16, device=DEV))
    for k in range(len(specs), len(a)):
        x = torch.rand(a[k].numel) * 0.2 - 0.1
        a[k].load_master([x.to(DEV)])
        b[k].load_master([x.to(DEV)])
    oa, ob = _odd_unit(F, 5000, 4, 1, 5), _odd_unit(F, 5000, 4, 1, 5)
    a.insert(2, oa)
    b.insert(2, ob)
    ha, hb = _odd_unit(F, 7777, 4, 0, 6, host_grads=True), _odd_unit(F, 7777, 4, 0, 6, host_grads=True)
    a.insert(4, ha)
    b.insert(4, hb)
    torch.cuda.synchronize()
    for t in (1, 2):
        g = torch.Generator().manual_seed(100 + t)
        for ua, ub in zip(a, b):
            for r in range(ua.world):
                x = (torch.randn(ua.numel, generator=g) * 1e-2).to(DEV, torch.bfloat16)
                for u in (ua, ub):
                    u.grads[r][:u.numel].copy_(x)
        F.fsdp_step_units(a, hp(F, t), gathers=2)
        for ub in b:
            F.fsdp_step_units([ub], hp(F, t), gathers=2)  # one unit per call: its own kernels
        torch.cuda.synchronize()
        assert_units_equal(a, b, 2)


@pytest.mark.parametrize("gathers", [1, 2])
def test_batched_units_in_a_captured_step(F, gathers):
    # the captured step holds batched update nodes; each launch rewrites their
    # scalars, and four launches over changing hyperparameters equal stepping
    # each unit alone, bit for bit
    rng = np.random.default_rng(40 + gathers)
    specs = [(int(n), 8, torch.bfloat16, torch.bfloat16) for n in rng.integers(1, 50000, 60)]
    specs += [(int(n), 2, torch.float16, torch.float16) for n in rng.integers(1, 50000, 10)]
    a, b = make_units(F, specs, 31)
    graph = F.UnitSequence(a).capture(gathers=gathers)
    for t in (1, 2, 3, 4):
        load_grads([a, b], t, 9)
        graph.launch(hp(F, t))
        for u in b:
            u.step(hp(F, t), gathers=gathers)
        torch.cuda.synchronize()
        assert_units_equal(a, b, gathers)
    graph.close()


def test_batched_units_match_oracle_and_count_nonfinite(F, orc):
    # a group of 40 units against the oracle, bit for bit; planted non-finite
    # gradients are counted as the per-unit kernel counts them
    rng = np.random.default_rng(7)
    specs = [(int(n), 4, torch.bfloat16, torch.bfloat16) for n in rng.integers(1, 30000, 40)]
    a, b = make_units(F, specs, 41)
    st = [[host(u.master), np.zeros(u.padded_numel, np.float32), np.zeros(u.padded_numel, np.float32)] for u in a]
    ca = torch.zeros(1, dtype=torch.int32, device=DEV)
    cb = torch.zeros(1, dtype=torch.int32, device=DEV)
    seq = F.UnitSequence(a)
    for t in (1, 2):
        load_grads([a, b], t, 17)
        if t == 2:
            for units in (a, b):
                units[5].grads[1][0] = float("inf")
                units[30].grads[3][units[30].numel - 1] = float("nan")
        seq.step(hp(F, t), gathers=1, nonfinite_count=ca)
        for u in b:
            u.step(hp(F, t), gathers=1, nonfinite_count=cb)
        torch.cuda.synchronize()
        assert_units_equal(a, b, 1)
        if t == 1:
            for u, (p, m, v) in zip(a, st):
                shards_o, _ = orc.fsdp_step([host(gr) for gr in u.grads], "bf16", u.world, p, m, v, "bf16",
                                            orc.hparams(1e-3 * t, 0.9, 0.999, 1e-8, 0.01, t))
                np.testing.assert_array_equal(host(u.master).view(np.uint32), p.view(np.uint32))
                np.testing.assert_array_equal(host(u.exp_avg).view(np.uint32), m.view(np.uint32))
                np.testing.assert_array_equal(host(u.exp_avg_sq).view(np.uint32), v.view(np.uint32))
                np.testing.assert_array_equal(host(u.shard_out), shards_o)
    assert int(ca.item()) == int(cb.item()) == 2


def make_variant_units(F, specs, seed, optimizer, state_dtype):
    g = torch.Generator().manual_seed(seed)
    a, b = [], []
    for numel, world, gdt, odt in specs:
        x = torch.rand(numel, generator=g) * 0.2 - 0.1
        for dst in (a, b):
            u = F.FlatParamUnit([("w", (numel,))], world, gdt, odt, device=DEV, optimizer=optimizer,
                                state_dtype=state_dtype)
            u.load_master([x.to(DEV)])
            dst.append(u)
    torch.cuda.synchronize()
    return a, b


def assert_variant_units_equal(a, b, gathers):
    for k, (ua, ub) in enumerate(zip(a, b)):
        for name in ("master", "exp_avg", "exp_avg_sq", "shard_out"):
            x, y = getattr(ua, name), getattr(ub, name)
            if x is not None:
                assert same(x, y), (k, name)
        for fa, fb in zip(ua.full, ub.full):
            assert same(fa, fb), k
        if gathers:
            for f in ua.full:
                assert same(f, ua.shard_out), k


VHP = {"adamw": (1e-3, 0.9, 0.999, 1e-8, 0.01), "sgd": (1e-2, 0.9, 0.0, 0.0, 1e-2),
       "adamax": (2e-3, 0.9, 0.999, 1e-8, 1e-2), "adadelta": (1.0, 0.9, 0.0, 1e-6, 1e-2)}


def vcfg(F, opt, t, lowp_dtype=None):
    lr, b1, b2, eps, wd = VHP[opt]
    return F.StepConfig(opt, lr * (1 + 0.1 * t), b1, b2, eps, wd, t, reduce_dtype=lowp_dtype)


@pytest.mark.parametrize("opt", ["sgd", "adamax", "adadelta", "adamw"])
@pytest.mark.parametrize("state", ["f32", "bf16"])
def test_small_variant_units_batched_equal_their_own_steps(F, opt, state):
    # the variant step batched: every optimizer, fp32 or bf16 state, a
    # bf16 reduce-scatter on the later steps, N in {1, 2, 4, 8}, sizes from 1
    # element to 40 k; bit-equal to each unit's own fsdp_reduce_scatter_step
    rng = np.random.default_rng(sum(map(ord, opt + state)))
    sdt = torch.float32 if state == "f32" else torch.bfloat16
    specs = [(int(n), int(w), torch.bfloat16, torch.bfloat16)
             for n, w in zip(rng.integers(1, 40000, 60), rng.choice([1, 2, 4, 8], 60))]
    specs[0] = (1, 8, torch.bfloat16, torch.bfloat16)
    a, b = make_variant_units(F, specs, 51, opt, sdt)
    seq = F.UnitSequence(a)
    for t in (1, 2, 3):
        load_grads([a, b], t, 23)
        cfg = vcfg(F, opt, t, torch.bfloat16 if t > 1 else None)
        seq.step(cfg, gathers=1)
        for u in b:
            u.step(cfg, gathers=1)
        torch.cuda.synchronize()
        assert_variant_units_equal(a, b, 1)


@pytest.mark.parametrize("opt,state", [("sgd", "f16"), ("adamw", "f16"), ("adadelta", "f32")])
def test_small_variant_units_fp16_with_loss_scale(F, opt, state):
    # fp16 gradients carrying a static loss scale of 1024 (unscaled inside the
    # step), fp16 or fp32 state, an fp16 reduce-scatter on the later steps
    rng = np.random.default_rng(len(opt) + len(state))
    sdt = torch.float16 if state == "f16" else torch.float32
    specs = [(int(n), int(w), torch.float16, torch.float16)
             for n, w in zip(rng.integers(1, 30000, 40), rng.choice([1, 2, 4, 8], 40))]
    a, b = make_variant_units(F, specs, 81, opt, sdt)
    seq = F.UnitSequence(a)
    lr, b1, b2, eps, wd = VHP[opt]
    for t in (1, 2, 3):
        g = torch.Generator().manual_seed(900 + t)
        for ua, ub in zip(a, b):
            for r in range(ua.world):
                x = (torch.randn(ua.numel, generator=g) * 1e-2 * 1024).to(DEV, torch.float16)
                ua.load_grad(r, [x])
                ub.load_grad(r, [x])
        cfg = F.StepConfig(opt, lr, b1, b2, eps, wd, t, 1024.0, reduce_dtype=torch.float16 if t > 1 else None)
        seq.step(cfg, gathers=1)
        for u in b:
            u.step(cfg, gathers=1)
        torch.cuda.synchronize()
        assert_variant_units_equal(a, b, 1)


def test_batched_variant_units_in_a_captured_step(F):
    # a captured SGD step with batched variant nodes: each launch rewrites
    # their scalars and reduction flag; equal to stepping each unit alone
    rng = np.random.default_rng(61)
    specs = [(int(n), 8, torch.bfloat16, torch.bfloat16) for n in rng.integers(1, 50000, 50)]
    a, b = make_variant_units(F, specs, 62, "sgd", torch.float32)
    graph = F.UnitSequence(a).capture(gathers=2, config=vcfg(F, "sgd", 1))
    for t in (1, 2, 3, 4):
        load_grads([a, b], t, 29)
        cfg = vcfg(F, "sgd", t, torch.bfloat16 if t % 2 == 0 else None)
        graph.launch(cfg)
        for u in b:
            u.step(cfg, gathers=2)
        torch.cuda.synchronize()
        assert_variant_units_equal(a, b, 2)
    graph.close()


def test_batched_variant_units_match_oracle(F, orc):
    # a batched Adamax group with bf16 state against the oracle, bit for bit
    rng = np.random.default_rng(71)
    specs = [(int(n), 4, torch.bfloat16, torch.bfloat16) for n in rng.integers(1, 20000, 30)]
    a, b = make_variant_units(F, specs, 72, "adamax", torch.bfloat16)
    st = [[host(u.master).copy(), np.zeros(u.padded_numel, np.uint16), np.zeros(u.padded_numel, np.uint16)]
          for u in a]
    seq = F.UnitSequence(a)
    lr, b1, b2, eps, wd = VHP["adamax"]
    for t in (1, 2):
        load_grads([a, b], t, 31)
        seq.step(vcfg(F, "adamax", t), gathers=1)
        torch.cuda.synchronize()
        for u, (p, s0, s1) in zip(a, st):
            orc.step_ex("adamax", False, [host(gr) for gr in u.grads], "bf16", u.world, p, s0, s1, "bf16", "bf16",
                        orc.hparams(lr * (1 + 0.1 * t), b1, b2, eps, wd, t))
            np.testing.assert_array_equal(host(u.master), p)
            np.testing.assert_array_equal(host(u.exp_avg), s0)
            np.testing.assert_array_equal(host(u.exp_avg_sq), s1)
