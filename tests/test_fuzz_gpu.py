"""Seeded random configurations of the fused step against the oracle: world
size, unit size, gradient/output dtypes, emulated rank subrange, pointer
offsets (vector or scalar path), the fused all-gather and the variant
optimizers, several steps each. Bars as in the other parity tests."""
import numpy as np
import pytest
import torch

import fsdp_inputs as fi
from gpu_util import assert_out_close, assert_state_close, host

pytestmark = pytest.mark.gpu
DEV = "cuda"
FMTS = ["bf16", "f16", "f32"]


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sharded_fsdp_reduce_gb300 as F
    return F


def _case(seed, max_p=40000):
    rng = np.random.default_rng(1000 + seed)
    world = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    P = int(rng.integers(1, max_p))
    gfmt, ofmt = str(rng.choice(FMTS)), str(rng.choice(FMTS))
    rb = int(rng.integers(0, world))
    re = int(rng.integers(rb + 1, world + 1))
    offset = int(rng.choice([0, 0, 1]))
    gather = bool(rng.integers(0, 2))
    scale = 1024.0 if gfmt == "f16" else 1.0
    return rng, world, P, gfmt, ofmt, rb, re, offset, gather, scale


@pytest.mark.parametrize("seed,max_p", [(s, 40000) for s in range(40)] + [(s, 3000000) for s in range(100, 108)])
def test_fuzz_fused_step(F, orc, seed, max_p):
    # max_p 3 M: units of up to ~1,500 CTAs of the vector path, many waves
    rng, world, P, gfmt, ofmt, rb, re, offset, gather, scale = _case(seed, max_p)
    P_pad = orc.padded_numel(P, world)
    S = P_pad // world
    gdt, odt = fi.torch_dtype(gfmt), fi.torch_dtype(ofmt)

    def alloc(n, dt):
        return torch.zeros(n + offset, dtype=dt, device=DEV)[offset:]

    grads = [alloc(P_pad, gdt) for _ in range(world)]
    master, m, v = (alloc(P_pad, torch.float32) for _ in range(3))
    out = alloc(P_pad, odt)
    fulls = [alloc(P_pad, odt) for _ in range(world)] if gather else []
    p0 = orc.flatten_pad([rng.uniform(-0.1, 0.1, P).astype(np.float32)], world)
    master.copy_(torch.from_numpy(p0))
    p_o, m_o, v_o = p0.copy(), np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)
    lo, hi = rb * S, re * S
    for t in (1, 2):
        rows = []
        for r in range(world):
            x = torch.from_numpy(orc.flatten_pad([(rng.standard_normal(P) * 1e-2 * scale).astype(np.float32)], world))
            rows.append(x.to(gdt))
            grads[r].copy_(rows[-1].to(DEV))
        hp = F.AdamWHParams(1e-3, 0.9, 0.999, 1e-8, 0.01, t, scale)
        if gather:
            F.fsdp_reduce_scatter_adam_cast_gather(grads, master, m, v, out, fulls, hp, rank_begin=rb, rank_end=re)
        else:
            F.fsdp_reduce_scatter_adam_cast(grads, master, m, v, out, hp, rank_begin=rb, rank_end=re)
        # the oracle updates every rank; only [lo, hi) is compared, the rest must be untouched
        before = p_o.copy(), m_o.copy(), v_o.copy()
        shards_o, _ = orc.fsdp_step([host(x) for x in rows], gfmt, world, p_o, m_o, v_o, ofmt,
                                    orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, t, scale))
        for arr, old in zip((p_o, m_o, v_o), before):  # ranks outside the subrange keep their state
            arr[:lo] = old[:lo]
            arr[hi:] = old[hi:]
        torch.cuda.synchronize()
        tag = f"seed={seed} N={world} P={P} {gfmt}->{ofmt} ranks=[{rb},{re}) off={offset} gather={gather} t={t}"
        assert_state_close(host(master), p_o, "master " + tag)
        assert_state_close(host(m), m_o, "exp_avg " + tag)
        assert_state_close(host(v), v_o, "exp_avg_sq " + tag)
        assert_out_close(host(out)[lo:hi], shards_o[lo:hi], ofmt, "shard_out " + tag)
        for f in fulls:
            np.testing.assert_array_equal(host(f)[lo:hi].view(np.uint8), host(out)[lo:hi].view(np.uint8))
    if rb > 0 or re < world:
        assert not host(out)[:lo].view(np.uint8).any() and not host(out)[hi:].view(np.uint8).any()


@pytest.mark.parametrize("seed,max_p", [(s, 30000) for s in range(24)] + [(s, 2000000) for s in range(100, 106)])
def test_fuzz_variant_step(F, orc, seed, max_p):
    rng = np.random.default_rng(5000 + seed)
    opt = str(rng.choice(["adamw", "sgd", "adamax", "adadelta"]))
    world = int(rng.choice([1, 2, 3, 8]))
    P = int(rng.integers(1, max_p))
    gfmt = str(rng.choice(FMTS))
    sfmt = str(rng.choice(["f32", "bf16", "f16"]))
    ofmt = str(rng.choice(FMTS)) if sfmt == "f32" else sfmt
    lowp = bool(rng.integers(0, 2)) and gfmt != "f32"
    scale = 1024.0 if gfmt == "f16" else 1.0
    lr, b1, b2, eps, wd = {"adamw": (1e-3, 0.9, 0.999, 1e-8, 0.01), "sgd": (1e-2, 0.9, 0.0, 0.0, 1e-2),
                           "adamax": (2e-3, 0.9, 0.999, 1e-8, 1e-2), "adadelta": (1.0, 0.9, 0.0, 1e-6, 1e-2)}[opt]
    P_pad = orc.padded_numel(P, world)
    gdt, sdt = fi.torch_dtype(gfmt), fi.torch_dtype(sfmt)
    ns = 1 if opt == "sgd" else 2
    grads = [torch.zeros(P_pad, dtype=gdt, device=DEV) for _ in range(world)]
    p0 = torch.from_numpy(orc.flatten_pad([rng.uniform(-0.1, 0.1, P).astype(np.float32)], world)).to(sdt)
    param = p0.to(DEV)
    states = [torch.zeros(P_pad, dtype=sdt, device=DEV) for _ in range(ns)]
    out = torch.zeros(P_pad, dtype=fi.torch_dtype(ofmt), device=DEV) if sfmt == "f32" else None
    p_o = host(p0)
    s_o = [np.zeros(P_pad, orc.np_storage(sfmt)) for _ in range(ns)]
    for t in (1, 2, 3):
        rows = [torch.from_numpy(orc.flatten_pad([(rng.standard_normal(P) * 1e-2 * scale).astype(np.float32)],
                                                 world)).to(gdt) for _ in range(world)]
        for g, r in zip(grads, rows):
            g.copy_(r.to(DEV))
        cfg = F.StepConfig(opt, lr, b1, b2, eps, wd, t, scale, reduce_dtype=gdt if lowp else None)
        F.fsdp_reduce_scatter_step(grads, param, states[0], states[1] if ns == 2 else None, out, cfg)
        shards_o, _ = orc.step_ex(opt, lowp, [host(r) for r in rows], gfmt, world, p_o, s_o[0],
                                  s_o[1] if ns == 2 else None, sfmt, ofmt, orc.hparams(lr, b1, b2, eps, wd, t, scale))
        torch.cuda.synchronize()
        tag = f"seed={seed} {opt} N={world} P={P} {gfmt} state={sfmt} out={ofmt} lowp={lowp} t={t}"
        cmp = assert_state_close if sfmt == "f32" else (lambda a, b, w: assert_out_close(a, b, sfmt, w))
        cmp(host(param), p_o, "param " + tag)
        for k in range(ns):
            cmp(host(states[k]), s_o[k], f"state{k} " + tag)
        if out is not None:
            assert_out_close(host(out), shards_o, ofmt, "shard_out " + tag)


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_step_units(F, orc, seed):
    # a random model: 1-5 units of random N, size and dtypes, some offloaded,
    # stepped by fsdp_step_units with random gathers and fusion
    rng = np.random.default_rng(5000 + seed)
    n_units = int(rng.integers(1, 6))
    gathers = int(rng.integers(0, 3))
    fuse = bool(rng.integers(0, 2))
    units, st = [], []
    for _ in range(n_units):
        world = int(rng.choice([1, 2, 3, 8]))
        P = int(rng.integers(1, 30000))
        gfmt, ofmt = str(rng.choice(FMTS)), str(rng.choice(FMTS))
        u = F.FlatParamUnit([("x", (P,))], world, fi.torch_dtype(gfmt), fi.torch_dtype(ofmt), device=DEV,
                            n_full=int(rng.integers(1, world + 1)), state_on_host=bool(rng.integers(0, 2)))
        p0 = orc.flatten_pad([rng.uniform(-0.1, 0.1, P).astype(np.float32)], world)
        u.master.copy_(torch.from_numpy(p0))
        units.append((u, gfmt, ofmt, P))
        st.append([p0.copy(), np.zeros_like(p0), np.zeros_like(p0)])
    seq = F.UnitSequence([u for u, *_ in units])
    for t in (1, 2):
        hp = F.AdamWHParams(1e-3, weight_decay=0.01, step=t)
        rows_all = []
        for u, gfmt, ofmt, P in units:
            rows = []
            for r in range(u.world):
                x = torch.from_numpy(orc.flatten_pad([(rng.standard_normal(P) * 1e-2).astype(np.float32)], u.world))
                x = x.to(fi.torch_dtype(gfmt))
                u.grads[r].copy_(x.to(DEV))
                rows.append(host(x))
            rows_all.append(rows)
        seq.step(hp, gathers=gathers, fuse_gather=fuse)
        torch.cuda.synchronize()
        for (u, gfmt, ofmt, P), rows, (p, m, v) in zip(units, rows_all, st):
            shards_o, _ = orc.fsdp_step(rows, gfmt, u.world, p, m, v, ofmt,
                                        orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, t, 1.0))
            assert_state_close(host(u.master), p, f"seed {seed} master t={t}")
            assert_state_close(host(u.exp_avg), m, f"seed {seed} exp_avg t={t}")
            assert_state_close(host(u.exp_avg_sq), v, f"seed {seed} exp_avg_sq t={t}")
            assert_out_close(host(u.shard_out), shards_o, ofmt, f"seed {seed} shard_out t={t}")
            for f in u.full:
                if gathers:
                    assert torch.equal(f, u.shard_out)
                else:
                    assert not f.view(torch.uint8).any()  # never gathered: still zero


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_step_graph(F, seed):
    # a random model captured once (AdamW, or a random variant optimizer) and
    # launched for a random sequence of steps with random hyperparameters,
    # against the native driver on a twin model, bit for bit
    rng = np.random.default_rng(7000 + seed)
    variant = bool(seed % 2)
    opt = str(rng.choice(["sgd", "adamax", "adadelta", "adamw"])) if variant else "adamw"
    n_units = int(rng.integers(1, 5))
    gathers = int(rng.integers(0, 3))
    fuse = (not variant) and gathers > 0 and bool(rng.integers(0, 2))
    specs = []
    for _ in range(n_units):
        world = int(rng.choice([1, 2, 3, 8]))
        P = int(rng.integers(1, 20000))
        gdt = fi.torch_dtype(str(rng.choice(["bf16", "f16", "f32"])))
        sdt = fi.torch_dtype(str(rng.choice(["bf16", "f32"]))) if variant else torch.float32
        odt = sdt if sdt != torch.float32 else fi.torch_dtype(str(rng.choice(FMTS)))
        host = sdt == torch.float32 and bool(rng.integers(0, 2))
        specs.append((world, P, gdt, sdt, odt, host, int(rng.integers(0, 1 << 30))))

    def build():
        units = []
        for world, P, gdt, sdt, odt, host, s in specs:
            u = F.FlatParamUnit([("x", (P,))], world, gdt, odt, device=DEV, optimizer=opt, state_dtype=sdt,
                                state_on_host=host)
            g = torch.Generator().manual_seed(s)
            u.load_master([(torch.rand(P, generator=g) * 0.2 - 0.1).to(DEV)])
            units.append(u)
        torch.cuda.synchronize()
        return units

    a, b = build(), build()

    def hp(t, lr, wd):
        if variant:
            return F.StepConfig(opt, lr, 0.9, 0.999, 1e-6, wd, t)
        return F.AdamWHParams(lr, 0.9, 0.999, 1e-8, wd, t)

    graph = F.UnitSequence(a).capture(gathers=gathers, fuse_gather=fuse, config=hp(1, 1e-3, 0.0) if variant else None)
    seq_b = F.UnitSequence(b)
    t = 0
    for _ in range(int(rng.integers(1, 4))):
        t += int(rng.integers(1, 3))
        lr, wd = float(10 ** rng.uniform(-4, -2)), float(rng.choice([0.0, 0.01, 0.1]))
        gg = torch.Generator().manual_seed(seed * 100 + t)
        for ua, ub in zip(a, b):
            for r in range(ua.world):
                x = (torch.randn(ua.padded_numel, generator=gg) * 1e-2).to(ua.grads[r].dtype)
                x[ua.numel:] = 0
                ua.grads[r].copy_(x)
                ub.grads[r].copy_(x)
        graph.launch(hp(t, lr, wd))
        seq_b.step(hp(t, lr, wd), gathers=gathers, fuse_gather=fuse)
    torch.cuda.synchronize()
    for ua, ub in zip(a, b):
        for name in ("master", "exp_avg", "exp_avg_sq", "shard_out"):
            x, y = getattr(ua, name), getattr(ub, name)
            if x is not None:
                iv = torch.int32 if x.element_size() == 4 else torch.int16
                assert torch.equal(x.cpu().view(iv), y.cpu().view(iv)), (seed, name)
        for fa, fb in zip(ua.full, ub.full):
            iv = torch.int32 if fa.element_size() == 4 else torch.int16
            assert torch.equal(fa.view(iv), fb.view(iv)), seed
    graph.close()


def _same(x, y):
    iv = torch.int32 if x.element_size() == 4 else torch.int16
    return torch.equal(x.view(iv), y.view(iv))


@pytest.mark.parametrize("seed", range(10))
def test_fuzz_batched_models(F, seed):
    # a random model of 2-320 units for the batched launches: mostly small
    # units of N in {1, 2, 4, 8} and two dtype pairs, 1-8 gathered buffers each,
    # among them units that keep their own launches (N = 3, host-resident
    # state, above the batching size), the first gather fused into the
    # update in half the seeds that gather; stepped by the planned native
    # step (even seeds) or a captured step (odd seeds) and compared bit for
    # bit with each unit stepped alone
    rng = np.random.default_rng(7000 + seed)
    n_units = int(rng.integers(2, 321))
    gathers = int(rng.integers(0, 3))
    fuse = gathers > 0 and bool(rng.random() < 0.5)
    pairs = [(torch.bfloat16, torch.bfloat16), (torch.bfloat16, torch.float16), (torch.float32, torch.bfloat16)]
    a, b = [], []
    g = torch.Generator().manual_seed(seed)
    for _ in range(n_units):
        kind = rng.random()
        world = 3 if kind < 0.05 else int(rng.choice([1, 2, 4, 8], p=[0.1, 0.2, 0.2, 0.5]))
        P = int(rng.integers((1 << 24) + 1, (1 << 24) + 5000)) if kind > 0.98 else int(rng.integers(1, 60000))
        host_state = 0.05 <= kind < 0.1
        gdt, odt = pairs[int(rng.integers(0, 2 if seed % 3 else 3))]
        n_full = int(rng.integers(1, 9))
        x = torch.rand(P, generator=g) * 0.2 - 0.1
        for dst in (a, b):
            u = F.FlatParamUnit([("x", (P,))], world, gdt, odt, device=DEV, n_full=n_full, state_on_host=host_state)
            u.load_master([x.to(DEV)])
            dst.append(u)
    torch.cuda.synchronize()
    graph = F.UnitSequence(a).capture(gathers=gathers, fuse_gather=fuse) if seed % 2 else None
    seq = F.UnitSequence(a)
    for t in (1, 2, 3):
        gg = torch.Generator().manual_seed(100 * seed + t)
        for ua, ub in zip(a, b):
            for r in range(ua.world):
                xg = (torch.randn(ua.numel, generator=gg) * 1e-2).to(DEV, ua.grads[r].dtype)
                ua.load_grad(r, [xg])
                ub.load_grad(r, [xg])
        hp = F.AdamWHParams(1e-3 * t, 0.9, 0.999, 1e-8, 0.01, t)
        if graph is not None:
            graph.launch(hp)
        else:
            seq.step(hp, gathers=gathers, fuse_gather=fuse)
        for u in b:
            u.step(hp, gathers=gathers, fuse_gather=fuse)
        torch.cuda.synchronize()
        for k, (ua, ub) in enumerate(zip(a, b)):
            for name in ("master", "exp_avg", "exp_avg_sq", "shard_out"):
                assert _same(getattr(ua, name), getattr(ub, name)), (seed, k, name, t)
            for fa, fb in zip(ua.full, ub.full):
                assert _same(fa, fb), (seed, k, t)
    if graph is not None:
        graph.close()
    del a, b
    torch.cuda.empty_cache()
