"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small units are compared element by element over their whole parity
trajectory; the 13B and 70B units run at full size in the launch
configuration the bench uses and are compared on sampled elements (the step
is pointwise, so the oracle computes each sampled element on its own), plus
the all-gather property full_k == shard_out at every element.

Bars: layout, gathered buffers and everything integer bit-exact; fp32 master,
exp_avg, exp_avg_sq within 1e-6 relative; bf16/fp16 outputs within 1 ulp.
The kernel performs the oracle's operations in the oracle's order, so the
results are in fact expected to be identical; test_bit_exact checks that.
"""
import numpy as np
import pytest
import torch

import fsdp_inputs as fi
from gpu_util import assert_out_close, assert_state_close, host

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


def split_views(unit, flat):
    return [flat.narrow(0, v.offset, v.numel).contiguous() for v in unit.views]


def new_unit(F, cfg, **kw):
    return F.FlatParamUnit(cfg.params, cfg.world, fi.torch_dtype(cfg.grad_dtype), fi.torch_dtype(cfg.out_dtype),
                           device=DEV, **kw)


# ------------------------------------------------------------------ whole trajectories

@pytest.mark.parametrize("name", ["tiny", "gpt2_small", "gpt2_large"])
def test_config_trajectory_elementwise(F, orc, name):
    cfg = fi.CONFIGS[name]
    N = cfg.world
    unit = new_unit(F, cfg)
    master = fi.gen_master(cfg)
    unit.load_master(split_views(unit, master.to(DEV)))
    p_o = orc.flatten_pad([master.numpy()], N)
    m_o = np.zeros_like(p_o)
    v_o = np.zeros_like(p_o)
    np.testing.assert_array_equal(host(unit.master), p_o)
    for t in range(1, cfg.steps + 1):
        grads = [fi.gen_grad(cfg, r, t) for r in range(N)]
        for r in range(N):
            unit.load_grad(r, split_views(unit, grads[r].to(DEV)))
        g_o = [orc.flatten_pad([host(g)], N) for g in grads]
        for r in range(N):
            np.testing.assert_array_equal(host(unit.grads[r]), g_o[r])  # flatten + zero pad, bit-exact
        unit.step(hp_for(F, cfg, t), gathers=cfg.gathers)
        shards_o, full_o = orc.fsdp_step(g_o, cfg.grad_dtype, N, p_o, m_o, v_o, cfg.out_dtype, ohp_for(orc, cfg, t))
        torch.cuda.synchronize()
        assert_state_close(host(unit.master), p_o, f"{name} master t={t}")
        assert_state_close(host(unit.exp_avg), m_o, f"{name} exp_avg t={t}")
        assert_state_close(host(unit.exp_avg_sq), v_o, f"{name} exp_avg_sq t={t}")
        assert_out_close(host(unit.shard_out), shards_o, cfg.out_dtype, f"{name} shard_out t={t}")
        for k, f in enumerate(unit.full):
            assert torch.equal(f, unit.shard_out), f"{name} full[{k}] t={t}"
        P = unit.numel
        assert not host(unit.master)[P:].any() and not host(unit.shard_out)[P:].any()  # pad stays zero


def test_bit_exact(F, orc):
    cfg = fi.CONFIGS["gpt2_small"]
    N = cfg.world
    unit = new_unit(F, cfg)
    master = fi.gen_master(cfg)
    unit.load_master([master.to(DEV)])
    p_o = master.numpy().copy()
    m_o = np.zeros_like(p_o)
    v_o = np.zeros_like(p_o)
    for t in (1, 2, 3):
        grads = [fi.gen_grad(cfg, r, t) for r in range(N)]
        for r in range(N):
            unit.load_grad(r, [grads[r].to(DEV)])
        unit.step(hp_for(F, cfg, t))
        shards_o, _ = orc.fsdp_step([host(g) for g in grads], cfg.grad_dtype, N, p_o, m_o, v_o, cfg.out_dtype,
                                    ohp_for(orc, cfg, t))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(unit.master).view(np.uint32), p_o.view(np.uint32))
        np.testing.assert_array_equal(host(unit.exp_avg).view(np.uint32), m_o.view(np.uint32))
        np.testing.assert_array_equal(host(unit.exp_avg_sq).view(np.uint32), v_o.view(np.uint32))
        np.testing.assert_array_equal(host(unit.shard_out), shards_o)


def _sample_indices(P_pad, N, k, seed):
    S = P_pad // N
    rng = np.random.default_rng(seed)
    idx = [rng.integers(0, P_pad, size=k)]
    for r in range(N):  # both ends of every rank block, and the last element
        idx.append(np.arange(r * S, r * S + 64))
        idx.append(np.arange((r + 1) * S - 64, (r + 1) * S))
    return np.unique(np.concatenate(idx)).astype(np.int64)


@pytest.mark.parametrize("name,fuse", [("gpt3_13b", False), ("llama70b", False), ("gpt3_13b", True), ("llama70b", True)])
def test_full_size_sampled(F, orc, name, fuse):
    # fuse: the first all-gather written by the update kernel itself
    cfg = fi.CONFIGS[name]
    N = cfg.world
    unit = new_unit(F, cfg)
    assert unit.padded_numel == unit.numel  # these units need no padding
    unit.load_master([fi.gen_master(cfg, device=DEV)])
    idx = _sample_indices(unit.padded_numel, N, 1 << 20, 7)
    idx_t = torch.from_numpy(idx).to(DEV)
    p_s = unit.master[idx_t].cpu().numpy()
    m_s = np.zeros_like(p_s)
    v_s = np.zeros_like(p_s)
    for t in range(1, cfg.steps + 1):
        for r in range(N):
            g = fi.gen_grad(cfg, r, t, device=DEV)
            unit.load_grad(r, [g])
            del g
        g_s = [host(unit.grads[r][idx_t]) for r in range(N)]
        unit.step(hp_for(F, cfg, t), gathers=cfg.gathers, fuse_gather=fuse)
        s = orc.scalars(ohp_for(orc, cfg, t), N)
        g_avg = orc.all_reduce_avg(g_s, cfg.grad_dtype, N, s.c)
        orc.adamw(p_s, m_s, v_s, g_avg, s)
        out_s = orc.cast_out(p_s, cfg.out_dtype)
        torch.cuda.synchronize()
        assert_state_close(host(unit.master[idx_t]), p_s, f"{name} master t={t}")
        assert_state_close(host(unit.exp_avg[idx_t]), m_s, f"{name} exp_avg t={t}")
        assert_state_close(host(unit.exp_avg_sq[idx_t]), v_s, f"{name} exp_avg_sq t={t}")
        assert_out_close(host(unit.shard_out[idx_t]), out_s, cfg.out_dtype, f"{name} shard_out t={t}")
        for k, f in enumerate(unit.full):
            assert torch.equal(f, unit.shard_out), f"{name} full[{k}] t={t}"
    del unit
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ sizes, dtypes, edge cases

def _run_flat(F, orc, world, P, gfmt, ofmt, steps=2, scale=1.0, seed=0, offset=0, n_dst=None):
    """Unit of one P-element tensor; tensors may start `offset` elements into
    larger allocations (offset 1 disables the 16-byte vector path)."""
    rng = np.random.default_rng(seed)
    P_pad = orc.padded_numel(P, world)
    gdt, odt = fi.torch_dtype(gfmt), fi.torch_dtype(ofmt)

    def alloc(n, dt):
        return torch.zeros(n + offset, dtype=dt, device=DEV)[offset:]

    grads = [alloc(P_pad, gdt) for _ in range(world)]
    master, m, v = (alloc(P_pad, torch.float32) for _ in range(3))
    out = alloc(P_pad, odt)
    fulls = [alloc(P_pad, odt) for _ in range(world if n_dst is None else n_dst)]
    p0 = rng.uniform(-0.1, 0.1, P).astype(np.float32)
    F.fsdp_flatten_pad([torch.from_numpy(p0).to(DEV)], world, out=master)
    p_o = orc.flatten_pad([p0], world)
    m_o = np.zeros(P_pad, np.float32)
    v_o = np.zeros(P_pad, np.float32)
    for t in range(1, steps + 1):
        rows = [torch.from_numpy((rng.standard_normal(P) * 1e-2 * scale).astype(np.float32)).to(gdt)
                for _ in range(world)]
        for r in range(world):
            F.fsdp_flatten_pad([rows[r].to(DEV)], world, out=grads[r])
        hp = F.AdamWHParams(1e-3, 0.9, 0.999, 1e-8, 0.01, t, scale)
        F.fsdp_reduce_scatter_adam_cast(grads, master, m, v, out, hp)
        F.fsdp_all_gather(out, fulls, world)
        g_o = [orc.flatten_pad([host(r_)], world) for r_ in rows]
        shards_o, full_o = orc.fsdp_step(g_o, gfmt, world, p_o, m_o, v_o, ofmt,
                                         orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, t, scale))
        torch.cuda.synchronize()
        assert_state_close(host(master), p_o, "master")
        assert_state_close(host(m), m_o, "exp_avg")
        assert_state_close(host(v), v_o, "exp_avg_sq")
        assert_out_close(host(out), shards_o, ofmt, "shard_out")
        for f in fulls:
            np.testing.assert_array_equal(host(f).view(np.uint8), host(out).view(np.uint8))
        assert not p_o[P:].any() and not host(master)[P:].any()


@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("P", [1, 2, 7, 8, 9, 17, 4099, 8 * 127 + 5])
def test_odd_sizes_bf16(F, orc, world, P):
    _run_flat(F, orc, world, P, "bf16", "bf16", seed=P * 10 + world)


@pytest.mark.parametrize("gfmt,ofmt,scale", [("f16", "f16", 1024.0), ("f32", "f32", 1.0), ("bf16", "f32", 1.0),
                                             ("f32", "bf16", 1.0), ("f16", "bf16", 1.0), ("bf16", "f16", 1.0)])
@pytest.mark.parametrize("world,P", [(2, 4099), (8, 8 * 1000 + 3), (4, 4 * 33)])
def test_dtype_combinations(F, orc, gfmt, ofmt, scale, world, P):
    _run_flat(F, orc, world, P, gfmt, ofmt, scale=scale, seed=world + P)


@pytest.mark.parametrize("gfmt,ofmt", [("bf16", "bf16"), ("f32", "f16")])
@pytest.mark.parametrize("world,P", [(2, 4099), (8, 8 * 200 + 1), (5, 1234)])
def test_unaligned_pointers_take_the_scalar_path(F, orc, gfmt, ofmt, world, P):
    _run_flat(F, orc, world, P, gfmt, ofmt, offset=1, seed=3)


def test_all_gather_fanouts(F, orc):
    for n_dst in (1, 2, 3, 8, 13):
        _run_flat(F, orc, 4, 4 * 77 + 1, "bf16", "bf16", steps=1, n_dst=n_dst, seed=n_dst)


def test_rank_subrange_touches_only_its_blocks(F, orc):
    cfg = fi.CONFIGS["tiny"]
    world, P = 4, 4 * 2050 - 3  # S = 2050: block starts are not 8-aligned
    rng = np.random.default_rng(11)
    P_pad = orc.padded_numel(P, world)
    S = P_pad // world
    grads = [torch.from_numpy(orc.flatten_pad([(rng.standard_normal(P) * 1e-2).astype(np.float32)], world))
             .to(torch.bfloat16).to(DEV) for _ in range(world)]
    master = torch.from_numpy(orc.flatten_pad([rng.uniform(-0.1, 0.1, P).astype(np.float32)], world)).to(DEV)
    m = torch.full((P_pad,), 1e-3, device=DEV)
    v = torch.full((P_pad,), 1e-6, device=DEV)
    out = torch.full((P_pad,), 7.0, dtype=torch.bfloat16, device=DEV)
    before = [host(x) for x in (master, m, v, out)]
    hp = F.AdamWHParams(1e-3, 0.9, 0.999, 1e-8, 0.01, 3)
    F.fsdp_reduce_scatter_adam_cast(grads, master, m, v, out, hp, rank_begin=1, rank_end=3)
    p_o, m_o, v_o = before[0].copy(), before[1].copy(), before[2].copy()
    shards_o, _ = orc.fsdp_step([host(g) for g in grads], "bf16", world, p_o, m_o, v_o, "bf16",
                                orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, 3))
    torch.cuda.synchronize()
    after = [host(x) for x in (master, m, v, out)]
    inside = slice(S, 3 * S)
    for k, (b, a) in enumerate(zip(before, after)):
        np.testing.assert_array_equal(a[:S], b[:S])  # rank 0's block untouched
        np.testing.assert_array_equal(a[3 * S:], b[3 * S:])  # rank 3's block untouched
    assert_state_close(after[0][inside], p_o[inside], "master")
    assert_state_close(after[1][inside], m_o[inside], "exp_avg")
    assert_state_close(after[2][inside], v_o[inside], "exp_avg_sq")
    assert_out_close(after[3][inside], shards_o[inside], "bf16", "shard_out")


def test_determinism(F):
    cfg = fi.CONFIGS["gpt2_small"]
    results = []
    for _ in range(2):
        unit = new_unit(F, cfg)
        unit.load_master([fi.gen_master(cfg, device=DEV)])
        for t in (1, 2):
            for r in range(cfg.world):
                unit.load_grad(r, [fi.gen_grad(cfg, r, t, device=DEV)])
            unit.step(hp_for(F, cfg, t))
        torch.cuda.synchronize()
        results.append([x.clone() for x in (unit.master, unit.exp_avg, unit.exp_avg_sq, unit.shard_out)])
    for a, b in zip(*results):
        assert torch.equal(a.view(torch.int8) if a.dtype != torch.float32 else a.view(torch.int32),
                           b.view(torch.int8) if b.dtype != torch.float32 else b.view(torch.int32))


def test_canary_guard_bands(F, orc):
    # every array sits between guard bands of NaN bit patterns; the step and the
    # gather must write inside their arrays only, and the pad must stay zero
    world, P, G = 8, 8 * 1001 - 5, 64
    P_pad = orc.padded_numel(P, world)
    rng = np.random.default_rng(5)
    CAN16, CAN32 = 0x7fc1, 0x7fc00001

    def guarded(n, dt):
        if dt == torch.float32:
            buf = torch.full((n + 2 * G,), CAN32, dtype=torch.int32, device=DEV).view(torch.float32)
        else:
            buf = torch.full((n + 2 * G,), CAN16, dtype=torch.int16, device=DEV).view(dt)
        return buf, buf[G:G + n]

    bufs = {}
    for name, dt in [("master", torch.float32), ("m", torch.float32), ("v", torch.float32),
                     ("out", torch.bfloat16)] + [(f"g{q}", torch.bfloat16) for q in range(world)] + \
                    [(f"f{q}", torch.bfloat16) for q in range(world)]:
        bufs[name] = guarded(P_pad, dt)
    grads = [bufs[f"g{q}"][1] for q in range(world)]
    for q in range(world):
        F.fsdp_flatten_pad([torch.from_numpy((rng.standard_normal(P) * 1e-3).astype(np.float32))
                            .to(torch.bfloat16).to(DEV)], world, out=grads[q])
    F.fsdp_flatten_pad([torch.from_numpy(rng.uniform(-0.1, 0.1, P).astype(np.float32)).to(DEV)], world,
                       out=bufs["master"][1])
    bufs["m"][1].zero_()
    bufs["v"][1].zero_()
    F.fsdp_reduce_scatter_adam_cast(grads, bufs["master"][1], bufs["m"][1], bufs["v"][1], bufs["out"][1],
                                    F.AdamWHParams(1e-3, 0.9, 0.999, 1e-8, 0.01, 1))
    F.fsdp_all_gather(bufs["out"][1], [bufs[f"f{q}"][1] for q in range(world)], world)
    torch.cuda.synchronize()
    for name, (buf, inner) in bufs.items():
        if buf.dtype == torch.float32:
            raw, can = buf.view(torch.int32).cpu().numpy().view(np.uint32), CAN32
        else:
            raw, can = buf.view(torch.int16).cpu().numpy().view(np.uint16), CAN16
        assert (raw[:G] == can).all() and (raw[G + P_pad:] == can).all(), f"guard band of {name} overwritten"
    for name in ("master", "m", "v", "out"):
        assert not host(bufs[name][1])[P:].any(), f"pad of {name} not zero"


def test_nonfinite_counter(F, orc):
    world, P = 2, 1024
    rng = np.random.default_rng(9)
    rows = (rng.standard_normal((world, P)) * 1e-2).astype(np.float32)
    rows[0, 10] = np.inf
    rows[1, 20] = np.nan
    rows[0, 30] = 3e38
    rows[1, 30] = 3e38   # finite inputs whose fp32 sum overflows
    rows[0, 40] = np.inf
    rows[1, 40] = -np.inf
    grads = [torch.from_numpy(r).to(torch.bfloat16).to(DEV) for r in rows]
    g_avg = orc.all_reduce_avg([host(g) for g in grads], "bf16", world, 0.5)
    expect = int(np.count_nonzero(~np.isfinite(g_avg)))
    assert expect == 4
    master = torch.zeros(P, device=DEV)
    m = torch.zeros(P, device=DEV)
    v = torch.zeros(P, device=DEV)
    out = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):
        F.fsdp_reduce_scatter_adam_cast(grads, master, m, v, out, F.AdamWHParams(1e-3), nonfinite_count=cnt)
    assert int(cnt.item()) == 2 * expect


def test_flatten_many_tensors_and_views(F, orc):
    rng = np.random.default_rng(21)
    for dt, fmt in ((torch.float32, "f32"), (torch.bfloat16, "bf16"), (torch.float16, "f16")):
        sizes = [int(s) for s in rng.integers(0, 300, size=70)] + [1, 4099, 0]
        world = 8
        host_parts = [rng.standard_normal(s).astype(np.float32) for s in sizes]
        parts = [torch.from_numpy(h).to(dt).to(DEV) for h in host_parts]
        # unaligned sources: every other tensor starts one element into its allocation
        parts = [torch.cat([torch.zeros(1, dtype=dt, device=DEV), p])[1:] if i % 2 else p
                 for i, p in enumerate(parts)]
        P_pad = orc.padded_numel(sum(sizes), world)
        dst = torch.full((P_pad,), float("nan"), dtype=dt, device=DEV)
        flat, views = F.fsdp_flatten_pad(parts, world, out=dst)
        want = orc.flatten_pad([host(p) for p in parts], world)
        np.testing.assert_array_equal(host(flat), want)
        np.testing.assert_array_equal([v.offset for v in views], orc.view_offsets(sizes))
        assert [v.numel for v in views] == sizes


def test_invalid_calls_enqueue_nothing(F):
    P = 64
    grads = [torch.ones(P, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    master = torch.full((P,), 0.5, device=DEV)
    m = torch.zeros(P, device=DEV)
    v = torch.zeros(P, device=DEV)
    out = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(F.FsdpError):
        F.fsdp_reduce_scatter_adam_cast(grads, master, m, v, out, F.AdamWHParams(1e-3, step=0))
    with pytest.raises(F.FsdpError):
        F.fsdp_reduce_scatter_adam_cast(grads, master, m, v, out, F.AdamWHParams(1e-3), rank_begin=2, rank_end=1)
    with pytest.raises(F.FsdpError):
        F.fsdp_reduce_scatter_adam_cast(grads, master, m, master, out, F.AdamWHParams(1e-3))  # v aliases master
    with pytest.raises(ValueError):
        F.fsdp_reduce_scatter_adam_cast(grads, master, m, v, out[:10], F.AdamWHParams(1e-3))
    torch.cuda.synchronize()
    assert torch.equal(master, torch.full((P,), 0.5, device=DEV))
    assert not m.any() and not v.any() and not out.any()
    assert F.fsdp_last_cuda_error() == 0
    assert F.fsdp_take_wait_timeouts() == 0


def test_a_bounded_wait_that_runs_out_is_counted_and_the_context_stays_usable(F):
    # the failure path of the bulk-copy pipelines' bounded waits, without a
    # fault: a wait on a barrier that nothing completes gives up after ~2^20
    # cycles (about half a millisecond), is counted, and the kernel returns
    assert F.fsdp_take_wait_timeouts() == 0
    s = torch.cuda.Stream()
    # each call's own counter, read in its stream's order: a copy to pinned
    # host memory and a wait on that one stream, no device-wide synchronize
    wt, wt_s = (torch.zeros(1, dtype=torch.int32, device=DEV) for _ in range(2))
    got, got_s = (torch.full((1,), -1, dtype=torch.int32, pin_memory=True) for _ in range(2))
    cur = torch.cuda.current_stream()
    F.fsdp_check_bounded_wait(1 << 20, wait_timeouts=wt)
    got.copy_(wt, non_blocking=True)
    s.wait_stream(cur)  # wt_s was zeroed on the current stream
    F.fsdp_check_bounded_wait(1 << 20, stream=s, wait_timeouts=wt_s)
    with torch.cuda.stream(s):
        got_s.copy_(wt_s, non_blocking=True)
    cur.synchronize()
    assert int(got.item()) == 1
    s.synchronize()
    assert int(got_s.item()) == 1
    # and on the device, over both calls
    assert F.fsdp_take_wait_timeouts() == 2
    assert F.fsdp_take_wait_timeouts() == 0  # the read resets the count
    assert F.fsdp_last_cuda_error() == 0
    # the context still works: a bulk-copy gather right after, with its own
    # counter at 0
    src = (torch.arange(1 << 20, device=DEV) % 251).to(torch.bfloat16)
    fulls = [torch.zeros_like(src) for _ in range(3)]
    wt.zero_()
    F.fsdp_all_gather(src, fulls, 1, wait_timeouts=wt)
    assert int(wt.item()) == 0
    torch.cuda.synchronize()
    assert all(torch.equal(f, src) for f in fulls)
    assert F.fsdp_take_wait_timeouts() == 0


def test_tensors_of_another_device_are_refused(F, monkeypatch):
    # the kernels run on the current device, so a tensor of another GPU is
    # refused by the binding before the library is called; with one GPU the
    # current device is made to read as another ordinal
    P = 64
    grads = [torch.ones(P, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    master = torch.full((P,), 0.5, device=DEV)
    m, v = torch.zeros(P, device=DEV), torch.zeros(P, device=DEV)
    out = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    full = [torch.zeros(P, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    hp = F.AdamWHParams(1e-3)
    calls = [lambda: F.fsdp_reduce_scatter_adam_cast(grads, master, m, v, out, hp),
             lambda: F.fsdp_reduce_scatter_adam_cast_gather(grads, master, m, v, out, full, hp),
             lambda: F.fsdp_reduce_scatter_step(grads, master, m, v, out, F.StepConfig("adamw", 1e-3)),
             lambda: F.fsdp_all_gather(out, full, 2),
             lambda: F.fsdp_flatten_pad([master], 2)]
    other = torch.cuda.current_device() + 1
    monkeypatch.setattr(torch.cuda, "current_device", lambda: other)
    for call in calls:
        with pytest.raises(ValueError, match="current device"):
            call()
    monkeypatch.undo()
    torch.cuda.synchronize()
    assert torch.equal(master, torch.full((P,), 0.5, device=DEV))
    assert not m.any() and not v.any() and not out.any() and not any(f.any() for f in full)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32, torch.float16])
@pytest.mark.parametrize("numel,n_dst", [((1 << 20) + 3, 8), (5 * (1 << 19) + 1, 3), ((1 << 21) + 7, 1),
                                         (3 * (1 << 20), 13), ((1 << 20) + 4096 * 3 + 5, 2)])
def test_all_gather_bulk_copy_path(F, dt, numel, n_dst):
    # >= 1 MB with 16-byte aligned pointers takes the TMA pipeline; the sizes
    # leave a partial last tile and (for odd element counts) a tail below 16 bytes
    world = 1
    src = torch.randn(numel, device=DEV).to(dt)
    fulls = [torch.full((numel,), float("nan"), device=DEV).to(dt) for _ in range(n_dst)]
    F.fsdp_all_gather(src, fulls, world)
    for k, f in enumerate(fulls):
        assert torch.equal(f.view(torch.int16 if dt != torch.float32 else torch.int32),
                           src.view(torch.int16 if dt != torch.float32 else torch.int32)), k
    assert F.fsdp_take_wait_timeouts() == 0


def test_step_from_host_matches_device_steps(F):
    # the pipelined host-buffer step (two gradient-buffer sets, copy streams)
    # must give the same bits as stepping on device-resident gradients
    cfg = fi.CONFIGS["gpt2_small"]
    N = cfg.world
    a, b = new_unit(F, cfg), new_unit(F, cfg)
    master = fi.gen_master(cfg, device=DEV)
    a.load_master([master])
    b.load_master([master])
    T = 5
    host = [[fi.gen_grad(cfg, r, t).pin_memory() for r in range(N)] for t in range(1, T + 1)]
    outs = [torch.empty(a.padded_numel, dtype=a.shard_out.dtype, pin_memory=True) for _ in range(T)]
    for t in range(1, T + 1):
        a.step_from_host(host[t - 1], outs[t - 1], hp_for(F, cfg, t), gathers=2)
    torch.cuda.synchronize()
    for t in range(1, T + 1):
        for r in range(N):
            b.grads[r].copy_(host[t - 1][r])
        b.step(hp_for(F, cfg, t), gathers=2)
        torch.cuda.synchronize()
        assert torch.equal(outs[t - 1].view(torch.int16), b.shard_out.cpu().view(torch.int16)), t
    for x, y in ((a.master, b.master), (a.exp_avg, b.exp_avg), (a.exp_avg_sq, b.exp_avg_sq)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    for f in a.full:
        assert torch.equal(f.view(torch.int16), b.shard_out.view(torch.int16))


def test_step_from_host_full_size_sampled(F, orc):
    # the 70B unit through the end-to-end path the bench times: its 13.7 GB
    # of gradients copied in from pinned host memory every step, the
    # non-finite count and the compute-dtype parameters read back; sampled
    # elements against the oracle
    cfg = fi.CONFIGS["llama70b"]
    N = cfg.world
    unit = new_unit(F, cfg)
    unit.load_master([fi.gen_master(cfg, device=DEV)])
    P_pad = unit.padded_numel
    idx = _sample_indices(P_pad, N, 1 << 19, 11)
    idx_c = torch.from_numpy(idx)
    idx_t = idx_c.to(DEV)
    p_s = host(unit.master[idx_t])
    m_s = np.zeros_like(p_s)
    v_s = np.zeros_like(p_s)
    hgrads = [torch.empty(P_pad, dtype=torch.bfloat16, pin_memory=True) for _ in range(N)]
    hout = torch.empty(P_pad, dtype=torch.bfloat16, pin_memory=True)
    counter = torch.zeros(1, dtype=torch.int32, device=DEV)
    hnf = torch.full((1,), -1, dtype=torch.int32, pin_memory=True)
    for t in range(1, cfg.steps + 1):
        for r in range(N):
            hgrads[r].copy_(fi.gen_grad(cfg, r, t, device=DEV))
        g_s = [host(hgrads[r][idx_c]) for r in range(N)]
        unit.step_from_host(hgrads, hout, hp_for(F, cfg, t), gathers=cfg.gathers, nonfinite_count=counter,
                            host_nonfinite=hnf)
        s = orc.scalars(ohp_for(orc, cfg, t), N)
        orc.adamw(p_s, m_s, v_s, orc.all_reduce_avg(g_s, cfg.grad_dtype, N, s.c), s)
        torch.cuda.synchronize()
        assert int(hnf.item()) == 0
        assert_state_close(host(unit.master[idx_t]), p_s, f"master t={t}")
        assert_state_close(host(unit.exp_avg[idx_t]), m_s, f"exp_avg t={t}")
        assert_state_close(host(unit.exp_avg_sq[idx_t]), v_s, f"exp_avg_sq t={t}")
        out_s = orc.cast_out(p_s, cfg.out_dtype)
        assert_out_close(host(hout[idx_c]), out_s, cfg.out_dtype, f"host_out t={t}")
        assert torch.equal(hout.view(torch.int16), unit.shard_out.cpu().view(torch.int16))
        for f in unit.full:
            assert torch.equal(f, unit.shard_out)
    del unit, hgrads, hout
    torch.cuda.empty_cache()


def test_zero_copy_step_full_size_sampled(F, orc):
    # the bench's other end-to-end form on the 70B unit: the 13.7 GB of
    # gradients stay in pinned host memory and the fused kernel reads them
    # in place through the C ABI (gradients are "device or mapped host"),
    # then the two gathers; the count comes back each step; sampled elements
    # against the oracle
    cfg = fi.CONFIGS["llama70b"]
    N = cfg.world
    unit = new_unit(F, cfg)
    unit.load_master([fi.gen_master(cfg, device=DEV)])
    P_pad = unit.padded_numel
    idx = _sample_indices(P_pad, N, 1 << 19, 17)
    idx_c = torch.from_numpy(idx)
    idx_t = idx_c.to(DEV)
    p_s = host(unit.master[idx_t])
    m_s = np.zeros_like(p_s)
    v_s = np.zeros_like(p_s)
    hgrads = [torch.empty(P_pad, dtype=torch.bfloat16, pin_memory=True) for _ in range(N)]
    counter = torch.zeros(1, dtype=torch.int32, device=DEV)
    hnf = torch.full((1,), -1, dtype=torch.int32, pin_memory=True)
    for t in (1, 2):
        for r in range(N):
            hgrads[r].copy_(fi.gen_grad(cfg, r, t, device=DEV))
        g_s = [host(hgrads[r][idx_c]) for r in range(N)]
        counter.zero_()
        F.fsdp_reduce_scatter_adam_cast(hgrads, unit.master, unit.exp_avg, unit.exp_avg_sq, unit.shard_out,
                                        hp_for(F, cfg, t), nonfinite_count=counter)
        hnf.copy_(counter, non_blocking=True)
        for _ in range(cfg.gathers):
            unit.all_gather()
        s = orc.scalars(ohp_for(orc, cfg, t), N)
        orc.adamw(p_s, m_s, v_s, orc.all_reduce_avg(g_s, cfg.grad_dtype, N, s.c), s)
        torch.cuda.synchronize()
        assert int(hnf.item()) == 0
        assert_state_close(host(unit.master[idx_t]), p_s, f"master t={t}")
        assert_state_close(host(unit.exp_avg[idx_t]), m_s, f"exp_avg t={t}")
        assert_state_close(host(unit.exp_avg_sq[idx_t]), v_s, f"exp_avg_sq t={t}")
        assert_out_close(host(unit.shard_out[idx_t]), orc.cast_out(p_s, cfg.out_dtype), cfg.out_dtype, f"t={t}")
        for f in unit.full:
            assert torch.equal(f, unit.shard_out)
    del unit, hgrads
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ fused all-gather

@pytest.mark.parametrize("name", ["tiny", "gpt2_small", "gpt2_large"])
def test_fused_gather_matches_oracle_and_unfused(F, orc, name):
    cfg = fi.CONFIGS[name]
    N = cfg.world
    a, b = new_unit(F, cfg), new_unit(F, cfg)
    master = fi.gen_master(cfg)
    for u in (a, b):
        u.load_master([master.to(DEV)] if u.padded_numel == u.numel else split_views(u, master.to(DEV)))
    p_o = orc.flatten_pad([master.numpy()], N)
    m_o = np.zeros_like(p_o)
    v_o = np.zeros_like(p_o)
    for t in range(1, 4):
        grads = [fi.gen_grad(cfg, r, t) for r in range(N)]
        for u in (a, b):
            for r in range(N):
                u.load_grad(r, split_views(u, grads[r].to(DEV)))
        a.step(hp_for(F, cfg, t), gathers=cfg.gathers, fuse_gather=True)
        b.step(hp_for(F, cfg, t), gathers=cfg.gathers)
        _, full_o = orc.fsdp_step([orc.flatten_pad([host(g)], N) for g in grads], cfg.grad_dtype, N, p_o, m_o, v_o,
                                  cfg.out_dtype, ohp_for(orc, cfg, t))
        torch.cuda.synchronize()
        assert_state_close(host(a.master), p_o, "master")
        for f in a.full:
            assert_out_close(host(f), full_o, cfg.out_dtype, "full")
        for x, y in zip((a.master, a.exp_avg, a.exp_avg_sq), (b.master, b.exp_avg, b.exp_avg_sq)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
        assert torch.equal(a.shard_out.view(torch.int16), b.shard_out.view(torch.int16))
        for fa, fb in zip(a.full, b.full):
            assert torch.equal(fa.view(torch.int16), fb.view(torch.int16))


@pytest.mark.parametrize("offset", [0, 1])
@pytest.mark.parametrize("world,P,ofmt", [(2, 4099, "bf16"), (3, 1000, "f16"), (8, 8 * 300 + 5, "f32")])
def test_fused_gather_without_shard_and_unaligned(F, orc, offset, world, P, ofmt):
    rng = np.random.default_rng(P + world + offset)
    P_pad = orc.padded_numel(P, world)
    odt = fi.torch_dtype(ofmt)

    def alloc(n, dt):
        return torch.zeros(n + offset, dtype=dt, device=DEV)[offset:]

    rows = (rng.standard_normal((world, P)) * 1e-2).astype(np.float32)
    g_o = [orc.flatten_pad([r], world) for r in rows]
    grads = [alloc(P_pad, torch.float32) for _ in range(world)]
    for g, r in zip(grads, g_o):
        g.copy_(torch.from_numpy(r))
    p0 = orc.flatten_pad([rng.uniform(-0.1, 0.1, P).astype(np.float32)], world)
    master, m, v = (alloc(P_pad, torch.float32) for _ in range(3))
    master.copy_(torch.from_numpy(p0))
    fulls = [alloc(P_pad, odt) for _ in range(world + 1)]
    F.fsdp_reduce_scatter_adam_cast_gather(grads, master, m, v, None, fulls, F.AdamWHParams(1e-3, weight_decay=0.01))
    p_o, m_o, v_o = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    _, full_o = orc.fsdp_step(g_o, "f32", world, p_o, m_o, v_o, ofmt, orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, 1))
    torch.cuda.synchronize()
    assert_state_close(host(master), p_o, "master")
    assert_state_close(host(m), m_o, "exp_avg")
    assert_state_close(host(v), v_o, "exp_avg_sq")
    for f in fulls:
        assert_out_close(host(f), full_o, ofmt, "full")


def test_fused_gather_rank_subrange(F, orc):
    world, P = 4, 4 * 2050
    rng = np.random.default_rng(3)
    grads = [torch.from_numpy((rng.standard_normal(P) * 1e-2).astype(np.float32)).to(torch.bfloat16).to(DEV)
             for _ in range(world)]
    master = torch.from_numpy(rng.uniform(-0.1, 0.1, P).astype(np.float32)).to(DEV)
    m = torch.zeros(P, device=DEV)
    v = torch.zeros(P, device=DEV)
    out = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    fulls = [torch.full((P,), 3.0, dtype=torch.bfloat16, device=DEV) for _ in range(world)]
    ref_master, ref_m, ref_v, ref_out = master.clone(), m.clone(), v.clone(), out.clone()
    hp = F.AdamWHParams(1e-3, weight_decay=0.01)
    F.fsdp_reduce_scatter_adam_cast_gather(grads, master, m, v, out, fulls, hp, rank_begin=1, rank_end=3)
    F.fsdp_reduce_scatter_adam_cast(grads, ref_master, ref_m, ref_v, ref_out, hp, rank_begin=1, rank_end=3)
    torch.cuda.synchronize()
    S = P // world
    assert torch.equal(master, ref_master) and torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    for f in fulls:
        assert torch.equal(f[S:3 * S].view(torch.int16), ref_out[S:3 * S].view(torch.int16))
        assert (f[:S] == 3.0).all() and (f[3 * S:] == 3.0).all()


def test_fused_gather_rejects_bad_arguments(F):
    P = 64
    grads = [torch.ones(P, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    master, m, v = (torch.zeros(P, device=DEV) for _ in range(3))
    out = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    fulls = [torch.zeros(P, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    hp = F.AdamWHParams(1e-3)
    with pytest.raises(ValueError):
        F.fsdp_reduce_scatter_adam_cast_gather(grads, master, m, v, out, [], hp)
    with pytest.raises(F.FsdpError):  # a gathered buffer aliasing shard_out
        F.fsdp_reduce_scatter_adam_cast_gather(grads, master, m, v, out, [fulls[0], out], hp)
    with pytest.raises(F.FsdpError):  # gathered buffers overlapping each other
        F.fsdp_reduce_scatter_adam_cast_gather(grads, master, m, v, None, [fulls[0], fulls[0]], hp)
    torch.cuda.synchronize()
    assert not master.any() and not out.any() and not fulls[0].any()


# ------------------------------------------------------------------ maximum and empty sizes

def test_unit_beyond_2_pow_31_elements(F, orc):
    # P_pad > 2^31: 64-bit indexing in the fused kernel, the bulk-copy gather
    # and flatten; sampled comparison around the 2^31 boundary, the rank
    # block boundary and random elements
    world = 2
    P = (1 << 31) + 24
    grads = [torch.empty(P, dtype=torch.bfloat16, device=DEV) for _ in range(world)]
    for r, g in enumerate(grads):
        gen = torch.Generator(device=DEV)
        gen.manual_seed(40 + r)
        g.copy_(torch.randn(P, generator=gen, device=DEV).mul_(1e-3))
    master = torch.empty(P, device=DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(39)
    src = torch.rand(P, generator=gen, device=DEV).mul_(0.2).sub_(0.1)
    F.fsdp_flatten_pad([src], world, out=master)
    assert torch.equal(master, src)
    del src
    m = torch.zeros(P, device=DEV)
    v = torch.zeros(P, device=DEV)
    out = torch.empty(P, dtype=torch.bfloat16, device=DEV)
    fulls = [torch.empty(P, dtype=torch.bfloat16, device=DEV) for _ in range(world)]
    rng = np.random.default_rng(41)
    S = P // world
    idx = np.unique(np.concatenate([rng.integers(0, P, 1 << 18), np.arange((1 << 31) - 64, P),
                                    np.arange(S - 64, S + 64), np.arange(64)]))
    idx_t = torch.from_numpy(idx).to(DEV)
    p_s = host(master[idx_t])
    g_s = [host(g[idx_t]) for g in grads]
    hp = F.AdamWHParams(1e-3, weight_decay=0.01)
    F.fsdp_reduce_scatter_adam_cast(grads, master, m, v, out, hp)
    F.fsdp_all_gather(out, fulls, world)
    s = orc.scalars(orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, 1), world)
    g_avg = orc.all_reduce_avg(g_s, "bf16", world, s.c)
    m_s = np.zeros_like(p_s)
    v_s = np.zeros_like(p_s)
    orc.adamw(p_s, m_s, v_s, g_avg, s)
    torch.cuda.synchronize()
    assert_state_close(host(master[idx_t]), p_s, "master")
    assert_state_close(host(m[idx_t]), m_s, "exp_avg")
    assert_out_close(host(out[idx_t]), orc.cast_out(p_s, "bf16"), "bf16", "shard_out")
    for f in fulls:
        assert torch.equal(f.view(torch.int16), out.view(torch.int16))
    assert F.fsdp_take_wait_timeouts() == 0
    del grads, master, m, v, out, fulls
    torch.cuda.empty_cache()


def test_maximum_world_64(F, orc):
    _run_flat(F, orc, 64, 64 * 37 + 11, "bf16", "bf16", steps=2, seed=64)
    _run_flat(F, orc, 64, 64 * 1024, "f16", "f16", steps=1, scale=1024.0, seed=65)


def test_empty_unit_is_a_no_op(F):
    e32 = torch.empty(0, device=DEV)
    e16 = torch.empty(0, dtype=torch.bfloat16, device=DEV)
    F.fsdp_reduce_scatter_adam_cast([e16, e16], e32, e32.clone(), e32.clone(), e16.clone(), F.AdamWHParams(1e-3))
    F.fsdp_all_gather(e16, [e16.clone()], 2)
    F.fsdp_reduce_scatter_step([e16, e16], e32, e32.clone(), e32.clone(), e16.clone(), F.StepConfig("adamw", 1e-3))
    flat, views = F.fsdp_flatten_pad([e16], 4)
    assert flat.numel() == 0 and views[0].numel == 0
    views, padded = F.fsdp_unflatten_views([(0,), (3, 0)], 8)
    assert padded == 0
    torch.cuda.synchronize()
    assert F.fsdp_last_cuda_error() == 0


def test_step_from_host_metric_readback(F):
    # the host-buffer step can hand back the step's non-finite count instead of
    # the parameters; planted non-finite gradients show up in it
    cfg = fi.CONFIGS["tiny"]
    N = cfg.world
    unit = new_unit(F, cfg)
    unit.load_master(split_views(unit, fi.gen_master(cfg).to(DEV)))
    counter = torch.zeros(1, dtype=torch.int32, device=DEV)
    results, keep = [], []
    for t in (1, 2, 3):
        host = [fi.gen_grad(cfg, r, t) for r in range(N)]
        padded = [torch.zeros(unit.padded_numel, dtype=host[0].dtype).pin_memory() for _ in range(N)]
        for h, p in zip(host, padded):
            p[:h.numel()].copy_(h)
        if t == 2:
            padded[0][5] = float("inf")
            padded[1][9] = float("nan")
        out = torch.zeros(1, dtype=torch.int32).pin_memory()
        unit.step_from_host(padded, None, hp_for(F, cfg, t), nonfinite_count=counter, host_nonfinite=out)
        results.append(out)
        keep.append(padded)  # host buffers stay alive until the copies are done
    torch.cuda.synchronize()
    assert [int(r.item()) for r in results] == [0, 2, 0]


def test_concurrent_host_threads(F):
    # two host threads step their own units on their own streams at once (the
    # library's launch caches are shared); results equal sequential runs
    import threading
    cfgs = [fi.CONFIGS["gpt2_small"], fi.CONFIGS["gpt2_large"]]

    def make(cfg):
        u = new_unit(F, cfg)
        u.load_master([fi.gen_master(cfg, device=DEV)])
        for r in range(cfg.world):
            u.load_grad(r, [fi.gen_grad(cfg, r, 1, device=DEV)])
        return u

    def run(u, cfg, stream, errors):
        try:
            with torch.cuda.stream(stream):
                for t in range(1, 6):
                    u.step(hp_for(F, cfg, t), gathers=2, stream=stream, fuse_gather=(t % 2 == 0))
            stream.synchronize()
        except Exception as e:  # surfaced below
            errors.append(e)

    seq = [make(c) for c in cfgs]
    for u, c in zip(seq, cfgs):
        run(u, c, torch.cuda.current_stream(), [])
    torch.cuda.synchronize()
    par = [make(c) for c in cfgs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in cfgs]
    errors = []
    threads = [threading.Thread(target=run, args=(u, c, s, errors)) for u, c, s in zip(par, cfgs, streams)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for a, b in zip(seq, par):
        for x, y in ((a.master, b.master), (a.exp_avg, b.exp_avg), (a.exp_avg_sq, b.exp_avg_sq)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
        assert torch.equal(a.shard_out.view(torch.int16), b.shard_out.view(torch.int16))
        for f, g in zip(a.full, b.full):
            assert torch.equal(f.view(torch.int16), g.view(torch.int16))


@pytest.mark.parametrize("ofmt", ["bf16", "f16"])
def test_cast_exhaustive_through_the_kernel(F, orc, ofmt):
    # with lr = 0, weight decay 0 and zero gradients the update leaves every
    # fp32 master value as it is (p*1 - 0*(0/eps)), so the kernel's output is
    # the cast of the master: all 2^32 fp32 bit patterns, in 2^30 chunks,
    # against the oracle's cast (itself pinned on all patterns against torch)
    n = 1 << 30
    odt = fi.torch_dtype(ofmt)
    exp_mask, man_mask = (0x7f80, 0x007f) if ofmt == "bf16" else (0x7c00, 0x03ff)
    grads = [torch.zeros(n, dtype=torch.bfloat16, device=DEV)]
    master = torch.empty(n, dtype=torch.float32, device=DEV)
    m = torch.empty(n, device=DEV)
    v = torch.empty(n, device=DEV)
    out = torch.empty(n, dtype=odt, device=DEV)
    ramp = np.arange(n, dtype=np.uint32)
    hp = F.AdamWHParams(0.0, weight_decay=0.0)
    for chunk in range(4):
        bits = ramp + np.uint32(chunk * n)
        master.copy_(torch.from_numpy(bits.view(np.float32)))
        m.zero_()
        v.zero_()
        F.fsdp_reduce_scatter_adam_cast(grads, master, m, v, out, hp)
        want = orc.cast(bits.view(np.float32), ofmt)
        got = host(out)
        nan_in = ((bits & 0x7f800000) == 0x7f800000) & ((bits & 0x007fffff) != 0)
        nan_out = ((got & exp_mask) == exp_mask) & ((got & man_mask) != 0)
        assert np.array_equal(nan_in, nan_out), chunk
        got[nan_in] = 0
        want[nan_in] = 0
        if not np.array_equal(got, want):
            i = int(np.flatnonzero(got != want)[0])
            raise AssertionError(f"{ofmt}: pattern {hex(int(bits[i]))} -> {hex(int(got[i]))}, oracle {hex(int(want[i]))}")
    del grads, master, m, v, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("gfmt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("lr", [1e-3, 1.0, 3e38])
def test_extreme_values_match_the_oracle(F, orc, gfmt, lr):
    # special master values x special gradients: zeros of both signs,
    # subnormals, the extremes of each format, infinities and NaN, through the
    # divide and square-root slow paths; bit-exact, NaN positions equal
    rng = np.random.default_rng(77)
    f32 = np.float32
    specials_p = np.array([0.0, -0.0, 1e-45, -1e-45, 1e-40, 1.17549435e-38, -1.17549435e-38, 1e-20, 0.1, -0.1,
                           1.0, 65504.0, 3.38953139e38, -3.38953139e38, np.inf, -np.inf, np.nan], f32)
    specials_g = np.array([0.0, -0.0, 1e-45, 5.96e-8, 6.1e-5, 1e-3, -1e-3, 1.0, 3.0e4, 65504.0, -65504.0,
                           3.38953139e38, np.inf, -np.inf, np.nan], f32)
    world = 2
    P = len(specials_p) * len(specials_g)
    p0 = np.repeat(specials_p, len(specials_g)).astype(f32)
    g_all = np.tile(specials_g, len(specials_p)).astype(f32)
    rows = [g_all, (rng.standard_normal(P) * 1e-3).astype(f32)]  # rank 1 adds ordinary noise
    P_pad = orc.padded_numel(P, world)
    tdt = fi.torch_dtype(gfmt)
    grads_t = [torch.from_numpy(orc.flatten_pad([r], world)).to(tdt) for r in rows]
    grads = [g.to(DEV) for g in grads_t]
    master = torch.from_numpy(orc.flatten_pad([p0], world)).to(DEV)
    m = torch.zeros(P_pad, device=DEV)
    v = torch.zeros(P_pad, device=DEV)
    out = torch.empty(P_pad, dtype=torch.bfloat16, device=DEV)
    p_o, m_o, v_o = host(master), np.zeros(P_pad, f32), np.zeros(P_pad, f32)
    for t in (1, 2):
        hp = F.AdamWHParams(lr, 0.9, 0.999, 1e-8, 0.01, t)
        F.fsdp_reduce_scatter_adam_cast(grads, master, m, v, out, hp)
        shards_o, _ = orc.fsdp_step([host(g) for g in grads_t], gfmt, world, p_o, m_o, v_o, "bf16",
                                    orc.hparams(lr, 0.9, 0.999, 1e-8, 0.01, t))
        torch.cuda.synchronize()
        for name, got, want in (("master", host(master), p_o), ("exp_avg", host(m), m_o),
                                ("exp_avg_sq", host(v), v_o)):
            gn, wn = np.isnan(got), np.isnan(want)
            assert np.array_equal(gn, wn), f"{name} NaN positions t={t}"
            np.testing.assert_array_equal(got[~gn].view(np.uint32), want[~wn].view(np.uint32), f"{name} t={t}")
        ob = host(out)
        onan = ((ob & 0x7f80) == 0x7f80) & ((ob & 0x7f) != 0)
        wnan = ((shards_o & 0x7f80) == 0x7f80) & ((shards_o & 0x7f) != 0)
        assert np.array_equal(onan, wnan)
        np.testing.assert_array_equal(ob[~onan], shards_o[~wnan])


# ------------------------------------------------------------------ snapshot / resume

@pytest.mark.parametrize("sharded,host_state", [(False, False), (True, False), (True, True)])
def test_resume_from_snapshot_is_bit_exact(F, sharded, host_state):
    # four steps in one go against two steps, a snapshot (whole, or one file
    # per rank shard), a fresh unit (optionally offloaded) restored from it,
    # and two more steps
    cfg = fi.CONFIGS["gpt2_small"]
    N = cfg.world
    a, b = new_unit(F, cfg), new_unit(F, cfg)
    master = fi.gen_master(cfg, device=DEV)
    a.load_master([master])
    b.load_master([master])

    def step(u, t):
        for r in range(N):
            u.grads[r].copy_(fi.gen_grad(cfg, r, t, device=DEV))
        u.step(hp_for(F, cfg, t), gathers=1)

    for t in (1, 2, 3, 4):
        step(a, t)
    for t in (1, 2):
        step(b, t)
    snap = [b.state_dict(rank=r) for r in range(N)] if sharded else b.state_dict()
    del b
    c = new_unit(F, cfg, state_on_host=host_state)
    if sharded:
        for r in reversed(range(N)):
            c.load_state_dict(snap[r], rank=r)
    else:
        c.load_state_dict(snap)
    for t in (3, 4):
        step(c, t)
    torch.cuda.synchronize()
    for name in ("master", "exp_avg", "exp_avg_sq"):
        assert torch.equal(getattr(a, name).cpu().view(torch.int32), getattr(c, name).cpu().view(torch.int32)), name
    assert torch.equal(a.shard_out.view(torch.int16), c.shard_out.view(torch.int16))
    assert torch.equal(a.full[0].view(torch.int16), c.full[0].view(torch.int16))
