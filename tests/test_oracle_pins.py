"""Pins of the CPU oracle against facts fixed outside it.

Each test checks the oracle against something other than itself: hand cases
with exact binary values (tests/golden/), brute force on tiny inputs, closed
forms, the identities the source pages state, and independent library routines
(numpy, torch's format conversions, torch.optim.AdamW). Every pin is chosen so
that a plausible slip (a dropped term, a wrong sign or index, a transposed
operand, a wrong rounding rule) fails it.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_kv(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = [s.strip() for s in line.split("=", 1)]
            vals[k] = v
    return vals


def floats(s):
    return np.array([float(x) for x in s.split()], dtype=np.float32)


def bf16_bits(x):
    """fp32 values -> bf16 bits via torch's own conversion (library routine)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def f16_bits(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


# ------------------------------------------------------------------ layout

def test_padded_numel_brute_force(orc):
    # smallest multiple of N that is >= P, found by search
    for world in range(1, 10):
        for numel in range(0, 60):
            expect = next(k for k in range(numel, numel + world + 1) if k % world == 0)
            assert orc.padded_numel(numel, world) == expect
            assert orc.shard_numel(expect, world) == expect // world
    assert orc.padded_numel(-1, 2) == -1
    assert orc.padded_numel(5, 0) == -1
    assert orc.shard_numel(7, 2) == -1


def test_unit_sizes_golden(orc):
    import fsdp_inputs as fi
    with open(os.path.join(GOLDEN, "unit_sizes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 5
    for name, world, P, P_pad, S in rows:
        cfg = fi.CONFIGS[name]
        assert cfg.world == int(world)
        assert fi.unit_numel(cfg) == int(P)
        assert orc.padded_numel(int(P), int(world)) == int(P_pad)
        assert orc.shard_numel(int(P_pad), int(world)) == int(S)


def test_view_offsets_are_prefix_sums(orc):
    rng = np.random.default_rng(1)
    numels = rng.integers(0, 1000, size=37)
    offs = orc.view_offsets(numels)
    np.testing.assert_array_equal(offs, np.concatenate([[0], np.cumsum(numels)[:-1]]))


def test_flatten_pad_matches_concatenate(orc):
    rng = np.random.default_rng(2)
    for world in (1, 2, 3, 8):
        parts = [rng.standard_normal(int(n)).astype(np.float32) for n in rng.integers(1, 50, size=5)]
        flat = orc.flatten_pad(parts, world)
        cat = np.concatenate(parts)
        pad = (-cat.size) % world
        np.testing.assert_array_equal(flat, np.concatenate([cat, np.zeros(pad, np.float32)]))


def test_shard_blocks_brute_force_n2(orc):
    # N=2, P in 1..9: rank r owns [r*S, (r+1)*S); the blocks tile the buffer in rank order
    for P in range(1, 10):
        P_pad = orc.padded_numel(P, 2)
        S = orc.shard_numel(P_pad, 2)
        owned = [list(range(r * S, (r + 1) * S)) for r in range(2)]
        assert owned[0] + owned[1] == list(range(P_pad))
        assert P_pad - P in (0, 1)


# ------------------------------------------------------------------ formats

_LOWS = np.array(sorted({0x0000, 0x0001, 0x0002, 0x0fff, 0x1000, 0x1001, 0x1fff, 0x2000, 0x2001,
                         0x3000, 0x3fff, 0x4000, 0x4001, 0x5000, 0x6000, 0x7000, 0x7fff, 0x8000,
                         0x8001, 0x9000, 0xa000, 0xbfff, 0xc000, 0xc001, 0xe000, 0xf000, 0xfffe,
                         0xffff, 0x0800, 0x17ff, 0x1800, 0x2800, 0x0400, 0x0c00, 0x6001, 0xdfff}),
                 dtype=np.uint32)


def _stratified_bits():
    # every upper 16-bit pattern (sign, exponent, top mantissa bits) combined
    # with every tie / near-tie lower pattern and a few random ones
    rng = np.random.default_rng(3)
    lows = np.concatenate([_LOWS, rng.integers(0, 1 << 16, size=28).astype(np.uint32)])
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    return (hi[:, None] | lows[None, :]).reshape(-1)


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_cast_round_to_nearest_even_vs_torch(orc, fmt):
    bits = _stratified_bits()
    x = bits.view(np.float32)
    got = orc.cast(x, fmt)
    want = bf16_bits(x) if fmt == "bf16" else f16_bits(x)
    nan = np.isnan(x)
    # NaN in, NaN out (payload conventions differ between implementations)
    if fmt == "bf16":
        got_nan = ((got & 0x7f80) == 0x7f80) & ((got & 0x007f) != 0)
    else:
        got_nan = ((got & 0x7c00) == 0x7c00) & ((got & 0x03ff) != 0)
    assert np.array_equal(got_nan, nan)
    bad = np.flatnonzero((got != want) & ~nan)
    assert bad.size == 0, [(hex(int(bits[i])), hex(int(got[i])), hex(int(want[i]))) for i in bad[:8]]


def test_cast_f16_vs_numpy_sample(orc):
    # numpy's own binary16 conversion, on a random sample spanning all exponents
    rng = np.random.default_rng(4)
    bits = rng.integers(0, 1 << 32, size=1 << 18, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(orc.cast(x, "f16"), want)


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_widen_all_patterns(orc, fmt):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = orc.widen(h, fmt)
    tdt = torch.bfloat16 if fmt == "bf16" else torch.float16
    want = torch.from_numpy(h.view(np.int16).copy()).view(tdt).to(torch.float32).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_cast_overflow_and_ties_by_hand(orc):
    # hand cases: largest finite, first overflow, halfway ties
    assert orc.cast(np.array([65504.0], np.float32), "f16")[0] == 0x7bff
    assert orc.cast(np.array([65519.99], np.float32), "f16")[0] == 0x7bff
    assert orc.cast(np.array([65520.0], np.float32), "f16")[0] == 0x7c00  # tie -> even = inf
    assert orc.cast(np.array([2.0 ** -25], np.float32), "f16")[0] == 0x0000  # tie -> even = 0
    assert orc.cast(np.array([2.0 ** -25 * 1.5], np.float32), "f16")[0] == 0x0001
    # bf16: 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> 1; 1 + 3*2^-8 -> 1 + 2^-6
    assert orc.cast(np.array([1 + 2.0 ** -8], np.float32), "bf16")[0] == 0x3f80
    assert orc.cast(np.array([1 + 3 * 2.0 ** -8], np.float32), "bf16")[0] == 0x3f82
    assert orc.cast(np.array([np.float32(3.4028235e38)], np.float32), "bf16")[0] == 0x7f80


# ------------------------------------------------------------------ reduce-scatter

def _grads_bf16(rows):
    return [bf16_bits(np.asarray(r, np.float32)) for r in rows]


def test_rs_hand_case_golden(orc):
    kv = read_kv("rs_hand_case.txt")
    world = int(kv["world"])
    grads = _grads_bf16([floats(kv["G0"]), floats(kv["G1"])])
    c = orc.scalars(orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1), world).c
    assert c == 0.5
    np.testing.assert_array_equal(orc.reduce_scatter(grads, "bf16", world, 0, c), floats(kv["rank0"]))
    np.testing.assert_array_equal(orc.reduce_scatter(grads, "bf16", world, 1, c), floats(kv["rank1"]))


def test_rs_fixed_rank_order_golden(orc):
    kv = read_kv("rs_order_case.txt")
    world = int(kv["world"])
    vals = floats(kv["G"])
    grads = [bf16_bits(np.array([vals[q], 0, 0, 0], np.float32)) for q in range(world)]
    c = orc.scalars(orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1), world).c
    g = orc.reduce_scatter(grads, "bf16", world, 0, c)
    assert g[0] == np.float32(kv["average"])
    assert g[0] != np.float32(kv["reverse_order_average"])


def test_rs_exact_on_integers_vs_numpy(orc):
    # small integers are exact in bf16 and their fp32 sums are exact, so the
    # fp32 average must equal numpy's fp64 mean exactly (N a power of two)
    rng = np.random.default_rng(5)
    for world in (2, 4, 8):
        P = 1000 * world
        rows = rng.integers(-100, 100, size=(world, P)).astype(np.float32)
        grads = _grads_bf16(rows)
        c = orc.scalars(orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1), world).c
        want = rows.astype(np.float64).sum(0) / world
        S = P // world
        for r in range(world):
            np.testing.assert_array_equal(orc.reduce_scatter(grads, "bf16", world, r, c),
                                          want[r * S:(r + 1) * S].astype(np.float32))


@pytest.mark.parametrize("world,fmt,scale", [(2, "bf16", 1.0), (3, "bf16", 1.0), (8, "bf16", 1.0),
                                             (2, "f16", 1024.0), (8, "f32", 1.0)])
def test_rs_within_fp32_bound_of_numpy(orc, world, fmt, scale):
    rng = np.random.default_rng(6 + world)
    P_pad = world * 777
    rows = (rng.standard_normal((world, P_pad)) * 1e-3 * scale).astype(np.float32)
    if fmt == "bf16":
        grads = _grads_bf16(rows)
        wide = np.stack([orc.widen(g, "bf16") for g in grads]).astype(np.float64)
    elif fmt == "f16":
        grads = [f16_bits(r) for r in rows]
        wide = np.stack([np.asarray(g).view(np.float16).astype(np.float64) for g in grads])
    else:
        grads = [r.copy() for r in rows]
        wide = rows.astype(np.float64)
    c = orc.scalars(orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, scale), world).c
    exact = wide.sum(0) / (world * scale)
    u = 2.0 ** -24
    bound = (world * u) * np.abs(wide).sum(0) / (world * scale) + u * np.abs(exact) + 1e-45
    S = P_pad // world
    for r in range(world):
        got = orc.reduce_scatter(grads, fmt, world, r, c).astype(np.float64)
        sl = slice(r * S, (r + 1) * S)
        assert np.all(np.abs(got - exact[sl]) <= bound[sl])


@pytest.mark.parametrize("world", [2, 3, 8])
def test_rs_then_ag_equals_allreduce(orc, world):
    # "the all-reduce ... can be decomposed into reduce-scatter and all-gather"
    rng = np.random.default_rng(7)
    P_pad = orc.padded_numel(1001, world)
    grads = _grads_bf16(rng.standard_normal((world, P_pad)).astype(np.float32) * 1e-2)
    c = orc.scalars(orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1), world).c
    shards = [orc.reduce_scatter(grads, "bf16", world, r, c) for r in range(world)]
    np.testing.assert_array_equal(orc.all_gather(shards, world), orc.all_reduce_avg(grads, "bf16", world, c))


def test_all_gather_is_rank_ordered_concatenation(orc):
    rng = np.random.default_rng(8)
    for world in (1, 2, 5):
        shards = [rng.integers(0, 1 << 16, size=13).astype(np.uint16) for _ in range(world)]
        np.testing.assert_array_equal(orc.all_gather(shards, world), np.concatenate(shards))


# ------------------------------------------------------------------ AdamW

def test_scalars_by_hand(orc):
    s = orc.scalars(orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, 1), 8)
    assert s.c == 0.125
    assert s.decay == np.float32(1 - 1e-3 * 0.01)
    assert s.alpha == np.float32(np.float64(np.float32(1e-3)) / (1 - np.float64(np.float32(0.9))))
    assert s.b2s == np.float32(math.sqrt(1 - np.float64(np.float32(0.999))))
    s2 = orc.scalars(orc.hparams(1e-4, 0.9, 0.999, 1e-8, 0.01, 3, 1024.0), 2)
    assert s2.c == 2.0 ** -11
    with pytest.raises(ValueError):
        orc.scalars(orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 0), 2)


def _adam_steps(orc, p0, gs, lr, wd, beta1=0.9, beta2=0.999, eps=1e-8):
    p = np.array(p0, np.float32).copy()
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    out = []
    for t, g in enumerate(gs, start=1):
        s = orc.scalars(orc.hparams(lr, beta1, beta2, eps, wd, t), 1)
        orc.adamw(p, m, v, np.asarray(g, np.float32), s)
        out.append((p.copy(), m.copy(), v.copy()))
    return out


def test_adamw_constant_gradient_golden(orc):
    kv = read_kv("adamw_closed_form.txt")
    lr, wd = float(kv["lr"]), float(kv["weight_decay"])
    p0 = float(kv["p0"])
    traj = _adam_steps(orc, [p0, p0], [np.array([1.0, -1.0])] * 2, lr, wd,
                       float(kv["beta1"]), float(kv["beta2"]), float(kv["eps"]))
    assert traj[0][0][0] == np.float32(kv["plus_p1"])
    assert traj[1][0][0] == np.float32(kv["plus_p2"])
    assert traj[0][0][1] == np.float32(kv["minus_p1"])
    assert traj[1][0][1] == np.float32(kv["minus_p2"])


def test_adamw_t1_closed_form(orc):
    # at t=1 with m0 = v0 = 0: m1 = (1-b1) g, v1 = (1-b2) g^2, mhat = g, vhat = g^2,
    # so p1 = p0 (1 - lr wd) - lr g / (|g| + eps); the g values span eps
    rng = np.random.default_rng(9)
    n = 4096
    p0 = rng.uniform(-0.1, 0.1, n).astype(np.float32)
    mag = 10.0 ** rng.uniform(-10, -1, n)
    g = (mag * rng.choice([-1, 1], n)).astype(np.float32)
    lr, wd, eps = 1e-3, 0.01, 1e-8
    (p1, m1, v1), = _adam_steps(orc, p0, [g], lr, wd, eps=eps)
    g64 = g.astype(np.float64)
    want = p0.astype(np.float64) * (1 - lr * wd) - lr * g64 / (np.abs(g64) + eps)
    u = 2.0 ** -24
    assert np.all(np.abs(p1 - want) <= 4 * u * (np.abs(want) + lr))
    # the hyperparameters are fp32 values: 1 - b1 is taken from fp32(0.9)
    omb1 = 1 - np.float64(np.float32(0.9))
    omb2 = 1 - np.float64(np.float32(0.999))
    np.testing.assert_allclose(m1, omb1 * g64, rtol=2 * u, atol=0)
    np.testing.assert_allclose(v1, omb2 * g64 * g64, rtol=4 * u, atol=0)


def test_adamw_zero_gradient_is_pure_decay(orc):
    p0 = np.array([0.5, -0.03125, 0.0, 1e-3], np.float32)
    traj = _adam_steps(orc, p0, [np.zeros(4)] * 3, 1e-3, 0.1)
    decay = np.float32(1 - 1e-3 * 0.1)
    p = p0.copy()
    for (pt, mt, vt) in traj:
        p = (p * decay).astype(np.float32)
        np.testing.assert_array_equal(pt, p)
        assert not mt.any() and not vt.any()


def test_adamw_pad_stays_zero(orc):
    traj = _adam_steps(orc, np.zeros(8), [np.zeros(8)] * 5, 1e-3, 0.1)
    for pt, mt, vt in traj:
        assert not pt.any() and not mt.any() and not vt.any()
        assert not np.signbit(pt).any()


def _torch_adamw_trajectory(p0, gs, lr, wd, beta1, beta2, eps):
    p = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    opt = torch.optim.AdamW([p], lr=lr, betas=(beta1, beta2), eps=eps, weight_decay=wd,
                            foreach=False, fused=False)
    st = []
    for g in gs:
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        state = opt.state[p]
        st.append((p.detach().numpy().copy(), state["exp_avg"].numpy().copy(),
                   state["exp_avg_sq"].numpy().copy()))
    return st


@pytest.mark.parametrize("lr,wd,sigma", [(1e-3, 0.01, 1e-2), (1e-4, 0.1, 1e-4), (3e-5, 0.1, 1e-4)])
def test_adamw_vs_torch_optim_trajectory(orc, lr, wd, sigma):
    # torch.optim.AdamW in fp64 (an independent library implementation of the
    # same update) against the oracle's fp32 trajectory, within a bound derived
    # from fp32 rounding; the gradients are the same fp32 values for both.
    rng = np.random.default_rng(10)
    n, T = 5000, 10
    beta1, beta2, eps = 0.9, 0.999, 1e-8
    p0 = rng.uniform(-0.1, 0.1, n).astype(np.float32)
    gs = [(rng.standard_normal(n) * sigma).astype(np.float32) for _ in range(T)]
    gs[3][:50] = 0.0
    ours = _adam_steps(orc, p0, gs, lr, wd, beta1, beta2, eps)
    ref = _torch_adamw_trajectory(p0.astype(np.float64), [g.astype(np.float64) for g in gs],
                                  np.float32(lr).item(), np.float32(wd).item(),
                                  np.float32(beta1).item(), np.float32(beta2).item(),
                                  np.float32(eps).item())
    u = 2.0 ** -24
    m_abs = np.zeros(n)
    for t, ((p, m, v), (rp, rm, rv)) in enumerate(zip(ours, ref), start=1):
        m_abs = 0.9 * m_abs + 0.1 * np.abs(gs[t - 1].astype(np.float64))
        # p: <= ~2 ulp of p per step plus the update's relative error
        assert np.all(np.abs(p - rp) <= t * 4 * u * (np.abs(rp) + lr)), t
        # m: error relative to the magnitude of its terms (cancellation-safe)
        assert np.all(np.abs(m - rm) <= t * 4 * u * m_abs + 1e-45), t
        # v: sum of nonnegative terms; (1-b2) is rounded once from fp32 0.999
        assert np.all(np.abs(v - rv) <= (t * 4 * u + 2e-6) * rv + 1e-45), t


def test_adamw_f64_shadow_matches_torch(orc):
    rng = np.random.default_rng(11)
    n, T = 3000, 6
    lr, wd = 1e-3, 0.01
    p = rng.uniform(-0.1, 0.1, n)
    m = np.zeros(n)
    v = np.zeros(n)
    gs = [rng.standard_normal(n) * 1e-3 for _ in range(T)]
    f = lambda x: np.float32(x).item()  # the oracle's hyperparameters are fp32 values
    ref = _torch_adamw_trajectory(p.copy(), gs, f(lr), f(wd), f(0.9), f(0.999), f(1e-8))
    for t, g in enumerate(gs, start=1):
        orc.adamw_f64(p, m, v, np.ascontiguousarray(g), orc.hparams(lr, 0.9, 0.999, 1e-8, wd, t))
        rp, rm, rv = ref[t - 1]
        np.testing.assert_allclose(m, rm, rtol=1e-12, atol=1e-20)
        np.testing.assert_allclose(v, rv, rtol=1e-12, atol=1e-25)
        np.testing.assert_allclose(p, rp, rtol=1e-12, atol=1e-15)


def test_adamw_is_pointwise(orc):
    # the optimizer is pointwise, so updating a shard alone equals the same
    # elements of the full update, bit for bit
    rng = np.random.default_rng(12)
    n = 1000
    p = rng.uniform(-0.1, 0.1, n).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = (rng.random(n) * 1e-6).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    s = orc.scalars(orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, 4), 1)
    full = [a.copy() for a in (p, m, v)]
    orc.adamw(*full, g, s)
    for lo, hi in ((0, 250), (250, 251), (251, 1000)):
        part = [a[lo:hi].copy() for a in (p, m, v)]
        orc.adamw(*part, np.ascontiguousarray(g[lo:hi]), s)
        for a, b in zip(part, full):
            np.testing.assert_array_equal(a, b[lo:hi])


# ------------------------------------------------------------------ whole step

@pytest.mark.parametrize("world,P,gfmt,ofmt,scale", [
    (2, 4099, "bf16", "bf16", 1.0), (3, 1000, "bf16", "bf16", 1.0), (8, 8 * 257 + 3, "bf16", "bf16", 1.0),
    (2, 2001, "f16", "f16", 1024.0), (4, 999, "f32", "f32", 1.0)])
def test_sharded_step_equals_ddp_step(orc, world, P, gfmt, ofmt, scale):
    # "FSDP produces results identical to standard DDP training": the sharded
    # step (reduce-scatter, shard AdamW, cast, all-gather) must equal the
    # full-replica all-reduce + AdamW + cast, bit for bit, over several steps
    rng = np.random.default_rng(13)
    P_pad = orc.padded_numel(P, world)
    master = orc.flatten_pad([rng.uniform(-0.1, 0.1, P).astype(np.float32)], world)
    a = [master.copy(), np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)]
    b = [master.copy(), np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)]
    for t in range(1, 4):
        rows = (rng.standard_normal((world, P)) * 1e-2 * scale).astype(np.float32)
        if gfmt == "bf16":
            gr = [orc.flatten_pad([bf16_bits(r)], world) for r in rows]
        elif gfmt == "f16":
            gr = [orc.flatten_pad([f16_bits(r)], world) for r in rows]
        else:
            gr = [orc.flatten_pad([r], world) for r in rows]
        hp = orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, t, scale)
        shards, full = orc.fsdp_step(gr, gfmt, world, *a, ofmt, hp)
        ddp_full = orc.ddp_step(gr, gfmt, world, *b, ofmt, hp)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)
        np.testing.assert_array_equal(full, ddp_full)
        np.testing.assert_array_equal(shards, full)
        # the pad stays exactly zero
        for x in a:
            assert not x[P:].any()
        assert not full[P:].any()


def test_tiny_trajectory_within_fp64_shadow(orc):
    # the fp32 step against the same definitions in fp64 (rounding bound only)
    import fsdp_inputs as fi
    cfg = fi.CONFIGS["tiny"]
    N = cfg.world
    P = fi.unit_numel(cfg)
    P_pad = orc.padded_numel(P, N)
    master = orc.flatten_pad([fi.gen_master(cfg).numpy()], N)
    p32, m32, v32 = master.copy(), np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)
    p64, m64, v64 = master.astype(np.float64), np.zeros(P_pad), np.zeros(P_pad)
    u = 2.0 ** -24
    for t in range(1, cfg.steps + 1):
        gr = [orc.flatten_pad([fi.gen_grad(cfg, r, t).view(torch.int16).numpy().view(np.uint16)], N)
              for r in range(N)]
        hp = orc.hparams(cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, t, cfg.grad_scale)
        orc.fsdp_step(gr, cfg.grad_dtype, N, p32, m32, v32, cfg.out_dtype, hp)
        g64 = orc.all_reduce_avg_f64(gr, cfg.grad_dtype, N, cfg.grad_scale)
        orc.adamw_f64(p64, m64, v64, g64, hp)
        assert np.all(np.abs(p32 - p64) <= t * 4 * u * (np.abs(p64) + cfg.lr))
        assert np.all(np.abs(v32 - v64) <= (t * 6 * u + 2e-6) * v64 + 1e-45)



def test_loss_scaled_fp16_trajectory_within_fp64_shadow(orc):
    # GPT-2 Large's form ("static loss scale 1024 to unscale in-kernel", N = 2,
    # fp16 gradients that carry the scale, reading R10): the fp32 step
    # multiplies by c = fp32(1/(N*1024)), the fp64 shadow divides by N*1024 in
    # double. Adam's update is almost blind to a gradient's scale, so the
    # moments and the averaged gradient are checked too: a shadow that kept
    # the scale would have m 1024x and v 1024^2 x the fp32 ones.
    import fsdp_inputs as fi
    cfg = fi.CONFIGS["gpt2_large"]
    assert cfg.grad_dtype == "f16" and cfg.grad_scale == 1024.0 and cfg.world == 2
    N, n = cfg.world, 1 << 16
    P_pad = orc.padded_numel(n, N)
    master = orc.flatten_pad([fi.gen_master(cfg, numel=n).numpy()], N)
    p32, m32, v32 = master.copy(), np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)
    p64, m64, v64 = master.astype(np.float64), np.zeros(P_pad), np.zeros(P_pad)
    mag = np.zeros(P_pad)  # the same recursion as m on |g|: the size of its terms, for a cancellation-safe bound
    u = 2.0 ** -24
    for t in range(1, 5):
        gr = [orc.flatten_pad([fi.gen_grad(cfg, r, t, numel=n).view(torch.int16).numpy().view(np.uint16)], N)
              for r in range(N)]
        hp = orc.hparams(cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, t, cfg.grad_scale)
        orc.fsdp_step(gr, cfg.grad_dtype, N, p32, m32, v32, cfg.out_dtype, hp)
        g64 = orc.all_reduce_avg_f64(gr, cfg.grad_dtype, N, cfg.grad_scale)
        # the average of N unscaled N(0, 1e-3) draws: standard deviation 1e-3 / sqrt(N)
        assert 0.9e-3 / np.sqrt(N) < np.std(g64) < 1.1e-3 / np.sqrt(N)
        orc.adamw_f64(p64, m64, v64, g64, hp)
        mag = cfg.beta1 * mag + (1 - cfg.beta1) * np.abs(g64)
        assert np.all(np.abs(p32 - p64) <= t * 4 * u * (np.abs(p64) + cfg.lr))
        assert np.all(np.abs(m32 - m64) <= t * 4 * u * mag)
        assert np.all(np.abs(v32 - v64) <= (t * 6 * u + 2e-6) * v64 + 1e-45)
