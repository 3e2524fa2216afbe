"""Pins of the oracle's variant paths: SGD with momentum,
Adamax, Adadelta, the reduce-scatter summed in the gradient dtype, and the
low-precision parameter/state step. Each is checked against hand cases,
closed forms, or torch's own implementations (torch.optim, torch's bf16/fp16
tensor arithmetic), never against the oracle itself."""
import os

import numpy as np
import pytest
import torch

from test_oracle_pins import GOLDEN, bf16_bits, f16_bits, floats, read_kv

U = 2.0 ** -24


def f32(x):
    return np.float32(x).item()


def _traj(orc, opt, p0, gs, lr, wd, beta1, beta2, eps):
    """The oracle's fp32 trajectory, one rank (N=1), fp32 gradients."""
    n = p0.size
    p = p0.astype(np.float32).copy()
    s0 = np.zeros(n, np.float32)
    s1 = None if opt == "sgd" else np.zeros(n, np.float32)
    out = []
    for t, g in enumerate(gs, start=1):
        hp = orc.hparams(lr, beta1, beta2, eps, wd, t)
        orc.step_ex(opt, False, [np.ascontiguousarray(g, np.float32)], "f32", 1, p, s0, s1, "f32", "f32", hp)
        out.append((p.copy(), s0.copy(), None if s1 is None else s1.copy()))
    return out


def _torch_traj(opt, p0, gs, lr, wd, beta1, beta2, eps):
    p = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    if opt == "sgd":
        o = torch.optim.SGD([p], lr=lr, momentum=beta1, weight_decay=wd, foreach=False)
    elif opt == "adamax":
        o = torch.optim.Adamax([p], lr=lr, betas=(beta1, beta2), eps=eps, weight_decay=wd, foreach=False)
    elif opt == "adadelta":
        o = torch.optim.Adadelta([p], lr=lr, rho=beta1, eps=eps, weight_decay=wd, foreach=False)
    else:
        o = torch.optim.AdamW([p], lr=lr, betas=(beta1, beta2), eps=eps, weight_decay=wd, foreach=False)
    out = []
    for g in gs:
        p.grad = torch.tensor(g, dtype=torch.float64)
        o.step()
        st = {k: v.clone() for k, v in o.state[p].items() if isinstance(v, torch.Tensor)}
        out.append((p.detach().numpy().copy(), st))
    return out


def test_sgd_momentum_golden(orc):
    kv = read_kv("sgd_momentum_closed_form.txt")
    traj = _traj(orc, "sgd", np.array([float(kv["p0"])]), [np.array([1.0])] * 3, float(kv["lr"]), 0.0,
                 float(kv["momentum"]), 0.0, 0.0)
    np.testing.assert_array_equal([t[1][0] for t in traj], floats(kv["b"]))
    np.testing.assert_array_equal([t[0][0] for t in traj], floats(kv["p"]))


@pytest.mark.parametrize("opt,lr,wd,beta1,beta2,eps", [
    ("sgd", 1e-2, 1e-2, 0.9, 0.0, 0.0),
    ("sgd", 1e-3, 0.0, 0.0, 0.0, 0.0),
    ("adamax", 2e-3, 1e-2, 0.9, 0.999, 1e-8),
    ("adadelta", 1.0, 1e-2, 0.9, 0.0, 1e-6),
])
def test_variant_optimizers_vs_torch(orc, opt, lr, wd, beta1, beta2, eps):
    rng = np.random.default_rng(30)
    n, T = 4000, 8
    p0 = rng.uniform(-0.1, 0.1, n).astype(np.float32)
    gs = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(T)]
    gs[2][:40] = 0.0
    ours = _traj(orc, opt, p0, gs, lr, wd, beta1, beta2, eps)
    ref = _torch_traj(opt, p0.astype(np.float64), [g.astype(np.float64) for g in gs], f32(lr), f32(wd),
                      f32(beta1), f32(beta2), f32(eps))
    # the states' recursions on magnitudes (d = g + wd*p can cancel, so the
    # bounds scale with the size of the terms, not of the result)
    b_abs, u_abs, s_abs, a_abs, m_abs = (np.zeros(n) for _ in range(5))
    a_prev = np.zeros(n)
    for t, ((p, s0, s1), (rp, st)) in enumerate(zip(ours, ref), start=1):
        prev = p0 if t == 1 else ref[t - 2][0]
        d_abs = np.abs(gs[t - 1]) + wd * np.abs(prev)
        b_abs = (0 if t == 1 else beta1) * b_abs + d_abs
        u_abs = np.maximum(beta2 * u_abs, d_abs + eps)
        s_abs = beta1 * s_abs + (1 - beta1) * d_abs ** 2
        m_abs = beta1 * m_abs + (1 - beta1) * d_abs
        if opt == "adadelta":
            delta_abs = np.sqrt(a_prev + eps) / np.sqrt(st["square_avg"].numpy() + eps) * d_abs
            a_abs = beta1 * a_abs + (1 - beta1) * delta_abs ** 2
            a_prev = st["acc_delta"].numpy()
            step_abs = lr * delta_abs
        elif opt == "adamax":
            step_abs = lr / (1 - beta1 ** t) * m_abs / st["exp_inf"].numpy()
        else:
            step_abs = lr * b_abs
        # the parameter within a few fp32 roundings per step of |p| and of the
        # magnitude of the step's terms
        bound = t * 6 * U * np.abs(rp) + t * 16 * U * step_abs
        assert np.all(np.abs(p - rp) <= bound), (opt, t, np.max(np.abs(p - rp) - bound))
        if opt == "sgd" and beta1 > 0:
            assert np.all(np.abs(s0 - st["momentum_buffer"].numpy()) <= t * 8 * U * b_abs + 1e-30), t
        if opt == "adamax":
            assert np.all(np.abs(s1 - st["exp_inf"].numpy()) <= t * 8 * U * u_abs), t
        if opt == "adadelta":
            assert np.all(np.abs(s0 - st["square_avg"].numpy()) <= t * 8 * U * s_abs + 1e-30), t
            assert np.all(np.abs(s1 - st["acc_delta"].numpy()) <= t * 32 * U * a_abs + 1e-30), t


def test_adamax_t1_closed_form(orc):
    # t=1, m0 = u0 = 0: m1 = (1-b1) g, u1 = |g| + eps, p1 = p0 - lr*g/(|g| + eps)
    rng = np.random.default_rng(31)
    n = 2048
    p0 = rng.uniform(-0.1, 0.1, n).astype(np.float32)
    g = (10.0 ** rng.uniform(-10, -1, n) * rng.choice([-1, 1], n)).astype(np.float32)
    (p1, m1, u1), = _traj(orc, "adamax", p0, [g], 1e-3, 0.0, 0.9, 0.999, 1e-8)
    g64 = g.astype(np.float64)
    want = p0 - 1e-3 * g64 / (np.abs(g64) + 1e-8)
    assert np.all(np.abs(p1 - want) <= 4 * U * (np.abs(want) + 1e-3))
    np.testing.assert_allclose(u1, np.abs(g64) + f32(1e-8), rtol=2 * U)


def test_adadelta_t1_closed_form(orc):
    # t=1, s0 = a0 = 0: s1 = (1-rho) g^2; delta = sqrt(eps)/sqrt(s1 + eps) * g;
    # a1 = (1-rho) delta^2; p1 = p0 - lr*delta
    rng = np.random.default_rng(32)
    n = 2048
    p0 = rng.uniform(-0.1, 0.1, n).astype(np.float32)
    g = (rng.standard_normal(n) * 10.0 ** rng.uniform(-6, -1, n)).astype(np.float32)
    rho, eps, lr = f32(0.9), f32(1e-6), 1.0
    (p1, s1, a1), = _traj(orc, "adadelta", p0, [g], lr, 0.0, 0.9, 0.0, 1e-6)
    g64 = g.astype(np.float64)
    sq = (1 - rho) * g64 * g64
    delta = np.sqrt(eps) / np.sqrt(sq + eps) * g64
    np.testing.assert_allclose(s1, sq, rtol=6 * U)
    np.testing.assert_allclose(a1, (1 - rho) * delta * delta, rtol=16 * U)
    assert np.all(np.abs(p1 - (p0 - lr * delta)) <= 8 * U * (np.abs(p0) + np.abs(delta)))


# ------------------------------------------------------------------ reduce-scatter in the gradient dtype

def test_rs_lowp_hand_case_golden(orc):
    kv = read_kv("rs_lowp_hand_case.txt")
    grads = [bf16_bits(np.array([float(kv["G0"]), 0], np.float32)),
             bf16_bits(np.array([float(kv["G1"]), 0], np.float32))]
    assert orc.reduce_scatter_lowp(grads, "bf16", 2, 0, 0.5)[0] == np.float32(kv["bf16_average"])
    assert orc.reduce_scatter(grads, "bf16", 2, 0, 0.5)[0] == np.float32(kv["fp32_average"])


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("world", [2, 3, 8])
def test_rs_lowp_vs_torch_sequential_adds(orc, fmt, world):
    # torch's own bf16/fp16 tensor addition rounds every sum to the dtype
    rng = np.random.default_rng(33 + world)
    P_pad = world * 1001
    rows = (rng.standard_normal((world, P_pad)) * 10.0 ** rng.uniform(-4, 0, (world, P_pad))).astype(np.float32)
    tdt = torch.bfloat16 if fmt == "bf16" else torch.float16
    ts = [torch.from_numpy(r).to(tdt) for r in rows]
    acc = ts[0].clone()
    for q in range(1, world):
        acc = acc + ts[q]
    c = np.float32(1.0 / world)
    want = (acc.to(torch.float32).numpy() * c).astype(np.float32)
    grads = [t.view(torch.int16).numpy().view(np.uint16).copy() for t in ts]
    S = P_pad // world
    for r in range(world):
        np.testing.assert_array_equal(orc.reduce_scatter_lowp(grads, fmt, world, r, c), want[r * S:(r + 1) * S])


# ------------------------------------------------------------------ the general step

def test_step_ex_adamw_equals_fsdp_step(orc):
    rng = np.random.default_rng(34)
    world, P = 4, 4 * 500 + 2
    P_pad = orc.padded_numel(P, world)
    master = orc.flatten_pad([rng.uniform(-0.1, 0.1, P).astype(np.float32)], world)
    a = [master.copy(), np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)]
    b = [master.copy(), np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)]
    for t in (1, 2, 3):
        gr = [orc.flatten_pad([bf16_bits(rng.standard_normal(P).astype(np.float32) * 1e-2)], world)
              for _ in range(world)]
        hp = orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, t)
        sh1, full1 = orc.fsdp_step(gr, "bf16", world, *a, "bf16", hp)
        sh2, full2 = orc.step_ex("adamw", False, gr, "bf16", world, b[0], b[1], b[2], "f32", "bf16", hp)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)
        np.testing.assert_array_equal(full1, full2)


@pytest.mark.parametrize("opt", ["adamw", "sgd", "adamax", "adadelta"])
def test_step_ex_sharded_equals_single_replica(orc, opt):
    # the N-rank step (each rank its own block) equals one replica updated
    # with the all-reduce average, bit for bit (pointwise update)
    rng = np.random.default_rng(35)
    world, P = 3, 3 * 400 + 1
    P_pad = orc.padded_numel(P, world)
    p0 = orc.flatten_pad([rng.uniform(-0.1, 0.1, P).astype(np.float32)], world)
    ns = 1 if opt == "sgd" else 2
    A = [p0.copy()] + [np.zeros(P_pad, np.float32) for _ in range(ns)]
    B = [p0.copy()] + [np.zeros(P_pad, np.float32) for _ in range(ns)]
    for t in (1, 2, 3):
        gr = [orc.flatten_pad([(rng.standard_normal(P) * 1e-2).astype(np.float32)], world) for _ in range(world)]
        hp = orc.hparams(1e-2, 0.9, 0.999, 1e-6, 0.01, t)
        orc.step_ex(opt, False, gr, "f32", world, A[0], A[1], A[2] if ns == 2 else None, "f32", "f32", hp)
        c = orc.scalars(hp, world).c
        g_avg = orc.all_reduce_avg(gr, "f32", world, c)
        orc.step_ex(opt, False, [g_avg], "f32", 1, B[0], B[1], B[2] if ns == 2 else None, "f32", "f32", hp)
        for x, y in zip(A, B):
            np.testing.assert_array_equal(x, y)
        assert not A[0][P:].any()


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_lowp_state_first_step_is_rounded_fp32_step(orc, fmt):
    # from values exact in the low-precision format and m = v = 0, the first
    # low-precision step equals the fp32 step rounded once per stored value
    rng = np.random.default_rng(36)
    world, P = 2, 2 * 700
    to_bits = bf16_bits if fmt == "bf16" else f16_bits
    p_bits = to_bits(rng.uniform(-0.1, 0.1, P).astype(np.float32))
    p32 = orc.widen(p_bits, fmt)
    gr = [to_bits((rng.standard_normal(P) * 1e-3).astype(np.float32)) for _ in range(world)]
    hp = orc.hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, 1)
    P_ = p_bits.copy()
    M_ = np.zeros(P, np.uint16)
    V_ = np.zeros(P, np.uint16)
    orc.step_ex("adamw", False, gr, fmt, world, P_, M_, V_, fmt, fmt, hp)
    p, m, v = p32.copy(), np.zeros(P, np.float32), np.zeros(P, np.float32)
    orc.step_ex("adamw", False, gr, fmt, world, p, m, v, "f32", "f32", hp)
    np.testing.assert_array_equal(P_, to_bits(p))
    np.testing.assert_array_equal(M_, to_bits(m))
    np.testing.assert_array_equal(V_, to_bits(v))


def test_lowp_state_constant_gradient_closed_form(orc):
    # bf16 param and state, constant gradient 1, lr = 2^-6, wd = 0, p0 = 0.5:
    # mhat ~ g and vhat ~ g^2 up to bf16 rounding of m and v (relative error
    # < 2^-6 per step), so each step moves p by 2^-6 (1 +- 2^-5); the exact
    # p_t = 0.5 - t 2^-6 is a bf16 value and the error is below half its ulp
    # (2^-9), so p_t rounds to it exactly
    world = 1
    p = bf16_bits(np.array([0.5, -0.5], np.float32))
    m = np.zeros(2, np.uint16)
    v = np.zeros(2, np.uint16)
    for t in range(1, 6):
        gr = [bf16_bits(np.array([1.0, -1.0], np.float32))]
        orc.step_ex("adamw", False, gr, "bf16", world, p, m, v, "bf16", "bf16",
                    orc.hparams(2.0 ** -6, 0.9, 0.999, 1e-8, 0.0, t))
        np.testing.assert_array_equal(orc.widen(p, "bf16"), np.array([0.5 - t / 64, -0.5 + t / 64], np.float32))
