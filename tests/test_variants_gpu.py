"""Parity of the variant steps (fsdp_reduce_scatter_step, through the C ABI)
with the oracle's general step: SGD with momentum, Adamax, Adadelta and AdamW;
fp32 or gradient-dtype reduce-scatter; fp32 master + fp32 state, or bf16/fp16
parameter and state. Bars: fp32 values within 1e-6 relative, bf16/fp16 values
within 1 ulp (the kernel performs the oracle's operations in its order, so the
results are expected to be identical, which test_variants_bit_exact checks).
"""
import numpy as np
import pytest
import torch

import fsdp_inputs as fi
from gpu_util import assert_out_close, assert_state_close, host

pytestmark = pytest.mark.gpu
DEV = "cuda"

HP = {  # lr, beta1, beta2, eps, weight_decay
    "adamw": (1e-3, 0.9, 0.999, 1e-8, 0.01),
    "sgd": (1e-2, 0.9, 0.0, 0.0, 1e-2),
    "adamax": (2e-3, 0.9, 0.999, 1e-8, 1e-2),
    "adadelta": (1.0, 0.9, 0.0, 1e-6, 1e-2),
}


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sharded_fsdp_reduce_gb300 as F
    return F


def _bits(x, fmt):
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(fi.torch_dtype(fmt))
    return t


def _compare(got, want, fmt, what):
    if fmt == "f32":
        assert_state_close(got, want, what)
    else:
        assert_out_close(got, want, fmt, what)


def run_variant(F, orc, opt, lowp_reduce, sfmt, ofmt, world, P, gfmt, steps=3, offset=0, scale=1.0, seed=0,
                exact=False):
    rng = np.random.default_rng(seed)
    P_pad = orc.padded_numel(P, world)
    gdt, sdt = fi.torch_dtype(gfmt), fi.torch_dtype(sfmt)
    lr, b1, b2, eps, wd = HP[opt]
    ns = 1 if opt == "sgd" else 2

    def alloc(n, dt):
        return torch.zeros(n + offset, dtype=dt, device=DEV)[offset:]

    grads = [alloc(P_pad, gdt) for _ in range(world)]
    param = alloc(P_pad, sdt)
    states = [alloc(P_pad, sdt) for _ in range(ns)]
    out = alloc(P_pad, fi.torch_dtype(ofmt)) if sfmt == "f32" else None
    p0 = _bits(orc.flatten_pad([rng.uniform(-0.1, 0.1, P).astype(np.float32)], world), sfmt)
    param.copy_(p0.to(DEV))
    p_o = host(p0)
    s_o = [np.zeros(P_pad, orc.np_storage(sfmt)) for _ in range(ns)]
    for t in range(1, steps + 1):
        rows = [_bits(orc.flatten_pad([(rng.standard_normal(P) * 1e-2 * scale).astype(np.float32)], world), gfmt)
                for _ in range(world)]
        for g, r in zip(grads, rows):
            g.copy_(r.to(DEV))
        cfg = F.StepConfig(opt, lr, b1, b2, eps, wd, t, scale, reduce_dtype=gdt if lowp_reduce else None)
        F.fsdp_reduce_scatter_step(grads, param, states[0], states[1] if ns == 2 else None, out, cfg)
        shards_o, _ = orc.step_ex(opt, lowp_reduce, [host(r) for r in rows], gfmt, world, p_o, s_o[0],
                                  s_o[1] if ns == 2 else None, sfmt, ofmt if sfmt == "f32" else sfmt,
                                  orc.hparams(lr, b1, b2, eps, wd, t, scale))
        torch.cuda.synchronize()
        if exact:
            np.testing.assert_array_equal(host(param).view(np.uint8), p_o.view(np.uint8))
            for k in range(ns):
                np.testing.assert_array_equal(host(states[k]).view(np.uint8), s_o[k].view(np.uint8))
            if out is not None:
                np.testing.assert_array_equal(host(out).view(np.uint8), shards_o.view(np.uint8))
            continue
        _compare(host(param), p_o, sfmt, f"{opt} param t={t}")
        for k in range(ns):
            _compare(host(states[k]), s_o[k], sfmt, f"{opt} state{k} t={t}")
        if out is not None:
            _compare(host(out), shards_o, ofmt, f"{opt} shard_out t={t}")
        assert not host(param)[P:].any()  # the pad stays zero


@pytest.mark.parametrize("opt", ["adamw", "sgd", "adamax", "adadelta"])
@pytest.mark.parametrize("lowp_reduce", [False, True])
@pytest.mark.parametrize("sfmt,ofmt", [("f32", "bf16"), ("bf16", "bf16"), ("f16", "f16")])
@pytest.mark.parametrize("world,P,gfmt", [(8, 8 * 1000 + 3, "bf16"), (2, 4099, "f16"), (3, 1001, "f32")])
def test_variant_step_matches_oracle(F, orc, opt, lowp_reduce, sfmt, ofmt, world, P, gfmt):
    run_variant(F, orc, opt, lowp_reduce, sfmt, ofmt, world, P, gfmt, seed=world + P)


@pytest.mark.parametrize("opt", ["adamw", "sgd", "adamax", "adadelta"])
def test_variants_bit_exact(F, orc, opt):
    run_variant(F, orc, opt, False, "f32", "bf16", 8, 8 * 4096, "bf16", steps=3, seed=1, exact=True)
    run_variant(F, orc, opt, True, "bf16", "bf16", 8, 8 * 4096, "bf16", steps=3, seed=2, exact=True)


@pytest.mark.parametrize("opt", ["adamw", "sgd"])
def test_variant_unaligned_and_fp16_scale(F, orc, opt):
    run_variant(F, orc, opt, False, "f32", "f16", 2, 2 * 777 + 1, "f16", offset=1, scale=1024.0, seed=5)
    run_variant(F, orc, opt, True, "f16", "f16", 4, 4 * 333, "f16", offset=1, scale=1024.0, seed=6)


def test_variant_step_adamw_equals_main_kernel(F):
    # the variant path with AdamW, fp32 reduction and fp32 state is the main path
    cfg = fi.CONFIGS["gpt2_small"]
    N = cfg.world
    grads = [fi.gen_grad(cfg, r, 1, device=DEV) for r in range(N)]
    master = fi.gen_master(cfg, device=DEV)
    a = [master.clone(), torch.zeros_like(master), torch.zeros_like(master)]
    b = [master.clone(), torch.zeros_like(master), torch.zeros_like(master)]
    oa = torch.empty(master.numel(), dtype=torch.bfloat16, device=DEV)
    ob = torch.empty_like(oa)
    for t in (1, 2):
        F.fsdp_reduce_scatter_adam_cast(grads, *a, oa, F.AdamWHParams(cfg.lr, weight_decay=cfg.weight_decay, step=t))
        F.fsdp_reduce_scatter_step(grads, b[0], b[1], b[2], ob,
                                   F.StepConfig("adamw", cfg.lr, weight_decay=cfg.weight_decay, step=t))
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))


def test_variant_full_size_sampled_bf16_state(F, orc):
    # the 70B unit at full size: pure-bf16 AdamW with a bf16 reduce-scatter,
    # compared on sampled elements (the step is pointwise)
    cfg = fi.CONFIGS["llama70b"]
    N = cfg.world
    P = fi.unit_numel(cfg)
    grads = [torch.empty(P, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    param = fi.gen_master(cfg, device=DEV).to(torch.bfloat16)
    s0 = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    s1 = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    rng = np.random.default_rng(8)
    idx = np.unique(np.concatenate([rng.integers(0, P, 1 << 19), np.arange(P - 64, P), np.arange(64)]))
    idx = idx[: len(idx) // N * N]
    idx_t = torch.from_numpy(idx).to(DEV)
    p_s = host(param[idx_t])
    m_s = np.zeros(len(idx), np.uint16)
    v_s = np.zeros(len(idx), np.uint16)
    for t in (1, 2, 3):
        for r in range(N):
            grads[r].copy_(fi.gen_grad(cfg, r, t, device=DEV))
        g_s = [host(grads[r][idx_t]) for r in range(N)]
        sc = F.StepConfig("adamw", cfg.lr, weight_decay=cfg.weight_decay, step=t, reduce_dtype=torch.bfloat16)
        F.fsdp_reduce_scatter_step(grads, param, s0, s1, None, sc)
        orc.step_ex("adamw", True, g_s, "bf16", N, p_s, m_s, v_s, "bf16", "bf16",
                    orc.hparams(cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, t))
        torch.cuda.synchronize()
        assert_out_close(host(param[idx_t]), p_s, "bf16", f"param t={t}")
        assert_out_close(host(s0[idx_t]), m_s, "bf16", f"exp_avg t={t}")
        assert_out_close(host(s1[idx_t]), v_s, "bf16", f"exp_avg_sq t={t}")
    del grads, param, s0, s1
    torch.cuda.empty_cache()


@pytest.mark.parametrize("opt,lowp", [("adamw", True), ("sgd", False), ("adamax", False), ("adadelta", False)])
def test_variant_full_size_sampled_fp32_state(F, orc, opt, lowp):
    # the 70B unit at full size with fp32 parameter and state, each variant
    # as the bench times it (AdamW with the bf16 reduce-scatter, SGD with
    # momentum, Adamax, Adadelta at lr 1), compared on sampled elements
    cfg = fi.CONFIGS["llama70b"]
    N = cfg.world
    P = fi.unit_numel(cfg)
    grads = [torch.empty(P, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    param = fi.gen_master(cfg, device=DEV)
    s0 = torch.zeros(P, device=DEV)
    s1 = None if opt == "sgd" else torch.zeros(P, device=DEV)
    out = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    rng = np.random.default_rng(9)
    idx = np.unique(np.concatenate([rng.integers(0, P, 1 << 19), np.arange(P - 64, P), np.arange(64)]))
    idx = idx[: len(idx) // N * N]
    idx_t = torch.from_numpy(idx).to(DEV)
    p_s = host(param[idx_t]).copy()
    s_s = [np.zeros(len(idx), np.float32) for _ in range(1 if s1 is None else 2)]
    lr = 1.0 if opt == "adadelta" else cfg.lr
    for t in (1, 2, 3):
        for r in range(N):
            grads[r].copy_(fi.gen_grad(cfg, r, t, device=DEV))
        g_s = [host(grads[r][idx_t]) for r in range(N)]
        sc = F.StepConfig(opt, lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, t,
                          reduce_dtype=torch.bfloat16 if lowp else None)
        F.fsdp_reduce_scatter_step(grads, param, s0, s1, out, sc)
        out_s, _ = orc.step_ex(opt, lowp, g_s, "bf16", N, p_s, s_s[0], s_s[1] if s1 is not None else None, "f32",
                               "bf16", orc.hparams(lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, t))
        torch.cuda.synchronize()
        assert_state_close(host(param[idx_t]), p_s, f"{opt} param t={t}")
        assert_state_close(host(s0[idx_t]), s_s[0], f"{opt} state0 t={t}")
        if s1 is not None:
            assert_state_close(host(s1[idx_t]), s_s[1], f"{opt} state1 t={t}")
        assert_out_close(host(out[idx_t]), out_s, "bf16", f"{opt} shard_out t={t}")
    del grads, param, s0, s1, out
    torch.cuda.empty_cache()


def test_variant_rejects_bad_arguments(F):
    P = 64
    grads = [torch.ones(P, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    p32, s32a, s32b = (torch.zeros(P, device=DEV) for _ in range(3))
    p16, s16a, s16b = (torch.zeros(P, dtype=torch.bfloat16, device=DEV) for _ in range(3))
    out = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(F.FsdpError):  # SGD takes one state
        F.fsdp_reduce_scatter_step(grads, p32, s32a, s32b, out, F.StepConfig("sgd", 1e-3))
    with pytest.raises(F.FsdpError):  # Adamax needs two
        F.fsdp_reduce_scatter_step(grads, p32, s32a, None, out, F.StepConfig("adamax", 1e-3))
    with pytest.raises(F.FsdpError):  # low-precision state: the param is the shard, no shard_out
        F.fsdp_reduce_scatter_step(grads, p16, s16a, s16b, out, F.StepConfig("adamw", 1e-3))
    with pytest.raises(F.FsdpError):  # fp32 state needs shard_out
        F.fsdp_reduce_scatter_step(grads, p32, s32a, s32b, None, F.StepConfig("adamw", 1e-3))
    with pytest.raises(F.FsdpError):  # reduce dtype must be fp32 or the gradient dtype
        F.fsdp_reduce_scatter_step(grads, p32, s32a, s32b, out,
                                   F.StepConfig("adamw", 1e-3, reduce_dtype=torch.float16))
    torch.cuda.synchronize()
    assert not p32.any() and not s32a.any() and not out.any()
