"""Host logic of FlatParamUnit that needs no GPU: layout of a unit's buffers
and the snapshot / resume of its optimizer state, whole or per rank shard."""
import pytest
import torch


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    import sharded_fsdp_reduce_gb300 as F
    return F


def cpu_unit(F, world=3):
    return F.FlatParamUnit([("w", (4, 5)), ("b", (3,))], world, torch.bfloat16, torch.bfloat16, device="cpu")


def test_unit_layout(F):
    u = cpu_unit(F)
    assert u.numel == 23 and u.padded_numel == 24 and u.shard_numel == 8
    assert [v.offset for v in u.views] == [0, 20]
    assert len(u.grads) == 3 and len(u.full) == 3
    pv = u.param_views(torch.arange(24.0))
    assert pv["w"].shape == (4, 5) and pv["b"].tolist() == [20.0, 21.0, 22.0]


def test_state_dict_whole_and_sharded_round_trip(F):
    a = cpu_unit(F)
    for k, name in enumerate(("master", "exp_avg", "exp_avg_sq")):
        getattr(a, name).copy_(torch.arange(24, dtype=torch.float32) + 100 * k)
    whole = a.state_dict()
    shards = [a.state_dict(rank=r) for r in range(3)]
    assert shards[1]["exp_avg"].tolist() == [float(x) for x in range(108, 116)]
    # the snapshot is a copy: later updates do not reach it
    a.master.zero_()
    assert whole["master"][5] == 5.0
    b, c = cpu_unit(F), cpu_unit(F)
    b.load_state_dict(whole)
    for r in (2, 0, 1):
        c.load_state_dict(shards[r], rank=r)
    for name in ("master", "exp_avg", "exp_avg_sq"):
        assert torch.equal(getattr(b, name), whole[name])
        assert torch.equal(getattr(c, name), whole[name])


def test_state_dict_rejects_bad_input(F):
    u = cpu_unit(F)
    with pytest.raises(ValueError):
        u.state_dict(rank=3)
    with pytest.raises(ValueError):
        u.load_state_dict(u.state_dict(rank=0))            # a shard is not the whole unit
    with pytest.raises(ValueError):
        u.load_state_dict(u.state_dict(), rank=1)          # nor the whole unit a shard
    bad = u.state_dict()
    bad["exp_avg"] = bad["exp_avg"].double()
    with pytest.raises(ValueError):
        u.load_state_dict(bad)


def test_variant_units_layout_and_bytes(F):
    # fp32 AdamW: N*2 + 3*(4+4) + 2 bytes per element (42 at N=8)
    u = F.FlatParamUnit([("w", (16,))], 8, torch.bfloat16, torch.bfloat16, device="cpu")
    assert not u.variant and u.step_bytes(2) == (16 * 42, 2 * 16 * 2 * 9)
    # SGD keeps one state buffer: 16 + 2*(4+4) + 2 = 34 bytes per element
    s = F.FlatParamUnit([("w", (16,))], 8, torch.bfloat16, torch.bfloat16, device="cpu", optimizer="sgd")
    assert s.variant and s.exp_avg_sq is None and s.step_bytes(1)[0] == 16 * 34
    # bf16 parameter + state: no fp32 master, the parameter is the shard; 16 + 3*(2+2) = 28
    b = F.FlatParamUnit([("w", (16,))], 8, torch.bfloat16, torch.bfloat16, device="cpu",
                        state_dtype=torch.bfloat16)
    assert b.variant and b.shard_out is b.master and b.master.dtype == torch.bfloat16
    assert b.step_bytes(1)[0] == 16 * 28
    assert set(b.state_dict()) == {"master", "exp_avg", "exp_avg_sq"}
    assert set(s.state_dict()) == {"master", "exp_avg"}
    # configurations the kernels do not take
    with pytest.raises(ValueError):
        F.FlatParamUnit([("w", (16,))], 8, torch.bfloat16, torch.float16, device="cpu", state_dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        F.FlatParamUnit([("w", (16,))], 8, torch.bfloat16, torch.bfloat16, device="cpu", optimizer="lamb")
    with pytest.raises(ValueError):
        F.FlatParamUnit([("w", (16,))], 8, torch.bfloat16, torch.bfloat16, device="cpu",
                        state_dtype=torch.bfloat16, state_on_host=True)
    with pytest.raises(ValueError):  # the state dict must match the unit's state buffers and dtype
        b.load_state_dict(u.state_dict())
    with pytest.raises(ValueError):
        s.load_state_dict(u.state_dict())


def test_step_config_matches_the_unit(F):
    s = F.FlatParamUnit([("w", (16,))], 8, torch.bfloat16, torch.bfloat16, device="cpu", optimizer="adamax")
    with pytest.raises(ValueError):
        s.step_config(F.StepConfig("sgd", 1e-3))
    with pytest.raises(ValueError):
        s.step_config(F.AdamWHParams(1e-3))               # an Adamax unit steps with a StepConfig
    a = F.FlatParamUnit([("w", (16,))], 8, torch.bfloat16, torch.bfloat16, device="cpu",
                        state_dtype=torch.bfloat16)
    cfg = a.step_config(F.AdamWHParams(2e-3, 0.8, 0.99, 1e-6, 0.1, 3, 4.0))
    assert (cfg.optimizer, cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, cfg.step, cfg.grad_scale) == \
        ("adamw", 2e-3, 0.8, 0.99, 1e-6, 0.1, 3, 4.0)


@pytest.mark.parametrize("fail_at", [1, 3, 5, 8])
def test_allocation_failure_reaches_the_caller(F, monkeypatch, fail_at):
    # a simulated out-of-memory at the fail_at-th buffer a unit allocates
    # (gradients, state, shard, gathered buffers): the error reaches the
    # caller unchanged, and a unit built afterwards is whole and zeroed
    real = torch.zeros
    count = {"n": 0}

    def zeros(*a, **k):
        count["n"] += 1
        if count["n"] == fail_at:
            raise torch.OutOfMemoryError("simulated allocation failure")
        return real(*a, **k)

    monkeypatch.setattr(torch, "zeros", zeros)
    with pytest.raises(torch.OutOfMemoryError, match="simulated"):
        cpu_unit(F)
    monkeypatch.undo()
    u = cpu_unit(F)
    bufs = u.grads + u.full + [u.master, u.exp_avg, u.exp_avg_sq, u.shard_out]
    assert len(bufs) == 10 and all(b.numel() == u.padded_numel and not b.any() for b in bufs)
