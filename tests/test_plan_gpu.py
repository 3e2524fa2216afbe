"""The validated model step (StepPlan, behind UnitSequence.step) and the
per-call counter of bounded waits that gave up.

A plan validates a model once; each launch checks only the step's scalars
and makes the launches fsdp_step_units would make. Its results must be the
same bits as the call that validates every time and as the captured graph,
over several steps, for models that mix batched small units, units with
their own launches and offloaded state; for the fused AdamW step and the
variant steps.
"""
import pytest
import torch

import fsdp_inputs as fi

pytestmark = pytest.mark.gpu

DEV = "cuda"


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


# (params, world, grad dtype, out dtype, state on host): small units that
# batch (N = 8 and N = 2), a GPT-2 small block (batched: under 2^24
# elements), a unit above 2^24 elements (its own launches), N = 3 (never
# batched) and an offloaded unit
def model_spec():
    small8 = ((("w", (40000,)),), 8, torch.bfloat16, torch.bfloat16, False)
    small2 = ((("w", (3000,)), ("b", (7,))), 2, torch.bfloat16, torch.bfloat16, False)
    return ([small8] * 5 + [small2] * 3
            + [(fi.CONFIGS["gpt2_small"].params, 8, torch.bfloat16, torch.bfloat16, False),
               ((("w", ((1 << 24) + 64,)),), 8, torch.bfloat16, torch.bfloat16, False),
               ((("w", (1001,)),), 3, torch.float32, torch.bfloat16, False),
               ((("w", (50000,)),), 8, torch.bfloat16, torch.bfloat16, True)])


def build(F, seed, optimizer="adamw", state_dtype=torch.float32):
    units = []
    g = torch.Generator().manual_seed(seed)
    for params, world, gdt, odt, on_host in model_spec():
        lowp = state_dtype != torch.float32
        u = F.FlatParamUnit(params, world, gdt, state_dtype if lowp else odt, device=DEV,
                            state_on_host=on_host and not lowp, optimizer=optimizer, state_dtype=state_dtype)
        u.load_master([(torch.rand(u.numel, generator=g) * 0.2 - 0.1).to(DEV)])
        units.append(u)
    torch.cuda.synchronize()
    return units


def load_grads(models, t):
    # identical gradients into every copy of the model
    g = torch.Generator().manual_seed(1000 + t)
    for k in range(len(models[0])):
        for r in range(models[0][k].world):
            x = (torch.randn(models[0][k].numel, generator=g) * 1e-2).to(DEV)
            for units in models:
                units[k].load_grad(r, [x.to(units[k].grads[r].dtype)])


def assert_models_equal(a, b):
    for ua, ub in zip(a, b):
        for name in ("master", "exp_avg", "exp_avg_sq", "shard_out"):
            x, y = getattr(ua, name), getattr(ub, name)
            if x is not None:
                assert same(x, y), name
        for fa, fb in zip(ua.full, ub.full):
            assert same(fa, fb)


@pytest.mark.parametrize("gathers,fuse", [(1, False), (2, False), (2, True)])
def test_plan_matches_unplanned_call_and_captured_graph(F, gathers, fuse):
    planned, unplanned, captured = build(F, 3), build(F, 3), build(F, 3)
    sp, su, sc = F.UnitSequence(planned), F.UnitSequence(unplanned), F.UnitSequence(captured)
    graph = sc.capture(gathers=gathers, fuse_gather=fuse)
    # one plan serves every step of the same kind
    assert sp.launches(gathers, fuse) == su.launches(gathers, fuse) < len(planned) * (1 + gathers)
    for t in (1, 2, 3, 4):
        load_grads([planned, unplanned, captured], t)
        hp = F.AdamWHParams(1e-3, weight_decay=0.01, step=t)
        sp.step(hp, gathers=gathers, fuse_gather=fuse)
        su.step_unplanned(hp, gathers=gathers, fuse_gather=fuse)
        graph.launch(hp)
        if t == 1:
            first = sp._plan
    torch.cuda.synchronize()
    assert sp._plan is first  # created once, launched four times
    assert_models_equal(planned, unplanned)
    assert_models_equal(planned, captured)
    for u in planned:
        if gathers:
            for f in u.full:
                assert same(f, u.shard_out)
    graph.close()


def test_a_plan_launched_from_other_host_threads(F):
    # a plan made on this thread, then launched from a new host thread at
    # each later step (that thread's own side streams and events; one launch
    # at a time, as the header requires of one plan): the same bits as the
    # same model planned and launched on this thread
    import threading
    a, b = build(F, 17), build(F, 17)
    sa, sb = F.UnitSequence(a), F.UnitSequence(b)
    for t in (1, 2, 3, 4):
        load_grads([a, b], t)
        hp = F.AdamWHParams(1e-3, weight_decay=0.01, step=t)
        sa.step(hp, gathers=2)
        if t == 1:
            sb.step(hp, gathers=2)
            first = sb._plan
            continue
        errors = []

        def launch():
            try:
                sb.step(hp, gathers=2)
                torch.cuda.synchronize()
            except Exception as e:  # reported on the main thread
                errors.append(e)

        th = threading.Thread(target=launch)
        th.start()
        th.join()
        assert not errors, errors
    torch.cuda.synchronize()
    assert sb._plan is first
    assert_models_equal(a, b)


@pytest.mark.parametrize("optimizer,state_dtype,lowp_reduce", [("adamw", torch.float32, True),
                                                               ("sgd", torch.float32, False),
                                                               ("adamax", torch.bfloat16, False),
                                                               ("adadelta", torch.float32, False)])
def test_variant_plan_matches_unplanned_call_and_captured_graph(F, optimizer, state_dtype, lowp_reduce):
    models = [build(F, 4, optimizer, state_dtype) for _ in range(3)]
    seqs = [F.UnitSequence(m) for m in models]
    # N = 3 with fp32 gradients takes part only with the fp32 reduction
    rd = torch.bfloat16 if lowp_reduce else None
    if lowp_reduce:
        models = [[u for u in m if u.grads[0].dtype == torch.bfloat16] for m in models]
        seqs = [F.UnitSequence(m) for m in models]
    cfg0 = F.StepConfig(optimizer, 1.0 if optimizer == "adadelta" else 1e-3, weight_decay=0.01, reduce_dtype=rd)
    graph = seqs[2].capture(gathers=1, config=cfg0)
    for t in (1, 2, 3):
        load_grads(models, t)
        cfg = F.StepConfig(optimizer, cfg0.lr, weight_decay=0.01, step=t, reduce_dtype=rd)
        seqs[0].step(cfg, gathers=1)
        seqs[1].step_unplanned(cfg, gathers=1)
        graph.launch(cfg)
    torch.cuda.synchronize()
    assert_models_equal(models[0], models[1])
    assert_models_equal(models[0], models[2])
    graph.close()


def test_plan_is_rebuilt_when_the_step_changes_kind(F):
    # the sequence keeps one plan per kind of step (gathers, fusion, optimizer,
    # counters): changing any of them validates anew, with the same results
    a, b = build(F, 5), build(F, 5)
    sa, sb = F.UnitSequence(a), F.UnitSequence(b)
    nf = torch.zeros(1, dtype=torch.int32, device=DEV)
    kinds = [dict(gathers=1), dict(gathers=2), dict(gathers=2, fuse_gather=True), dict(gathers=1, nonfinite_count=nf),
             dict(gathers=1)]
    plans = []
    for t, kw in enumerate(kinds, start=1):
        load_grads([a, b], t)
        hp = F.AdamWHParams(1e-3, step=t)
        sa.step(hp, **kw)
        sb.step_unplanned(hp, **kw)
        plans.append(sa._plan)
    torch.cuda.synchronize()
    assert len({id(p) for p in plans}) == len(plans)
    assert int(nf.item()) == 0
    assert_models_equal(a, b)


def test_a_refused_plan_enqueues_nothing(F):
    # two units sharing a written buffer, or one reading what another writes:
    # the plan is refused when it is made and no unit is touched
    for share in ("exp_avg", "grads"):
        units = build(F, 6)[:3]
        before = [u.master.clone() for u in units]
        if share == "exp_avg":
            units[1].exp_avg = units[0].exp_avg
        else:
            units[2].grads[0] = units[0].master.view(torch.bfloat16)[: units[2].padded_numel]
        seq = F.UnitSequence(units)
        with pytest.raises(F.FsdpError):
            seq.step(F.AdamWHParams(1e-3), gathers=1)
        with pytest.raises(F.FsdpError):
            seq.step_unplanned(F.AdamWHParams(1e-3), gathers=1)
        torch.cuda.synchronize()
        for u, m in zip(units, before):
            assert same(u.master, m)
            assert not u.shard_out.any() and not any(f.any() for f in u.full)


def test_wait_timeouts_counter_reads_zero_on_every_step_path(F):
    # the per-call counter of bounded waits that gave up: 0 in normal
    # operation on every path that gathers, read in stream order
    units = build(F, 7)
    wt = torch.zeros(1, dtype=torch.int32, device=DEV)
    seq = F.UnitSequence(units)
    load_grads([units], 1)
    hp = F.AdamWHParams(1e-3, step=1)
    for u in units[-4:]:
        u.step(hp, gathers=2, wait_timeouts=wt)
        u.all_gather(wait_timeouts=wt)
    seq.step(F.AdamWHParams(1e-3, step=2), gathers=2, wait_timeouts=wt)
    seq.step_unplanned(F.AdamWHParams(1e-3, step=3), gathers=2, wait_timeouts=wt)
    graph = seq.capture(gathers=2, wait_timeouts=wt)
    graph.launch(F.AdamWHParams(1e-3, step=4))
    assert int(wt.item()) == 0  # .item() waits for the current stream only
    for u in units:
        for f in u.full:
            assert same(f, u.shard_out)
    graph.close()
    with pytest.raises(ValueError):
        units[0].all_gather(wait_timeouts=torch.zeros(1, dtype=torch.float32, device=DEV))


def test_descriptors_keep_the_buffers_they_point_at_alive(F):
    # a plan or a captured step writes to the addresses its descriptors were
    # made with; a buffer replaced in a unit afterwards must not be freed and
    # handed to another allocation while they exist
    units = build(F, 8)[:3]
    seq = F.UnitSequence(units)
    seq.step(F.AdamWHParams(1e-3, step=1), gathers=1)
    old = units[1].exp_avg
    ptr = old.data_ptr()
    units[1].exp_avg = torch.zeros_like(old)  # replaced after the descriptors were made
    del old
    fresh = [torch.empty_like(units[1].exp_avg) for _ in range(4)]
    assert all(t.data_ptr() != ptr for t in fresh)
    kept = [t for t in seq.descs._keep if isinstance(t, torch.Tensor)]
    assert any(t.data_ptr() == ptr for t in kept)
    seq.step(F.AdamWHParams(1e-3, step=2), gathers=1)  # still writes the old buffer, which is still allocated
    torch.cuda.synchronize()
