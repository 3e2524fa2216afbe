"""Where a model's buffers live, as the multi-unit calls see it: the library
classifies each buffer as device or host memory (host buffers are refused
by the bulk-copy gather, and host-resident state keeps a unit out of the
batched launches), asking the driver once per device allocation. Buffers
carved from one device allocation must batch and step exactly as separate
allocations do, and a host buffer among them must still be found, wherever
it sits in the model. Called through the C ABI with raw descriptors.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def E():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sharded_fsdp_reduce_gb300 import _lib as E
    E.load()
    return E


class Arena:
    """One device allocation handing out 256-byte aligned views."""

    def __init__(self, nbytes):
        self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
        self.at = 0

    def take(self, n, dtype):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        assert self.at + nbytes <= self.buf.numel()
        t = self.buf[self.at:self.at + nbytes].view(dtype)
        self.at += (nbytes + 255) // 256 * 256
        return t


def unit_bytes(P, world):
    # grads, master/m/v, shard, gathered buffers (bf16 / fp32), with alignment slack
    return world * 2 * P + 3 * 4 * P + 2 * P + world * 2 * P + (2 * world + 5) * 256


def make_model(U, P, world, seed, arena=None):
    """U units of P elements, N = world, bf16 gradients and output; every
    buffer a view into `arena` (one allocation), or its own allocation."""
    g = torch.Generator().manual_seed(seed)
    take = arena.take if arena else (lambda n, dt: torch.zeros(n, dtype=dt, device=DEV))
    units = []
    for _ in range(U):
        u = {"grads": [take(P, torch.bfloat16) for _ in range(world)],
             "master": take(P, torch.float32), "m": take(P, torch.float32), "v": take(P, torch.float32),
             "shard": take(P, torch.bfloat16),
             "full": [take(P, torch.bfloat16) for _ in range(world)]}
        u["master"].copy_(torch.rand(P, generator=g) * 0.2 - 0.1)
        u["m"].zero_()
        u["v"].zero_()
        for x in u["grads"]:
            x.copy_((torch.randn(P, generator=g) * 1e-2).to(torch.bfloat16))
        units.append(u)
    torch.cuda.synchronize()
    return units


def descs(E, units, P, world):
    keep, arr = [], (E.FsdpUnit * len(units))()
    for k, u in enumerate(units):
        grads = (ctypes.c_void_p * world)(*[x.data_ptr() for x in u["grads"]])
        full = (ctypes.c_void_p * len(u["full"]))(*[x.data_ptr() for x in u["full"]])
        keep += [grads, full]
        d = arr[k]
        d.grads, d.full_bufs = ctypes.addressof(grads), ctypes.addressof(full)
        d.master, d.exp_avg, d.exp_avg_sq = u["master"].data_ptr(), u["m"].data_ptr(), u["v"].data_ptr()
        d.shard_out = u["shard"].data_ptr()
        d.padded_numel, d.world, d.n_full = P, world, len(u["full"])
        d.grad_dtype, d.out_dtype = E.FSDP_BF16, E.FSDP_BF16
    return arr, keep


def hp(E, t):
    return E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.01, t, 1.0)


def same(a, b):
    iv = torch.int32 if a.element_size() == 4 else torch.int16
    return torch.equal(a.view(iv), b.view(iv))


@pytest.mark.parametrize("world", [1, 2, 8])
def test_buffers_carved_from_one_allocation_batch_and_match_own_steps(E, world):
    # 40 units whose every buffer is a view into one device allocation: the
    # model batches into one update and one gather launch, and three steps
    # equal each unit stepped alone (its own update and gather launches) on
    # buffers that are separate allocations
    lib = E.load()
    U, P = 40, world * 3000
    arena = Arena(U * unit_bytes(P, world))
    a = make_model(U, P, world, 5, arena)
    b = make_model(U, P, world, 5)
    arr, keep = descs(E, a, P, world)
    n = ctypes.c_int64(-1)
    assert lib.fsdp_step_units_launches(arr, U, ctypes.byref(hp(E, 1)), 1, 0, ctypes.byref(n)) == E.FSDP_OK
    assert n.value == 2
    for t in (1, 2, 3):
        h = hp(E, t)
        assert lib.fsdp_step_units(arr, U, ctypes.byref(h), 1, 0, None, None, None) == E.FSDP_OK
        for u in b:
            grads = (ctypes.c_void_p * world)(*[x.data_ptr() for x in u["grads"]])
            full = (ctypes.c_void_p * world)(*[x.data_ptr() for x in u["full"]])
            assert lib.fsdp_reduce_scatter_adam_cast(grads, E.FSDP_BF16, world, P, u["master"].data_ptr(),
                                                     u["m"].data_ptr(), u["v"].data_ptr(), u["shard"].data_ptr(),
                                                     E.FSDP_BF16, ctypes.byref(h), 0, world, None, None) == E.FSDP_OK
            assert lib.fsdp_all_gather(u["shard"].data_ptr(), E.FSDP_BF16, world, P, full, world, None,
                                       None) == E.FSDP_OK
    torch.cuda.synchronize()
    for ua, ub in zip(a, b):
        for key in ("master", "m", "v", "shard"):
            assert same(ua[key], ub[key]), key
        for fa, fb in zip(ua["full"], ub["full"]):
            assert same(fa, fb)
            assert same(fa, ua["shard"])
    del keep


@pytest.mark.parametrize("where", ["first", "last"])
@pytest.mark.parametrize("kind", ["pinned", "pageable"])
def test_a_host_buffer_among_carved_device_buffers_is_refused(E, where, kind):
    # one gathered buffer or one shard in host memory, in the model's first
    # unit (before any device allocation is known) or in its last (after
    # every other buffer was found in the one device allocation): the call
    # is refused and nothing is enqueued
    lib = E.load()
    U, P, world = 24, 2 * 2048, 2
    arena = Arena(U * unit_bytes(P, world))
    units = make_model(U, P, world, 9, arena)
    before = [u["master"].clone() for u in units]
    k = 0 if where == "first" else U - 1
    host = torch.zeros(P, dtype=torch.bfloat16, pin_memory=(kind == "pinned"))
    for field in ("full", "shard"):
        saved = units[k]["full"][1] if field == "full" else units[k]["shard"]
        if field == "full":
            units[k]["full"][1] = host
        else:
            units[k]["shard"] = host
        arr, keep = descs(E, units, P, world)
        n = ctypes.c_int64(-1)
        assert lib.fsdp_step_units_launches(arr, U, ctypes.byref(hp(E, 1)), 1, 0,
                                            ctypes.byref(n)) == E.FSDP_ERR_INVALID_ARG
        assert lib.fsdp_step_units(arr, U, ctypes.byref(hp(E, 1)), 1, 0, None, None, None) == E.FSDP_ERR_INVALID_ARG
        plan = ctypes.c_void_p()
        assert lib.fsdp_step_plan_create(arr, U, 1, 0, None, None, ctypes.byref(plan)) == E.FSDP_ERR_INVALID_ARG
        assert not plan.value
        if field == "full":
            units[k]["full"][1] = saved
        else:
            units[k]["shard"] = saved
    torch.cuda.synchronize()
    for u, m0 in zip(units, before):
        assert same(u["master"], m0)
    assert lib.fsdp_last_cuda_error() == 0


def test_host_state_among_carved_units_keeps_its_own_launches(E):
    # a unit whose master, m and v are pinned host memory, placed after 20
    # units carved from one device allocation, is not batched with them (the
    # batched kernels' build is for state in HBM): one batch of 20 (update and
    # gather) plus the host-state unit's own two launches; the device-state
    # unit after it joins the batch of the first 20
    lib = E.load()
    U, P, world = 22, 2 * 2048, 2
    arena = Arena(U * unit_bytes(P, world))
    units = make_model(U, P, world, 13, arena)
    hs = [torch.zeros(P, pin_memory=True) for _ in range(3)]
    units[20]["master"], units[20]["m"], units[20]["v"] = hs
    arr, keep = descs(E, units, P, world)
    n = ctypes.c_int64(-1)
    assert lib.fsdp_step_units_launches(arr, U, ctypes.byref(hp(E, 1)), 1, 0, ctypes.byref(n)) == E.FSDP_OK
    assert n.value == 2 + 2
    del keep


_EXPANDABLE_SCRIPT = r"""
import ctypes, sys
import torch
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[2])
import sharded_fsdp_reduce_gb300 as F
from sharded_fsdp_reduce_gb300 import _lib as E
import test_residency_gpu as T

def same(a, b):
    iv = torch.int32 if a.element_size() == 4 else torch.int16
    return torch.equal(a.view(iv), b.view(iv))

# FlatParamUnits (each buffer its own torch allocation, inside the
# allocator's expandable segments): the planned and the unplanned model step
# equal each unit's own step
g = torch.Generator().manual_seed(3)
specs = [(int(n), w) for n, w in zip(torch.randint(1, 30000, (30,), generator=g), [1, 2, 8] * 10)]
a, b, c = ([F.FlatParamUnit([("w", (n,))], w, torch.bfloat16, torch.bfloat16, device="cuda") for n, w in specs]
           for _ in range(3))
for k, (n, w) in enumerate(specs):
    x = (torch.rand(n, generator=g) * 0.2 - 0.1).cuda()
    for u in (a[k], b[k], c[k]):
        u.load_master([x])
seq_a, seq_b = F.UnitSequence(a), F.UnitSequence(b)
assert seq_a.launches(gathers=1) < 2 * len(specs)
for t in (1, 2, 3):
    for k, (n, w) in enumerate(specs):
        for r in range(w):
            gr = (torch.randn(n, generator=g) * 1e-2).cuda().to(torch.bfloat16)
            for u in (a[k], b[k], c[k]):
                u.load_grad(r, [gr])
    hp = F.AdamWHParams(1e-3, weight_decay=0.01, step=t)
    seq_a.step(hp, gathers=1)
    seq_b.step_unplanned(hp, gathers=1)
    for u in c:
        u.step(hp, gathers=1)
torch.cuda.synchronize()
for ua, ub, uc in zip(a, b, c):
    for name in ("master", "exp_avg", "exp_avg_sq", "shard_out"):
        assert same(getattr(ua, name), getattr(uc, name)) and same(getattr(ub, name), getattr(uc, name)), name
    for fa, fc in zip(ua.full, uc.full):
        assert same(fa, fc)

# raw descriptors over one expandable-segment allocation: one batch; a
# pinned host gathered buffer in the last unit is refused
lib = E.load()
U, P, world = 16, 2 * 1024, 2
arena = T.Arena(U * T.unit_bytes(P, world))
units = T.make_model(U, P, world, 4, arena)
arr, keep = T.descs(E, units, P, world)
n = ctypes.c_int64(-1)
assert lib.fsdp_step_units_launches(arr, U, ctypes.byref(T.hp(E, 1)), 1, 0, ctypes.byref(n)) == E.FSDP_OK
assert n.value == 2, n.value
units[-1]["full"][0] = torch.zeros(P, dtype=torch.bfloat16, pin_memory=True)
arr, keep = T.descs(E, units, P, world)
assert lib.fsdp_step_units(arr, U, ctypes.byref(T.hp(E, 1)), 1, 0, None, None, None) == E.FSDP_ERR_INVALID_ARG
print("expandable ok")
"""


def test_models_under_the_allocators_expandable_segments(E):
    # the caching allocator's expandable segments map device memory into one
    # reserved address range (driver virtual memory management): the
    # residency answers and the batching must hold there too. The allocator
    # mode is fixed when CUDA starts, so this runs in a child process.
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, PYTORCH_CUDA_ALLOC_CONF="expandable_segments:True")
    r = subprocess.run([sys.executable, "-c", _EXPANDABLE_SCRIPT, os.path.dirname(here), here],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "expandable ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
