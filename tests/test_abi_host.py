"""Host-side checks of the C ABI: the library loads, exports every function the
header declares, and its host-only functions (layout, status strings, argument
validation that returns before any CUDA call) behave as documented. No GPU is
needed and no device work is enqueued: every call here is rejected on the host
or is host-only.
"""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from sharded_fsdp_reduce_gb300 import _lib
    return _lib.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fsdp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fsdp_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    from sharded_fsdp_reduce_gb300 import _lib
    names = declared_functions()
    assert names, "no declarations parsed"
    assert sorted(_lib.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_padded_numel_matches_oracle(lib, orc):
    for world in (1, 2, 3, 7, 8, 64):
        for numel in list(range(0, 40)) + [4099, 7087872, 855654400, 2**40 + 3]:
            assert lib.fsdp_padded_numel(numel, world) == orc.padded_numel(numel, world)
    assert lib.fsdp_padded_numel(-1, 2) == -1
    assert lib.fsdp_padded_numel(3, 0) == -1


def test_unflatten_views_match_oracle_offsets(orc):
    import fsdp_inputs as fi
    import sharded_fsdp_reduce_gb300 as F
    for cfg in fi.CONFIGS.values():
        shapes = [s for _, s in cfg.params]
        views, padded = F.fsdp_unflatten_views(shapes, cfg.world)
        numels = [int(np.prod(s)) for s in shapes]
        np.testing.assert_array_equal([v.offset for v in views], orc.view_offsets(numels))
        assert [v.numel for v in views] == numels
        assert [v.shape for v in views] == [tuple(s) for s in shapes]
        assert padded == orc.padded_numel(sum(numels), cfg.world)


def test_unflatten_views_edge_cases():
    import sharded_fsdp_reduce_gb300 as F
    views, padded = F.fsdp_unflatten_views([(), (0,), (3, 0), (5,)], 4)
    assert [v.numel for v in views] == [1, 0, 0, 5]
    assert [v.offset for v in views] == [0, 1, 1, 1]
    assert padded == 8
    views, padded = F.fsdp_unflatten_views([], 3)
    assert views == [] and padded == 0
    with pytest.raises(F.FsdpError):
        F.fsdp_unflatten_views([(2, -1)], 2)
    with pytest.raises(F.FsdpError):
        F.fsdp_unflatten_views([(1,) * 9], 2)
    with pytest.raises(F.FsdpError):
        F.fsdp_unflatten_views([(3,)], 0)
    with pytest.raises(F.FsdpError):
        F.fsdp_unflatten_views([(2**62,), (2**62,)], 1)  # offset overflow


def test_status_strings(lib):
    from sharded_fsdp_reduce_gb300 import _lib
    for code in range(6):
        assert lib.fsdp_status_string(code).decode().startswith(
            ["FSDP_OK", "FSDP_ERR_INVALID_ARG", "FSDP_ERR_ALIGNMENT", "FSDP_ERR_CUDA",
             "FSDP_ERR_UNSUPPORTED_DTYPE", "FSDP_ERR_HOST_MEMORY"][code])
    assert lib.fsdp_status_string(99).decode().startswith("FSDP_ERR_UNKNOWN")
    assert lib.fsdp_last_cuda_error() == 0
    assert _lib.FSDP_OK == 0


# ---------------------------------------------------------------- validation (host only)

FAKE = 0x7f0000000000  # never dereferenced: every call below fails validation first


def _rsa(lib, **kw):
    from sharded_fsdp_reduce_gb300 import _lib
    world = kw.get("world", 2)
    P = kw.get("P", 16)
    grads = kw.get("grads", [FAKE + 0x100000 * (q + 1) for q in range(world)])
    garr = None if grads is None else (ctypes.c_void_p * max(len(grads), 1))(*grads)
    hp = kw.get("hp", _lib.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0))
    return lib.fsdp_reduce_scatter_adam_cast(
        garr, kw.get("gdt", 1), world, P, kw.get("master", FAKE + 0x1000000), kw.get("m", FAKE + 0x2000000),
        kw.get("v", FAKE + 0x3000000), kw.get("out", FAKE + 0x4000000), kw.get("odt", 1),
        None if hp is None else ctypes.byref(hp), kw.get("rb", 0), kw.get("re", world),
        kw.get("nf", None), None)


def test_rsa_rejects_invalid_arguments(lib):
    from sharded_fsdp_reduce_gb300 import _lib
    E = _lib
    assert _rsa(lib, gdt=7) == E.FSDP_ERR_UNSUPPORTED_DTYPE
    assert _rsa(lib, odt=-1) == E.FSDP_ERR_UNSUPPORTED_DTYPE
    assert _rsa(lib, world=0, grads=[]) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, world=65, grads=[FAKE] * 65) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, grads=None) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, hp=None) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, P=15) == E.FSDP_ERR_INVALID_ARG            # not a multiple of N
    assert _rsa(lib, P=-2) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, rb=1, re=0) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, rb=0, re=3) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, rb=-1) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, hp=E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 0, 1.0)) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, hp=E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 0.0)) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, hp=E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, float("inf"))) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, master=None) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, out=None) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, grads=[FAKE, None]) == E.FSDP_ERR_INVALID_ARG
    # misalignment to the element size
    assert _rsa(lib, master=FAKE + 0x1000002) == E.FSDP_ERR_ALIGNMENT
    assert _rsa(lib, out=FAKE + 0x4000001) == E.FSDP_ERR_ALIGNMENT
    assert _rsa(lib, grads=[FAKE + 1, FAKE + 0x100000]) == E.FSDP_ERR_ALIGNMENT
    assert _rsa(lib, nf=FAKE + 2) == E.FSDP_ERR_ALIGNMENT
    # aliasing: shard_out inside a state buffer, state buffers overlapping, grads on the state
    assert _rsa(lib, out=FAKE + 0x1000000 + 16) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, m=FAKE + 0x1000000 + 8) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, grads=[FAKE + 0x3000000, FAKE]) == E.FSDP_ERR_INVALID_ARG
    assert _rsa(lib, grads=[FAKE + 0x4000000, FAKE]) == E.FSDP_ERR_INVALID_ARG
    # empty work is a no-op that succeeds without touching anything
    assert _rsa(lib, P=0) == E.FSDP_OK
    assert _rsa(lib, rb=1, re=1) == E.FSDP_OK
    assert lib.fsdp_last_cuda_error() == 0


def test_all_gather_rejects_invalid_arguments(lib):
    from sharded_fsdp_reduce_gb300 import _lib as E
    arr = lambda *p: (ctypes.c_void_p * len(p))(*p)
    ag = lambda src, dt, world, P, dsts, n, wt=None: lib.fsdp_all_gather(src, dt, world, P, dsts, n, wt, None)
    assert ag(FAKE, 9, 2, 16, arr(FAKE + 4096), 1) == E.FSDP_ERR_UNSUPPORTED_DTYPE
    assert ag(FAKE, 1, 0, 16, arr(FAKE + 4096), 1) == E.FSDP_ERR_INVALID_ARG
    assert ag(FAKE, 1, 2, 15, arr(FAKE + 4096), 1) == E.FSDP_ERR_INVALID_ARG
    assert ag(FAKE, 1, 2, 16, arr(FAKE + 4096), 0) == E.FSDP_ERR_INVALID_ARG
    assert ag(FAKE, 1, 2, 16, None, 1) == E.FSDP_ERR_INVALID_ARG
    assert ag(None, 1, 2, 16, arr(FAKE + 4096), 1) == E.FSDP_ERR_INVALID_ARG
    assert ag(FAKE + 1, 1, 2, 16, arr(FAKE + 4096), 1) == E.FSDP_ERR_ALIGNMENT
    assert ag(FAKE, 1, 2, 16, arr(FAKE + 4097), 1) == E.FSDP_ERR_ALIGNMENT
    assert ag(FAKE, 1, 2, 16, arr(FAKE + 16), 1) == E.FSDP_ERR_INVALID_ARG      # overlaps the source
    assert ag(FAKE, 1, 2, 16, arr(FAKE + 4096, FAKE + 4100), 2) == E.FSDP_ERR_INVALID_ARG  # dsts overlap
    assert ag(FAKE, 1, 2, 16, arr(FAKE + 4096, None), 2) == E.FSDP_ERR_INVALID_ARG
    assert ag(FAKE, 1, 2, 0, arr(FAKE + 4096), 1) == E.FSDP_OK                   # empty: no-op
    assert ag(FAKE, 1, 2, 16, arr(FAKE + 4096), 1, FAKE + 2) == E.FSDP_ERR_ALIGNMENT  # counter off 4 bytes


def test_flatten_rejects_invalid_arguments(lib):
    from sharded_fsdp_reduce_gb300 import _lib as E
    arr = lambda *p: (ctypes.c_void_p * len(p))(*p)
    i64 = lambda *n: (ctypes.c_int64 * len(n))(*n)
    fl = lambda srcs, numels, n, dt, world, dst, dn: lib.fsdp_flatten_pad(srcs, numels, n, dt, world, dst, dn,
                                                                          None, None)
    assert fl(arr(FAKE), i64(5), 1, 3, 2, FAKE + 4096, 6) == E.FSDP_ERR_UNSUPPORTED_DTYPE
    assert fl(arr(FAKE), i64(5), 1, 1, 2, FAKE + 4096, 5) == E.FSDP_ERR_INVALID_ARG   # dst_numel != padded
    assert fl(arr(FAKE), i64(5), 1, 1, 0, FAKE + 4096, 5) == E.FSDP_ERR_INVALID_ARG
    assert fl(arr(FAKE), i64(-5), 1, 1, 2, FAKE + 4096, 0) == E.FSDP_ERR_INVALID_ARG
    assert fl(arr(None), i64(5), 1, 1, 2, FAKE + 4096, 6) == E.FSDP_ERR_INVALID_ARG
    assert fl(arr(FAKE), i64(5), 1, 1, 2, None, 6) == E.FSDP_ERR_INVALID_ARG
    assert fl(arr(FAKE + 1), i64(5), 1, 1, 2, FAKE + 4096, 6) == E.FSDP_ERR_ALIGNMENT
    assert fl(arr(FAKE), i64(5), 1, 0, 2, FAKE + 4098, 6) == E.FSDP_ERR_ALIGNMENT    # f32 dst on 2 bytes
    assert fl(arr(FAKE + 4), i64(5), 1, 1, 2, FAKE, 6) == E.FSDP_ERR_INVALID_ARG     # source inside dst
    assert fl(None, None, 0, 1, 2, None, 0) == E.FSDP_OK                              # nothing to do


def test_take_wait_timeouts_rejects_null(lib):
    from sharded_fsdp_reduce_gb300 import _lib as E
    assert lib.fsdp_take_wait_timeouts(None) == E.FSDP_ERR_INVALID_ARG


def test_check_bounded_wait_rejects_limits_out_of_range(lib):
    from sharded_fsdp_reduce_gb300 import _lib as E
    for limit in (0, -1, (1 << 31) + 1):
        assert lib.fsdp_check_bounded_wait(limit, None, None) == E.FSDP_ERR_INVALID_ARG
    assert lib.fsdp_check_bounded_wait(1 << 20, FAKE + 1, None) == E.FSDP_ERR_ALIGNMENT


def test_fused_gather_rejects_invalid_arguments(lib):
    from sharded_fsdp_reduce_gb300 import _lib as E
    arr = lambda *p: (ctypes.c_void_p * len(p))(*p)
    hp = E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
    g = arr(FAKE + 0x100000, FAKE + 0x200000)

    def call(out, fulls, n, **kw):
        return lib.fsdp_reduce_scatter_adam_cast_gather(g, 1, 2, 16, FAKE + 0x1000000, FAKE + 0x2000000,
                                                        FAKE + 0x3000000, out, 1, fulls, n, ctypes.byref(hp),
                                                        0, 2, None, None)
    assert call(FAKE + 0x4000000, arr(FAKE + 0x5000000), 0) == E.FSDP_ERR_INVALID_ARG   # no destination
    assert call(FAKE + 0x4000000, None, 1) == E.FSDP_ERR_INVALID_ARG
    assert call(FAKE + 0x4000000, arr(None), 1) == E.FSDP_ERR_INVALID_ARG
    assert call(FAKE + 0x4000000, arr(FAKE + 0x5000001), 1) == E.FSDP_ERR_ALIGNMENT
    assert call(FAKE + 0x4000000, arr(FAKE + 0x4000010), 1) == E.FSDP_ERR_INVALID_ARG  # overlaps shard_out
    assert call(None, arr(FAKE + 0x1000000), 1) == E.FSDP_ERR_INVALID_ARG              # overlaps master
    assert call(None, arr(FAKE + 0x100010), 1) == E.FSDP_ERR_INVALID_ARG               # overlaps a gradient
    assert call(None, arr(FAKE + 0x5000000, FAKE + 0x5000008), 2) == E.FSDP_ERR_INVALID_ARG
    assert lib.fsdp_reduce_scatter_adam_cast(g, 1, 2, 16, FAKE + 0x1000000, FAKE + 0x2000000, FAKE + 0x3000000,
                                             None, 1, ctypes.byref(hp), 0, 2, None, None) == E.FSDP_ERR_INVALID_ARG


def test_variant_step_rejects_invalid_arguments(lib):
    from sharded_fsdp_reduce_gb300 import _lib as E
    arr = lambda *p: (ctypes.c_void_p * len(p))(*p)
    g = arr(FAKE + 0x100000, FAKE + 0x200000)

    def call(opt=0, rd=0, sdt=0, odt=1, p=FAKE + 0x1000000, s0=FAKE + 0x2000000, s1=FAKE + 0x3000000,
             out=FAKE + 0x4000000, step=1, P=16, gdt=1):
        cfg = E.FsdpStepConfig(opt, rd, 1e-3, 0.9, 0.999, 1e-8, 0.0, step, 1.0)
        return lib.fsdp_reduce_scatter_step(g, gdt, 2, P, p, s0, s1, sdt, out, odt, ctypes.byref(cfg), 0, 2, None,
                                            None)
    assert call(opt=4) == E.FSDP_ERR_INVALID_ARG
    assert call(opt=-1) == E.FSDP_ERR_INVALID_ARG
    assert call(rd=2) == E.FSDP_ERR_UNSUPPORTED_DTYPE            # f16 reduction of bf16 gradients
    assert call(sdt=1, odt=2, out=None) == E.FSDP_ERR_UNSUPPORTED_DTYPE  # bf16 state, f16 out
    assert call(sdt=7) == E.FSDP_ERR_UNSUPPORTED_DTYPE
    assert call(opt=1) == E.FSDP_ERR_INVALID_ARG                 # SGD with a second state
    assert call(opt=2, s1=None) == E.FSDP_ERR_INVALID_ARG        # Adamax without one
    assert call(sdt=1, odt=1) == E.FSDP_ERR_INVALID_ARG          # bf16 state with a shard_out
    assert call(out=None) == E.FSDP_ERR_INVALID_ARG              # fp32 state without shard_out
    assert call(step=0) == E.FSDP_ERR_INVALID_ARG
    assert call(P=15) == E.FSDP_ERR_INVALID_ARG
    assert call(p=FAKE + 0x1000002) == E.FSDP_ERR_ALIGNMENT
    assert call(s0=FAKE + 0x1000000 + 8) == E.FSDP_ERR_INVALID_ARG   # state overlaps the param
    assert call(out=FAKE + 0x100000) == E.FSDP_ERR_INVALID_ARG       # shard_out on a gradient
    assert call(P=0) == E.FSDP_OK
    assert lib.fsdp_last_cuda_error() == 0


def test_exports_nothing_but_the_c_abi(lib):
    # host code is built with hidden visibility: the dynamic symbol table holds
    # the declared entry points and nothing else
    import shutil
    import subprocess
    from sharded_fsdp_reduce_gb300 import _lib
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True, check=True)
    exported = sorted(line.split()[-1] for line in out.stdout.splitlines() if " T " in line)
    assert exported == declared_functions()


def test_binding_refuses_unpinned_host_tensors(lib):
    # the kernels stream device memory or pinned (mapped) host memory only;
    # the binding refuses an ordinary host tensor before calling the library
    import torch
    import sharded_fsdp_reduce_gb300 as F
    P = 8
    g = [torch.ones(P, dtype=torch.bfloat16)] * 2
    st = [torch.zeros(P) for _ in range(3)]
    out = torch.zeros(P, dtype=torch.bfloat16)
    hp = F.AdamWHParams(1e-3, step=1)
    with pytest.raises(ValueError, match="grads"):
        F.fsdp_reduce_scatter_adam_cast(g, *st, out, hp)
    with pytest.raises(ValueError):
        F.fsdp_reduce_scatter_adam_cast_gather(g, *st, None, [out], hp)
    with pytest.raises(ValueError, match="grads"):
        F.fsdp_reduce_scatter_step(g, st[0], st[1], st[2], out, F.StepConfig("adamw", 1e-3))
    with pytest.raises(ValueError, match="shard_out"):
        F.fsdp_all_gather(out, [out.clone()], 2)


def _unit(E, base, world=2, P=16, n_full=2, gd=1, od=1):
    """An fsdp_unit descriptor over fake, non-overlapping addresses (never
    dereferenced: every call below is rejected on the host)."""
    arr = lambda *p: (ctypes.c_void_p * len(p))(*p)
    g = arr(*[base + 0x100000 * (q + 1) for q in range(world)])
    f = arr(*[base + 0x1000000 * (8 + d) for d in range(n_full)]) if n_full else None
    u = E.FsdpUnit()
    u.grads = ctypes.addressof(g)
    u.full_bufs = ctypes.addressof(f) if f is not None else None
    u.master, u.exp_avg, u.exp_avg_sq = base + 0x1000000, base + 0x2000000, base + 0x3000000
    u.shard_out = base + 0x4000000
    u.padded_numel, u.world, u.grad_dtype, u.out_dtype, u.n_full = P, world, gd, od, n_full
    return u, (g, f)


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host-only: needs a machine without a GPU")
def test_step_units_validates_every_unit_before_launching(lib):
    # unit 0 is valid; the call must still fail on unit 1 without launching
    # unit 0 (a launch here would report FSDP_ERR_CUDA: there is no device)
    from sharded_fsdp_reduce_gb300 import _lib as E
    hp = E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
    keep = []

    def call(units, gathers=1, fuse=0, hpp=ctypes.byref(hp), n=None):
        arr = (E.FsdpUnit * max(len(units), 1))(*units)
        return lib.fsdp_step_units(arr, len(units) if n is None else n, hpp, gathers, fuse, None, None, None)

    def unit(base, **kw):
        u, k = _unit(E, base, **kw)
        keep.append(k)
        return u

    A, B = FAKE, FAKE + 0x100000000
    assert call([]) == E.FSDP_OK
    assert lib.fsdp_step_units(None, 0, ctypes.byref(hp), 1, 0, None, None, None) == E.FSDP_OK
    assert lib.fsdp_step_units(None, 1, ctypes.byref(hp), 1, 0, None, None, None) == E.FSDP_ERR_INVALID_ARG
    assert lib.fsdp_step_units(None, 0, ctypes.byref(hp), 1, 0, None, FAKE + 2, None) == E.FSDP_ERR_ALIGNMENT
    assert call([unit(A)], hpp=None) == E.FSDP_ERR_INVALID_ARG
    assert call([unit(A)], gathers=-1) == E.FSDP_ERR_INVALID_ARG
    assert call([unit(A)], gathers=65) == E.FSDP_ERR_INVALID_ARG
    assert call([unit(A), unit(B, gd=7)]) == E.FSDP_ERR_UNSUPPORTED_DTYPE
    assert call([unit(A), unit(B, n_full=0)]) == E.FSDP_ERR_INVALID_ARG        # gathers without buffers
    assert call([unit(A), unit(B, P=15)]) == E.FSDP_ERR_INVALID_ARG            # not a multiple of N
    assert call([unit(A), unit(B, world=65)]) == E.FSDP_ERR_INVALID_ARG
    bad = unit(B)
    bad.master = B + 0x1000002
    assert call([unit(A), bad]) == E.FSDP_ERR_ALIGNMENT
    bad = unit(B)
    bad.shard_out = None
    assert call([unit(A), bad]) == E.FSDP_ERR_INVALID_ARG
    bad = unit(B)
    bad.exp_avg = A + 0x1000000                                                # shares unit 0's master
    assert call([unit(A), bad]) == E.FSDP_ERR_INVALID_ARG
    bad = unit(B)
    bad.shard_out = A + 0x1000000 * 9                                          # unit 0's gathered buffer
    assert call([unit(A), bad]) == E.FSDP_ERR_INVALID_ARG
    bad = unit(B)
    bad.master = B + 0x100000                                                  # master on its own gradient
    assert call([unit(A), bad]) == E.FSDP_ERR_INVALID_ARG
    assert call([unit(A, n_full=0), unit(B, n_full=0)], gathers=1, fuse=1) == E.FSDP_ERR_INVALID_ARG
    assert call([unit(A, P=0), unit(B, P=0)]) == E.FSDP_OK                     # empty units: nothing to launch
    assert lib.fsdp_last_cuda_error() == 0


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host-only: needs a machine without a GPU")
def test_step_units_ex_validates_every_unit_before_launching(lib):
    from sharded_fsdp_reduce_gb300 import _lib as E
    keep = []

    def unit(base, world=2, P=16, n_full=2, sdt=0, odt=1, opt_states=2, out=True):
        arr = lambda *p: (ctypes.c_void_p * len(p))(*p)
        g = arr(*[base + 0x100000 * (q + 1) for q in range(world)])
        f = arr(*[base + 0x1000000 * (8 + d) for d in range(n_full)]) if n_full else None
        keep.append((g, f))
        u = E.FsdpUnitEx()
        u.grads, u.full_bufs = ctypes.addressof(g), (ctypes.addressof(f) if f is not None else None)
        u.param, u.state0 = base + 0x1000000, base + 0x2000000
        u.state1 = base + 0x3000000 if opt_states == 2 else None
        u.shard_out = base + 0x4000000 if out else None
        u.padded_numel, u.world, u.n_full = P, world, n_full
        u.grad_dtype, u.state_dtype, u.out_dtype = 1, sdt, odt
        return u

    def call(units, opt=0, gathers=1):
        cfg = E.FsdpStepConfig(opt, 0, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
        arr = (E.FsdpUnitEx * max(len(units), 1))(*units)
        return lib.fsdp_step_units_ex(arr, len(units), ctypes.byref(cfg), gathers, None, None, None)

    A, B = FAKE, FAKE + 0x100000000
    assert call([]) == E.FSDP_OK
    assert call([unit(A), unit(B, sdt=7)]) == E.FSDP_ERR_UNSUPPORTED_DTYPE
    assert call([unit(A), unit(B)], opt=1) == E.FSDP_ERR_INVALID_ARG          # SGD with a second state
    assert call([unit(A, opt_states=1), unit(B, opt_states=1)], opt=2) == E.FSDP_ERR_INVALID_ARG  # Adamax without
    assert call([unit(A), unit(B, sdt=1, odt=1)]) == E.FSDP_ERR_INVALID_ARG   # bf16 state with a shard_out
    assert call([unit(A), unit(B, n_full=0)]) == E.FSDP_ERR_INVALID_ARG       # gathers without buffers
    bad = unit(B)
    bad.state0 = A + 0x2000000                                                 # unit 0's first state
    assert call([unit(A), bad]) == E.FSDP_ERR_INVALID_ARG
    assert call([unit(A, P=0), unit(B, P=0)]) == E.FSDP_OK                     # empty units: nothing to launch
    flagged = unit(B)
    flagged.reserved = 1                                                       # a reserved field that is not 0
    assert call([unit(A), flagged]) == E.FSDP_ERR_INVALID_ARG
    assert lib.fsdp_last_cuda_error() == 0


def test_step_graph_rejects_invalid_arguments_on_the_host(lib):
    from sharded_fsdp_reduce_gb300 import _lib as E
    out = ctypes.c_void_p(123)
    assert lib.fsdp_step_graph_create(None, 0, 1, 0, None, None, None) == E.FSDP_ERR_INVALID_ARG     # no handle
    assert lib.fsdp_step_graph_create(None, 1, 1, 0, None, None, ctypes.byref(out)) == E.FSDP_ERR_INVALID_ARG
    assert out.value is None                                                                          # cleared
    assert lib.fsdp_step_graph_create(None, 0, -1, 0, None, None, ctypes.byref(out)) == E.FSDP_ERR_INVALID_ARG
    hp = E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
    assert lib.fsdp_step_graph_launch(None, ctypes.byref(hp), None) == E.FSDP_ERR_INVALID_ARG
    assert lib.fsdp_step_graph_destroy(None) == E.FSDP_OK


def _fake_units(E, specs, ex=False):
    """fsdp_unit (or fsdp_unit_ex) descriptors over never-dereferenced
    addresses, one 4 GB region per unit so that no written buffers overlap;
    specs are (padded_numel, world, n_full, misaligned)."""
    keep, units = [], []
    for u, (P, world, n_full, misaligned) in enumerate(specs):
        base = FAKE + (u << 32) + (4 if misaligned else 0)
        grads = (ctypes.c_void_p * world)(*[base + 0x80000000 + (q << 26) for q in range(world)])
        full = (ctypes.c_void_p * n_full)(*[base + 0x40000000 + (d << 26) for d in range(n_full)])
        keep += [grads, full]
        x = E.FsdpUnitEx() if ex else E.FsdpUnit()
        x.grads, x.full_bufs = ctypes.addressof(grads), ctypes.addressof(full)
        if ex:
            x.param, x.state0, x.state1 = base, base + 0x10000000, base + 0x20000000
            x.state_dtype = 0
        else:
            x.master, x.exp_avg, x.exp_avg_sq = base, base + 0x10000000, base + 0x20000000
        x.shard_out = base + 0x30000000
        x.padded_numel, x.world, x.n_full = P, world, n_full
        x.grad_dtype, x.out_dtype = 1, 1
        units.append(x)
    arr = ((E.FsdpUnitEx if ex else E.FsdpUnit) * max(len(units), 1))(*units)
    return arr, keep


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host-only: fake addresses need a machine without a GPU")
def test_step_units_launches_follow_the_batching(lib):
    # the planning query: nothing is enqueued; small units batch
    # bench.GROUP_MAX_UNITS (the header's batch size) per launch, larger or
    # misaligned units or N = 3 keep their own launches
    from sharded_fsdp_reduce_gb300 import _lib as E
    import bench
    hp = E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
    out = ctypes.c_int64(-1)

    def count(specs, gathers=1, fuse=0):
        arr, keep = _fake_units(E, specs)
        st = lib.fsdp_step_units_launches(arr, len(specs), ctypes.byref(hp), gathers, fuse, ctypes.byref(out))
        assert st == E.FSDP_OK, st
        return out.value

    small = (50000, 8, 8, False)
    G = bench.GROUP_MAX_UNITS
    for n, gathers in ((200, 1), (200, 2), (200, 0), (G, 1), (G + 1, 1), (2 * G + 3, 1), (1, 1), (2, 1)):
        assert count([small] * n, gathers) == bench.model_launches(n, 50000, gathers), (n, gathers)
    assert count([(7087872, 8, 8, False)] * 12) == bench.model_launches(12, 7087872, 1) == 2
    big = ((1 << 24) + 8, 8, 8, False)
    assert count([big] * 3) == 6                                     # above the size limit: own launches
    assert count([small] * 5 + [(50000, 8, 8, True)]) == 2 + 2       # a misaligned unit keeps its own
    assert count([small] * 5 + [(50000 - 2, 2, 1, False)] * 3) == 2 + 2   # another N: a second batch
    assert count([(3 * 1000, 3, 3, False)] * 4) == 8                 # N = 3 is not batched
    assert count([(1000, 1, 1, False)] * 4) == 2                     # N = 1 is (a single rank)
    assert count([small] * 5, gathers=2, fuse=1) == 2                # fused gather: one batch, then a gather
    assert count([small] * 300, gathers=1, fuse=1) == 3              # fused batches take 128 units each
    assert count([small] * 5 + [(50000, 8, 8, True)], gathers=1, fuse=1) == 1 + 1  # misaligned: its own
    assert count([small] * 3 + [(0, 8, 8, False)]) == 2              # an empty unit launches nothing
    assert lib.fsdp_step_units_launches(None, 0, ctypes.byref(hp), 1, 0, None) == E.FSDP_ERR_INVALID_ARG
    arr, keep = _fake_units(E, [small, small])
    arr[1].master = arr[0].master                                     # two units writing one buffer
    assert lib.fsdp_step_units_launches(arr, 2, ctypes.byref(hp), 1, 0, ctypes.byref(out)) == E.FSDP_ERR_INVALID_ARG
    # the variant call
    cfg = E.FsdpStepConfig(1, 0, 1e-2, 0.9, 0.0, 0.0, 0.0, 1, 1.0)  # SGD: one state
    arr, keep = _fake_units(E, [small] * (G + 22), ex=True)
    for k in range(G + 22):
        arr[k].state1 = None
    assert lib.fsdp_step_units_ex_launches(arr, G + 22, ctypes.byref(cfg), 1, ctypes.byref(out)) == E.FSDP_OK
    assert out.value == 4
    assert lib.fsdp_last_cuda_error() == 0


def _expected_launches(specs, gathers):
    """The batching rule restated: units of N in {1, 2, 4, 8}, at most 2^24
    elements, 16-byte aligned and not empty batch with the earlier ones of
    the same N (every fake unit here shares the dtypes and gathers), the
    header's batch size per batch; a batch of one is a unit on its own; one
    update and `gathers` gathers per work item."""
    import bench
    G = bench.GROUP_MAX_UNITS
    items, open_ = 0, {}
    for P, world, n_full, misaligned in specs:
        if P == 0:
            continue
        if world not in (1, 2, 4, 8) or P > (1 << 24) or misaligned or n_full > 8:
            items += 1
            continue
        if open_.get(world, G) == G:
            items += 1
            open_[world] = 0
        open_[world] += 1
    return items * (1 + gathers)


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host-only: fake addresses need a machine without a GPU")
@pytest.mark.parametrize("seed", range(20))
def test_step_units_launches_random_models(lib, seed):
    # random models of 1-400 units mixing batchable and non-batchable units:
    # the library's count equals the rule restated above
    import numpy as np
    from sharded_fsdp_reduce_gb300 import _lib as E
    rng = np.random.default_rng(seed)
    specs = []
    for _ in range(int(rng.integers(1, 401))):
        world = int(rng.choice([1, 2, 3, 4, 8]))
        r = rng.random()
        P = 0 if r < 0.03 else (int(rng.integers(1 << 24, (1 << 24) + 64)) // world * world if r < 0.06
                                else int(rng.integers(1, 5000)) * world)
        specs.append((P, world, int(rng.integers(1, world + 1)), bool(rng.random() < 0.05)))
    gathers = int(rng.integers(0, 3))
    arr, keep = _fake_units(E, specs)
    hp = E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
    out = ctypes.c_int64(-1)
    assert lib.fsdp_step_units_launches(arr, len(specs), ctypes.byref(hp), gathers, 0, ctypes.byref(out)) == E.FSDP_OK
    assert out.value == _expected_launches(specs, gathers)


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host-only: fake addresses need a machine without a GPU")
def test_a_unit_may_not_read_what_another_unit_writes(lib):
    # units run at the same time (side streams, batched launches): a unit
    # whose gradients lie in another unit's master, state, shard or gathered
    # buffer would race, so the model is refused; gradients shared by two
    # units (both only read them) are fine
    from sharded_fsdp_reduce_gb300 import _lib as E
    hp = E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
    out = ctypes.c_int64(-1)
    small = (50000, 8, 8, False)

    def count(arr, n, ex=False):
        if ex:
            cfg = E.FsdpStepConfig(0, 0, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
            return lib.fsdp_step_units_ex_launches(arr, n, ctypes.byref(cfg), 1, ctypes.byref(out))
        return lib.fsdp_step_units_launches(arr, n, ctypes.byref(hp), 1, 0, ctypes.byref(out))

    for ex in (False, True):
        arr, keep = _fake_units(E, [small] * 3, ex=ex)
        assert count(arr, 3, ex) == E.FSDP_OK and out.value == 2
        g1 = ctypes.cast(arr[1].grads, ctypes.POINTER(ctypes.c_void_p))
        written = (arr[0].param, arr[0].state0, arr[0].shard_out) if ex else \
            (arr[0].master, arr[0].exp_avg, arr[0].shard_out)
        fulls0 = ctypes.cast(arr[0].full_bufs, ctypes.POINTER(ctypes.c_void_p))
        for target in (*written, fulls0[3], written[1] + 2 * 1000):  # starts inside, or at, a written range
            saved = g1[5]
            g1[5] = target
            assert count(arr, 3, ex) == E.FSDP_ERR_INVALID_ARG, (ex, hex(target))
            g1[5] = saved
        # the range just before unit 0's master, ending where it starts: no overlap
        g1[5] = written[0] - 2 * 50000
        assert count(arr, 3, ex) == E.FSDP_OK
        # unit 2 reads unit 1's gradients (read only): allowed
        g2 = ctypes.cast(arr[2].grads, ctypes.POINTER(ctypes.c_void_p))
        for q in range(8):
            g2[q] = g1[q]
        assert count(arr, 3, ex) == E.FSDP_OK and out.value == 2
    assert lib.fsdp_last_cuda_error() == 0


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host-only: fake addresses need a machine without a GPU")
def test_step_plan_validates_once_and_checks_only_the_scalars_per_launch(lib):
    from sharded_fsdp_reduce_gb300 import _lib as E
    small = (50000, 8, 8, False)
    plan = ctypes.c_void_p(123)
    # invalid models: refused at creation, the handle cleared
    assert lib.fsdp_step_plan_create(None, 0, 1, 0, None, None, None) == E.FSDP_ERR_INVALID_ARG
    assert lib.fsdp_step_plan_create(None, 1, 1, 0, None, None, ctypes.byref(plan)) == E.FSDP_ERR_INVALID_ARG
    assert plan.value is None
    arr, keep = _fake_units(E, [small, small])
    arr[1].exp_avg = arr[0].master                                        # two units writing one buffer
    assert lib.fsdp_step_plan_create(arr, 2, 1, 0, None, None, ctypes.byref(plan)) == E.FSDP_ERR_INVALID_ARG
    assert plan.value is None
    assert lib.fsdp_step_plan_create(arr, 1, 1, 0, None, FAKE + 2, ctypes.byref(plan)) == E.FSDP_ERR_ALIGNMENT
    # a valid model: created without touching a device
    arr, keep = _fake_units(E, [small] * 3)
    assert lib.fsdp_step_plan_create(arr, 3, 1, 0, None, None, ctypes.byref(plan)) == E.FSDP_OK and plan.value
    bad = [E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 0, 1.0),            # step 0
           E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 0.0),            # grad_scale 0
           E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, float("inf"))]
    for hp in bad:
        assert lib.fsdp_step_plan_launch(plan, ctypes.byref(hp), None) == E.FSDP_ERR_INVALID_ARG
    assert lib.fsdp_step_plan_launch(plan, None, None) == E.FSDP_ERR_INVALID_ARG
    cfg = E.FsdpStepConfig(0, 0, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
    assert lib.fsdp_step_plan_launch_ex(plan, ctypes.byref(cfg), None) == E.FSDP_ERR_INVALID_ARG  # not a variant plan
    assert lib.fsdp_last_cuda_error() == 0                                   # nothing was launched
    assert lib.fsdp_step_plan_destroy(plan) == E.FSDP_OK
    assert lib.fsdp_step_plan_destroy(None) == E.FSDP_OK
    # a variant plan: the launch's optimizer and reduction dtype are checked
    arr, keep = _fake_units(E, [small] * 2, ex=True)
    assert lib.fsdp_step_plan_create_ex(arr, 2, ctypes.byref(cfg), 1, None, None, ctypes.byref(plan)) == E.FSDP_OK
    other = E.FsdpStepConfig(2, 0, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)      # Adamax
    assert lib.fsdp_step_plan_launch_ex(plan, ctypes.byref(other), None) == E.FSDP_ERR_INVALID_ARG
    f16 = E.FsdpStepConfig(0, 2, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)        # fp16 sum of bf16 gradients
    assert lib.fsdp_step_plan_launch_ex(plan, ctypes.byref(f16), None) == E.FSDP_ERR_UNSUPPORTED_DTYPE
    hp = E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
    assert lib.fsdp_step_plan_launch(plan, ctypes.byref(hp), None) == E.FSDP_ERR_INVALID_ARG  # not an AdamW plan
    assert lib.fsdp_last_cuda_error() == 0
    assert lib.fsdp_step_plan_destroy(plan) == E.FSDP_OK


def test_running_out_of_host_memory_is_a_status_not_an_abort(tmp_path):
    # a model the library cannot even hold its bookkeeping for (2^31 - 1
    # units): every call that plans a model returns FSDP_ERR_HOST_MEMORY and
    # the process goes on. Run in a child whose address space is capped, so
    # that the allocation fails whatever the machine's overcommit policy.
    import subprocess
    import sys
    code = r"""
import ctypes, resource, sys
resource.setrlimit(resource.RLIMIT_AS, (16 << 30, 16 << 30))
sys.path.insert(0, ROOT)
from sharded_fsdp_reduce_gb300 import _lib as E
lib = E.load()
hp = E.FsdpAdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
cfg = E.FsdpStepConfig(0, 0, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
arr, arr_ex = (E.FsdpUnit * 1)(), (E.FsdpUnitEx * 1)()
n = 2**31 - 1
out, handle = ctypes.c_int64(-1), ctypes.c_void_p(None)
got = [lib.fsdp_step_units_launches(arr, n, ctypes.byref(hp), 1, 0, ctypes.byref(out)),
       lib.fsdp_step_units_ex_launches(arr_ex, n, ctypes.byref(cfg), 1, ctypes.byref(out)),
       lib.fsdp_step_units(arr, n, ctypes.byref(hp), 1, 0, None, None, None),
       lib.fsdp_step_units_ex(arr_ex, n, ctypes.byref(cfg), 1, None, None, None),
       lib.fsdp_step_plan_create(arr, n, 1, 0, None, None, ctypes.byref(handle)),
       lib.fsdp_step_plan_create_ex(arr_ex, n, ctypes.byref(cfg), 1, None, None, ctypes.byref(handle)),
       lib.fsdp_step_graph_create(arr, n, 1, 0, None, None, ctypes.byref(handle))]
print(got, out.value, handle.value)
""".replace("ROOT", repr(ROOT))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == "[5, 5, 5, 5, 5, 5, 5] -1 None", r.stdout
