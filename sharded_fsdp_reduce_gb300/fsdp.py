"""Python binding of the C ABI in include/fsdp.h, one function per entry point
with the same name. Argument marshalling only: every step of the path runs in
the CUDA library; these functions turn torch tensors into device pointers and
sizes, pass the current CUDA stream, and raise FsdpError on a non-OK status.
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import List, Optional, Sequence, Tuple

import torch

from . import _lib
from ._lib import FsdpAdamwHparams, FsdpStepConfig, FsdpUnit, FsdpUnitEx, FsdpView

__all__ = [
    "AdamWHParams", "StepConfig", "OPTIMIZERS", "FsdpError", "View", "fsdp_reduce_scatter_step",
    "fsdp_padded_numel", "fsdp_unflatten_views", "fsdp_flatten_pad",
    "fsdp_reduce_scatter_adam_cast", "fsdp_reduce_scatter_adam_cast_gather", "fsdp_all_gather",
    "fsdp_status_string",
    "fsdp_last_cuda_error", "fsdp_take_wait_timeouts", "fsdp_check_bounded_wait", "dtype_code",
    "UnitDescs", "fsdp_step_units", "fsdp_step_units_ex", "StepGraph", "StepPlan",
    "fsdp_step_units_launches", "fsdp_step_units_ex_launches",
]

_DTYPES = {torch.float32: _lib.FSDP_F32, torch.bfloat16: _lib.FSDP_BF16, torch.float16: _lib.FSDP_F16}


class FsdpError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = fsdp_status_string(status)
        if status == _lib.FSDP_ERR_CUDA:
            msg += f" (cudaError {fsdp_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")
        self.status = status


@dataclasses.dataclass(frozen=True)
class AdamWHParams:
    lr: float
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    step: int = 1
    grad_scale: float = 1.0

    def to_c(self) -> FsdpAdamwHparams:
        return FsdpAdamwHparams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay,
                                int(self.step), self.grad_scale)


OPTIMIZERS = {"adamw": _lib.FSDP_OPT_ADAMW, "sgd": _lib.FSDP_OPT_SGD, "adamax": _lib.FSDP_OPT_ADAMAX,
              "adadelta": _lib.FSDP_OPT_ADADELTA}


@dataclasses.dataclass(frozen=True)
class StepConfig:
    """fsdp_step_config: optimizer ("adamw", "sgd", "adamax", "adadelta"), the
    reduction dtype (None = fp32 reduce-scatter, else the gradient dtype) and
    the hyperparameters (beta1 is SGD's momentum and Adadelta's rho)."""
    optimizer: str
    lr: float
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    step: int = 1
    grad_scale: float = 1.0
    reduce_dtype: Optional[torch.dtype] = None

    def to_c(self) -> FsdpStepConfig:
        rd = _lib.FSDP_F32 if self.reduce_dtype is None else dtype_code(self.reduce_dtype)
        return FsdpStepConfig(OPTIMIZERS[self.optimizer], rd, self.lr, self.beta1, self.beta2, self.eps,
                              self.weight_decay, int(self.step), self.grad_scale)


@dataclasses.dataclass(frozen=True)
class View:
    offset: int
    numel: int
    shape: Tuple[int, ...]


def dtype_code(dt: torch.dtype) -> int:
    try:
        return _DTYPES[dt]
    except KeyError:
        raise TypeError(f"unsupported dtype {dt}; expected float32, bfloat16 or float16") from None


def _check(status: int, where: str) -> None:
    if status != _lib.FSDP_OK:
        raise FsdpError(status, where)


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _on_current_device(t: torch.Tensor, name: str) -> None:
    """The kernels run on the current device: a tensor of another GPU would
    reach them as a foreign address, so it is refused here."""
    d, cur = t.get_device(), torch.cuda.current_device()
    if d != cur:
        raise ValueError(f"{name} is on cuda:{d} but the current device is cuda:{cur}")


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    _on_current_device(t, name)
    return t.data_ptr()


def _mem(t: torch.Tensor, name: str) -> int:
    """A buffer the update kernels stream through: CUDA memory, or page-locked
    host memory (mapped into the device's address space; the kernel then
    reads and writes it over the host link, the offload mode)."""
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or (t.device.type == "cpu" and t.is_pinned())):
        raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.is_cuda:
        _on_current_device(t, name)
    return t.data_ptr()


def _ptrs(ts: Sequence[torch.Tensor], name: str, host_ok: bool = False):
    get = _mem if host_ok else _dev
    return (ctypes.c_void_p * len(ts))(*[get(t, f"{name}[{i}]") for i, t in enumerate(ts)])


def _grad_dtype(grads: Sequence[torch.Tensor], P_pad: int, name: str = "grads") -> torch.dtype:
    """The gradients' common dtype, after checking every buffer's length and dtype."""
    gdt = grads[0].dtype if len(grads) else torch.bfloat16
    for i, g in enumerate(grads):
        if g.numel() != P_pad or g.dtype != gdt:
            raise ValueError(f"{name}[{i}] must hold {P_pad} elements of {gdt}")
    return gdt


def _check_fp32_state(P_pad: int, prefix: str = "", **bufs: torch.Tensor) -> None:
    for name, t in bufs.items():
        if t.dtype != torch.float32 or t.numel() != P_pad:
            raise ValueError(f"{prefix}{name} must be float32 with {P_pad} elements")


def _counter(t: Optional[torch.Tensor], name: str = "nonfinite_count"):
    """Device address of an optional counter (a CUDA int32/uint32 tensor): the
    non-finite gradient count, or a call's count of bounded waits that gave up."""
    if t is None:
        return None
    if t.dtype not in (torch.int32, torch.uint32) or t.numel() < 1:
        raise ValueError(f"{name} must be a CUDA int32/uint32 tensor")
    return _dev(t, name)


def _views(c_views, n) -> List[View]:
    return [View(int(c_views[k].offset), int(c_views[k].numel),
                 tuple(int(c_views[k].shape[d]) for d in range(c_views[k].ndim))) for k in range(n)]


def fsdp_status_string(status: int) -> str:
    return _lib.load().fsdp_status_string(int(status)).decode()


def fsdp_last_cuda_error() -> int:
    return int(_lib.load().fsdp_last_cuda_error())


def fsdp_take_wait_timeouts() -> int:
    """Bounded in-kernel waits that gave up since the last call, on the whole
    device (synchronizes the device). A call's own count: its wait_timeouts."""
    n = ctypes.c_uint32(0)
    _check(_lib.load().fsdp_take_wait_timeouts(ctypes.byref(n)), "fsdp_take_wait_timeouts")
    return int(n.value)


def fsdp_check_bounded_wait(limit_cycles: int, stream: Optional[torch.cuda.Stream] = None,
                            wait_timeouts: Optional[torch.Tensor] = None) -> None:
    """Self-test of the bounded waits' failure path: one kernel waits on a
    barrier that nothing completes and gives up after about limit_cycles SM
    cycles; fsdp_take_wait_timeouts() then counts it, and so does
    wait_timeouts (a CUDA int32/uint32 counter) when given. Asynchronous."""
    _check(_lib.load().fsdp_check_bounded_wait(int(limit_cycles), _counter(wait_timeouts, "wait_timeouts"),
                                               _stream(stream)), "fsdp_check_bounded_wait")


def fsdp_padded_numel(numel: int, world: int) -> int:
    return int(_lib.load().fsdp_padded_numel(int(numel), int(world)))


def fsdp_unflatten_views(shapes: Sequence[Sequence[int]], world: int) -> Tuple[List[View], int]:
    """Views (offset, numel, shape) of the parameters in a FlatParameter and its padded length."""
    n = len(shapes)
    dims = [int(d) for s in shapes for d in s]
    c_dims = (ctypes.c_int64 * max(len(dims), 1))(*dims)
    c_nd = (ctypes.c_int32 * max(n, 1))(*[len(s) for s in shapes])
    c_views = (FsdpView * max(n, 1))()
    padded = ctypes.c_int64(0)
    _check(_lib.load().fsdp_unflatten_views(c_dims, c_nd, n, int(world), c_views, ctypes.byref(padded)),
           "fsdp_unflatten_views")
    return _views(c_views, n), int(padded.value)


def fsdp_flatten_pad(tensors: Sequence[torch.Tensor], world: int, out: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, List[View]]:
    """Flatten the tensors (one dtype, CUDA, contiguous) into a zero-padded flat buffer."""
    if not tensors:
        raise ValueError("fsdp_flatten_pad needs at least one tensor")
    dt = tensors[0].dtype
    if any(t.dtype != dt for t in tensors):
        raise TypeError("all tensors of a unit must share one dtype")
    total = sum(t.numel() for t in tensors)
    padded = fsdp_padded_numel(total, world)
    if out is None:
        out = torch.empty(padded, dtype=dt, device=tensors[0].device)
    elif out.dtype != dt or out.numel() != padded:
        raise ValueError(f"out must hold {padded} elements of {dt}")
    n = len(tensors)
    c_views = (FsdpView * n)()
    numels = (ctypes.c_int64 * n)(*[t.numel() for t in tensors])
    _check(_lib.load().fsdp_flatten_pad(_ptrs(tensors, "tensors"), numels, n, dtype_code(dt), int(world),
                                        _dev(out, "out"), out.numel(), c_views, _stream(stream)),
           "fsdp_flatten_pad")
    return out, _views(c_views, n)


def fsdp_reduce_scatter_adam_cast(grads: Sequence[torch.Tensor], master: torch.Tensor, exp_avg: torch.Tensor,
                                  exp_avg_sq: torch.Tensor, shard_out: torch.Tensor, hparams: AdamWHParams,
                                  rank_begin: int = 0, rank_end: Optional[int] = None,
                                  nonfinite_count: Optional[torch.Tensor] = None,
                                  stream: Optional[torch.cuda.Stream] = None) -> None:
    """Fused reduce-scatter + AdamW + cast for the emulated ranks [rank_begin, rank_end).

    grads: N tensors (or the rows of an [N, P_pad] tensor) of one dtype.
    master / exp_avg / exp_avg_sq: fp32 [P_pad], updated in place.
    grads, master, exp_avg and exp_avg_sq may be pinned host tensors (the
    offload mode: the kernel streams them over the host link).
    shard_out: [P_pad] of the compute dtype, CUDA; rank r writes [r*S, (r+1)*S).
    nonfinite_count: optional CUDA uint32/int32 scalar, incremented by the
    number of non-finite averaged gradient elements.
    """
    world = len(grads)
    P_pad = master.numel()
    gdt = _grad_dtype(grads, P_pad)
    _check_fp32_state(P_pad, master=master, exp_avg=exp_avg, exp_avg_sq=exp_avg_sq)
    if shard_out.numel() != P_pad:
        raise ValueError(f"shard_out must hold {P_pad} elements")
    nf = _counter(nonfinite_count)
    hp = hparams.to_c()
    re = world if rank_end is None else int(rank_end)
    args = (_ptrs(grads, "grads", host_ok=True) if world else None, dtype_code(gdt), world, P_pad,
            _mem(master, "master"), _mem(exp_avg, "exp_avg"), _mem(exp_avg_sq, "exp_avg_sq"),
            _dev(shard_out, "shard_out"), dtype_code(shard_out.dtype), ctypes.byref(hp), int(rank_begin), re,
            nf, _stream(stream))
    _check(_lib.load().fsdp_reduce_scatter_adam_cast(*args), "fsdp_reduce_scatter_adam_cast")


def fsdp_reduce_scatter_adam_cast_gather(grads: Sequence[torch.Tensor], master: torch.Tensor,
                                         exp_avg: torch.Tensor, exp_avg_sq: torch.Tensor,
                                         shard_out: Optional[torch.Tensor], full_bufs: Sequence[torch.Tensor],
                                         hparams: AdamWHParams, rank_begin: int = 0,
                                         rank_end: Optional[int] = None,
                                         nonfinite_count: Optional[torch.Tensor] = None,
                                         stream: Optional[torch.cuda.Stream] = None) -> None:
    """The fused update with the all-gather fused in: as fsdp_reduce_scatter_adam_cast,
    and each updated element is also written to every buffer of full_bufs.
    shard_out may be None (not written)."""
    world = len(grads)
    P_pad = master.numel()
    if not full_bufs:
        raise ValueError("full_bufs must hold at least one buffer")
    odt = full_bufs[0].dtype
    for i, f in enumerate(full_bufs):
        if f.numel() != P_pad or f.dtype != odt:
            raise ValueError(f"full_bufs[{i}] must hold {P_pad} elements of {odt}")
    if shard_out is not None and (shard_out.numel() != P_pad or shard_out.dtype != odt):
        raise ValueError(f"shard_out must hold {P_pad} elements of {odt}")
    gdt = _grad_dtype(grads, P_pad)
    _check_fp32_state(P_pad, master=master, exp_avg=exp_avg, exp_avg_sq=exp_avg_sq)
    nf = _counter(nonfinite_count)
    hp = hparams.to_c()
    re = world if rank_end is None else int(rank_end)
    args = (_ptrs(grads, "grads", host_ok=True) if world else None, dtype_code(gdt), world, P_pad,
            _mem(master, "master"), _mem(exp_avg, "exp_avg"), _mem(exp_avg_sq, "exp_avg_sq"),
            _dev(shard_out, "shard_out") if shard_out is not None else None, dtype_code(odt),
            _ptrs(full_bufs, "full_bufs"), len(full_bufs), ctypes.byref(hp), int(rank_begin), re, nf,
            _stream(stream))
    _check(_lib.load().fsdp_reduce_scatter_adam_cast_gather(*args), "fsdp_reduce_scatter_adam_cast_gather")


def fsdp_reduce_scatter_step(grads: Sequence[torch.Tensor], param: torch.Tensor, state0: torch.Tensor,
                             state1: Optional[torch.Tensor], shard_out: Optional[torch.Tensor], config: StepConfig,
                             rank_begin: int = 0, rank_end: Optional[int] = None,
                             nonfinite_count: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None) -> None:
    """Variant step: fused reduce-scatter + (AdamW | SGD | Adamax | Adadelta) + cast.

    param/state0/state1: [P_pad], fp32 (then shard_out receives the cast) or
    all bf16/fp16 (then param is the shard and shard_out must be None).
    state1 is None for SGD. grads, param and the states may be pinned host
    tensors (offload mode)."""
    world = len(grads)
    P_pad = param.numel()
    gdt = _grad_dtype(grads, P_pad)
    sdt = param.dtype
    for name, t in (("state0", state0), ("state1", state1)):
        if t is not None and (t.dtype != sdt or t.numel() != P_pad):
            raise ValueError(f"{name} must hold {P_pad} elements of {sdt}")
    if shard_out is not None and shard_out.numel() != P_pad:
        raise ValueError(f"shard_out must hold {P_pad} elements")
    odt = shard_out.dtype if shard_out is not None else sdt
    nf = _counter(nonfinite_count)
    cfg = config.to_c()
    re = world if rank_end is None else int(rank_end)
    args = (_ptrs(grads, "grads", host_ok=True) if world else None, dtype_code(gdt), world, P_pad,
            _mem(param, "param"), _mem(state0, "state0"), _mem(state1, "state1") if state1 is not None else None,
            dtype_code(sdt), _dev(shard_out, "shard_out") if shard_out is not None else None, dtype_code(odt),
            ctypes.byref(cfg), int(rank_begin), re, nf, _stream(stream))
    _check(_lib.load().fsdp_reduce_scatter_step(*args), "fsdp_reduce_scatter_step")


def fsdp_all_gather(shard_out: torch.Tensor, full_bufs: Sequence[torch.Tensor], world: int,
                    stream: Optional[torch.cuda.Stream] = None, wait_timeouts: Optional[torch.Tensor] = None) -> None:
    """Copy the rank-ordered shards (shard_out, [P_pad]) into every full buffer.
    wait_timeouts: optional CUDA int32/uint32 counter, incremented by each of
    this call's bounded waits that gave up (non-zero: the copy is incomplete)."""
    P_pad = shard_out.numel()
    for i, f in enumerate(full_bufs):
        if f.numel() != P_pad or f.dtype != shard_out.dtype:
            raise ValueError(f"full_bufs[{i}] must hold {P_pad} elements of {shard_out.dtype}")
    _check(_lib.load().fsdp_all_gather(_dev(shard_out, "shard_out"), dtype_code(shard_out.dtype), int(world),
                                       P_pad, _ptrs(full_bufs, "full_bufs"), len(full_bufs),
                                       _counter(wait_timeouts, "wait_timeouts"), _stream(stream)),
           "fsdp_all_gather")


class UnitDescs:
    """The C descriptors of a sequence of FSDP units, built once for
    fsdp_step_units (fsdp_unit: fp32 master and AdamW state, built when every
    unit has them) and fsdp_step_units_ex (fsdp_unit_ex: any unit). A unit is
    any object holding FlatParamUnit's buffers: grads (N tensors), full
    (gathered buffers), master (the parameter), exp_avg and exp_avg_sq (the
    optimizer states; exp_avg_sq None for SGD), shard_out (for fp32 state;
    the parameter itself for bf16/fp16 state). The descriptors hold the
    buffers' addresses: build new ones if a unit's buffers are replaced.
    The units and the very tensors whose addresses are held are kept alive
    while the descriptors exist, so that a buffer replaced in a unit is not
    freed and its memory handed to another allocation while a plan or a
    captured step made from these descriptors still writes to it."""

    def __init__(self, units: Sequence):
        self.units = list(units)
        self.n = len(self.units)
        self.array_ex = (FsdpUnitEx * max(self.n, 1))()
        self.adamw = all(u.master.dtype == torch.float32 and u.exp_avg_sq is not None for u in self.units)
        self.array = (FsdpUnit * max(self.n, 1))() if self.adamw else None
        self._keep = []
        for k, u in enumerate(self.units):
            pre = f"units[{k}]."
            P = u.master.numel()
            gdt = _grad_dtype(u.grads, P, pre + "grads")
            sdt = u.master.dtype
            for name in ("exp_avg", "exp_avg_sq"):
                t = getattr(u, name)
                if t is not None and (t.dtype != sdt or t.numel() != P):
                    raise ValueError(f"{pre}{name} must hold {P} elements of {sdt}")
            lowp = sdt != torch.float32
            odt = sdt if lowp else u.shard_out.dtype
            if not lowp and u.shard_out.numel() != P:
                raise ValueError(f"{pre}shard_out must hold {P} elements")
            for i, f in enumerate(u.full):
                if f.numel() != P or f.dtype != odt:
                    raise ValueError(f"{pre}full[{i}] must hold {P} elements of {odt}")
            grads = _ptrs(u.grads, pre + "grads", host_ok=True)
            full = _ptrs(u.full, pre + "full") if u.full else None
            self._keep += [grads, full, list(u.grads), list(u.full), u.master, u.exp_avg, u.exp_avg_sq,
                           u.shard_out]
            param = _mem(u.master, pre + "master")
            s0 = _mem(u.exp_avg, pre + "exp_avg")
            s1 = _mem(u.exp_avg_sq, pre + "exp_avg_sq") if u.exp_avg_sq is not None else None
            out = None if lowp else _dev(u.shard_out, pre + "shard_out")
            e = self.array_ex[k]
            e.grads, e.full_bufs = ctypes.addressof(grads), ctypes.addressof(full) if full is not None else None
            e.param, e.state0, e.state1, e.shard_out = param, s0, s1, out
            e.padded_numel, e.world, e.n_full = P, len(u.grads), len(u.full)
            e.grad_dtype, e.state_dtype, e.out_dtype = dtype_code(gdt), dtype_code(sdt), dtype_code(odt)
            if self.adamw:
                d = self.array[k]
                d.grads, d.full_bufs = e.grads, e.full_bufs
                d.master, d.exp_avg, d.exp_avg_sq, d.shard_out = param, s0, s1, out
                d.padded_numel, d.world, d.n_full = P, len(u.grads), len(u.full)
                d.grad_dtype, d.out_dtype = dtype_code(gdt), dtype_code(odt)


def fsdp_step_units(units, hparams: AdamWHParams, gathers: int = 1, fuse_first_gather: bool = False,
                    nonfinite_count: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None, wait_timeouts: Optional[torch.Tensor] = None) -> None:
    """The step of a whole model in one call: for each unit in order, its
    fused reduce-scatter + AdamW + cast, then `gathers` all-gathers into its
    full buffers (the first written by the update kernel itself with
    fuse_first_gather). `units` is a UnitDescs or a sequence of units (then
    descriptors are built for this call). Every call validates every unit;
    StepPlan validates once for repeated steps."""
    descs = units if isinstance(units, UnitDescs) else UnitDescs(units)
    if not descs.adamw:
        raise ValueError("fsdp_step_units needs fp32 master and AdamW state in every unit; use fsdp_step_units_ex")
    nf = _counter(nonfinite_count)
    wt = _counter(wait_timeouts, "wait_timeouts")
    hp = hparams.to_c()
    _check(_lib.load().fsdp_step_units(descs.array, descs.n, ctypes.byref(hp), int(gathers),
                                       1 if fuse_first_gather else 0, nf, wt, _stream(stream)), "fsdp_step_units")


def fsdp_step_units_ex(units, config: StepConfig, gathers: int = 1, nonfinite_count: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None,
                       wait_timeouts: Optional[torch.Tensor] = None) -> None:
    """The variant step of a whole model in one call: for each unit in order,
    fsdp_reduce_scatter_step's update under `config`, then `gathers`
    all-gathers of its compute-dtype shards into its full buffers. `units` is
    a UnitDescs or a sequence of units."""
    descs = units if isinstance(units, UnitDescs) else UnitDescs(units)
    nf = _counter(nonfinite_count)
    wt = _counter(wait_timeouts, "wait_timeouts")
    cfg = config.to_c()
    _check(_lib.load().fsdp_step_units_ex(descs.array_ex, descs.n, ctypes.byref(cfg), int(gathers), nf, wt,
                                          _stream(stream)), "fsdp_step_units_ex")


def fsdp_step_units_launches(units, hparams: Optional[AdamWHParams] = None, gathers: int = 1,
                             fuse_first_gather: bool = False) -> int:
    """How many kernel launches fsdp_step_units makes for these units (small
    units batched); the units are validated, nothing is enqueued. Arguments
    as fsdp_step_units (hparams only validated; default lr 1e-3)."""
    descs = units if isinstance(units, UnitDescs) else UnitDescs(units)
    if not descs.adamw:
        raise ValueError("fsdp_step_units needs fp32 master and AdamW state in every unit; use the _ex query")
    hp = (hparams if hparams is not None else AdamWHParams(1e-3)).to_c()
    n = ctypes.c_int64(0)
    _check(_lib.load().fsdp_step_units_launches(descs.array, descs.n, ctypes.byref(hp), int(gathers),
                                                1 if fuse_first_gather else 0, ctypes.byref(n)),
           "fsdp_step_units_launches")
    return int(n.value)


def fsdp_step_units_ex_launches(units, config: StepConfig, gathers: int = 1) -> int:
    """How many kernel launches fsdp_step_units_ex makes for these units under
    `config` (small units batched); nothing is enqueued."""
    descs = units if isinstance(units, UnitDescs) else UnitDescs(units)
    cfg = config.to_c()
    n = ctypes.c_int64(0)
    _check(_lib.load().fsdp_step_units_ex_launches(descs.array_ex, descs.n, ctypes.byref(cfg), int(gathers),
                                                   ctypes.byref(n)), "fsdp_step_units_ex_launches")
    return int(n.value)


class _StepHandle:
    """A model step prepared once by the library (a captured graph or a
    validated plan) and launched with each step's scalars. The units'
    buffers must stay allocated (the library holds their addresses; the units
    are kept alive here)."""

    _CREATE, _CREATE_EX, _LAUNCH, _LAUNCH_EX, _DESTROY = "", "", "", "", ""

    def __init__(self, units, gathers: int = 1, fuse_first_gather: bool = False,
                 nonfinite_count: Optional[torch.Tensor] = None, config: Optional[StepConfig] = None,
                 wait_timeouts: Optional[torch.Tensor] = None):
        self.descs = units if isinstance(units, UnitDescs) else UnitDescs(units)
        self.config = config
        self._counters = (nonfinite_count, wait_timeouts)
        self._handle = ctypes.c_void_p(None)
        lib = _lib.load()
        nf, wt = _counter(nonfinite_count), _counter(wait_timeouts, "wait_timeouts")
        if config is None:
            if not self.descs.adamw:
                raise ValueError("an AdamW model step needs fp32 master and AdamW state in every unit")
            st = getattr(lib, self._CREATE)(self.descs.array, self.descs.n, int(gathers),
                                            1 if fuse_first_gather else 0, nf, wt, ctypes.byref(self._handle))
        else:
            if fuse_first_gather:
                raise ValueError("the variant step has no fused gather")
            cfg = config.to_c()
            st = getattr(lib, self._CREATE_EX)(self.descs.array_ex, self.descs.n, ctypes.byref(cfg), int(gathers),
                                               nf, wt, ctypes.byref(self._handle))
        _check(st, self._CREATE)

    def launch(self, hparams, stream: Optional[torch.cuda.Stream] = None) -> None:
        """Run one step: hparams is AdamWHParams for an AdamW step, a
        StepConfig of the same optimizer for a variant step."""
        if not self._handle:
            raise RuntimeError("the model step was destroyed")
        lib = _lib.load()
        c = hparams.to_c()
        name = self._LAUNCH if self.config is None else self._LAUNCH_EX
        _check(getattr(lib, name)(self._handle, ctypes.byref(c), _stream(stream)), name)

    def close(self) -> None:
        if self._handle:
            _check(getattr(_lib.load(), self._DESTROY)(self._handle), self._DESTROY)
            self._handle = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class StepGraph(_StepHandle):
    """A model step captured as a CUDA graph (fsdp_step_graph_create, or
    fsdp_step_graph_create_ex when `config` is given): one launch runs every
    unit's update and gathers, with the scalars of the step given to
    launch()."""

    _CREATE, _CREATE_EX = "fsdp_step_graph_create", "fsdp_step_graph_create_ex"
    _LAUNCH, _LAUNCH_EX, _DESTROY = "fsdp_step_graph_launch", "fsdp_step_graph_launch_ex", "fsdp_step_graph_destroy"


class StepPlan(_StepHandle):
    """A model step validated once (fsdp_step_plan_create, or
    fsdp_step_plan_create_ex when `config` is given): launch() enqueues the
    launches fsdp_step_units would make, checking only the step's scalars."""

    _CREATE, _CREATE_EX = "fsdp_step_plan_create", "fsdp_step_plan_create_ex"
    _LAUNCH, _LAUNCH_EX, _DESTROY = "fsdp_step_plan_launch", "fsdp_step_plan_launch_ex", "fsdp_step_plan_destroy"
