"""One FSDP unit (FlatParameter) with N emulated ranks in one GPU's memory,
and its stream-ordered step.

The buffers are plain torch allocations; every operation on them is a call
into the CUDA library. Per rank q: its flat gradient buffer (P_pad elements of
the gradient dtype) and its gathered full-parameter buffer (P_pad elements of
the compute dtype). Shared by all ranks, as the concatenation of their shards:
the fp32 master weights, exp_avg (m), exp_avg_sq (v) and the compute-dtype
shards (shard_out); rank r's shard is [r*S, (r+1)*S).

Offload mode (state_on_host=True): master, exp_avg and exp_avg_sq live in
pinned host memory instead of HBM ("FSDP (Fully Sharded Data Parallel)", "CPU
Offloading"; "fairseq ... FSDP 实战指南", --cpu-offload keeps the optimizer
state and the FP32 copy of the model on the CPU). The same update kernel
reads and writes them in place over the host link; the gradients, the
compute-dtype shards and the gathered buffers stay in HBM.

The step of one unit ("FSDP (Fully Sharded Data Parallel)", "The Per-Layer
Communication"; "Fully Sharded Data Parallel: faster AI training with fewer
GPUs", "From all-reduce to sharded parameters"): the gradients are
reduce-scattered, each rank's shard is updated by AdamW and cast, and the
updated shards are all-gathered for the next forward (and, with
reshard-after-forward, once more for the backward).
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import torch

from .fsdp import (AdamWHParams, UnitDescs, View, fsdp_all_gather, fsdp_flatten_pad, fsdp_reduce_scatter_adam_cast,
                   fsdp_reduce_scatter_adam_cast_gather, fsdp_step_units, fsdp_unflatten_views)


class FlatParamUnit:
    def __init__(self, params: Sequence[Tuple[str, Tuple[int, ...]]], world: int, grad_dtype: torch.dtype,
                 out_dtype: torch.dtype, device="cuda", n_full: Optional[int] = None,
                 state_on_host: bool = False):
        self.names = [n for n, _ in params]
        self.shapes = [tuple(s) for _, s in params]
        self.world = int(world)
        self.views, self.padded_numel = fsdp_unflatten_views(self.shapes, self.world)
        self.numel = sum(math.prod(s) for s in self.shapes)
        self.shard_numel = self.padded_numel // self.world
        self.device = torch.device(device)
        P = self.padded_numel
        self.grads = [torch.zeros(P, dtype=grad_dtype, device=self.device) for _ in range(self.world)]
        self.state_on_host = bool(state_on_host)
        if self.state_on_host:
            state = [torch.zeros(P, dtype=torch.float32, pin_memory=True) for _ in range(3)]
        else:
            state = [torch.zeros(P, dtype=torch.float32, device=self.device) for _ in range(3)]
        self.master, self.exp_avg, self.exp_avg_sq = state
        self.shard_out = torch.zeros(P, dtype=out_dtype, device=self.device)
        nf = self.world if n_full is None else int(n_full)
        self.full = [torch.zeros(P, dtype=out_dtype, device=self.device) for _ in range(nf)]
        self._host = None

    # ---------------------------------------------------------------- set-up

    def load_master(self, tensors: Sequence[torch.Tensor], stream=None) -> None:
        """Flatten the unit's initial fp32 parameters into the master buffer."""
        if not self.state_on_host:
            fsdp_flatten_pad(list(tensors), self.world, out=self.master, stream=stream)
            return
        flat, _ = fsdp_flatten_pad(list(tensors), self.world, stream=stream)
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        with torch.cuda.stream(s):
            self.master.copy_(flat, non_blocking=True)
            flat.record_stream(s)

    def load_grad(self, rank: int, tensors: Sequence[torch.Tensor], stream=None) -> None:
        """Flatten rank ``rank``'s per-parameter gradients into its flat buffer (pad zeroed)."""
        fsdp_flatten_pad(list(tensors), self.world, out=self.grads[rank], stream=stream)

    def param_views(self, flat: torch.Tensor) -> Dict[str, torch.Tensor]:
        """The original parameters as views into a flat buffer (pad not visible)."""
        return {n: flat.narrow(0, v.offset, v.numel).view(v.shape) for n, v in zip(self.names, self.views)}

    # ---------------------------------------------------------------- the step

    def reduce_scatter_adam_cast(self, hp: AdamWHParams, rank_begin: int = 0, rank_end: Optional[int] = None,
                                 nonfinite_count: Optional[torch.Tensor] = None, stream=None) -> None:
        fsdp_reduce_scatter_adam_cast(self.grads, self.master, self.exp_avg, self.exp_avg_sq, self.shard_out,
                                      hp, rank_begin, rank_end, nonfinite_count, stream)

    def all_gather(self, stream=None) -> None:
        fsdp_all_gather(self.shard_out, self.full, self.world, stream)

    def step(self, hp: AdamWHParams, gathers: int = 1, nonfinite_count: Optional[torch.Tensor] = None,
             stream=None, fuse_gather: bool = False) -> None:
        """Reduce-scatter + AdamW + cast, then ``gathers`` all-gathers, in stream order.

        gathers=2 is reshard-after-forward (gathered before forward and again
        before backward), gathers=1 the no-reshard mode. With fuse_gather the
        first gather is written by the update kernel itself."""
        if fuse_gather and gathers >= 1:
            fsdp_reduce_scatter_adam_cast_gather(self.grads, self.master, self.exp_avg, self.exp_avg_sq,
                                                 self.shard_out, self.full, hp, nonfinite_count=nonfinite_count,
                                                 stream=stream)
            gathers -= 1
        else:
            self.reduce_scatter_adam_cast(hp, nonfinite_count=nonfinite_count, stream=stream)
        for _ in range(gathers):
            self.all_gather(stream)

    def step_from_host(self, host_grads: Sequence[torch.Tensor], host_out: Optional[torch.Tensor], hp: AdamWHParams,
                       gathers: int = 1, nonfinite_count: Optional[torch.Tensor] = None,
                       host_nonfinite: Optional[torch.Tensor] = None) -> None:
        """One step whose N gradient buffers come from pinned host memory.
        Its results go back to pinned host memory as asked: host_out receives
        the compute-dtype parameters (shard_out, all ranks' shards);
        host_nonfinite receives the step's count of non-finite averaged
        gradients (nonfinite_count is then required; it is zeroed first).
        Asynchronous; consecutive calls overlap: the host-to-device copy of a
        step runs on its own stream into a second set of gradient buffers
        while the previous step's kernels and device-to-host copies run. The
        host buffers are complete once the current stream is synchronized."""
        if host_nonfinite is not None and nonfinite_count is None:
            raise ValueError("host_nonfinite needs a device nonfinite_count")
        if self._host is None:
            self._host = _HostPipeline(self)
        self._host.step(host_grads, host_out, hp, gathers, nonfinite_count, host_nonfinite)

    # ---------------------------------------------------------------- snapshot / resume

    def state_dict(self, rank: Optional[int] = None) -> Dict[str, torch.Tensor]:
        """Host copies of the optimizer state: the whole unit (rank=None), or
        rank r's shard [r*S, (r+1)*S) alone, the per-rank file of a sharded
        checkpoint ("fairseq ... FSDP 实战指南", --use-sharded-state: each
        rank saves its own shard). Synchronizes with the current stream."""
        lo, hi = self._range(rank)
        if self.device.type == "cuda":
            torch.cuda.current_stream(self.device).synchronize()
        return {name: getattr(self, name)[lo:hi].detach().to("cpu", copy=True)
                for name in ("master", "exp_avg", "exp_avg_sq")}

    def load_state_dict(self, state: Dict[str, torch.Tensor], rank: Optional[int] = None) -> None:
        """Restore what state_dict(rank) returned (rank=None: the whole unit)."""
        lo, hi = self._range(rank)
        for name in ("master", "exp_avg", "exp_avg_sq"):
            src = state[name]
            if src.dtype != torch.float32 or src.numel() != hi - lo:
                raise ValueError(f"{name} must be float32 with {hi - lo} elements")
            getattr(self, name)[lo:hi].copy_(src.reshape(-1))

    def _range(self, rank: Optional[int]) -> Tuple[int, int]:
        if rank is None:
            return 0, self.padded_numel
        if not 0 <= int(rank) < self.world:
            raise ValueError(f"rank must be in [0, {self.world})")
        S = self.shard_numel
        return int(rank) * S, (int(rank) + 1) * S

    def step_bytes(self, gathers: int = 1) -> Tuple[int, int]:
        """Algorithmic bytes of one step: (fused kernel, all-gathers)."""
        gs = self.grads[0].element_size()
        os_ = self.shard_out.element_size()
        P = self.padded_numel
        rsa = P * (self.world * gs + 3 * (4 + 4) + os_)
        ag = gathers * P * os_ * (1 + len(self.full))
        return rsa, ag


class _HostPipeline:
    """Stream plumbing of FlatParamUnit.step_from_host: two gradient-buffer
    sets, a copy-in stream, a copy-out stream, and events that order each
    buffer's reuse after the work that reads it."""

    def __init__(self, unit: FlatParamUnit):
        self.unit = unit
        self.sets = [unit.grads, [torch.empty_like(g) for g in unit.grads]]
        self.read_done = [None, None]   # compute finished reading set k
        self.out_read = None            # copy-out finished reading shard_out
        self.copy_in = torch.cuda.Stream(device=unit.device)
        self.copy_out = torch.cuda.Stream(device=unit.device)
        self.i = 0

    def step(self, host_grads, host_out, hp, gathers, nonfinite_count, host_nonfinite):
        u = self.unit
        if len(host_grads) != u.world:
            raise ValueError(f"need {u.world} host gradient buffers")
        k = self.i % 2
        gset = self.sets[k]
        compute = torch.cuda.current_stream(u.device)
        if self.read_done[k] is not None:
            self.copy_in.wait_event(self.read_done[k])
        with torch.cuda.stream(self.copy_in):
            for g, h in zip(gset, host_grads):
                g.copy_(h, non_blocking=True)
        compute.wait_stream(self.copy_in)
        if self.out_read is not None:
            compute.wait_event(self.out_read)   # shard_out / the counter are about to be rewritten
        if host_nonfinite is not None:
            nonfinite_count.zero_()
        fsdp_reduce_scatter_adam_cast(gset, u.master, u.exp_avg, u.exp_avg_sq, u.shard_out, hp,
                                      nonfinite_count=nonfinite_count, stream=compute)
        self.read_done[k] = compute.record_event()
        self.copy_out.wait_event(self.read_done[k])
        with torch.cuda.stream(self.copy_out):
            if host_out is not None:
                host_out.copy_(u.shard_out, non_blocking=True)
            if host_nonfinite is not None:
                host_nonfinite.copy_(nonfinite_count, non_blocking=True)
        self.out_read = self.copy_out.record_event()
        for _ in range(gathers):
            fsdp_all_gather(u.shard_out, u.full, u.world, stream=compute)
        compute.wait_stream(self.copy_out)  # the step ends when its result is on the host
        self.i += 1


class UnitSequence:
    """The FSDP units of a model, stepped in order by one call into the
    library (fsdp_step_units): per unit the fused update and its all-gathers,
    all on one stream, with the per-unit loop in native code."""

    def __init__(self, units: Sequence[FlatParamUnit]):
        self.units = list(units)
        self.descs = UnitDescs(self.units)

    def step(self, hp: AdamWHParams, gathers: int = 1, nonfinite_count: Optional[torch.Tensor] = None,
             stream=None, fuse_gather: bool = False) -> None:
        fsdp_step_units(self.descs, hp, gathers, fuse_gather, nonfinite_count, stream)

    def step_bytes(self, gathers: int = 1) -> Tuple[int, int]:
        """Algorithmic bytes of one model step: (fused kernels, all-gathers)."""
        rsa = ag = 0
        for u in self.units:
            a, b = u.step_bytes(gathers)
            rsa += a
            ag += b
        return rsa, ag
