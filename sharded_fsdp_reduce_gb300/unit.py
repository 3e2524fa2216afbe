"""One FSDP unit (FlatParameter) with N emulated ranks in one GPU's memory,
and its stream-ordered step.

The buffers are plain torch allocations; every operation on them is a call
into the CUDA library. Per rank q: its flat gradient buffer (P_pad elements of
the gradient dtype) and its gathered full-parameter buffer (P_pad elements of
the compute dtype). Shared by all ranks, as the concatenation of their shards:
the fp32 master weights, exp_avg (m), exp_avg_sq (v) and the compute-dtype
shards (shard_out); rank r's shard is [r*S, (r+1)*S).

Optimizers and precisions: AdamW with fp32 master and state (the fused
kernel, optionally with the first gather fused in) by default; with
optimizer "sgd", "adamax" or "adadelta", or state_dtype bf16/fp16, the unit
holds that optimizer's state (one buffer for SGD, two otherwise) in that
dtype and steps through the variant kernel (fsdp_reduce_scatter_step). With
bf16/fp16 state there is no fp32 master: the parameter buffer is the rank's
compute-dtype shard and shard_out is that same buffer.

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
from typing import Dict, Optional, Sequence, Tuple

import torch

from .fsdp import (OPTIMIZERS, AdamWHParams, StepConfig, StepGraph, StepPlan, UnitDescs, fsdp_all_gather,
                   fsdp_flatten_pad, fsdp_reduce_scatter_adam_cast, fsdp_reduce_scatter_adam_cast_gather,
                   fsdp_reduce_scatter_step, fsdp_step_units, fsdp_step_units_ex, fsdp_step_units_ex_launches,
                   fsdp_step_units_launches, fsdp_unflatten_views)


class FlatParamUnit:
    """One FSDP unit's buffers and step.

    params: (name, shape) per original parameter, in registration order (the
    flatten order). world: N emulated ranks. grad_dtype / out_dtype: the
    gradients' dtype and the compute dtype of the shards and gathered
    buffers. n_full: gathered buffers (default N, one per rank).
    state_on_host: fp32 master and state in pinned host memory (offload).
    optimizer / state_dtype: the update ("adamw", "sgd", "adamax",
    "adadelta") and the dtype of the parameter and state (fp32 keeps an fp32
    master beside the compute-dtype shard; bf16/fp16 keeps none)."""

    def __init__(self, params: Sequence[Tuple[str, Tuple[int, ...]]], world: int, grad_dtype: torch.dtype,
                 out_dtype: torch.dtype, device="cuda", n_full: Optional[int] = None,
                 state_on_host: bool = False, optimizer: str = "adamw",
                 state_dtype: torch.dtype = torch.float32):
        self.names = [n for n, _ in params]
        self.shapes = [tuple(s) for _, s in params]
        self.world = int(world)
        self.views, self.padded_numel = fsdp_unflatten_views(self.shapes, self.world)
        self.numel = sum(math.prod(s) for s in self.shapes)
        self.shard_numel = self.padded_numel // self.world
        self.device = torch.device(device)
        P = self.padded_numel
        self.grads = [torch.zeros(P, dtype=grad_dtype, device=self.device) for _ in range(self.world)]
        if optimizer not in OPTIMIZERS:
            raise ValueError(f"optimizer must be one of {sorted(OPTIMIZERS)}")
        self.optimizer = optimizer
        self.state_dtype = state_dtype
        lowp = state_dtype != torch.float32
        if lowp and out_dtype != state_dtype:
            raise ValueError("with bf16/fp16 state the compute dtype is the state dtype (the parameter is the shard)")
        if lowp and state_on_host:
            raise ValueError("a bf16/fp16 parameter is the gathered shard and stays in HBM: no offload")
        self.state_on_host = bool(state_on_host)

        def state_buf():
            if self.state_on_host:
                return torch.zeros(P, dtype=state_dtype, pin_memory=True)
            return torch.zeros(P, dtype=state_dtype, device=self.device)

        self.master = state_buf()
        self.exp_avg = state_buf()
        self.exp_avg_sq = None if optimizer == "sgd" else state_buf()
        self.shard_out = self.master if lowp else torch.zeros(P, dtype=out_dtype, device=self.device)
        nf = self.world if n_full is None else int(n_full)
        self.full = [torch.zeros(P, dtype=out_dtype, device=self.device) for _ in range(nf)]
        self._host = None

    # ---------------------------------------------------------------- set-up

    def load_master(self, tensors: Sequence[torch.Tensor], stream=None) -> None:
        """Flatten the unit's initial parameters into the master buffer (the
        parameter buffer, rounded to nearest even for bf16/fp16 state)."""
        if not self.state_on_host and all(t.dtype == self.master.dtype for t in tensors):
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

    @property
    def variant(self) -> bool:
        """Whether the unit steps through the variant kernel (another
        optimizer or bf16/fp16 state) rather than the fused AdamW kernel."""
        return self.optimizer != "adamw" or self.state_dtype != torch.float32

    def step_config(self, hp) -> StepConfig:
        """The variant step's configuration for hp (a StepConfig naming this
        unit's optimizer, or AdamWHParams for an AdamW unit)."""
        if isinstance(hp, StepConfig):
            if hp.optimizer != self.optimizer:
                raise ValueError(f"this unit's optimizer is {self.optimizer}, not {hp.optimizer}")
            return hp
        if self.optimizer != "adamw":
            raise ValueError(f"a {self.optimizer} unit steps with a StepConfig")
        return StepConfig("adamw", hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.step, hp.grad_scale)

    def reduce_scatter_adam_cast(self, hp, rank_begin: int = 0, rank_end: Optional[int] = None,
                                 nonfinite_count: Optional[torch.Tensor] = None, stream=None) -> None:
        """The unit's update: the fused AdamW kernel for AdamWHParams on fp32
        state, else the variant kernel."""
        self._update(self.grads, hp, rank_begin, rank_end, nonfinite_count, stream)

    def _update(self, grads, hp, rank_begin=0, rank_end=None, nonfinite_count=None, stream=None) -> None:
        if isinstance(hp, AdamWHParams) and not self.variant:
            fsdp_reduce_scatter_adam_cast(grads, self.master, self.exp_avg, self.exp_avg_sq, self.shard_out,
                                          hp, rank_begin, rank_end, nonfinite_count, stream)
            return
        lowp = self.state_dtype != torch.float32
        fsdp_reduce_scatter_step(grads, self.master, self.exp_avg, self.exp_avg_sq,
                                 None if lowp else self.shard_out, self.step_config(hp), rank_begin, rank_end,
                                 nonfinite_count, stream)

    def all_gather(self, stream=None, wait_timeouts: Optional[torch.Tensor] = None) -> None:
        fsdp_all_gather(self.shard_out, self.full, self.world, stream, wait_timeouts=wait_timeouts)

    def step(self, hp: AdamWHParams, gathers: int = 1, nonfinite_count: Optional[torch.Tensor] = None,
             stream=None, fuse_gather: bool = False, wait_timeouts: Optional[torch.Tensor] = None) -> None:
        """Reduce-scatter + AdamW + cast, then ``gathers`` all-gathers, in stream order.

        gathers=2 is reshard-after-forward (gathered before forward and again
        before backward), gathers=1 the no-reshard mode. With fuse_gather the
        first gather is written by the update kernel itself (the fused AdamW
        kernel only). hp: AdamWHParams, or a StepConfig for the variant step.
        wait_timeouts: optional CUDA int32 counter of the gathers' bounded
        waits that gave up (zeroed by the caller; non-zero after the step's
        work: the gathered buffers are incomplete and the device is suspect)."""
        if fuse_gather and gathers >= 1 and (self.variant or not isinstance(hp, AdamWHParams)):
            raise ValueError("fuse_gather needs the fused AdamW kernel (fp32 state, AdamWHParams)")
        if fuse_gather and gathers >= 1:
            fsdp_reduce_scatter_adam_cast_gather(self.grads, self.master, self.exp_avg, self.exp_avg_sq,
                                                 self.shard_out, self.full, hp, nonfinite_count=nonfinite_count,
                                                 stream=stream)
            gathers -= 1
        else:
            self.reduce_scatter_adam_cast(hp, nonfinite_count=nonfinite_count, stream=stream)
        for _ in range(gathers):
            self.all_gather(stream, wait_timeouts)

    def step_from_host(self, host_grads: Sequence[torch.Tensor], host_out: Optional[torch.Tensor], hp: AdamWHParams,
                       gathers: int = 1, nonfinite_count: Optional[torch.Tensor] = None,
                       host_nonfinite: Optional[torch.Tensor] = None,
                       wait_timeouts: Optional[torch.Tensor] = None) -> None:
        """One step whose N gradient buffers come from pinned host memory.
        Its results go back to pinned host memory as asked: host_out receives
        the compute-dtype parameters (shard_out, all ranks' shards);
        host_nonfinite receives the step's count of non-finite averaged
        gradients (nonfinite_count is then required; it is zeroed first).
        Asynchronous; consecutive calls overlap: the host-to-device copy of a
        step runs on its own stream into a second set of gradient buffers
        while the previous step's kernels and device-to-host copies run. The
        host buffers are complete once the current stream is synchronized.
        wait_timeouts: as in step()."""
        if host_nonfinite is not None and nonfinite_count is None:
            raise ValueError("host_nonfinite needs a device nonfinite_count")
        if self._host is None:
            self._host = _HostPipeline(self)
        self._host.step(host_grads, host_out, hp, gathers, nonfinite_count, host_nonfinite, wait_timeouts)

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
                for name in ("master", "exp_avg", "exp_avg_sq") if getattr(self, name) is not None}

    def load_state_dict(self, state: Dict[str, torch.Tensor], rank: Optional[int] = None) -> None:
        """Restore what state_dict(rank) returned (rank=None: the whole unit)."""
        lo, hi = self._range(rank)
        names = [n for n in ("master", "exp_avg", "exp_avg_sq") if getattr(self, n) is not None]
        if sorted(state) != sorted(names):
            raise ValueError(f"state must hold exactly {names}")
        for name in names:
            src = state[name]
            if src.dtype != self.state_dtype or src.numel() != hi - lo:
                raise ValueError(f"{name} must be {self.state_dtype} with {hi - lo} elements")
            getattr(self, name)[lo:hi].copy_(src.reshape(-1))

    def _range(self, rank: Optional[int]) -> Tuple[int, int]:
        if rank is None:
            return 0, self.padded_numel
        if not 0 <= int(rank) < self.world:
            raise ValueError(f"rank must be in [0, {self.world})")
        S = self.shard_numel
        return int(rank) * S, (int(rank) + 1) * S

    def step_bytes(self, gathers: int = 1) -> Tuple[int, int]:
        """Algorithmic bytes of one step: (update kernel, all-gathers). The
        update reads N gradients, reads and writes the parameter and each
        state, and writes the compute-dtype shard when the state is fp32."""
        gs = self.grads[0].element_size()
        ss = self.master.element_size()
        os_ = self.shard_out.element_size()
        P = self.padded_numel
        nbuf = 2 if self.exp_avg_sq is None else 3
        rsa = P * (self.world * gs + nbuf * 2 * ss + (0 if self.state_dtype != torch.float32 else os_))
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

    def step(self, host_grads, host_out, hp, gathers, nonfinite_count, host_nonfinite, wait_timeouts=None):
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
        u._update(gset, hp, nonfinite_count=nonfinite_count, stream=compute)
        self.read_done[k] = compute.record_event()
        self.copy_out.wait_event(self.read_done[k])
        with torch.cuda.stream(self.copy_out):
            if host_out is not None:
                host_out.copy_(u.shard_out, non_blocking=True)
            if host_nonfinite is not None:
                host_nonfinite.copy_(nonfinite_count, non_blocking=True)
        self.out_read = self.copy_out.record_event()
        for _ in range(gathers):
            fsdp_all_gather(u.shard_out, u.full, u.world, stream=compute, wait_timeouts=wait_timeouts)
        compute.wait_stream(self.copy_out)  # the step ends when its result is on the host
        self.i += 1


class UnitSequence:
    """The FSDP units of a model, stepped by one call into the library: per
    unit the update and its all-gathers, ordered on the caller's stream. The
    native loop spreads the units over two side streams and batches units of
    up to 2^24 elements that share N, dtypes and gathers into one launch per
    kernel (256 units at most); the results are those of stepping each unit
    on its own.

    step() validates the model once and keeps that plan (StepPlan) for the
    steps that follow with the same gathers, fusion, optimizer and counters,
    so a step pays only its launches; step_unplanned() validates every
    unit on every call (fsdp_step_units / fsdp_step_units_ex). Both hold the
    units' buffer addresses from construction: build a new UnitSequence if a
    unit's buffers are replaced. One host thread at a time steps a given
    sequence (each planned step rewrites the plan's kernel arguments)."""

    def __init__(self, units: Sequence[FlatParamUnit]):
        self.units = list(units)
        self.descs = UnitDescs(self.units)
        self._plan = None       # the last StepPlan made by step()
        self._plan_key = None   # what it was made for

    def _adamw_fused(self, hp) -> bool:
        return isinstance(hp, AdamWHParams) and all(not u.variant for u in self.units)

    def _variant_config(self, hp, fuse_gather: bool) -> StepConfig:
        if fuse_gather:
            raise ValueError("fuse_gather needs the fused AdamW kernel in every unit")
        cfg = hp if isinstance(hp, StepConfig) else StepConfig(
            "adamw", hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.step, hp.grad_scale)
        for u in self.units:
            u.step_config(cfg)  # every unit takes this optimizer
        return cfg

    def step(self, hp, gathers: int = 1, nonfinite_count: Optional[torch.Tensor] = None,
             stream=None, fuse_gather: bool = False, wait_timeouts: Optional[torch.Tensor] = None) -> None:
        """hp: AdamWHParams (every unit AdamW; the fused kernel where the state
        is fp32) or a StepConfig (the variant kernel in every unit).
        nonfinite_count / wait_timeouts: optional CUDA int32 counters, summed
        over the units (see FlatParamUnit.step)."""
        ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        if self._adamw_fused(hp):
            config, kind = None, "adamw"
        else:
            config = self._variant_config(hp, fuse_gather)
            kind = config.optimizer
        key = (kind, int(gathers), bool(fuse_gather), ptr(nonfinite_count), ptr(wait_timeouts))
        if key != self._plan_key:
            if self._plan is not None:
                self._plan.close()
                self._plan, self._plan_key = None, None
            self._plan = StepPlan(self.descs, gathers, fuse_gather, nonfinite_count, config, wait_timeouts)
            self._plan_key = key
        self._plan.launch(hp if config is None else config, stream)

    def step_unplanned(self, hp, gathers: int = 1, nonfinite_count: Optional[torch.Tensor] = None,
                       stream=None, fuse_gather: bool = False, wait_timeouts: Optional[torch.Tensor] = None) -> None:
        """The same step through the call that validates every unit each time."""
        if self._adamw_fused(hp):
            fsdp_step_units(self.descs, hp, gathers, fuse_gather, nonfinite_count, stream, wait_timeouts)
            return
        cfg = self._variant_config(hp, fuse_gather)
        fsdp_step_units_ex(self.descs, cfg, gathers, nonfinite_count, stream, wait_timeouts)

    def capture(self, gathers: int = 1, fuse_gather: bool = False,
                nonfinite_count: Optional[torch.Tensor] = None, config: Optional[StepConfig] = None,
                wait_timeouts: Optional[torch.Tensor] = None) -> StepGraph:
        """The model's step captured as one CUDA graph; StepGraph.launch runs it
        for any step. Without `config`: the fused AdamW step (every unit
        AdamW with fp32 state), launched with AdamWHParams. With a StepConfig
        (required when a unit takes the variant step): the variant step of
        that optimizer, launched with StepConfigs."""
        if config is None and any(u.variant for u in self.units):
            raise ValueError("units that take the variant step are captured with a StepConfig")
        if config is not None:
            for u in self.units:
                u.step_config(config)  # every unit takes this optimizer
        return StepGraph(self.descs, gathers, fuse_gather, nonfinite_count, config, wait_timeouts)

    def launches(self, gathers: int = 1, fuse_gather: bool = False, config: Optional[StepConfig] = None) -> int:
        """Kernel launches of one model step as step() (or capture()) makes
        it, small units batched; nothing runs."""
        if config is None and all(not u.variant for u in self.units):
            return fsdp_step_units_launches(self.descs, gathers=gathers, fuse_first_gather=fuse_gather)
        if fuse_gather:
            raise ValueError("fuse_gather needs the fused AdamW kernel in every unit")
        cfg = config if config is not None else StepConfig(self.units[0].optimizer, 1e-3)
        return fsdp_step_units_ex_launches(self.descs, cfg, gathers)

    def step_bytes(self, gathers: int = 1) -> Tuple[int, int]:
        """Algorithmic bytes of one model step: (fused kernels, all-gathers)."""
        rsa = ag = 0
        for u in self.units:
            a, b = u.step_bytes(gathers)
            rsa += a
            ag += b
        return rsa, ag
