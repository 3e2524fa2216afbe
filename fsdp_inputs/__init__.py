"""Seeded synthetic inputs for the FSDP FlatParameter step.

This module is shared by the CPU oracle's tests and the CUDA path's tests and
bench. It holds only workload definitions (the parameter shapes of each
synthetic transformer-block unit, the optimizer hyperparameters, the gradient
distribution) and seeded random draws. It performs none of the method's
arithmetic: no padding, no reduction, no optimizer update, no cast of the
step's outputs.

Workloads (synthetic stand-ins; there is no dataset or checkpoint):

* ``tiny``        one 4,099-element unit, N=2, bf16 grads ~N(0, 1e-2).
* ``gpt2_small``  one GPT-2 small block (d=768), N=8, bf16 grads ~N(0, 1e-3).
* ``gpt2_large``  one GPT-2 Large block (d=1280), N=2, fp16 compute dtype,
                  grads ~N(0, 1e-3) stored pre-multiplied by a static loss scale
                  of 1024.
* ``gpt3_13b``    one GPT-3 13B-style block (d=5120, MLP 20480), N=8, bf16
                  grads ~N(0, 1e-4).
* ``llama70b``    one Llama-70B-style block (d=8192, GQA 64 q / 8 kv heads of
                  128, SwiGLU 28672, RMSNorm weights only), N=8, bf16 grads
                  ~N(0, 1e-4); the all-gather runs twice per step (fwd + bwd).

Draws: master ~ U(-0.1, 0.1) in fp32 with seed ``base`` (identical on every
rank, since FSDP does not broadcast the initial weights and all workers must
start from the same values); the gradient of rank r at step t is an fp32
N(0, sigma) draw with seed ``base + 1000*r + t``, multiplied by the loss scale
(a power of two, so exact) and rounded to the gradient dtype by torch's own
round-to-nearest-even conversion. sigma is a standard deviation.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Tuple

import torch

__all__ = [
    "UnitConfig",
    "CONFIGS",
    "unit_numel",
    "torch_dtype",
    "gen_master",
    "gen_grad",
    "gen_uniform",
]


@dataclasses.dataclass(frozen=True)
class UnitConfig:
    name: str
    world: int                                   # N emulated ranks
    params: Tuple[Tuple[str, Tuple[int, ...]], ...]  # registration order = flatten order
    grad_dtype: str                              # "bf16" | "f16" | "f32"
    out_dtype: str                               # compute dtype of the gathered params
    sigma: float                                 # std of the true gradient
    grad_scale: float                            # static loss scale (1.0 if none)
    lr: float
    beta1: float
    beta2: float
    eps: float
    weight_decay: float
    steps: int                                   # steps of the parity trajectory
    gathers: int                                 # all-gathers per step (fwd, bwd)
    description: str = ""


def _gpt2_block(d: int, mlp: int) -> Tuple[Tuple[str, Tuple[int, ...]], ...]:
    # weights stored [in, out]
    return (
        ("ln1.weight", (d,)), ("ln1.bias", (d,)),
        ("attn.qkv.weight", (d, 3 * d)), ("attn.qkv.bias", (3 * d,)),
        ("attn.proj.weight", (d, d)), ("attn.proj.bias", (d,)),
        ("ln2.weight", (d,)), ("ln2.bias", (d,)),
        ("mlp.fc.weight", (d, mlp)), ("mlp.fc.bias", (mlp,)),
        ("mlp.proj.weight", (mlp, d)), ("mlp.proj.bias", (d,)),
    )


def _llama_block(d: int, kv: int, ffn: int) -> Tuple[Tuple[str, Tuple[int, ...]], ...]:
    return (
        ("attn_norm.weight", (d,)),
        ("attn.wq", (d, d)), ("attn.wk", (d, kv)), ("attn.wv", (d, kv)),
        ("attn.wo", (d, d)),
        ("ffn_norm.weight", (d,)),
        ("ffn.w_gate", (d, ffn)), ("ffn.w_up", (d, ffn)), ("ffn.w_down", (ffn, d)),
    )


_ADAM = dict(beta1=0.9, beta2=0.999, eps=1e-8)

CONFIGS: Dict[str, UnitConfig] = {
    "tiny": UnitConfig(
        name="tiny", world=2,
        params=(("w", (64, 64)), ("b", (3,))),
        grad_dtype="bf16", out_dtype="bf16", sigma=1e-2, grad_scale=1.0,
        lr=1e-3, weight_decay=0.01, steps=3, gathers=1, **_ADAM,
        description="tiny unit, 4,099 fp32 params, N=2"),
    "gpt2_small": UnitConfig(
        name="gpt2_small", world=8, params=_gpt2_block(768, 3072),
        grad_dtype="bf16", out_dtype="bf16", sigma=1e-3, grad_scale=1.0,
        lr=1e-3, weight_decay=0.01, steps=10, gathers=1, **_ADAM,
        description="GPT-2 small block unit (d=768), N=8"),
    "gpt2_large": UnitConfig(
        name="gpt2_large", world=2, params=_gpt2_block(1280, 5120),
        grad_dtype="f16", out_dtype="f16", sigma=1e-3, grad_scale=1024.0,
        lr=1e-4, weight_decay=0.01, steps=10, gathers=1, **_ADAM,
        description="GPT-2 Large block unit (d=1280), N=2, fp16, loss scale 1024"),
    "gpt3_13b": UnitConfig(
        name="gpt3_13b", world=8, params=_gpt2_block(5120, 20480),
        grad_dtype="bf16", out_dtype="bf16", sigma=1e-4, grad_scale=1.0,
        lr=1e-4, weight_decay=0.1, steps=5, gathers=1, **_ADAM,
        description="GPT-3 13B-style block unit (d=5120, MLP 20480), N=8"),
    "llama70b": UnitConfig(
        name="llama70b", world=8, params=_llama_block(8192, 1024, 28672),
        grad_dtype="bf16", out_dtype="bf16", sigma=1e-4, grad_scale=1.0,
        lr=3e-5, weight_decay=0.1, steps=3, gathers=2, **_ADAM,
        description="Llama-70B-style block unit (d=8192, GQA 64q/8kv x128, SwiGLU 28672), N=8"),
}


def unit_numel(cfg: UnitConfig) -> int:
    """Number of parameters in the unit (sum of the shapes' products)."""
    return sum(math.prod(shape) for _, shape in cfg.params)


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[name]


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gen_uniform(numel: int, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    """fp32 U(lo, hi) draw of ``numel`` values."""
    g = _generator(seed, device)
    x = torch.rand(numel, generator=g, device=device, dtype=torch.float32)
    return x.mul_(hi - lo).add_(lo)


def gen_master(cfg: UnitConfig, device="cpu", seed_base: int = 0, numel: int | None = None) -> torch.Tensor:
    """Initial fp32 master weights, U(-0.1, 0.1), identical for every rank."""
    n = unit_numel(cfg) if numel is None else int(numel)
    return gen_uniform(n, -0.1, 0.1, seed_base, device)


def gen_grad(cfg: UnitConfig, rank: int, step: int, device="cpu", seed_base: int = 0,
             numel: int | None = None, sigma: float | None = None) -> torch.Tensor:
    """Rank ``rank``'s unpadded flat gradient at step ``step`` (1-based), in the
    gradient dtype, pre-multiplied by the static loss scale."""
    n = unit_numel(cfg) if numel is None else int(numel)
    s = cfg.sigma if sigma is None else sigma
    g = _generator(seed_base + 1000 * rank + step, device)
    x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
    x.mul_(s)
    if cfg.grad_scale != 1.0:
        x.mul_(cfg.grad_scale)
    return x.to(torch_dtype(cfg.grad_dtype))
