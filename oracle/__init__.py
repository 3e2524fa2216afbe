"""CPU oracle for the FSDP FlatParameter step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package. The product (the CUDA library and its
binding) never does. The arithmetic lives in ``fsdp_oracle.c`` (plain C, fp32
one IEEE operation at a time, plus an fp64 shadow); this module only builds it,
loads it and moves numpy arrays in and out.

Parity of every function here is pinned by the ``-m "not gpu"`` tests against
facts the sources and mathematics fix (hand cases with exact binary values, the
all-reduce = reduce-scatter + all-gather identity, sharded == DDP, closed forms
of AdamW, numpy/torch's own format conversions and torch.optim.AdamW).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, BF16, F16 = 0, 1, 2
OPT_ADAMW, OPT_SGD, OPT_ADAMAX, OPT_ADADELTA = 0, 1, 2, 3
OPTIMIZERS = {"adamw": OPT_ADAMW, "sgd": OPT_SGD, "adamax": OPT_ADAMAX, "adadelta": OPT_ADADELTA}
_DT = {"f32": F32, "bf16": BF16, "f16": F16}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fsdp_oracle.c")
# FSDP_ORACLE_LIB points the tests at another build of fsdp_oracle.c (the
# mutation test plants one mistake per build and expects the pins to fail).
_LIB_PATH = os.environ.get("FSDP_ORACLE_LIB") or os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """gcc build of an oracle source file (no FMA contraction, no fast-math)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``fsdp_oracle.c`` into ``liboracle.so``."""
    if os.environ.get("FSDP_ORACLE_LIB"):
        return _LIB_PATH
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


class HParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("step", ctypes.c_int64), ("grad_scale", ctypes.c_float)]


class Scalars(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in
                ("c", "decay", "beta1", "beta2", "one_minus_beta1", "one_minus_beta2",
                 "alpha", "b2s", "eps")]


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        sig = {
            "orc_set_threads": (None, [i32]),
            "orc_get_threads": (i32, []),
            "orc_padded_numel": (i64, [i64, i64]),
            "orc_shard_numel": (i64, [i64, i64]),
            "orc_view_offsets": (None, [vp, i32, vp]),
            "orc_flatten_pad": (None, [vp, vp, i32, i32, i64, vp]),
            "orc_f32_to_bf16": (ctypes.c_uint16, [f32]),
            "orc_f32_to_f16": (ctypes.c_uint16, [f32]),
            "orc_bf16_to_f32": (f32, [ctypes.c_uint16]),
            "orc_f16_to_f32": (f32, [ctypes.c_uint16]),
            "orc_cast_array": (None, [vp, i64, i32, vp]),
            "orc_widen_array": (None, [vp, i64, i32, vp]),
            "orc_scalars_from_hparams": (i32, [ctypes.POINTER(HParams), i64, ctypes.POINTER(Scalars)]),
            "orc_reduce_scatter": (None, [vp, i32, i64, i64, i64, f32, vp]),
            "orc_all_reduce_avg": (None, [vp, i32, i64, i64, f32, vp]),
            "orc_adamw": (None, [vp, vp, vp, vp, i64, ctypes.POINTER(Scalars)]),
            "orc_cast": (None, [vp, i64, i32, vp]),
            "orc_all_gather": (None, [vp, i32, i64, i64, vp]),
            "orc_fsdp_step": (i32, [vp, i32, i64, i64, vp, vp, vp, i32, vp, vp,
                                    ctypes.POINTER(HParams), vp]),
            "orc_ddp_step": (i32, [vp, i32, i64, i64, vp, vp, vp, i32, vp,
                                   ctypes.POINTER(HParams), vp]),
            "orc_reduce_scatter_lowp": (None, [vp, i32, i64, i64, i64, f32, vp]),
            "orc_step_ex": (i32, [i32, i32, vp, i32, i64, i64, vp, vp, vp, i32, i32, vp, vp,
                                  ctypes.POINTER(HParams), vp]),
            "orc_all_reduce_avg_f64": (None, [vp, i32, i64, i64, ctypes.c_double, vp]),
            "orc_adamw_f64": (None, [vp, vp, vp, vp, i64, ctypes.POINTER(HParams)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


# ---------------------------------------------------------------- helpers

def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def dtype_code(name: str) -> int:
    return _DT[name]


def np_storage(name: str):
    """numpy storage dtype of a format: bf16/f16 are held as raw uint16 bits."""
    return np.float32 if name == "f32" else np.uint16


def hparams(lr, beta1, beta2, eps, weight_decay, step, grad_scale=1.0) -> HParams:
    return HParams(lr, beta1, beta2, eps, weight_decay, int(step), grad_scale)


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def get_threads() -> int:
    return int(_load().orc_get_threads())


# ---------------------------------------------------------------- layout

def padded_numel(numel: int, world: int) -> int:
    return int(_load().orc_padded_numel(numel, world))


def shard_numel(padded: int, world: int) -> int:
    return int(_load().orc_shard_numel(padded, world))


def view_offsets(numels) -> np.ndarray:
    n = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
    out = np.zeros(len(n), dtype=np.int64)
    _load().orc_view_offsets(_ptr(n), len(n), _ptr(out))
    return out


def flatten_pad(tensors, world: int) -> np.ndarray:
    """Concatenate contiguous numpy arrays (one dtype) and zero-pad to a multiple of N."""
    ts = [np.ascontiguousarray(t).reshape(-1) for t in tensors]
    dt = ts[0].dtype
    assert all(t.dtype == dt for t in ts)
    numels = np.array([t.size for t in ts], dtype=np.int64)
    padded = padded_numel(int(numels.sum()), world)
    out = np.empty(padded, dtype=dt)
    _load().orc_flatten_pad(_ptr_array(ts), _ptr(numels), len(ts), dt.itemsize, padded, _ptr(out))
    return out


# ---------------------------------------------------------------- formats

def cast(x: np.ndarray, fmt: str) -> np.ndarray:
    """fp32 -> bf16/f16 bits (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_cast_array(_ptr(x), x.size, _DT[fmt], _ptr(out))
    return out


def widen(h: np.ndarray, fmt: str) -> np.ndarray:
    """bf16/f16 bits (uint16) -> fp32, exact."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().orc_widen_array(_ptr(h), h.size, _DT[fmt], _ptr(out))
    return out


# ---------------------------------------------------------------- the step

def scalars(hp: HParams, world: int) -> Scalars:
    s = Scalars()
    rc = _load().orc_scalars_from_hparams(ctypes.byref(hp), world, ctypes.byref(s))
    if rc:
        raise ValueError("invalid hyperparameters")
    return s


def reduce_scatter(grads, grad_fmt: str, world: int, rank: int, c: float) -> np.ndarray:
    padded = grads[0].size
    S = shard_numel(padded, world)
    out = np.empty(S, dtype=np.float32)
    _load().orc_reduce_scatter(_ptr_array(grads), _DT[grad_fmt], world, S, rank, c, _ptr(out))
    return out


def all_reduce_avg(grads, grad_fmt: str, world: int, c: float) -> np.ndarray:
    padded = grads[0].size
    out = np.empty(padded, dtype=np.float32)
    _load().orc_all_reduce_avg(_ptr_array(grads), _DT[grad_fmt], world, padded, c, _ptr(out))
    return out


def adamw(p: np.ndarray, m: np.ndarray, v: np.ndarray, g: np.ndarray, s: Scalars) -> None:
    """In place on p, m, v (fp32)."""
    n = p.size
    assert m.size == n and v.size == n and g.size == n
    _load().orc_adamw(_ptr(p), _ptr(m), _ptr(v), _ptr(g), n, ctypes.byref(s))


def cast_out(p: np.ndarray, fmt: str) -> np.ndarray:
    out = np.empty(p.size, dtype=np_storage(fmt))
    _load().orc_cast(_ptr(p), p.size, _DT[fmt], _ptr(out))
    return out


def all_gather(shards, world: int) -> np.ndarray:
    S = shards[0].size
    dt = shards[0].dtype
    out = np.empty(S * world, dtype=dt)
    _load().orc_all_gather(_ptr_array(shards), dt.itemsize, world, S, _ptr(out))
    return out


def fsdp_step(grads, grad_fmt: str, world: int, master, m, v, out_fmt: str, hp: HParams):
    """Sharded step, ranks emulated in turn. Updates master/m/v in place.
    Returns (shards_out concatenated [P_pad], gathered full buffer [P_pad])."""
    padded = master.size
    S = shard_numel(padded, world)
    shards = np.empty(padded, dtype=np_storage(out_fmt))
    full = np.empty(padded, dtype=np_storage(out_fmt))
    scratch = np.empty(max(S, 1), dtype=np.float32)
    rc = _load().orc_fsdp_step(_ptr_array(grads), _DT[grad_fmt], world, padded, _ptr(master), _ptr(m),
                               _ptr(v), _DT[out_fmt], _ptr(shards), _ptr(full), ctypes.byref(hp),
                               _ptr(scratch))
    if rc:
        raise ValueError("oracle fsdp_step: bad arguments")
    return shards, full


def ddp_step(grads, grad_fmt: str, world: int, master, m, v, out_fmt: str, hp: HParams):
    """Full-replica DDP step: all-reduce average, AdamW on everything, cast."""
    padded = master.size
    full = np.empty(padded, dtype=np_storage(out_fmt))
    scratch = np.empty(max(padded, 1), dtype=np.float32)
    rc = _load().orc_ddp_step(_ptr_array(grads), _DT[grad_fmt], world, padded, _ptr(master), _ptr(m),
                              _ptr(v), _DT[out_fmt], _ptr(full), ctypes.byref(hp), _ptr(scratch))
    if rc:
        raise ValueError("oracle ddp_step: bad arguments")
    return full


def reduce_scatter_lowp(grads, grad_fmt: str, world: int, rank: int, c: float) -> np.ndarray:
    """Block `rank` of the reduce-scatter summed in the gradient dtype."""
    padded = grads[0].size
    S = shard_numel(padded, world)
    out = np.empty(S, dtype=np.float32)
    _load().orc_reduce_scatter_lowp(_ptr_array(grads), _DT[grad_fmt], world, S, rank, c, _ptr(out))
    return out


def step_ex(optimizer: str, reduce_lowp: bool, grads, grad_fmt: str, world: int, param, s0, s1, state_fmt: str,
            out_fmt: str, hp: HParams):
    """General step (optimizer, reduce precision, state precision), ranks in
    turn then the all-gather. Updates param/s0/s1 in place (numpy arrays of
    the state format: float32, or uint16 bits for bf16/f16; s1 None for SGD).
    Returns (shards_out, gathered full buffer)."""
    padded = param.size
    S = shard_numel(padded, world)
    shards = np.empty(padded, dtype=np_storage(out_fmt))
    full = np.empty(padded, dtype=np_storage(out_fmt))
    scratch = np.empty(max(S, 1), dtype=np.float32)
    rc = _load().orc_step_ex(OPTIMIZERS[optimizer], int(bool(reduce_lowp)), _ptr_array(grads), _DT[grad_fmt],
                             world, padded, _ptr(param), _ptr(s0), _ptr(s1) if s1 is not None else None,
                             _DT[state_fmt], _DT[out_fmt], _ptr(shards), _ptr(full), ctypes.byref(hp),
                             _ptr(scratch))
    if rc:
        raise ValueError("oracle step_ex: bad arguments")
    return shards, full


def all_reduce_avg_f64(grads, grad_fmt: str, world: int, grad_scale: float = 1.0) -> np.ndarray:
    padded = grads[0].size
    out = np.empty(padded, dtype=np.float64)
    _load().orc_all_reduce_avg_f64(_ptr_array(grads), _DT[grad_fmt], world, padded, grad_scale, _ptr(out))
    return out


def adamw_f64(p, m, v, g, hp: HParams) -> None:
    n = p.size
    _load().orc_adamw_f64(_ptr(p), _ptr(m), _ptr(v), _ptr(g), n, ctypes.byref(hp))
