"""ctypes loader for libfsdpreduce.so and the C structs of include/fsdp.h.

Loading fails loudly (RuntimeError) when the library has not been built: there
is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfsdpreduce.so")

FSDP_MAX_WORLD = 64
FSDP_MAX_NDIM = 8

FSDP_OK = 0
FSDP_ERR_INVALID_ARG = 1
FSDP_ERR_ALIGNMENT = 2
FSDP_ERR_CUDA = 3
FSDP_ERR_UNSUPPORTED_DTYPE = 4
FSDP_ERR_HOST_MEMORY = 5

FSDP_F32, FSDP_BF16, FSDP_F16 = 0, 1, 2
FSDP_OPT_ADAMW, FSDP_OPT_SGD, FSDP_OPT_ADAMAX, FSDP_OPT_ADADELTA = 0, 1, 2, 3

# every symbol include/fsdp.h declares
EXPORTS = (
    "fsdp_padded_numel",
    "fsdp_unflatten_views",
    "fsdp_flatten_pad",
    "fsdp_reduce_scatter_adam_cast",
    "fsdp_reduce_scatter_adam_cast_gather",
    "fsdp_reduce_scatter_step",
    "fsdp_all_gather",
    "fsdp_status_string",
    "fsdp_last_cuda_error",
    "fsdp_take_wait_timeouts",
    "fsdp_check_bounded_wait",
    "fsdp_step_units",
    "fsdp_step_units_ex",
    "fsdp_step_units_launches",
    "fsdp_step_units_ex_launches",
    "fsdp_step_graph_create",
    "fsdp_step_graph_launch",
    "fsdp_step_graph_destroy",
    "fsdp_step_graph_create_ex",
    "fsdp_step_graph_launch_ex",
    "fsdp_step_plan_create",
    "fsdp_step_plan_create_ex",
    "fsdp_step_plan_launch",
    "fsdp_step_plan_launch_ex",
    "fsdp_step_plan_destroy",
)


class FsdpView(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("shape", ctypes.c_int64 * FSDP_MAX_NDIM), ("offset", ctypes.c_int64),
                ("numel", ctypes.c_int64)]


class FsdpAdamwHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("step", ctypes.c_int64),
                ("grad_scale", ctypes.c_float)]


class FsdpStepConfig(ctypes.Structure):
    _fields_ = [("optimizer", ctypes.c_int32), ("reduce_dtype", ctypes.c_int32), ("lr", ctypes.c_float),
                ("beta1", ctypes.c_float), ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float), ("step", ctypes.c_int64), ("grad_scale", ctypes.c_float)]


class FsdpUnit(ctypes.Structure):
    _fields_ = [("grads", ctypes.c_void_p), ("full_bufs", ctypes.c_void_p), ("master", ctypes.c_void_p),
                ("exp_avg", ctypes.c_void_p), ("exp_avg_sq", ctypes.c_void_p), ("shard_out", ctypes.c_void_p),
                ("padded_numel", ctypes.c_int64), ("world", ctypes.c_int32), ("grad_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("n_full", ctypes.c_int32)]


class FsdpUnitEx(ctypes.Structure):
    _fields_ = [("grads", ctypes.c_void_p), ("full_bufs", ctypes.c_void_p), ("param", ctypes.c_void_p),
                ("state0", ctypes.c_void_p), ("state1", ctypes.c_void_p), ("shard_out", ctypes.c_void_p),
                ("padded_numel", ctypes.c_int64), ("world", ctypes.c_int32), ("grad_dtype", ctypes.c_int32),
                ("state_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32), ("n_full", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load the in-tree CUDA library (build it first with ``build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: the CUDA library must be built "
                "(python -c 'import __graft_entry__ as g; g.build()'); there is no fallback")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        sigs = {
            "fsdp_padded_numel": (i64, [i64, i32]),
            "fsdp_unflatten_views": (i32, [vp, vp, i32, i32, ctypes.POINTER(FsdpView), ctypes.POINTER(i64)]),
            "fsdp_flatten_pad": (i32, [vp, vp, i32, i32, i32, vp, i64, ctypes.POINTER(FsdpView), vp]),
            "fsdp_reduce_scatter_adam_cast": (i32, [vp, i32, i32, i64, vp, vp, vp, vp, i32,
                                                    ctypes.POINTER(FsdpAdamwHparams), i32, i32, vp, vp]),
            "fsdp_reduce_scatter_adam_cast_gather": (i32, [vp, i32, i32, i64, vp, vp, vp, vp, i32, vp, i32,
                                                           ctypes.POINTER(FsdpAdamwHparams), i32, i32, vp, vp]),
            "fsdp_reduce_scatter_step": (i32, [vp, i32, i32, i64, vp, vp, vp, i32, vp, i32,
                                               ctypes.POINTER(FsdpStepConfig), i32, i32, vp, vp]),
            "fsdp_all_gather": (i32, [vp, i32, i32, i64, vp, i32, vp, vp]),
            "fsdp_status_string": (ctypes.c_char_p, [i32]),
            "fsdp_last_cuda_error": (i32, []),
            "fsdp_take_wait_timeouts": (i32, [ctypes.POINTER(ctypes.c_uint32)]),
            "fsdp_check_bounded_wait": (i32, [i64, vp, vp]),
            "fsdp_step_units": (i32, [ctypes.POINTER(FsdpUnit), i32, ctypes.POINTER(FsdpAdamwHparams), i32, i32,
                                      vp, vp, vp]),
            "fsdp_step_units_ex": (i32, [ctypes.POINTER(FsdpUnitEx), i32, ctypes.POINTER(FsdpStepConfig), i32,
                                         vp, vp, vp]),
            "fsdp_step_units_launches": (i32, [ctypes.POINTER(FsdpUnit), i32, ctypes.POINTER(FsdpAdamwHparams), i32,
                                               i32, ctypes.POINTER(i64)]),
            "fsdp_step_units_ex_launches": (i32, [ctypes.POINTER(FsdpUnitEx), i32, ctypes.POINTER(FsdpStepConfig),
                                                  i32, ctypes.POINTER(i64)]),
            "fsdp_step_graph_create": (i32, [ctypes.POINTER(FsdpUnit), i32, i32, i32, vp, vp, ctypes.POINTER(vp)]),
            "fsdp_step_graph_launch": (i32, [vp, ctypes.POINTER(FsdpAdamwHparams), vp]),
            "fsdp_step_graph_destroy": (i32, [vp]),
            "fsdp_step_graph_create_ex": (i32, [ctypes.POINTER(FsdpUnitEx), i32, ctypes.POINTER(FsdpStepConfig), i32,
                                                vp, vp, ctypes.POINTER(vp)]),
            "fsdp_step_graph_launch_ex": (i32, [vp, ctypes.POINTER(FsdpStepConfig), vp]),
            "fsdp_step_plan_create": (i32, [ctypes.POINTER(FsdpUnit), i32, i32, i32, vp, vp, ctypes.POINTER(vp)]),
            "fsdp_step_plan_create_ex": (i32, [ctypes.POINTER(FsdpUnitEx), i32, ctypes.POINTER(FsdpStepConfig), i32,
                                               vp, vp, ctypes.POINTER(vp)]),
            "fsdp_step_plan_launch": (i32, [vp, ctypes.POINTER(FsdpAdamwHparams), vp]),
            "fsdp_step_plan_launch_ex": (i32, [vp, ctypes.POINTER(FsdpStepConfig), vp]),
            "fsdp_step_plan_destroy": (i32, [vp]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib
