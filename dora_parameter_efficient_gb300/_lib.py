"""ctypes loader for ``libdora.so`` (the C ABI declared in include/dora.h).

There is no fallback: if the library is missing or fails to load, every call
raises.  Build it with ``dora_parameter_efficient_gb300.build.build()``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdora.so")

DORA_OK = 0
DORA_ERR_INVALID_ARG = 1
DORA_ERR_UNSUPPORTED = 2
DORA_ERR_WORKSPACE = 3
DORA_ERR_CUDA = 4
DORA_ERR_TIMEOUT = 5
DORA_ERR_NO_DEVICE = 6

DORA_BF16 = 0
DORA_F32 = 1

# name -> (restype, argtypes), mirroring include/dora.h
_P = ctypes.c_void_p
_I64 = ctypes.c_int64


class NormModule(ctypes.Structure):
    """struct dora_norm_module"""
    _fields_ = [("W", _P), ("A", _P), ("B", _P), ("m", _P), ("wnorm", _P), ("g", _P),
                ("d_out", _I64), ("d_in", _I64)]


class ComposeModule(ctypes.Structure):
    """struct dora_compose_module"""
    _fields_ = [("base", _P), ("lora", _P), ("g", _P), ("out", _P), ("T", _I64), ("d_out", _I64)]


SIGNATURES = {
    "dora_norm_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64, ctypes.c_int]),
    "dora_factored_norm": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64,
                                          ctypes.c_float, _P, ctypes.c_float, _P, _P, _P,
                                          ctypes.c_size_t, _P]),
    "dora_factored_norm_timed": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64,
                                                ctypes.c_float, _P, ctypes.c_float, _P, _P, _P,
                                                ctypes.c_size_t, _P, _P, _P]),
    "dora_factored_norm_noalloc": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64,
                                                  ctypes.c_float, _P, ctypes.c_float, _P, _P,
                                                  _P]),
    "dora_norm_partials_floats": (ctypes.c_size_t, [_I64, _I64]),
    "dora_norm_partials": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64, _P, _P,
                                          ctypes.c_size_t, _P]),
    "dora_norm_finalize_workspace_size": (ctypes.c_size_t, [_I64, _I64, ctypes.c_int]),
    "dora_norm_finalize_partials": (ctypes.c_int, [_P, _P, ctypes.c_int, _I64, _I64,
                                                   ctypes.c_float, _P, ctypes.c_float, _P, _P, _P,
                                                   ctypes.c_size_t, _P]),
    "dora_compose": (ctypes.c_int, [_P, _P, _P, ctypes.c_float, ctypes.c_int, _I64, _I64, _P, _P]),
    "dora_norm_grouped_workspace_size": (ctypes.c_size_t, [_P, ctypes.c_int, _I64, ctypes.c_int]),
    "dora_factored_norm_grouped": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, _I64,
                                                  ctypes.c_float, ctypes.c_float, _P,
                                                  ctypes.c_size_t, _P]),
    "dora_norm_grouped_plan_create": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, _I64, _P,
                                                     ctypes.c_size_t, _P,
                                                     ctypes.POINTER(_P)]),
    "dora_norm_grouped_plan_run": (ctypes.c_int, [_P, ctypes.c_float, ctypes.c_float, _P]),
    "dora_norm_grouped_plan_destroy": (None, [_P]),
    "dora_compose_grouped_workspace_size": (ctypes.c_size_t, [ctypes.c_int]),
    "dora_compose_grouped": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_float, ctypes.c_int, _P,
                                            ctypes.c_size_t, _P]),
    "dora_compose_train": (ctypes.c_int, [_P, _P, _P, ctypes.c_float, ctypes.c_int, _I64, _I64,
                                          _P, _P, _P]),
    "dora_compose_backward_workspace_size": (ctypes.c_size_t, [_I64, _I64]),
    "dora_compose_backward": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_float, ctypes.c_float,
                                             ctypes.c_int, _I64, _I64, _P, _P, _P, _P,
                                             ctypes.c_size_t, _P]),
    "dora_check_status": (ctypes.c_int, [_P, _P]),
    "dora_selftest_timeout": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.c_uint, _P]),
    "dora_selftest_grouped_schedule": (ctypes.c_int, [_P, _P, ctypes.c_int, _I64, ctypes.c_int,
                                                      ctypes.POINTER(ctypes.c_int),
                                                      ctypes.POINTER(ctypes.c_int64)]),
    "dora_selftest_schedule": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_int,
                                              ctypes.POINTER(ctypes.c_int),
                                              ctypes.POINTER(ctypes.c_int),
                                              ctypes.POINTER(ctypes.c_int64)]),
    "dora_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dora_version": (ctypes.c_int, []),
    "dora_launch_count": (ctypes.c_uint64, []),
}

_lib = None
_lock = threading.Lock()


class DoraError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load():
    """Load libdora.so once; raises if it is not there."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "dora_parameter_efficient_gb300.build.build() (there is no fallback path)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().dora_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != DORA_OK:
        raise DoraError(status, where)
