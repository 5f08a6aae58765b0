"""ctypes loader for libplmla.so (the C ABI in include/plmla.h).

The library must have been built (``python -m paged_latent_attention_gb300.build``
or ``__graft_entry__.build()``); there is no fallback implementation, and a
missing library raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import re

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libplmla.so")
HEADER_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "include", "plmla.h")

_i32, _i64, _sz, _p, _f = (ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p,
                           ctypes.c_float)

# name -> (restype, argtypes); mirrors include/plmla.h
SIGNATURES = {
    "mla_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "mla_split_budget": (_i32, [_i32, _i32, _i32, _i32, _i32]),
    "mla_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "mla_plan_splits": (ctypes.c_int, [_p, _i32, _i32, _p, _p, _p]),
    "mla_decode": (ctypes.c_int, [_p, _p, _p, _p, _i64, _i64, _p, _i64, _p, _i32, _i32, _i32,
                                  _f, _p, _p, _p, _sz, _i32, _i32, _p]),
    "mla_decode_ex": (ctypes.c_int, [_p, _p, _p, _p, _i64, _i64, _p, _i64, _p, _i32, _i32, _i32,
                                     _f, _p, _p, _p, _sz, _i32, _i32, _p, _p]),
    "mla_decode_layers": (ctypes.c_int, [_i32, _p, _p, _p, _p, _i64, _i64, _p, _i64, _p, _i32,
                                         _i32, _i32, _f, _p, _p, _p, _sz, _i32, _i32, _p]),
    "mla_decode_layers_fp8": (ctypes.c_int, [_i32, _p, _p, _p, _p, _p, _i64, _i64, _p, _i64, _p,
                                             _i32, _i32, _i32, _f, _p, _p, _p, _sz, _i32, _i32,
                                             _p]),
    "mla_split_combine": (ctypes.c_int, [_p, _p, _p, _p, _i32, _i32, _i32, _p, _p, _p]),
    "mla_decode_static_scratch": (ctypes.c_int, [_p, _p, _p, _p, _i64, _i64, _p, _i64, _p, _i32,
                                                 _i32, _i32, _f, _p, _p, _i32, _i32, _p]),
    "mla_static_scratch_status": (ctypes.c_int, [_p, _p]),
    "mla_kv_append": (ctypes.c_int, [_p, _p, _p, _i64, _i64, _p, _i64, _p, _i32, _i32, _p, _p]),
    "mla_workspace_size_fp8": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "mla_decode_fp8": (ctypes.c_int, [_p, _p, _p, _p, _i64, _i64, _f, _p, _i64, _p, _i32, _i32,
                                      _i32, _f, _p, _p, _p, _sz, _i32, _i32, _p]),
    "mla_decode_fp8_ex": (ctypes.c_int, [_p, _p, _p, _p, _i64, _i64, _f, _p, _i64, _p, _i32,
                                         _i32, _i32, _f, _p, _p, _p, _sz, _i32, _i32, _p, _p]),
    "mla_kv_append_fp8": (ctypes.c_int, [_p, _p, _p, _i64, _i64, _f, _p, _i64, _p, _i32, _i32,
                                         _p, _p]),
    "mla_quantize_queries_fp8": (ctypes.c_int, [_p, _p, _i64, _p, _p, _p]),
    "mla_merge_partials": (ctypes.c_int, [_p, _p, _i32, _i64, _p, _p, _p]),
    "mla_dcp_shard": (ctypes.c_int, [_p, _i64, _p, _i32, _i32, _i32, _p, _i64, _p, _p]),
    "mla_set_page_checks": (None, [_i32]),
    "mla_set_split_mode": (ctypes.c_int, [_i32]),
    "mla_get_split_mode": (_i32, []),
    "mla_set_team_clusters": (ctypes.c_int, [_i32]),
    "mla_get_team_clusters": (_i32, []),
    "mla_get_page_checks": (_i32, []),
}

_lib = None


class StageEvents(ctypes.Structure):
    """plmla_stage_events: cudaEvent_t handles (or None) recorded between kernels."""
    _fields_ = [("plan_begin", _p), ("decode_begin", _p), ("combine_begin", _p),
                ("combine_end", _p)]


class PlmlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} ({status})")


def header_functions():
    """Names of the functions include/plmla.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def lib():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is not built; run `python -m paged_latent_attention_gb300.build`")
    handle = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    _lib = handle
    return handle


def strerror(status: int) -> str:
    return lib().mla_strerror(int(status)).decode()


def check(status: int, where: str):
    if status != 0:
        raise PlmlaError(status, where)
