"""ctypes view of libpa.so.  Argument marshalling only; no arithmetic of the path.

The library must have been built (``__graft_entry__.build()`` or
``python -m paged_kv_cache_08_gb300.build``).  There is no fallback: if the
shared library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "_build" / "libpa.so"
HEADER = _PKG.parent / "include" / "pa.h"

c_int, c_i64, c_u64, c_size, c_f32, c_vp = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t,
                                            ctypes.c_float, ctypes.c_void_p)
c_i32p = ctypes.POINTER(ctypes.c_int32)
c_i64p = ctypes.POINTER(ctypes.c_int64)
c_u32p = ctypes.POINTER(ctypes.c_uint32)


class DecodeOptions(ctypes.Structure):
    _fields_ = [("tokens_per_split", c_int), ("math", c_int), ("num_ctas", c_int), ("flags", c_int),
                ("timeline", c_vp)]


PA_OK = 0
STATUS = {0: "PA_OK", -1: "PA_ERR_INVALID_ARG", -2: "PA_ERR_UNSUPPORTED", -3: "PA_ERR_CUDA",
          -4: "PA_ERR_POOL_EXHAUSTED", -5: "PA_ERR_DEVICE_TIMEOUT", -6: "PA_ERR_BOUNDS",
          -7: "PA_ERR_WORKSPACE", -8: "PA_ERR_SCRATCH_LIMIT"}
DEV_BAD_BLOCK_ID, DEV_BAD_CONTEXT, DEV_BAD_SLOT, DEV_TIMEOUT, DEV_BAD_PLAN = 0x1, 0x2, 0x4, 0x8, 0x10
MATH = {"auto": 0, "fma": 1, "mma": 2, "mma_split": 3}
EARLY_READS = 1
PREFILL_MMA_SYNC = 4
PLAN_ADAPTIVE = 8
PLAN_RUNS = 16

_SIGNATURES = {
    "pa_cache_write": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_int, c_int, c_int, c_vp]),
    "pa_copy_blocks": (c_int, [c_vp, c_vp, c_int, c_vp, c_vp, c_int, c_vp, c_vp, c_int, c_int, c_int, c_int, c_int,
                               c_vp]),
    "pa_decode": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f32, c_int, c_int, c_int, c_int, c_int, c_int,
                          c_int, c_int, c_vp, c_size, c_vp]),
    "pa_decode_ex": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f32, c_int, c_int, c_int, c_int, c_int, c_int,
                             c_int, c_int, c_vp, c_size, c_vp, ctypes.POINTER(DecodeOptions)]),
    "pa_decode_append": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f32, c_int, c_int, c_int, c_int,
                                 c_int, c_int, c_int, c_int, c_vp, c_size, c_vp, ctypes.POINTER(DecodeOptions)]),
    "pa_multi_query": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f32, c_int, c_int, c_int, c_int, c_int,
                               c_int, c_int, c_int, c_int, c_int, c_vp, c_size, c_vp, ctypes.POINTER(DecodeOptions)]),
    "pa_multi_query_append": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f32, c_int, c_int,
                                      c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_vp, c_size, c_vp,
                                      ctypes.POINTER(DecodeOptions)]),
    "pa_decode_runs": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f32, c_int, c_int, c_int, c_int, c_int, c_int,
                               c_int, c_int, c_vp, c_size, c_vp]),
    "pa_decode_runs_workspace_size": (c_size, [c_int, c_int, c_int, c_int, c_int, c_int]),
    "pa_gather_runs": (c_int, [c_vp, c_vp, c_int, c_vp, c_vp, c_int, c_vp, c_int, c_int, c_int, c_int, c_int, c_vp]),
    "pa_slots_create": (c_vp, [c_int, c_int]),
    "pa_slots_destroy": (None, [c_vp]),
    "pa_slots_alloc": (c_int, [c_vp, c_int, c_i32p, c_i32p]),
    "pa_slots_release": (c_int, [c_vp, c_int, c_int, c_int]),
    "pa_slots_tail": (c_int, [c_vp, c_int]),
    "pa_slots_live": (c_int, [c_vp, c_int]),
    "pa_slots_num_free": (c_int, [c_vp]),
    "pa_decode_static": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f32, c_int, c_int, c_int, c_int, c_int,
                                 c_int, c_int, c_int, c_vp]),
    "pa_decode_plan_size": (c_size, [c_int, c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(DecodeOptions)]),
    "pa_decode_plan": (c_int, [c_vp, c_size, c_vp, c_vp, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_vp,
                               ctypes.POINTER(DecodeOptions)]),
    "pa_decode_plan_sections": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(DecodeOptions),
                                        ctypes.POINTER(c_int), ctypes.POINTER(c_size), ctypes.POINTER(c_size)]),
    "pa_decode_planned_workspace_size": (c_size, [ctypes.POINTER(DecodeOptions)]),
    "pa_decode_plan_runs": (c_int, [c_vp, c_size, c_vp, c_vp, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_vp,
                                    ctypes.POINTER(DecodeOptions)]),
    "pa_decode_planned_workspace_init": (c_int, [c_vp, c_size, c_vp]),
    "pa_decode_planned": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_f32, c_int, c_int, c_int, c_int,
                                  c_int, c_int, c_int, c_int, c_vp, c_size, c_vp, ctypes.POINTER(DecodeOptions)]),
    "pa_decode_workspace_size": (c_size, [c_int, c_int, c_int, c_int, c_int, c_int]),
    "pa_decode_workspace_size_ex": (c_size, [c_int, c_int, c_int, c_int, c_int, c_int,
                                             ctypes.POINTER(DecodeOptions)]),
    "pa_decode_workspace_init": (c_int, [c_vp, c_size, c_vp]),
    "pa_decode_kernel_kind": (c_int, [c_int, c_int, c_int, ctypes.POINTER(DecodeOptions)]),
    "pa_decode_plan_tokens_per_split": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int,
                                                ctypes.POINTER(DecodeOptions)]),
    "pa_status_string": (ctypes.c_char_p, [c_int]),
    "pa_read_device_status": (c_int, [c_vp, c_int, c_u32p]),
    "pa_kernel_launch_count": (c_u64, []),
    "pa_pool_create": (c_vp, [c_int]),
    "pa_pool_destroy": (None, [c_vp]),
    "pa_pool_alloc": (c_int, [c_vp]),
    "pa_pool_incref": (c_int, [c_vp, c_int]),
    "pa_pool_decref": (c_int, [c_vp, c_int]),
    "pa_pool_refcount": (c_int, [c_vp, c_int]),
    "pa_pool_num_free": (c_int, [c_vp]),
    "pa_pool_num_blocks": (c_int, [c_vp]),
    "pa_pool_assign": (c_int, [c_vp, c_i32p, c_int, c_int, c_int, c_i32p, c_int]),
    "pa_pool_append_token": (c_int, [c_vp, c_i32p, c_int, c_int, c_int, c_i64p, c_i32p, c_i32p]),
    "pa_pool_release": (c_int, [c_vp, c_i32p, c_int, c_int, c_int]),
    "pa_pool_move_blocks": (c_int, [c_vp, c_vp, c_i32p, c_int, c_i32p, c_i32p]),
    "pa_build_slot_mapping": (c_int, [c_i32p, c_int, c_i32p, c_int, c_int, c_i64p]),
}

_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/pa.h declares."""
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not LIB_PATH.exists():
        raise RuntimeError(f"libpa.so not built ({LIB_PATH}); run `python -m paged_kv_cache_08_gb300.build` "
                           "or __graft_entry__.build() first")
    lib = ctypes.CDLL(str(LIB_PATH))
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class PAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({code})")


def check(fn: str, code: int) -> int:
    if code < 0:
        raise PAError(fn, code)
    return code
