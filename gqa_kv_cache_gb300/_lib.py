"""ctypes declarations of libgqa.so (the C ABI in include/gqa_decode.h)."""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgqa.so")

P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t

# name -> (restype, argtypes); the exported C functions of include/gqa_decode.h
SIGNATURES = {
    "gqa_status_string": (ctypes.c_char_p, [I]),
    "gqa_workspace_bytes": (Z, [I, I, I, I, I, P]),
    "gqa_workspace_reset": (I, [P, Z, P]),
    "gqa_decode_step": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, Z, P, P]),
    "gqa_decode_step_paged": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, Z, P, P]),
    "gqa_decode_step_ex": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, Z, P, P, P]),
    "gqa_decode_step_paged_ex": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, Z, P, P, P]),
    "gqa_validate": (I, [P, P, P, I, I, I, I, I, I, P, P]),
    "gqa_validate_attend": (I, [P, P, P, I, I, I, I, I, I, P, P]),
    "gqa_attend": (I, [P, I, P, P, P, P, P, I, I, I, I, I, I, I, P, Z, P, P, P]),
    "gqa_workspace_bytes_multi": (Z, [I, I, I, I, I, I, P]),
    "gqa_decode_multi": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, Z, P, P, P]),
    "gqa_decode_multi_paged": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, P, Z, P, P,
                                   P]),
    "gqa_validate_multi": (I, [P, P, P, P, I, I, I, I, I, I, I, P, P]),
    "gqa_attend_paged": (I, [P, I, P, P, P, P, P, I, I, I, I, I, I, I, I, P, Z, P, P, P]),
    "gqa_trace_enable": (I, [I]),
    "gqa_trace_collect": (I, [I, P, P]),
    "gqa_kernel_name": (ctypes.c_char_p, [I]),
    "gqa_version": (I, []),
    "gqa_noalloc_scratch_bytes": (Z, []),
    "gqa_decode_step_noalloc": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P]),
}


class GqaOptions(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("grid_ctas", ctypes.c_int),
                ("sched_pad", ctypes.c_int), ("window", ctypes.c_int),
                ("kept_prefix", ctypes.c_int), ("wait_limit_cycles", ctypes.c_int),
                ("test_stall", ctypes.c_int), ("reserved", ctypes.c_int * 1),
                ("head_sink", ctypes.c_void_p), ("kept_prefix_rows", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """The loaded library. Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                    "g.build()'` (or python gqa_kv_cache_gb300/build.py)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
