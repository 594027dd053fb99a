"""ctypes binding of libh3kern.so (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_LOCK = threading.Lock()
_LIB = None

c_int, c_int64, c_float, c_void_p = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p


class AttnGroup(ctypes.Structure):
    """h3_attn_group: one query group and its two KV views."""
    _fields_ = [("q_start", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("kv_start", ctypes.c_int32), ("kv_len", ctypes.c_int32),
                ("cache_start", ctypes.c_int32), ("cache_len", ctypes.c_int32)]
c_i32p = ctypes.POINTER(ctypes.c_int32)
c_u32p = ctypes.POINTER(ctypes.c_uint32)

# name -> (restype, argtypes); the symbols include/h3kern.h and
# include/h3kern_debug.h declare.
SIGNATURES = {
    "h3_qk_norm_rope": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_void_p,
                                c_void_p, c_int64, c_int, c_int, c_int, c_int, c_int,
                                c_float, c_float, c_void_p]),
    "h3_qk_norm_rope_varlen": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_void_p,
                                       c_void_p, c_i32p, c_i32p, c_int, c_int, c_int, c_int, c_int,
                                       c_int, c_float, c_float, c_void_p]),
    "h3_qk_norm_rope_lora": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int64,
                                     c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_int64,
                                     c_int, c_int, c_int, c_int, c_int, c_float, c_float,
                                     c_void_p]),
    "h3_attention": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int64,
                             c_void_p, c_int64, c_i32p, c_i32p, c_i32p, c_int, c_int, c_int,
                             c_float, c_void_p]),
    "h3_attention_groups": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int64,
                                    c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int64,
                                    c_void_p, c_int, c_int, c_int, c_float, c_void_p]),
    "h3_block_means": (c_int, [c_void_p, c_int64, c_int64, c_int, c_int, c_void_p, c_void_p]),
    "h3_block_means_qk": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_int64, c_int, c_int,
                                  c_void_p, c_void_p, c_void_p]),
    "h3_block_select": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_float, c_float, c_int,
                                c_void_p, c_void_p, c_void_p, c_void_p]),
    "h3_sparse_attention": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int64,
                                    c_void_p, c_int64, c_int64, c_int, c_int, c_void_p, c_void_p,
                                    c_int, c_float, c_void_p]),
    "h3_wire_record_bytes": (c_int, [c_int, c_int]),
    "h3_pack_qkv": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int64, c_int64,
                            c_int, c_int, c_int, c_void_p, c_void_p]),
    "h3_unpack_qkv": (c_int, [c_void_p, c_int64, c_int, c_int, c_void_p, c_int64, c_void_p,
                              c_int64, c_void_p, c_int64, c_void_p]),
    "h3_pack_out": (c_int, [c_void_p, c_int64, c_int64, c_int, c_int, c_void_p, c_void_p]),
    "h3_merge_heads": (c_int, [c_void_p, c_int64, c_int, c_int, c_int, c_void_p, c_int64,
                               c_void_p]),
    "h3_copy_2d": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_int64, c_int64, c_void_p]),
    "h3_last_error": (ctypes.c_char_p, []),
    "h3_status_word": (c_int, [c_u32p]),
    "h3_version": (c_int, []),
    "h3_debug_fault_next_attention": (c_int, [c_int]),
}

STATUS = {0: "H3_OK", -1: "H3_ERR_ARG", -2: "H3_ERR_ALIGN", -3: "H3_ERR_SHAPE",
          -4: "H3_ERR_ARCH", -5: "H3_ERR_LAUNCH", -6: "H3_ERR_TIMEOUT", -7: "H3_ERR_DEVICE"}


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libh3kern.so (building it first if asked).  Raises if absent:
    there is no fallback implementation."""
    global _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        path = lib_path()
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libh3kern.so not found at {path}; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
        return lib
