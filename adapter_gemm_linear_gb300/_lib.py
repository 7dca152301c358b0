"""ctypes declarations of the C ABI in include/lora.h (argument marshalling only).

The library is loaded from the package's in-tree ``_build/liblora.so``.  If it
is missing, ``lib()`` raises: there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

LORA_BLOCK_ROWS = 16
LORA_MAX_PROJ = 4

STATUS_NAMES = {
    0: "LORA_OK",
    1: "LORA_ERR_INVALID_ARG",
    2: "LORA_ERR_ALIGNMENT",
    3: "LORA_ERR_DTYPE",
    4: "LORA_ERR_RANK",
    5: "LORA_ERR_SLOT",
    6: "LORA_ERR_OUT_OF_BLOCKS",
    7: "LORA_ERR_ADAPTER_ID",
    8: "LORA_ERR_SEGMENTS",
    9: "LORA_ERR_CUDA",
    10: "LORA_ERR_DEVICE_TIMEOUT",
    11: "LORA_ERR_DEVICE_INDEX",
    12: "LORA_ERR_WORKSPACE",
    13: "LORA_ERR_UNSUPPORTED",
}
STATUS = {v: k for k, v in STATUS_NAMES.items()}

LORA_BF16 = 0
LORA_FP32 = 1
ABI_VERSION = 5  # include/lora.h LORA_ABI_VERSION


class PoolDesc(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("K", ctypes.c_int32),
        ("N", ctypes.c_int32),
        ("max_slots", ctypes.c_int32),
        ("max_rank", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("a_arena", ctypes.c_void_p),
        ("b_arena", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("ranks", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("free_list_seed", ctypes.c_uint64),
    ]


class Proj(ctypes.Structure):
    _fields_ = [
        ("W", ctypes.c_void_p),
        ("pool", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("ldo", ctypes.c_int32),
        ("w_scale", ctypes.c_void_p),
        ("w_bits", ctypes.c_int32),
    ]


class ForwardArgs(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("M", ctypes.c_int32),
        ("K", ctypes.c_int32),
        ("x", ctypes.c_void_p),
        ("ldx", ctypes.c_int32),
        ("n_proj", ctypes.c_int32),
        ("proj", ctypes.POINTER(Proj)),
        ("row_adapter", ctypes.c_void_p),
        ("seg_offsets", ctypes.c_void_p),
        ("seg_adapter", ctypes.c_void_p),
        ("perm", ctypes.c_void_p),
        ("num_segs", ctypes.c_int32),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("stage_events", ctypes.POINTER(ctypes.c_void_p)),
        ("num_stage_events", ctypes.c_int32),
        ("scales", ctypes.c_void_p),
    ]


# (name, restype, argtypes) of every entry point declared in include/lora.h
SIGNATURES = [
    ("lora_pool_create", ctypes.c_int,
     [ctypes.POINTER(PoolDesc), ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]),
    ("lora_pool_destroy", ctypes.c_int, [ctypes.c_void_p]),
    ("lora_pool_load_slot", ctypes.c_int,
     [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p,
      ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    ("lora_pool_unload_slot", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    ("lora_pool_touch", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    ("lora_pool_pin", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    ("lora_pool_unpin", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    ("lora_pool_evict_lru", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    ("lora_pool_slot_use", ctypes.c_int,
     [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)]),
    ("lora_pool_slot_info", ctypes.c_int,
     [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
      ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int32)]),
    ("lora_pool_free_blocks", ctypes.c_int32, [ctypes.c_void_p]),
    ("lora_pool_get_desc", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(PoolDesc)]),
    ("lora_pool_slot_bytes", ctypes.c_size_t,
     [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int]),
    ("lora_pool_arena_bytes", ctypes.c_size_t,
     [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int]),
    ("lora_segment_rows", ctypes.c_int,
     [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
      ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    ("lora_forward_workspace_bytes", ctypes.c_size_t, [ctypes.POINTER(ForwardArgs)]),
    ("lora_linear_forward", ctypes.c_int, [ctypes.POINTER(ForwardArgs), ctypes.c_void_p]),
    ("lora_linear_forward_noalloc", ctypes.c_int, [ctypes.POINTER(ForwardArgs), ctypes.c_void_p]),
    ("lora_get_device_status", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    ("lora_test_arm_wait_timeout", ctypes.c_int, [ctypes.c_uint64]),
    ("lora_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("lora_last_cuda_error", ctypes.c_int32, []),
    ("lora_cuda_error_name", ctypes.c_char_p, [ctypes.c_int32]),
    ("lora_abi_version", ctypes.c_int32, []),
    ("lora_kernel_launches", ctypes.c_uint64, []),
]

_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def lib():
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"liblora.so not found at {path}; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(path)
            for name, res, args in SIGNATURES:
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            if L.lora_abi_version() != ABI_VERSION:  # the structs below follow this version's layout
                raise RuntimeError(f"{path} has ABI {L.lora_abi_version()}, this binding {ABI_VERSION}; rebuild it")
            _lib = L
    return _lib
