"""ctypes declarations of the C ABI in include/pa.h (argument marshalling only).

``load()`` opens the in-tree ``libpa_gb300.so`` and raises if it is missing:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa_gb300.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_CUDA = 3
PA_ERR_OOM = 4
PA_ERR_WORKSPACE = 5
PA_ERR_DEVICE_TIMEOUT = 6

PA_DTYPE_F32 = 0
PA_DTYPE_BF16 = 1

i32 = C.c_int32
i64 = C.c_int64
vp = C.c_void_p
P_i32 = C.POINTER(C.c_int32)
P_i64 = C.POINTER(C.c_int64)

# name -> (restype, argtypes); every symbol include/pa.h declares
SIGNATURES = {
    "pa_status_string": (C.c_char_p, [i32]),
    "pa_version": (C.c_char_p, []),
    "pa_reshape_and_cache": (i32, [vp, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, vp]),
    "pa_copy_blocks": (i32, [vp, vp, i32, i32, i32, i32, i32, vp, i32, vp]),
    "pa_reshape_and_cache_checked": (i32, [vp, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]),
    "pa_copy_blocks_checked": (i32, [vp, vp, i32, i32, i32, i32, i32, vp, i32, vp, vp]),
    "pa_reshape_and_cache_layers": (i32, [vp, vp, i64, i32, i32, vp, vp, vp, i64, i32, i32, i32,
                                          i32, i32, vp]),
    "pa_copy_blocks_layers": (i32, [vp, vp, i64, i32, i32, i32, i32, i32, i32, vp, i32, vp]),
    "pa_decode_workspace_size": (C.c_size_t, [i32, i32, i32, i32, i32, i32, i32, i32]),
    "pa_decode_shared_prefix_workspace_size": (C.c_size_t, [i32, i32, i32, i32, i32, i32]),
    "pa_decode_shared_prefix": (i32, [vp, i32, vp, i32, i32, vp, vp, i32, i32, i32, i32, i32, vp, i32, vp,
                                      i32, vp, vp, i32, i32, i32, C.c_float, vp, vp, C.c_size_t, vp]),
    "pa_prefill": (i32, [vp, i32, vp, i32, vp, vp, i32, i32, i32, vp, vp, i32, i32, i32, i32, i32, vp,
                         i32, C.c_float, vp, vp]),
    "pa_decode": (i32, [vp, i32, vp, i32, i32, vp, vp, i32, i32, i32, i32, i32, vp, i32, vp, i32,
                        C.c_float, i32, vp, C.c_size_t, vp]),
    "pa_decode_no_alloc": (i32, [vp, i32, vp, i32, i32, vp, vp, i32, i32, i32, i32, i32, vp, i32,
                                 vp, i32, C.c_float, i32, vp]),
    "pa_decode_no_alloc_error": (i32, [vp, P_i32]),
    "pa_set_decode_kv_per_item": (i32, [i32]),
    "pa_decode_plan": (i32, [i32, i32, i32, i32, i32, i32, i32, i32, P_i32, P_i32]),
    "pa_workspace_init": (i32, [vp, C.c_size_t, vp]),
    "pa_test_stall_decode": (None, [C.c_uint64]),
    "pa_workspace_error": (i32, [vp, vp, P_i32]),
    "pa_alloc_create": (i32, [i32, i32, P_i32, C.POINTER(vp)]),
    "pa_alloc_destroy": (None, [vp]),
    "pa_alloc_num_blocks": (i32, [vp]),
    "pa_alloc_block_size": (i32, [vp]),
    "pa_alloc_num_free": (i32, [vp]),
    "pa_alloc_refcount": (i32, [vp, i32]),
    "pa_alloc_allocate": (i32, [vp, P_i32]),
    "pa_alloc_incref": (i32, [vp, i32]),
    "pa_alloc_decref": (i32, [vp, i32]),
    "pa_alloc_seq_create": (i32, [vp, P_i32]),
    "pa_alloc_fork": (i32, [vp, i32, P_i32]),
    "pa_alloc_append_slot": (i32, [vp, i32, P_i64, P_i32, P_i32]),
    "pa_alloc_append_slots": (i32, [vp, P_i32, i32, P_i64, P_i64, P_i32, P_i32]),
    "pa_alloc_append_tokens": (i32, [vp, i32, i32, P_i64]),
    "pa_alloc_free_seq": (i32, [vp, i32]),
    "pa_alloc_seq_len": (i32, [vp, i32]),
    "pa_alloc_num_seqs": (i32, [vp]),
    "pa_alloc_block_table": (i32, [vp, i32, P_i32, i32, P_i32]),
    "pa_alloc_export_tables": (i32, [vp, P_i32, i32, P_i32, i32, P_i32, i32]),
    "pa_alloc_free_list": (i32, [vp, P_i32, i32, P_i32]),
    "pa_alloc_live_seqs": (i32, [vp, P_i32, i32, P_i32]),
    "pa_alloc_enable_prefix_cache": (i32, [vp]),
    "pa_alloc_seq_create_prefix": (i32, [vp, P_i32, i32, vp, i32, P_i32, P_i32, P_i64]),
    "pa_alloc_append_token_ids": (i32, [vp, i32, P_i32, i32, P_i64]),
    "pa_alloc_num_cached": (i32, [vp]),
    "pa_alloc_block_key": (i32, [vp, i32, C.c_char_p]),
    "pa_sha256": (i32, [vp, C.c_size_t, C.c_char_p]),
}

_lib = None
_lock = threading.Lock()


class PAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = status_string(status) if _lib is not None else str(status)
        super().__init__(f"{what}: {name}" if what else name)


def load() -> C.CDLL:
    """Open libpa_gb300.so (built by ``paged_kv_cache_142_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m paged_kv_cache_142_gb300.build` (no CPU fallback exists)")
            lib = C.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def check(status: int, what: str = "") -> None:
    if status != PA_OK:
        raise PAError(status, what)
