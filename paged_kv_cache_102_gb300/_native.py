"""ctypes loader for libpagedkv.so (built in-tree by ``build.py``).

There is no fallback: if the library is missing or fails to load, every call
raises.  Argument types mirror include/pagedkv.h one to one.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedkv.so")

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I32 = ctypes.c_int
I64 = ctypes.c_int64
SZ = ctypes.c_size_t
F32 = ctypes.c_float

# name -> (restype, argtypes), in the order of include/pagedkv.h
SIGNATURES = {
    "paged_kv_append": (I32, [P, P, P, I32, P, P, I32, I32, I32, I32, I32, I32, P, P, P]),
    "paged_attention_decode": (I32, [P, P, P, P, I32, P, I32, I32, I32, I32, I32, I32, F32, P, I32, I32, P, P,
                                     I32, P, SZ, P]),
    "paged_attention_decode_append": (I32, [P, P, P, P, P, P, P, I32, P, I32, I32, I32, I32, I32, I32, F32, P,
                                            I32, I32, P, P, I32, P, SZ, P]),
    "paged_attention_decode_noalloc": (I32, [P, P, P, P, I32, P, I32, I32, I32, I32, I32, I32, F32, P, I32, I32,
                                             P, P, I32, P]),
    "paged_attention_decode_sparse": (I32, [P, P, P, P, I32, P, I32, I32, I32, I32, I32, I32, F32, P, I32, I32, P,
                                            P, I32, P, SZ, P]),
    "quest_block_minmax": (I32, [P, P, I32, P, I32, I32, I32, I32, I32, I32, I32, P, P]),
    "quest_append_minmax": (I32, [P, P, I32, I32, I32, I32, I32, I32, I32, P, P, P]),
    "quest_select": (I32, [P, P, P, I32, P, I32, I32, I32, I32, I32, I32, I32, I32, P, P, P, SZ, P]),
    "quest_workspace_size": (SZ, [I32, I32, I32]),
    "pkv_workspace_size": (SZ, [I32, I32, I32, I32, I32, I32, I32]),
    "pkv_resolve_partition_size": (I32, [I32, I32, I32, I32, I32, I32, I32]),
    "paged_block_copy": (I32, [P, P, P, I32, I32, SZ, P]),
    "paged_block_swap": (I32, [P, P, P, I32, I32, SZ, P, I32, P]),
    "pkv_last_error": (ctypes.c_char_p, []),
    "pkv_device_error": (I32, [P, I32, P]),
    "pkv_version": (I32, []),
    "pkv_selftest_wait_timeout": (I32, [I32, P]),
    "pkv_set_kernel_path": (I32, [I32]),
    "pkv_bm_create": (P, [I32, I32, P, I32]),
    "pkv_bm_destroy": (None, [P]),
    "pkv_bm_add_sequence": (I32, [P, I64, I32]),
    "pkv_bm_append_slots": (I32, [P, P, I32, P, P, P]),
    "pkv_bm_append_tokens": (I32, [P, P, P, I32, P, P, P]),
    "pkv_bm_fork": (I32, [P, I64, I64]),
    "pkv_bm_free_sequence": (I32, [P, I64]),
    "pkv_bm_get_tables": (I32, [P, P, I32, P, I32, I32, P]),
    "pkv_bm_add_sequence_cached": (I32, [P, I64, P, I32, P]),
    "pkv_bm_num_cached_blocks": (I32, [P]),
    "pkv_bm_swap_out_group": (I32, [P, P, I32, P, I32, P]),
    "pkv_bm_swap_in_group": (I32, [P, P, I32, P, I32, P]),
    "pkv_bm_swap_out": (I32, [P, I64, P, I32, P]),
    "pkv_bm_swap_in": (I32, [P, I64, P, I32, P]),
    "pkv_bm_num_free": (I32, [P]),
    "pkv_bm_ref_count": (I32, [P, I32]),
    "pkv_bm_context_len": (I32, [P, I64]),
    "pkv_bm_num_seq_blocks": (I32, [P, I64]),
    "pkv_bm_free_list": (I32, [P, P, I32]),
}


class PagedKVError(RuntimeError):
    def __init__(self, func: str, code: int, msg: str):
        super().__init__(f"{func} failed with status {code}: {msg}")
        self.code = code


_fns: dict = {}


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: run paged_kv_cache_102_gb300.build.build() "
                                  "(or __graft_entry__.build()) first; there is no CPU fallback")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def check(func: str, code: int) -> None:
    if code != 0:
        raise PagedKVError(func, code, lib().pkv_last_error().decode())


def function(func: str):
    """The library's C function `func` with its declared argument types."""
    fn = _fns.get(func)
    if fn is None:
        fn = _fns[func] = getattr(lib(), func)
    return fn


def call(func: str, *args) -> None:
    fn = _fns.get(func)
    if fn is None:
        fn = _fns[func] = getattr(lib(), func)
    code = fn(*args)
    if code != 0:
        raise PagedKVError(func, code, lib().pkv_last_error().decode())
