"""Float64 CPU oracle for the paged KV-cache decode path.

TEST INFRASTRUCTURE ONLY.  The product package never imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may load it.  It shares no code with the CUDA library: the
arithmetic lives in ``oracle.c`` (float64 attention, element-format
decoders, the E4M3 encoder, scatter append and block copy) and in
``block_manager_ref.py`` (a naive re-statement of the block allocator).

All arrays passed here are numpy arrays holding raw element bits: uint16 for
binary16/bfloat16, uint8 for E4M3.  Element-type codes: ``F16 = 0``,
``BF16 = 1``, ``E4M3 = 2``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, BF16, E4M3 = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc (OpenMP on)."""
    stale = not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64, f32, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_float, ctypes.c_size_t
            lib.oracle_paged_decode.argtypes = [P, i32, P, P, i32, f64, f64, P, i32, P,
                                                i32, i32, i32, i32, i32, i32, f64, P]
            lib.oracle_paged_decode.restype = i32
            lib.oracle_append.argtypes = [P, P, i32, P, i32, P, P, i32, i32, i32, i32, i32, f32, f32]
            lib.oracle_append.restype = i32
            lib.oracle_block_copy.argtypes = [P, P, P, i32, i32, sz]
            lib.oracle_block_copy.restype = i32
            lib.oracle_block_swap.argtypes = [P, P, P, i32, i32, sz, P, i32]
            lib.oracle_block_swap.restype = i32
            lib.oracle_decode_array.argtypes = [P, i32, sz, P]
            lib.oracle_decode_array.restype = None
            lib.oracle_e4m3_encode_array.argtypes = [P, sz, P]
            lib.oracle_e4m3_encode_array.restype = None
            lib.oracle_quest_select.argtypes = [P, i32, P, i32, f64, P, i32, P, i32, i32, i32, i32, i32, i32, i32,
                                                P, P, P]
            lib.oracle_quest_select.restype = i32
            lib.oracle_sparse_decode.argtypes = [P, i32, P, P, i32, f64, f64, P, i32, P, i32, i32, i32, i32, i32,
                                                 i32, f64, P]
            lib.oracle_sparse_decode.restype = i32
            lib.oracle_quest_block_minmax.argtypes = [P, i32, P, i32, P, i32, i32, i32, i32, i32, P, P]
            lib.oracle_quest_block_minmax.restype = i32
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i32
            del i64
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(a: np.ndarray, dtype: int) -> np.ndarray:
    want = np.uint8 if dtype == E4M3 else np.uint16
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        a = a.view(want)
    return a


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def decode_elements(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Element bits -> float64 (E4M3 without any scale)."""
    bits = _bits(bits, dtype)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode_array(_ptr(bits), dtype, bits.size, _ptr(out))
    return out


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """binary32 -> E4M3 codes, round to nearest even, saturating to +-448."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def paged_decode(q, q_dtype, k_cache, v_cache, cache_dtype, block_tables, context_lens,
                 scale, k_scale=1.0, v_scale=1.0):
    """Float64 paged decode attention.

    q: [B, Hq, D] bits; k_cache, v_cache: [NB, Hkv, bs, D] bits;
    block_tables: int32 [B, max_blocks]; context_lens: int32 [B].
    Returns float64 [B, Hq, D].
    """
    q = _bits(q, q_dtype)
    k_cache = _bits(k_cache, cache_dtype)
    v_cache = _bits(v_cache, cache_dtype)
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape
    assert block_tables.shape[0] == B and context_lens.shape == (B,)
    out = np.empty((B, Hq, D), dtype=np.float64)
    rc = _load().oracle_paged_decode(_ptr(q), q_dtype, _ptr(k_cache), _ptr(v_cache), cache_dtype,
                                     float(k_scale), float(v_scale), _ptr(block_tables),
                                     block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, bs, D, NB,
                                     float(scale), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_paged_decode rejected its arguments (rc={rc})")
    return out


def append(k, v, act_dtype, slot_mapping, k_cache, v_cache, cache_dtype, k_scale=1.0, v_scale=1.0):
    """Scatter new K/V rows into the caches in place (see oracle.c)."""
    k = _bits(k, act_dtype)
    v = _bits(v, act_dtype)
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
    T, Hkv, D = k.shape
    NB, Hkv2, bs, D2 = k_cache.shape
    assert Hkv2 == Hkv and D2 == D
    rc = _load().oracle_append(_ptr(k), _ptr(v), act_dtype, _ptr(slot_mapping), T,
                               _ptr(k_cache), _ptr(v_cache), cache_dtype, NB, Hkv, bs, D,
                               float(k_scale), float(v_scale))
    if rc != 0:
        raise ValueError("oracle_append: slot outside the pool or unsupported types")


def block_copy(k_cache, v_cache, src_dst_pairs):
    """Copy whole physical blocks, K and V, for every (src, dst) pair, in order."""
    pairs = np.ascontiguousarray(src_dst_pairs, dtype=np.int32).reshape(-1, 2)
    NB = k_cache.shape[0]
    block_bytes = k_cache[0].nbytes
    rc = _load().oracle_block_copy(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), pairs.shape[0], NB, block_bytes)
    if rc != 0:
        raise ValueError("oracle_block_copy: block id outside the pool")


def block_swap_out(k_cache, v_cache, block_ids) -> np.ndarray:
    """Staging bytes [n, 2, block_bytes]: entry i = K block ids[i], then V block ids[i]."""
    ids = np.ascontiguousarray(block_ids, dtype=np.int32).reshape(-1)
    assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
    NB = k_cache.shape[0]
    block_bytes = k_cache[0].nbytes
    staging = np.zeros((len(ids), 2, block_bytes), np.uint8)
    rc = _load().oracle_block_swap(_ptr(k_cache), _ptr(v_cache), _ptr(ids), len(ids), NB, block_bytes,
                                   _ptr(staging), 0)
    if rc != 0:
        raise ValueError("oracle_block_swap: block id outside the pool")
    return staging


def block_swap_in(k_cache, v_cache, block_ids, staging) -> None:
    """Write staging entry i back into block ids[i] of both caches, in place."""
    ids = np.ascontiguousarray(block_ids, dtype=np.int32).reshape(-1)
    staging = np.ascontiguousarray(staging, dtype=np.uint8)
    NB = k_cache.shape[0]
    block_bytes = k_cache[0].nbytes
    assert staging.shape == (len(ids), 2, block_bytes)
    rc = _load().oracle_block_swap(_ptr(k_cache), _ptr(v_cache), _ptr(ids), len(ids), NB, block_bytes,
                                   _ptr(staging), 1)
    if rc != 0:
        raise ValueError("oracle_block_swap: block id outside the pool")


def quest_select(q, q_dtype, k_cache, cache_dtype, block_tables, context_lens, budget_blocks, k_scale=1.0):
    """QUEST top-K block selection per (sequence, kv head) (see oracle.c).
    Returns (sel_tables int32 [B, Hkv, budget], sel_lens int32 [B, Hkv],
    bounds float64 [B, Hkv, max_blocks])."""
    q = _bits(q, q_dtype)
    k_cache = _bits(k_cache, cache_dtype)
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    sel = np.zeros((B, Hkv, budget_blocks), np.int32)
    lens = np.zeros((B, Hkv), np.int32)
    bounds = np.full((B, Hkv, block_tables.shape[1]), np.nan)
    rc = _load().oracle_quest_select(_ptr(q), q_dtype, _ptr(k_cache), cache_dtype, float(k_scale),
                                     _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, bs,
                                     D, NB, int(budget_blocks), _ptr(sel), _ptr(lens), _ptr(bounds))
    if rc != 0:
        raise ValueError(f"oracle_quest_select rejected its arguments (rc={rc})")
    return sel, lens, bounds


def quest_block_minmax(k_cache, cache_dtype, block_tables, context_lens):
    """Channel-wise min and max of each (sequence, logical block, kv head)'s filled keys:
    two float64 arrays [B, max_blocks, Hkv, D] (NaN past the context)."""
    k_cache = _bits(k_cache, cache_dtype)
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    NB, Hkv, bs, D = k_cache.shape
    B, maxb = block_tables.shape
    mn = np.empty((B, maxb, Hkv, D))
    mx = np.empty((B, maxb, Hkv, D))
    rc = _load().oracle_quest_block_minmax(_ptr(k_cache), cache_dtype, _ptr(block_tables), maxb, _ptr(context_lens),
                                           B, Hkv, bs, D, NB, _ptr(mn), _ptr(mx))
    if rc != 0:
        raise ValueError("oracle_quest_block_minmax rejected its arguments")
    return mn, mx


def sparse_decode(q, q_dtype, k_cache, v_cache, cache_dtype, tables, lens, scale, k_scale=1.0, v_scale=1.0):
    """Attention over per-(sequence, kv head) block lists: tables [B, Hkv, max_blocks], lens [B, Hkv]."""
    q = _bits(q, q_dtype)
    k_cache = _bits(k_cache, cache_dtype)
    v_cache = _bits(v_cache, cache_dtype)
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    out = np.empty((B, Hq, D), np.float64)
    rc = _load().oracle_sparse_decode(_ptr(q), q_dtype, _ptr(k_cache), _ptr(v_cache), cache_dtype, float(k_scale),
                                      float(v_scale), _ptr(tables), tables.shape[2], _ptr(lens), B, Hq, Hkv, bs, D,
                                      NB, float(scale), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_sparse_decode rejected its arguments (rc={rc})")
    return out


def slot_of(block_table, pos: int, block_size: int) -> int:
    """Flat slot of token ``pos``: table[pos // bs] * bs + pos % bs
    (Ultralytics glossary "PagedAttention", section "How paging works")."""
    return int(block_table[pos // block_size]) * block_size + pos % block_size
