"""Paged KV-cache decode on GB300 (sm_103a).

Python binding over the C ABI of ``libpagedkv.so`` (include/pagedkv.h).  The
functions here only marshal torch tensors into pointers and sizes; all device
work runs in the library's CUDA kernels, and the block manager runs in the
library's C++ host code.  There is no CPU fallback: a missing library raises.

    paged_kv_append(k, v, slot_mapping, k_cache, v_cache, ...)
    paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, ...)
    paged_attention_decode_append(q, k_new, v_new, slot_mapping, k_cache, v_cache, ...)
    DecodePlan(...).run()   # either of the two above, marshalled once for fixed buffers
    paged_block_copy(k_cache, v_cache, src_dst_pairs, ...)
    BlockManager(num_blocks, block_size, free_list=None)

Cache tensors are [num_blocks, num_kv_heads, block_size, head_dim], float16 or
bfloat16, or uint8 / float8_e4m3fn holding E4M3 codes with float32 per-tensor
scales (1-element CUDA tensors).
"""
from __future__ import annotations

import ctypes
import threading

import numpy as np
import torch

from . import _native
from ._native import PagedKVError

F16, BF16, E4M3 = 0, 1, 2
PARTITION_SINGLE = 0
PARTITION_AUTO = -1

ERR_INVALID, ERR_SHAPE, ERR_CUDA, ERR_NO_SPACE, ERR_NOT_FOUND = 1, 2, 3, 4, 5
DEV_BAD_BLOCK, DEV_BAD_CONTEXT_LEN, DEV_BAD_SLOT, DEV_BAD_PAIR, DEV_WAIT_TIMEOUT = 1, 2, 4, 8, 16
PATH_AUTO, PATH_CUDA_CORE, PATH_TENSOR, PATH_TENSOR_2CTA = 0, 1, 2, 3
SWAP_OUT, SWAP_IN = 0, 1

__all__ = ["paged_kv_append", "paged_attention_decode", "paged_attention_decode_append", "DecodePlan",
           "paged_block_copy",
           "paged_block_swap", "paged_attention_decode_sparse", "quest_block_minmax", "quest_append_minmax",
           "quest_select", "workspace_size",
           "resolve_partition_size", "device_error", "set_kernel_path", "BlockManager", "OutOfBlocks", "PagedKVError",
           "F16", "BF16", "E4M3", "PARTITION_SINGLE", "PARTITION_AUTO", "load"]


class OutOfBlocks(PagedKVError):
    pass


def load():
    """Load libpagedkv.so (raises if it was not built)."""
    return _native.lib()


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return E4M3
    raise TypeError(f"unsupported element type {t.dtype}")


def _ptr(t):
    # ctypes converts a Python int for a c_void_p argument
    return None if t is None else t.data_ptr()


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _require_out(device, out):
    """`out` may be a CUDA tensor on `device` or a pinned host tensor, which the
    kernels write directly over the host link."""
    if out.is_pinned() and not out.is_cuda:
        if not out.is_contiguous():
            raise ValueError("out must be contiguous")
        return
    _require_cuda(device, out=out)


def _require_cuda(device, **tensors):
    index = device.index if device.index is not None else torch.cuda.current_device()
    for name, t in tensors.items():
        if t is None:
            continue
        if t.get_device() != index:  # -1 for a CPU tensor
            raise ValueError(f"{name} must be a CUDA tensor on {device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


def paged_kv_append(k, v, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None, stream=None):
    """Write k, v [T, Hkv, D] into their slots (int64 [T], negative = skip)."""
    T, Hkv, D = k.shape
    NB, Hkv2, bs, D2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or Hkv2 != Hkv or D2 != D:
        raise ValueError("paged_kv_append: shape mismatch")
    if slot_mapping.dtype != torch.int64 or slot_mapping.shape != (T,):
        raise ValueError("paged_kv_append: slot_mapping must be int64 [num_tokens]")
    _require_cuda(k.device, k=k, v=v, slot_mapping=slot_mapping, k_cache=k_cache, v_cache=v_cache,
                  k_scale=k_scale, v_scale=v_scale)
    _native.call("paged_kv_append", _ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache), _ptr(v_cache),
                 NB, Hkv, bs, D, _code(k), _code(k_cache), _ptr(k_scale), _ptr(v_scale),
                 _stream(stream, k.device))


def set_kernel_path(path: int) -> int:
    """Select the decode kernel (PATH_*) for later calls; returns the previous choice."""
    prev = int(_native.lib().pkv_set_kernel_path(int(path)))
    if prev < 0:
        raise ValueError(f"unknown kernel path {path}")
    return prev


def resolve_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
                           partition_size=PARTITION_AUTO):
    return int(_native.lib().pkv_resolve_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                        max_blocks_per_seq, block_size, partition_size))


def workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
                   partition_size=PARTITION_AUTO) -> int:
    return int(_native.lib().pkv_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                max_blocks_per_seq, block_size, partition_size))


_ws_lock = threading.Lock()
_ws_cache: dict = {}


def _workspace(device, stream_ptr: int, nbytes: int) -> torch.Tensor:
    """A reusable workspace per (device, stream): calls on one stream are ordered."""
    key = (device.index, stream_ptr)
    with _ws_lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
            _ws_cache[key] = buf
        return buf


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out=None, k_scale=None,
                           v_scale=None, partition_size=PARTITION_AUTO, workspace=None, stream=None):
    """Decode attention for q [B, Hq, D] over the paged cache; returns out [B, Hq, D]."""
    args, out, _ = _decode_args(q, k_cache, v_cache, block_tables, context_lens, scale, out, k_scale, v_scale,
                                partition_size, workspace, stream)
    _native.call("paged_attention_decode", *args)
    return out


def _decode_args(q, k_cache, v_cache, block_tables, context_lens, scale, out, k_scale, v_scale, partition_size,
                 workspace, stream):
    """Validated C arguments of paged_attention_decode, the output and the workspace."""
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("paged_attention_decode: shape mismatch")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("paged_attention_decode: block_tables and context_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("paged_attention_decode: block_tables [B, max_blocks], context_lens [B]")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("paged_attention_decode: out must match q")
    _require_out(q.device, out)
    _require_cuda(q.device, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
                  context_lens=context_lens, k_scale=k_scale, v_scale=v_scale, workspace=workspace)
    max_blocks = block_tables.shape[1]
    s = _stream(stream, q.device)
    if workspace is None:
        need = workspace_size(B, Hq, Hkv, D, max_blocks, bs, partition_size)
        if need:
            workspace = _workspace(q.device, s, need)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_blocks, _ptr(context_lens), B, Hq, Hkv,
            bs, D, NB, float(scale), _ptr(out), _code(q), _code(k_cache), _ptr(k_scale), _ptr(v_scale),
            int(partition_size), _ptr(workspace), ws_bytes, s)
    return args, out, workspace


def paged_attention_decode_append(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, context_lens, scale,
                                  out=None, k_scale=None, v_scale=None, partition_size=PARTITION_AUTO, workspace=None,
                                  stream=None):
    """Append each sequence's new K/V row (k_new, v_new [B, Hkv, D] at slot_mapping int64 [B]) and decode, in one
    launch; context_lens count the new token.  Returns out [B, Hq, D]."""
    args, out, _ = _decode_append_args(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, context_lens,
                                       scale, out, k_scale, v_scale, partition_size, workspace, stream)
    _native.call("paged_attention_decode_append", *args)
    return out


def _decode_append_args(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, context_lens, scale, out,
                        k_scale, v_scale, partition_size, workspace, stream):
    """Validated C arguments of paged_attention_decode_append, the output and the workspace."""
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or k_new.shape != (B, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("paged_attention_decode_append: shape mismatch")
    if slot_mapping.dtype != torch.int64 or slot_mapping.shape != (B,):
        raise ValueError("paged_attention_decode_append: slot_mapping must be int64 [num_seqs]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("paged_attention_decode_append: block_tables and context_lens must be int32")
    if out is None:
        out = torch.empty_like(q)
    _require_out(q.device, out)
    _require_cuda(q.device, q=q, k_new=k_new, v_new=v_new, slot_mapping=slot_mapping, k_cache=k_cache,
                  v_cache=v_cache, block_tables=block_tables, context_lens=context_lens, k_scale=k_scale,
                  v_scale=v_scale, workspace=workspace)
    max_blocks = block_tables.shape[1]
    s = _stream(stream, q.device)
    if workspace is None:
        need = workspace_size(B, Hq, Hkv, D, max_blocks, bs, partition_size)
        if need:
            workspace = _workspace(q.device, s, need)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
            max_blocks, _ptr(context_lens), B, Hq, Hkv, bs, D, NB, float(scale), _ptr(out), _code(q),
            _code(k_cache), _ptr(k_scale), _ptr(v_scale), int(partition_size), _ptr(workspace), ws_bytes, s)
    return args, out, workspace


class DecodePlan:
    """One decode step for fixed tensors, validated and marshalled once.

    With k_new, v_new and slot_mapping it is paged_attention_decode_append,
    else paged_attention_decode; the arguments mean the same.  run() issues
    the step with a single C call and returns `out`.  Between runs the
    tensors' contents may change (new queries, tables, lengths), their
    storage, shapes and types may not.  Every run goes on the stream given
    here (default: the current stream at construction)."""

    def __init__(self, q, k_cache, v_cache, block_tables, context_lens, scale, out=None, k_scale=None, v_scale=None,
                 partition_size=PARTITION_AUTO, workspace=None, stream=None, k_new=None, v_new=None,
                 slot_mapping=None):
        given = [t is not None for t in (k_new, v_new, slot_mapping)]
        if any(given) and not all(given):
            raise ValueError("DecodePlan: k_new, v_new and slot_mapping go together")
        if all(given):
            self.func = "paged_attention_decode_append"
            self._args, self.out, ws = _decode_append_args(q, k_new, v_new, slot_mapping, k_cache, v_cache,
                                                           block_tables, context_lens, scale, out, k_scale, v_scale,
                                                           partition_size, workspace, stream)
        else:
            self.func = "paged_attention_decode"
            self._args, self.out, ws = _decode_args(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                                                    k_scale, v_scale, partition_size, workspace, stream)
        # the plan holds its tensors so that their storage outlives it
        self._tensors = (q, k_cache, v_cache, block_tables, context_lens, k_scale, v_scale, ws, k_new, v_new,
                         slot_mapping)
        self._fn = _native.function(self.func)

    def run(self):
        code = self._fn(*self._args)
        if code != 0:
            _native.check(self.func, code)
        return self.out


def quest_block_minmax(k_cache, block_tables, context_lens, kmeta=None, stream=None, meta_dtype=None):
    """Per-block channel min/max of the keys (QUEST metadata) for every block the sequences use;
    returns kmeta [num_blocks, Hkv, 2, D] in the queries' 16-bit type (meta_dtype: default the
    cache's type, bfloat16 for an E4M3 cache, whose metadata holds the unscaled code values)."""
    NB, Hkv, bs, D = k_cache.shape
    if meta_dtype is None:
        meta_dtype = kmeta.dtype if kmeta is not None else (
            torch.bfloat16 if _code(k_cache) == E4M3 else k_cache.dtype)
    if kmeta is None:
        kmeta = torch.zeros(NB, Hkv, 2, D, dtype=meta_dtype, device=k_cache.device)
    if kmeta.dtype != meta_dtype:
        raise ValueError("quest_block_minmax: kmeta must be of meta_dtype")
    _require_cuda(k_cache.device, k_cache=k_cache, block_tables=block_tables, context_lens=context_lens, kmeta=kmeta)
    _native.call("quest_block_minmax", _ptr(k_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                 block_tables.shape[0], Hkv, bs, D, NB, _code(k_cache), _code(kmeta), _ptr(kmeta),
                 _stream(stream, k_cache.device))
    return kmeta


def quest_append_minmax(k_new, slot_mapping, kmeta, block_size, stream=None, k_scale=None):
    """Widen QUEST metadata with newly appended keys k_new [T, Hkv, D] at slot_mapping (int64 [T]).
    For an E4M3 cache pass its k_scale (device float32 [1]): each key enters as the append stores it."""
    T, Hkv, D = k_new.shape
    _require_cuda(k_new.device, k_new=k_new, slot_mapping=slot_mapping, kmeta=kmeta, k_scale=k_scale)
    _native.call("quest_append_minmax", _ptr(k_new), _ptr(slot_mapping), T, Hkv, block_size, D, kmeta.shape[0],
                 _code(k_new), E4M3 if k_scale is not None else _code(k_new), _ptr(k_scale), _ptr(kmeta),
                 _stream(stream, k_new.device))


def quest_select(q, kmeta, block_tables, context_lens, block_size, budget_blocks, sel_tables=None, sel_lens=None,
                 workspace=None, stream=None):
    """QUEST top-K blocks per (sequence, kv head); returns (sel_tables [B, Hkv, budget], sel_lens [B, Hkv])."""
    B, Hq, D = q.shape
    NB, Hkv = kmeta.shape[0], kmeta.shape[1]
    if sel_tables is None:
        sel_tables = torch.empty(B, Hkv, budget_blocks, dtype=torch.int32, device=q.device)
    if sel_lens is None:
        sel_lens = torch.empty(B, Hkv, dtype=torch.int32, device=q.device)
    _require_cuda(q.device, q=q, kmeta=kmeta, block_tables=block_tables, context_lens=context_lens,
                  sel_tables=sel_tables, sel_lens=sel_lens, workspace=workspace)
    s = _stream(stream, q.device)
    need = int(_native.lib().quest_workspace_size(B, Hkv, block_tables.shape[1]))
    if workspace is None:
        workspace = _workspace(q.device, -s - 1, need)  # separate from the decode workspace
    _native.call("quest_select", _ptr(q), _ptr(kmeta), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                 B, Hq, Hkv, block_size, D, NB, _code(q), int(budget_blocks), _ptr(sel_tables), _ptr(sel_lens),
                 _ptr(workspace), workspace.numel() * workspace.element_size(), s)
    return sel_tables, sel_lens


def paged_attention_decode_sparse(q, k_cache, v_cache, sel_tables, sel_lens, scale, out=None, k_scale=None,
                                  v_scale=None, partition_size=PARTITION_AUTO, workspace=None, stream=None):
    """Decode over per-(sequence, kv head) block lists sel_tables [B, Hkv, max_sel], sel_lens [B, Hkv]."""
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _require_out(q.device, out)
    _require_cuda(q.device, q=q, k_cache=k_cache, v_cache=v_cache, sel_tables=sel_tables, sel_lens=sel_lens,
                  k_scale=k_scale, v_scale=v_scale, workspace=workspace)
    max_sel = sel_tables.shape[2]
    s = _stream(stream, q.device)
    need = workspace_size(B, Hq, Hkv, D, max_sel, bs, partition_size)
    if need and workspace is None:
        workspace = _workspace(q.device, s, need)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _native.call("paged_attention_decode_sparse", _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(sel_tables), max_sel,
                 _ptr(sel_lens), B, Hq, Hkv, bs, D, NB, float(scale), _ptr(out), _code(q), _code(k_cache),
                 _ptr(k_scale), _ptr(v_scale), int(partition_size), _ptr(workspace), ws_bytes, s)
    return out


def paged_block_copy(k_cache, v_cache, src_dst_pairs, stream=None):
    """Copy whole blocks (K and V) for each (src, dst) row of int32 [P, 2]."""
    if src_dst_pairs.dtype != torch.int32 or src_dst_pairs.dim() != 2 or src_dst_pairs.shape[1] != 2:
        raise ValueError("paged_block_copy: src_dst_pairs must be int32 [P, 2]")
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype:
        raise ValueError("paged_block_copy: k_cache and v_cache must match")
    _require_cuda(k_cache.device, k_cache=k_cache, v_cache=v_cache, src_dst_pairs=src_dst_pairs)
    block_bytes = k_cache[0].numel() * k_cache.element_size()
    _native.call("paged_block_copy", _ptr(k_cache), _ptr(v_cache), _ptr(src_dst_pairs), src_dst_pairs.shape[0],
                 k_cache.shape[0], block_bytes, _stream(stream, k_cache.device))


def paged_block_swap(k_cache, v_cache, block_ids, staging, direction, stream=None):
    """Copy whole blocks between the pools and staging [n, 2, block_bytes] (uint8,
    pinned host or device).  direction: SWAP_OUT (pools -> staging) or SWAP_IN."""
    if block_ids.dtype != torch.int32 or block_ids.dim() != 1:
        raise ValueError("paged_block_swap: block_ids must be int32 [n]")
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype:
        raise ValueError("paged_block_swap: k_cache and v_cache must match")
    _require_cuda(k_cache.device, k_cache=k_cache, v_cache=v_cache, block_ids=block_ids)
    block_bytes = k_cache[0].numel() * k_cache.element_size()
    if staging.numel() * staging.element_size() < block_ids.numel() * 2 * block_bytes or not staging.is_contiguous():
        raise ValueError("paged_block_swap: staging must be contiguous with room for [n, 2, block_bytes]")
    if not staging.is_cuda and not staging.is_pinned():
        raise ValueError("paged_block_swap: host staging must be pinned memory")
    _native.call("paged_block_swap", _ptr(k_cache), _ptr(v_cache), _ptr(block_ids), block_ids.numel(),
                 k_cache.shape[0], block_bytes, _ptr(staging), int(direction), _stream(stream, k_cache.device))


def device_error(reset: bool = True, stream=None, device=None) -> int:
    """Read (and by default clear) the current device's kernel error bits."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    bits = ctypes.c_int(0)
    _native.call("pkv_device_error", ctypes.byref(bits), int(reset), _stream(stream, device))
    return bits.value


def selftest_wait_timeout(limit_us: int = 1000, stream=None, device=None) -> None:
    """Run the bounded-wait check kernel (a wait on a barrier nothing arrives
    at, given up after limit_us); read the outcome with device_error()."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    _native.call("pkv_selftest_wait_timeout", int(limit_us), _stream(stream, device))


class BlockManager:
    """Host-side block allocator (C++ in libpagedkv.so): FIFO free list,
    per-block reference counts, copy-on-write of a shared last block."""

    def __init__(self, num_blocks: int, block_size: int, free_list=None):
        lib = _native.lib()
        fl = None if free_list is None else np.ascontiguousarray(free_list, dtype=np.int32)
        self._h = lib.pkv_bm_create(num_blocks, block_size,
                                    None if fl is None else fl.ctypes.data_as(ctypes.c_void_p),
                                    0 if fl is None else len(fl))
        if not self._h:
            raise PagedKVError("pkv_bm_create", 1, lib.pkv_last_error().decode())
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _native.lib().pkv_bm_destroy(h)
            self._h = None

    def _check(self, func, code):
        if code == ERR_NO_SPACE:
            raise OutOfBlocks(func, code, _native.lib().pkv_last_error().decode())
        _native.check(func, code)

    def add_sequence(self, seq_id: int, num_tokens: int) -> None:
        self._check("pkv_bm_add_sequence", _native.lib().pkv_bm_add_sequence(self._h, int(seq_id), int(num_tokens)))

    def add_sequence_cached(self, seq_id: int, tokens) -> int:
        """Register a prompt by token ids, sharing the longest cached prefix of
        full blocks; returns how many leading tokens are already in the pool."""
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        cached = ctypes.c_int(0)
        self._check("pkv_bm_add_sequence_cached", _native.lib().pkv_bm_add_sequence_cached(
            self._h, int(seq_id), toks.ctypes.data_as(ctypes.c_void_p), len(toks), ctypes.byref(cached)))
        return cached.value

    def swap_out(self, seq_id: int) -> np.ndarray:
        """Release a sequence's blocks, keeping it as swapped out; returns the
        blocks (logical order) whose contents must be staged out first."""
        n = max(self.num_seq_blocks(seq_id), 0)
        out = np.empty(max(n, 1), np.int32)
        cnt = ctypes.c_int(0)
        self._check("pkv_bm_swap_out", _native.lib().pkv_bm_swap_out(
            self._h, int(seq_id), out.ctypes.data_as(ctypes.c_void_p), len(out), ctypes.byref(cnt)))
        return out[: cnt.value].copy()

    def swap_in(self, seq_id: int, max_blocks: int) -> np.ndarray:
        """Give a swapped-out sequence fresh blocks; returns them (logical order)."""
        out = np.empty(max(max_blocks, 1), np.int32)
        cnt = ctypes.c_int(0)
        self._check("pkv_bm_swap_in", _native.lib().pkv_bm_swap_in(
            self._h, int(seq_id), out.ctypes.data_as(ctypes.c_void_p), len(out), ctypes.byref(cnt)))
        return out[: cnt.value].copy()

    def swap_out_group(self, seq_ids) -> np.ndarray:
        """Swap out sequences together (e.g. one prompt's samples): returns their
        distinct blocks, first-use order, each to be staged once."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        cap = max(sum(max(self.num_seq_blocks(s), 0) for s in ids), 1)
        out = np.empty(cap, np.int32)
        cnt = ctypes.c_int(0)
        self._check("pkv_bm_swap_out_group", _native.lib().pkv_bm_swap_out_group(
            self._h, ids.ctypes.data_as(ctypes.c_void_p), len(ids), out.ctypes.data_as(ctypes.c_void_p), cap,
            ctypes.byref(cnt)))
        return out[: cnt.value].copy()

    def swap_in_group(self, seq_ids, max_blocks: int) -> np.ndarray:
        """Bring a group swapped out together back: one fresh block per staged
        entry (returned in staging order); shared blocks are shared again."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        out = np.empty(max(max_blocks, 1), np.int32)
        cnt = ctypes.c_int(0)
        self._check("pkv_bm_swap_in_group", _native.lib().pkv_bm_swap_in_group(
            self._h, ids.ctypes.data_as(ctypes.c_void_p), len(ids), out.ctypes.data_as(ctypes.c_void_p), len(out),
            ctypes.byref(cnt)))
        return out[: cnt.value].copy()

    @property
    def num_cached_blocks(self) -> int:
        return int(_native.lib().pkv_bm_num_cached_blocks(self._h))

    def append_slots(self, seq_ids):
        """Reserve the next slot of each sequence; returns (slots int64 [n], cow_pairs int32 [k, 2])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = len(ids)
        slots = np.empty(n, np.int64)
        pairs = np.empty((max(n, 1), 2), np.int32)
        npairs = ctypes.c_int(0)
        self._check("pkv_bm_append_slots", _native.lib().pkv_bm_append_slots(
            self._h, ids.ctypes.data_as(ctypes.c_void_p), n, slots.ctypes.data_as(ctypes.c_void_p),
            pairs.ctypes.data_as(ctypes.c_void_p), ctypes.byref(npairs)))
        return slots, pairs[: npairs.value].copy()

    def append_tokens(self, seq_ids, token_ids):
        """append_slots with each new token's id: a token that fills its block
        registers the block in the prefix cache (sequences added by
        add_sequence_cached).  Returns (slots int64 [n], cow_pairs int32 [k, 2])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        toks = np.ascontiguousarray(token_ids, dtype=np.int32)
        n = len(ids)
        if len(toks) != n:
            raise ValueError("append_tokens: one token id per sequence id")
        slots = np.empty(n, np.int64)
        pairs = np.empty((max(n, 1), 2), np.int32)
        npairs = ctypes.c_int(0)
        self._check("pkv_bm_append_tokens", _native.lib().pkv_bm_append_tokens(
            self._h, ids.ctypes.data_as(ctypes.c_void_p), toks.ctypes.data_as(ctypes.c_void_p), n,
            slots.ctypes.data_as(ctypes.c_void_p), pairs.ctypes.data_as(ctypes.c_void_p), ctypes.byref(npairs)))
        return slots, pairs[: npairs.value].copy()

    def fork(self, parent_id: int, child_id: int) -> None:
        self._check("pkv_bm_fork", _native.lib().pkv_bm_fork(self._h, int(parent_id), int(child_id)))

    def free_sequence(self, seq_id: int) -> None:
        self._check("pkv_bm_free_sequence", _native.lib().pkv_bm_free_sequence(self._h, int(seq_id)))

    def tables(self, seq_ids, max_blocks_per_seq: int | None = None, pad: int = 0):
        """Block tables int32 [n, max_blocks_per_seq] (pad-filled) and context lengths int32 [n]."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        if max_blocks_per_seq is None:
            max_blocks_per_seq = max([self.num_seq_blocks(s) for s in ids] + [1])
        t = np.empty((len(ids), max_blocks_per_seq), np.int32)
        lens = np.empty(len(ids), np.int32)
        self._check("pkv_bm_get_tables", _native.lib().pkv_bm_get_tables(
            self._h, ids.ctypes.data_as(ctypes.c_void_p), len(ids), t.ctypes.data_as(ctypes.c_void_p),
            max_blocks_per_seq, pad, lens.ctypes.data_as(ctypes.c_void_p)))
        return t, lens

    @property
    def num_free(self) -> int:
        return int(_native.lib().pkv_bm_num_free(self._h))

    def ref_count(self, block: int) -> int:
        return int(_native.lib().pkv_bm_ref_count(self._h, int(block)))

    def context_len(self, seq_id: int) -> int:
        return int(_native.lib().pkv_bm_context_len(self._h, int(seq_id)))

    def num_seq_blocks(self, seq_id: int) -> int:
        return int(_native.lib().pkv_bm_num_seq_blocks(self._h, int(seq_id)))

    def free_list(self) -> np.ndarray:
        n = int(_native.lib().pkv_bm_free_list(self._h, None, 0))
        out = np.empty(n, np.int32)
        _native.lib().pkv_bm_free_list(self._h, out.ctypes.data_as(ctypes.c_void_p), n)
        return out
