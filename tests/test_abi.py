"""The C-ABI library loads, exports every function include/pagedkv.h
declares, and rejects bad arguments on the host (no GPU needed)."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    skip = {"if", "sizeof", "defined"}
    return sorted({n for n in names if n not in skip and (n.startswith("pkv_") or n.startswith("paged_"))})


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("paged_kv_append", "paged_attention_decode", "paged_block_copy", "pkv_workspace_size",
                 "pkv_last_error"):
        assert must in names


def test_every_declared_symbol_is_exported(pkv_lib):
    lib = ctypes.CDLL(pkv_lib._native.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding knows the signature of each
    assert set(_declared_functions()) <= set(pkv_lib._native.SIGNATURES)


def test_version(pkv_lib):
    assert pkv_lib._native.lib().pkv_version() == 100


def _decode(lib, **kw):
    args = dict(q=1 << 12, k=1 << 12, v=1 << 12, tables=1 << 12, maxb=4, lens=1 << 12, B=2, Hq=8, Hkv=8, bs=16, D=128,
                NB=16, scale=0.1, out=1 << 12, act=1, cache=1, ks=None, vs=None, part=-1, ws=None, wsb=0,
                stream=None)
    args.update(kw)
    return lib.paged_attention_decode(*args.values())


def test_decode_argument_checks(pkv_lib):
    lib = pkv_lib._native.lib()
    assert _decode(lib, Hq=12, Hkv=8) == 2          # not a multiple
    assert _decode(lib, Hq=24, Hkv=8) == 1          # group 3 unsupported
    assert _decode(lib, D=96) == 1
    assert _decode(lib, bs=8) == 1
    assert _decode(lib, act=2) == 1                 # E4M3 queries
    assert _decode(lib, act=0, cache=1) == 1        # mixed 16-bit types
    assert _decode(lib, cache=2) == 1               # E4M3 without scales
    assert _decode(lib, q=None) == 1
    assert _decode(lib, q=(1 << 12) + 8) == 1       # misaligned
    assert _decode(lib, part=48) == 1               # not a multiple of 32
    assert _decode(lib, maxb=200, part=512) == 1    # needs a workspace, none given
    assert "workspace" in lib.pkv_last_error().decode()
    assert _decode(lib, B=0) == 0                   # nothing to do
    assert _decode(lib, maxb=4, ws=None) == 1       # the header is always needed


def test_partition_and_workspace_sizes(pkv_lib):
    lib = pkv_lib._native.lib()
    assert lib.pkv_resolve_partition_size(4, 8, 8, 128, 129, 16, 0) == 2080   # single pass: 2064 -> 2080
    assert lib.pkv_resolve_partition_size(4, 8, 8, 128, 129, 16, 512) == 512
    assert lib.pkv_resolve_partition_size(4, 8, 8, 128, 129, 16, -1) == 1024  # CUDA-core shapes
    # tensor-core shapes: 512 tokens, or 256 with 256..1023 (sequence, kv head, 512-token partition) items
    assert lib.pkv_resolve_partition_size(4, 64, 8, 128, 129, 16, -1) == 512   # 4 * 8 * 5 = 160 items
    assert lib.pkv_resolve_partition_size(16, 64, 8, 128, 129, 16, -1) == 256  # 16 * 8 * 5 = 640 items
    assert lib.pkv_resolve_partition_size(32, 64, 8, 128, 129, 16, -1) == 512  # 32 * 8 * 5 = 1280 items
    # head_dim 64: items cover pairs of kv heads; an odd kv-head count has no pairs (CUDA-core shapes)
    assert lib.pkv_resolve_partition_size(4, 64, 8, 64, 129, 16, -1) == 512    # 4 * 4 * 5 = 80 items
    assert lib.pkv_resolve_partition_size(16, 64, 8, 64, 129, 16, -1) == 256   # 16 * 4 * 5 = 320 items
    assert lib.pkv_resolve_partition_size(16, 24, 3, 64, 129, 16, -1) == 1024
    assert lib.pkv_resolve_partition_size(4, 8, 8, 128, 8, 16, 512) == 128    # whole context fits one
    assert lib.pkv_resolve_partition_size(4, 8, 8, 128, 129, 32, 48) == -1
    assert lib.pkv_workspace_size(4, 8, 8, 128, 8, 16, 512) == 256  # the work-counter header only
    parts = -(-129 * 16 // 512)
    rows = 4 * 8 * parts
    ml = -(-(rows * 2 * 4) // 256) * 256
    assert lib.pkv_workspace_size(4, 8, 8, 128, 129, 16, 512) == 256 + ml + rows * 128 * 4
    assert lib.pkv_workspace_size(4, 8, 8, 128, 129, 16, 48) == 0  # invalid partition size


def test_append_and_copy_argument_checks(pkv_lib):
    lib = pkv_lib._native.lib()
    a = 1 << 12
    assert lib.paged_kv_append(a, a, a, 4, a, a, 16, 8, 16, 100, 1, 1, None, None, None) == 1  # D % 8
    assert lib.paged_kv_append(a, a, a, 4, a, a, 16, 8, 16, 128, 1, 0, None, None, None) == 1  # mixed types
    assert lib.paged_kv_append(a, a, a, 4, a, a, 16, 8, 16, 128, 1, 2, None, None, None) == 1  # no scales
    assert lib.paged_kv_append(None, a, a, 4, a, a, 16, 8, 16, 128, 1, 1, None, None, None) == 1
    assert lib.paged_kv_append(a, a, a, 0, a, a, 16, 8, 16, 128, 1, 1, None, None, None) == 0  # empty
    assert lib.paged_block_copy(a, a, a, 1, 16, 100, None) == 1  # not a multiple of 16
    assert lib.paged_block_copy(a, a, a, 0, 16, 4096, None) == 0  # empty
    assert lib.paged_block_copy(None, a, a, 1, 16, 4096, None) == 1


def test_decode_plan_wants_all_append_tensors(pkv_lib):
    """A fused plan needs k_new, v_new and slot_mapping together (checked before any device work)."""
    with pytest.raises(ValueError):
        pkv_lib.DecodePlan(None, None, None, None, None, 0.1, k_new=object())
