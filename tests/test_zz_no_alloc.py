"""paged_attention_decode_noalloc, the decode entry point for callers that
cannot allocate device memory (for example an engine that has reserved all
free device memory for its own pool, or a host framework that forbids
cudaMalloc on its decode path).  Its split-K scratch is a fixed 16 MiB array
inside the library instead of a caller-provided workspace.

Checked through the C ABI: on two calls in a row (different inputs, so stale
scratch from the first call would show up in the second), its output matches
paged_attention_decode with a caller-allocated workspace, within the
attention tolerance; a request that needs more scratch than the array holds
is refused with a clear message.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.parity import TOL

pytestmark = pytest.mark.gpu


def _case(seed, B, Hq, Hkv, D, bs, max_len, dev):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, max_len + 1, (B,), generator=g).to(torch.int32)
    lens[0] = max_len
    nblk = (lens + bs - 1) // bs
    maxb = int(nblk.max())
    NB = int(nblk.sum()) + 3
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.zeros(B, maxb, dtype=torch.int32)
    o = 0
    for i in range(B):
        n = int(nblk[i])
        tables[i, :n] = perm[o:o + n]
        o += n
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
    kc = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.bfloat16)
    return [t.to(dev) for t in (q, kc, vc, tables, lens)] + [NB, maxb]


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point(pkv_lib, cuda_device):
    lib = pkv_lib._native.lib()
    B, Hq, Hkv, D, bs, scale, part = 24, 32, 8, 128, 16, 0.088, 512
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, (seed, max_len) in enumerate([(1, 3000), (2, 1700)]):
        q, kc, vc, tables, lens, NB, maxb = _case(seed, B, Hq, Hkv, D, bs, max_len, cuda_device)
        need = lib.pkv_workspace_size(B, Hq, Hkv, D, maxb, bs, part)
        assert 0 < need <= lib_limit(), "the case must exercise the split-K scratch"
        ws = torch.empty(need, dtype=torch.uint8, device=cuda_device)
        want = torch.empty_like(q)
        got = torch.full_like(q, float("nan"))
        rc = lib.paged_attention_decode(_p(q), _p(kc), _p(vc), _p(tables), maxb, _p(lens), B, Hq, Hkv, bs, D, NB,
                                        scale, _p(want), 1, 1, None, None, part, _p(ws), need, stream)
        assert rc == 0, lib.pkv_last_error()
        rc = lib.paged_attention_decode_noalloc(_p(q), _p(kc), _p(vc), _p(tables), maxb, _p(lens), B, Hq, Hkv, bs,
                                                D, NB, scale, _p(got), 1, 1, None, None, part, stream)
        assert rc == 0, lib.pkv_last_error()
        torch.cuda.synchronize()
        err = (got.float() - want.float()).abs().max().item()
        assert np.isfinite(err) and err <= TOL["bf16"], f"call {call}: max |diff| {err}"
    assert pkv_lib.device_error(reset=True) == 0


def lib_limit():
    return 16 << 20


def test_noalloc_refuses_oversized_requests(pkv_lib, cuda_device):
    lib = pkv_lib._native.lib()
    # 128 sequences x 64 heads x 17 partitions of a 8193-token table need ~72 MB of scratch
    B, Hq, Hkv, D, bs, maxb = 128, 64, 8, 128, 16, 513
    need = lib.pkv_workspace_size(B, Hq, Hkv, D, maxb, bs, 512)
    assert need > lib_limit()
    dummy = torch.zeros(64, dtype=torch.uint8, device=cuda_device)
    p = _p(dummy)
    rc = lib.paged_attention_decode_noalloc(p, p, p, p, maxb, p, B, Hq, Hkv, bs, D, 4, 0.1, p, 1, 1, None, None,
                                            512, None)
    assert rc == 1
    msg = lib.pkv_last_error().decode()
    assert str(need) in msg and str(lib_limit()) in msg
