"""paged_attention_decode_noalloc, the decode entry point for callers that
cannot allocate device memory (for example an engine that has reserved all
free device memory for its own pool, or a host framework that forbids
cudaMalloc on its decode path).  Its split-K scratch is a fixed array inside
the library instead of a caller-provided workspace.

Checked through the C ABI, on both decode kernels (the tensor-core kernel for
grouped heads and the CUDA-core kernel for one query head per KV head, each
writing split-K partials into the fixed array) and on 16-bit and E4M3 caches:
on two calls in a row with the same shapes but different inputs and shorter
contexts (so stale partials left by the first call would show up in the
second), its output is bit-identical to paged_attention_decode with a
caller-allocated workspace -- the same kernels on the same inputs -- and the
second call leaves the device's free memory unchanged.  A request that needs
more scratch than the array holds is refused with a clear message.  This
file is collected last on purpose.
"""
import ctypes
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

_HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pagedkv.h")


def lib_limit():
    """PKV_NOALLOC_MAX_WORKSPACE_BYTES as the public header defines it."""
    with open(_HEADER) as f:
        m = re.search(r"#define\s+PKV_NOALLOC_MAX_WORKSPACE_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", f.read())
    assert m, "PKV_NOALLOC_MAX_WORKSPACE_BYTES not found in the header"
    return int(m.group(1)) << int(m.group(2))


def _case(seed, B, Hq, Hkv, D, bs, max_len, cache, dev, shrink=None):
    """A random paged batch; with `shrink`, the lengths are cut to at most
    that many tokens (same table width, fewer partitions in use)."""
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
    if shrink is not None:
        lens = torch.clamp(lens // 3, min=1, max=shrink).to(torch.int32)
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
    if cache == "e4m3":
        kc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=torch.uint8, generator=g)
        vc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=torch.uint8, generator=g)
        kc[(kc & 0x7F) == 0x7F] = 0x3C  # no NaN codes
        vc[(vc & 0x7F) == 0x7F] = 0x3C
        scales = [torch.tensor([0.02], dtype=torch.float32).to(dev), torch.tensor([0.03], dtype=torch.float32).to(dev)]
    else:
        kc = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.bfloat16)
        vc = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.bfloat16)
        scales = [None, None]
    return [t.to(dev) for t in (q, kc, vc, tables, lens)] + [NB, maxb] + scales


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


CASES = [
    # (query heads, kv heads, cache, max context): kernel the library picks
    (32, 8, "bf16", 3000),   # 4 query heads per kv head: tensor-core kernel, 512-token partitions
    (8, 8, "bf16", 5000),    # 1 query head per kv head: CUDA-core kernel
    (32, 8, "e4m3", 2600),   # tensor-core kernel, E4M3 operands
    (8, 8, "e4m3", 4100),    # CUDA-core kernel, E4M3 cache
]


@pytest.mark.parametrize("Hq,Hkv,cache,max_len", CASES, ids=lambda c: str(c))
def test_noalloc_bit_identical_to_workspace_entry_point(pkv_lib, cuda_device, Hq, Hkv, cache, max_len):
    lib = pkv_lib._native.lib()
    B, D, bs, scale, part = 24, 128, 16, 0.088, 512
    cache_code = 2 if cache == "e4m3" else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    free_after = []
    # two calls in a row: same shapes, new inputs, and the second with shorter
    # contexts, so partitions the first call filled are not written again
    for call, (seed, shrink) in enumerate([(1, None), (2, 700)]):
        q, kc, vc, tables, lens, NB, maxb, ks, vs = _case(seed, B, Hq, Hkv, D, bs, max_len, cache, cuda_device,
                                                          shrink)
        need = lib.pkv_workspace_size(B, Hq, Hkv, D, maxb, bs, part)
        assert 256 < need <= lib_limit(), "the case must exercise the split-K scratch"
        ws = torch.empty(need, dtype=torch.uint8, device=cuda_device)
        want = torch.empty_like(q)
        got = torch.full_like(q, float("nan"))
        rc = lib.paged_attention_decode(_p(q), _p(kc), _p(vc), _p(tables), maxb, _p(lens), B, Hq, Hkv, bs, D, NB,
                                        scale, _p(want), 1, cache_code, _p(ks), _p(vs), part, _p(ws), need, stream)
        assert rc == 0, lib.pkv_last_error()
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        rc = lib.paged_attention_decode_noalloc(_p(q), _p(kc), _p(vc), _p(tables), maxb, _p(lens), B, Hq, Hkv, bs,
                                                D, NB, scale, _p(got), 1, cache_code, _p(ks), _p(vs), part, stream)
        assert rc == 0, lib.pkv_last_error()
        torch.cuda.synchronize()
        free_after.append((free_before, torch.cuda.mem_get_info()[0]))
        assert torch.equal(got, want), f"call {call}: max |diff| {(got.float() - want.float()).abs().max().item()}"
    # the first call on a device may load the library's device code (and with
    # it the fixed array); the second call must not take any device memory
    before, after = free_after[1]
    assert after >= before, f"the second call took {before - after} bytes of device memory"
    assert pkv_lib.device_error(reset=True) == 0


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
