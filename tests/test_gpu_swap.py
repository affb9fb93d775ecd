"""Block swap between the pools and pinned host memory: bit-exact against a
plain gather/scatter, and decode after a swap round trip is unchanged."""
import numpy as np
import pytest
import torch

import oracle
from oracle.block_manager_ref import RefBlockManager
from tests.parity import TOL, assert_attention_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture
def pkv(pkv_lib, cuda_device):
    pkv_lib.device_error(reset=True)
    yield pkv_lib
    assert pkv_lib.device_error(reset=True) == 0


@pytest.mark.parametrize("Hkv,bs,D,dtype", [(32, 16, 128, torch.bfloat16), (8, 32, 64, torch.float16),
                                            (40, 16, 128, torch.uint8)])
def test_swap_bit_exact(pkv, Hkv, bs, D, dtype):
    g = torch.Generator().manual_seed(Hkv + bs)
    NB = 40
    if dtype == torch.uint8:
        kc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=dtype, generator=g)
        vc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=dtype, generator=g)
    else:
        kc = torch.randn(NB, Hkv, bs, D, generator=g).to(dtype)
        vc = torch.randn(NB, Hkv, bs, D, generator=g).to(dtype)
    ids = torch.randperm(NB, generator=g)[:13].to(torch.int32)
    block_bytes = kc[0].numel() * kc.element_size()
    staging = torch.zeros(13, 2, block_bytes, dtype=torch.uint8).pin_memory()
    dk, dv = kc.cuda(), vc.cuda()
    pkv.paged_block_swap(dk, dv, ids.cuda(), staging, pkv.SWAP_OUT)
    torch.cuda.synchronize()
    kb, vb = bits(kc).reshape(NB, -1).view(np.uint8), bits(vc).reshape(NB, -1).view(np.uint8)
    want = np.stack([np.stack([kb[i], vb[i]]) for i in ids.numpy()])
    assert np.array_equal(staging.numpy(), want)
    # swap back in to other blocks
    dst = torch.randperm(NB, generator=g)[:13].to(torch.int32)
    pkv.paged_block_swap(dk, dv, dst.cuda(), staging, pkv.SWAP_IN)
    torch.cuda.synchronize()
    rk, rv = bits(kc).copy(), bits(vc).copy()
    rkb, rvb = rk.reshape(NB, -1).view(np.uint8), rv.reshape(NB, -1).view(np.uint8)
    for j, b in enumerate(dst.numpy()):
        rkb[b] = want[j, 0]
        rvb[b] = want[j, 1]
    assert np.array_equal(bits(dk), rk) and np.array_equal(bits(dv), rv)


def test_swap_refuses_pageable_staging_and_flags_bad_ids(pkv):
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    with pytest.raises(ValueError):
        pkv.paged_block_swap(kc, vc, torch.tensor([1], dtype=torch.int32, device="cuda"),
                             torch.zeros(1, 2, 4096, dtype=torch.uint8), pkv.SWAP_OUT)
    staging = torch.zeros(2, 2, 4096, dtype=torch.uint8, device="cuda")
    pkv.paged_block_swap(kc, vc, torch.tensor([1, 9], dtype=torch.int32, device="cuda"), staging, pkv.SWAP_OUT)
    assert pkv.device_error(reset=True) == pkv.DEV_BAD_PAIR


def test_decode_unchanged_after_swap_round_trip(pkv):
    """Swap two sequences out, let other requests overwrite the freed blocks,
    swap them back in to fresh blocks: decode output is bit-identical."""
    bs, Hq, Hkv, D, NB = 16, 16, 4, 128, 96
    g = torch.Generator().manual_seed(1)
    kc = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.bfloat16).cuda()
    vc = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.bfloat16).cuda()
    lens = [130, 33, 517, 64]
    bm = pkv.BlockManager(NB, bs)
    ref = RefBlockManager(NB, bs)
    for i, L in enumerate(lens):
        bm.add_sequence(i, L)
        ref.add_sequence(i, L)
    ids = np.arange(4)
    q = torch.randn(4, Hq, D, generator=g).to(torch.bfloat16).cuda()
    t, l = bm.tables(ids)
    before = pkv.paged_attention_decode(q, kc, vc, torch.from_numpy(t).cuda(), torch.from_numpy(l).cuda(), 0.09)
    want = oracle.paged_decode(bits(q), oracle.BF16, bits(kc), bits(vc), oracle.BF16, t, l, 0.09)
    assert_attention_close(before, want, TOL["bf16"])
    block_bytes = kc[0].numel() * kc.element_size()
    stage = {}
    for s in (0, 2):
        blocks = bm.swap_out(s)
        assert list(blocks) == ref.swap_out(s)
        buf = torch.empty(len(blocks), 2, block_bytes, dtype=torch.uint8).pin_memory()
        pkv.paged_block_swap(kc, vc, torch.from_numpy(blocks).cuda(), buf, pkv.SWAP_OUT)
        stage[s] = buf
    # another request takes the freed blocks and writes into them
    bm.add_sequence(10, 40 * bs)
    ref.add_sequence(10, 40 * bs)
    t10, _ = bm.tables([10])
    kc[torch.from_numpy(t10[0]).long().cuda()] = 0
    vc[torch.from_numpy(t10[0]).long().cuda()] = 7
    bm.free_sequence(10)
    ref.free_sequence(10)
    for s in (0, 2):
        blocks = bm.swap_in(s, 64)
        assert list(blocks) == ref.swap_in(s)
        pkv.paged_block_swap(kc, vc, torch.from_numpy(blocks).cuda(), stage[s], pkv.SWAP_IN)
    t, l = bm.tables(ids)
    after = pkv.paged_attention_decode(q, kc, vc, torch.from_numpy(t).cuda(), torch.from_numpy(l).cuda(), 0.09)
    torch.cuda.synchronize()
    assert torch.equal(before, after)
