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
    rk, rv = bits(kc).copy(), bits(vc).copy()
    want = oracle.block_swap_out(rk, rv, ids.numpy())
    assert np.array_equal(staging.numpy(), want)
    # swap back in to other blocks
    dst = torch.randperm(NB, generator=g)[:13].to(torch.int32)
    pkv.paged_block_swap(dk, dv, dst.cuda(), staging, pkv.SWAP_IN)
    torch.cuda.synchronize()
    oracle.block_swap_in(rk, rv, dst.numpy(), want)
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


def test_group_swap_keeps_sharing_and_decode(pkv):
    """Parallel sampling preempted as a group: 3 prompts x 4 samples share their
    prompt blocks (count 4), each sample appends divergent tokens (copy-on-write
    of the partial block).  Each prompt's samples are swapped out together --
    every shared block staged once -- the freed blocks are overwritten, and the
    group is swapped back in: the tables share blocks again (counts as before),
    the staging bytes and caches equal the oracle's gather/scatter on the oracle
    allocator's blocks, and decode is bit-identical to the decode before the
    swap and within tolerance of the float64 oracle."""
    bs, Hq, Hkv, D, NB, n = 16, 8, 8, 64, 200, 4
    g = torch.Generator().manual_seed(4)
    dev = torch.device("cuda")
    kc = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.float16).to(dev)
    vc = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.float16).to(dev)
    rk, rv = bits(kc).copy(), bits(vc).copy()
    bm = pkv.BlockManager(NB, bs)
    ref = RefBlockManager(NB, bs)
    prompts = [203, 77, 130]
    for p, L in enumerate(prompts):
        for m in (bm, ref):
            m.add_sequence(p * n, L)
            for j in range(1, n):
                m.fork(p * n, p * n + j)
    seqs = list(range(len(prompts) * n))
    for step in range(20):
        active = [s for s in seqs if step < 3 + 4 * (s % n)]
        slots, pairs = bm.append_slots(active)
        want = [ref.append_slot(s) for s in active]
        assert list(slots) == [w[0] for w in want]
        if len(pairs):
            pkv.paged_block_copy(kc, vc, torch.from_numpy(pairs).to(dev))
            oracle.block_copy(rk, rv, pairs)
        kn = torch.randn(len(active), Hkv, D, generator=g).half()
        vn = torch.randn(len(active), Hkv, D, generator=g).half()
        pkv.paged_kv_append(kn.to(dev), vn.to(dev), torch.from_numpy(slots).to(dev), kc, vc)
        oracle.append(bits(kn), bits(vn), oracle.F16, slots, rk, rv, oracle.F16)
    q = torch.randn(len(seqs), Hq, D, generator=g).half().to(dev)
    t, l = bm.tables(seqs)
    before = pkv.paged_attention_decode(q, kc, vc, torch.from_numpy(t).to(dev), torch.from_numpy(l).to(dev), 0.125)
    def used(tables, s):
        return [int(b) for b in tables[s][: -(-int(l[s]) // bs)]]

    counts_before = sorted(bm.ref_count(b) for b in {b for s in seqs for b in used(t, s)})
    assert max(counts_before) == n  # full prompt blocks shared by all four samples
    block_bytes = kc[0].numel() * kc.element_size()
    stage = {}
    for p in range(len(prompts)):
        members = [p * n + j for j in range(n)]
        blocks = bm.swap_out_group(members)
        assert list(blocks) == ref.swap_out_group(members)
        assert len(blocks) == len({b for m in members for b in used(t, m)}) < sum(len(used(t, m)) for m in members)
        buf = torch.empty(len(blocks), 2, block_bytes, dtype=torch.uint8).pin_memory()
        pkv.paged_block_swap(kc, vc, torch.from_numpy(blocks).to(dev), buf, pkv.SWAP_OUT)
        torch.cuda.synchronize()
        staged = oracle.block_swap_out(rk, rv, blocks)
        assert np.array_equal(buf.numpy(), staged)
        stage[p] = (buf, staged)
    # the freed blocks are overwritten by another request
    kc.fill_(0)
    vc.fill_(0)
    rk[...] = 0
    rv[...] = 0
    for p in (2, 0, 1):
        members = [p * n + j for j in range(n)][::-1]
        blocks = bm.swap_in_group(members, NB)
        assert list(blocks) == ref.swap_in_group(members)
        buf, staged = stage[p]
        pkv.paged_block_swap(kc, vc, torch.from_numpy(blocks).to(dev), buf, pkv.SWAP_IN)
        oracle.block_swap_in(rk, rv, blocks, staged)
    t2, l2 = bm.tables(seqs)
    assert np.array_equal(l2, l)
    for s in seqs:
        assert list(t2[s][: -(-int(l[s]) // bs)]) == ref.tables[s]
    assert sorted(bm.ref_count(b) for b in {b for s in seqs for b in used(t2, s)}) == counts_before
    after = pkv.paged_attention_decode(q, kc, vc, torch.from_numpy(t2).to(dev), torch.from_numpy(l2).to(dev), 0.125)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)
    assert torch.equal(before, after)
    want = oracle.paged_decode(bits(q), oracle.F16, rk, rv, oracle.F16, t2, l2, 0.125)
    assert_attention_close(after, want, TOL["f16"])
