"""Prefix caching in the C++ block manager against the oracle allocator (which
keys blocks by the exact token prefix instead of a hash)."""
import numpy as np
import pytest

from oracle.block_manager_ref import OutOfBlocks as RefOutOfBlocks
from oracle.block_manager_ref import RefBlockManager


def _state(bm, ref, NB):
    assert [bm.ref_count(b) for b in range(NB)] == ref.ref
    assert list(bm.free_list()) == ref.free
    assert bm.num_free == ref.available()
    assert bm.num_cached_blocks == len(ref.block_of_prefix)


def test_shared_system_prompt_reuses_full_blocks(pkv_lib):
    bs = 16
    system = list(range(1000, 1040))  # 40 tokens: two full blocks and a partial one
    bm = pkv_lib.BlockManager(32, bs)
    ref = RefBlockManager(32, bs)
    first = system + [1, 2, 3]
    second = system + [7, 8]
    assert bm.add_sequence_cached(0, first) == 0 == ref.add_sequence_cached(0, first)
    assert bm.add_sequence_cached(1, second) == 32 == ref.add_sequence_cached(1, second)
    t, _ = bm.tables([0, 1])
    assert list(t[0][:2]) == list(t[1][:2])  # the two full system-prompt blocks are shared
    assert t[0][2] != t[1][2]  # the partial block is per request
    assert bm.ref_count(int(t[0][0])) == 2
    _state(bm, ref, 32)
    # a prompt that differs inside the first block shares nothing
    third = [5] + system[1:] + [9]
    assert bm.add_sequence_cached(2, third) == 0 == ref.add_sequence_cached(2, third)
    _state(bm, ref, 32)


def test_freed_cached_blocks_survive_until_evicted(pkv_lib):
    bs = 4
    bm = pkv_lib.BlockManager(6, bs)
    ref = RefBlockManager(6, bs)
    prompt = [1, 2, 3, 4, 5, 6, 7, 8, 9]  # two full blocks + one partial
    for m in (bm, ref):
        m.add_sequence_cached(0, prompt)
        m.free_sequence(0)
    _state(bm, ref, 6)
    assert bm.num_cached_blocks == 2 and bm.num_free == 6
    # the same prompt later is still a hit
    assert bm.add_sequence_cached(1, prompt) == 8 == ref.add_sequence_cached(1, prompt)
    _state(bm, ref, 6)
    bm.free_sequence(1)
    ref.free_sequence(1)
    # fill the pool: the free list goes first, then the least recently freed cached block
    bm.add_sequence(2, 4 * 5)
    ref.add_sequence(2, 4 * 5)
    _state(bm, ref, 6)
    assert bm.num_cached_blocks == 1 and bm.num_free == 1
    with pytest.raises(pkv_lib.OutOfBlocks):
        bm.add_sequence_cached(3, prompt)
    bm.free_sequence(2)
    ref.free_sequence(2)
    # the prompt's first block was evicted, so the chain misses from the start
    assert bm.add_sequence_cached(3, prompt) == 0 == ref.add_sequence_cached(3, prompt)
    _state(bm, ref, 6)


@pytest.mark.parametrize("seed", range(10))
def test_random_requests_match_oracle(pkv_lib, seed):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([2, 4, 16]))
    NB = int(rng.integers(12, 80))
    fl = rng.permutation(NB).astype(np.int32)
    bm = pkv_lib.BlockManager(NB, bs, free_list=fl)
    ref = RefBlockManager(NB, bs, free_list=fl)
    systems = [list(rng.integers(0, 50, size=int(rng.integers(0, 4 * bs)))) for _ in range(3)]
    live, nid = [], 0
    for _ in range(300):
        op = int(rng.integers(0, 5))
        if op <= 1 or not live:
            toks = systems[int(rng.integers(0, 3))] + list(rng.integers(0, 3, size=int(rng.integers(0, 2 * bs))))
            try:
                want = ref.add_sequence_cached(nid, toks)
                ok = True
            except RefOutOfBlocks:
                ok = False
            if ok:
                assert bm.add_sequence_cached(nid, toks) == want
                live.append(nid)
            else:
                with pytest.raises(pkv_lib.OutOfBlocks):
                    bm.add_sequence_cached(nid, toks)
            nid += 1
        elif op == 2:
            s = int(rng.choice(live))
            snap = (list(ref.free), list(ref.ref), {k: list(v) for k, v in ref.tables.items()}, dict(ref.lens),
                    dict(ref.prefix_of_block), dict(ref.block_of_prefix), list(ref.lru))
            try:
                want = ref.append_slot(s)
                ok = True
            except RefOutOfBlocks:
                (ref.free, ref.ref, ref.tables, ref.lens, ref.prefix_of_block, ref.block_of_prefix,
                 ref.lru) = snap
                ok = False
            if ok:
                slots, pairs = bm.append_slots([s])
                assert slots[0] == want[0]
            else:
                with pytest.raises(pkv_lib.OutOfBlocks):
                    bm.append_slots([s])
        elif op == 3:
            parent = int(rng.choice(live))
            bm.fork(parent, nid)
            ref.fork(parent, nid)
            live.append(nid)
            nid += 1
        else:
            s = live.pop(int(rng.integers(0, len(live))))
            bm.free_sequence(s)
            ref.free_sequence(s)
        _state(bm, ref, NB)
    for s in live:
        t, lens = bm.tables([s])
        assert list(t[0][: len(ref.tables[s])]) == ref.tables[s] and lens[0] == ref.lens[s]
