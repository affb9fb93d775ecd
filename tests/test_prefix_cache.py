"""Prefix caching in the C++ block manager against the oracle allocator (which
keys blocks by the exact token prefix instead of a hash): prompt blocks, and
blocks filled by decoding when each appended token's id is given."""
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
        op = int(rng.integers(0, 6))
        op = 2 if op == 5 else op  # appends twice as often: decoding fills blocks
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
            with_id = rng.random() < 0.9
            tok = int(rng.integers(0, 3))
            snap = (list(ref.free), list(ref.ref), {k: list(v) for k, v in ref.tables.items()}, dict(ref.lens),
                    dict(ref.prefix_of_block), dict(ref.block_of_prefix), list(ref.lru),
                    {k: list(v) for k, v in ref.tokens.items()})
            try:
                want = ref.append_token(s, tok) if with_id else ref.append_slot(s)
                ok = True
            except RefOutOfBlocks:
                (ref.free, ref.ref, ref.tables, ref.lens, ref.prefix_of_block, ref.block_of_prefix,
                 ref.lru, ref.tokens) = snap
                ok = False
            if ok:
                slots, pairs = bm.append_tokens([s], [tok]) if with_id else bm.append_slots([s])
                assert slots[0] == want[0]
                assert [tuple(p) for p in pairs] == ([want[1]] if want[1] is not None else [])
            else:
                with pytest.raises(pkv_lib.OutOfBlocks):
                    if with_id:
                        bm.append_tokens([s], [tok])
                    else:
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


def test_multi_turn_hand_example_matches_oracle(pkv_lib):
    """The oracle's hand-worked two-turn dialogue (block size 4, free list
    [5, 2, 7, 0, 1, 3, 4, 6]) through the C++ manager: the answer's tokens
    fill block 2, which the second turn finds by its prefix."""
    fl = [5, 2, 7, 0, 1, 3, 4, 6]
    bm = pkv_lib.BlockManager(8, 4, free_list=fl)
    ref = RefBlockManager(8, 4, free_list=fl)
    assert bm.add_sequence_cached(1, [11, 12, 13, 14, 15, 16]) == 0 == ref.add_sequence_cached(1, [11, 12, 13, 14,
                                                                                                   15, 16])
    for t, slot in ((17, 10), (18, 11), (19, 28)):
        s, p = bm.append_tokens([1], [t])
        assert s[0] == slot == ref.append_token(1, t)[0] and len(p) == 0
    assert bm.num_cached_blocks == 2
    bm.free_sequence(1)
    ref.free_sequence(1)
    _state(bm, ref, 8)
    second = [11, 12, 13, 14, 15, 16, 17, 18, 19, 30, 31, 32]
    assert bm.add_sequence_cached(2, second) == 8 == ref.add_sequence_cached(2, second)
    t, _ = bm.tables([2])
    assert list(t[0]) == [5, 2, 0] == ref.tables[2]
    _state(bm, ref, 8)


@pytest.mark.parametrize("bs", [4, 16])
def test_next_turn_reuses_prompt_and_answer_blocks(pkv_lib, bs):
    """A dialogue: turn 1's prompt, then its answer decoded token by token with
    ids; turn 2's prompt is turn 1's prompt + answer + a new user turn.  Every
    full block of turn 1 (prompt blocks and answer blocks alike) is reused,
    whether turn 1 is still running or has finished."""
    rng = np.random.default_rng(bs)
    NB = 64
    for finished in (False, True):
        bm = pkv_lib.BlockManager(NB, bs)
        ref = RefBlockManager(NB, bs)
        prompt = list(rng.integers(0, 32000, size=3 * bs + 5))
        answer = list(rng.integers(0, 32000, size=2 * bs + 7))
        assert bm.add_sequence_cached(0, prompt) == 0 == ref.add_sequence_cached(0, prompt)
        for t in answer:
            s, _ = bm.append_tokens([0], [t])
            assert s[0] == ref.append_token(0, t)[0]
        n1 = len(prompt) + len(answer)
        t1, _ = bm.tables([0])
        if finished:
            bm.free_sequence(0)
            ref.free_sequence(0)
        follow = prompt + answer + list(rng.integers(0, 32000, size=bs + 3))
        cached = bm.add_sequence_cached(1, follow)
        assert cached == ref.add_sequence_cached(1, follow) == (n1 // bs) * bs
        t2, _ = bm.tables([1])
        assert list(t2[0][: n1 // bs]) == list(t1[0][: n1 // bs])  # every full block of turn 1
        _state(bm, ref, NB)


def test_append_without_ids_stops_registration_and_forks_inherit(pkv_lib):
    bs = 4
    bm = pkv_lib.BlockManager(16, bs)
    ref = RefBlockManager(16, bs)
    for m in (bm, ref):
        m.add_sequence_cached(0, [1, 2, 3])
        m.add_sequence_cached(1, [1, 2, 3])
        m.fork(0, 2)
    # sequence 1 appends without an id: its block is not registered when it fills
    bm.append_slots([1])
    ref.append_slot(1)
    # the fork (2) and its parent (0) append the same token with ids: the parent
    # copies the shared partial block, the last holder writes in place, and the
    # first of them to fill registers the prefix 1, 2, 3, 9
    s, p = bm.append_tokens([0, 2], [9, 9])
    w0, w2 = ref.append_token(0, 9), ref.append_token(2, 9)
    assert list(s) == [w0[0], w2[0]] and [tuple(x) for x in p] == [w0[1]]
    _state(bm, ref, 16)
    assert bm.num_cached_blocks == 1
    assert bm.add_sequence_cached(3, [1, 2, 3, 9, 5]) == 4 == ref.add_sequence_cached(3, [1, 2, 3, 9, 5])
    _state(bm, ref, 16)
    with pytest.raises(ValueError):
        bm.append_tokens([0], [1, 2])
