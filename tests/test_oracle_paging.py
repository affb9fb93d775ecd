"""Pins for the oracle's append, block copy and naive allocator, from the
pages' worked examples (fixtures under tests/golden/, each naming its page)."""
import math

import numpy as np
import pytest
import torch

from oracle.block_manager_ref import (OutOfBlocks, RefBlockManager, kv_bytes_per_sequence,
                                      reserved_unused_slots)
from tests.conftest import golden


def test_t1_forty_tokens_scatter_and_gather(oracle_mod):
    g = golden("t1_ultralytics_40_tokens.json")
    bs, D, n = g["block_size"], g["head_dim"], g["num_tokens"]
    bm = RefBlockManager(g["pool_blocks"], bs, free_list=g["free_list"])
    table = bm.add_sequence(0, n)
    assert len(table) == g["expected_num_blocks"] == math.ceil(n / bs)
    assert table == g["expected_block_table"]
    # write every key through its slot, as the example does, with the oracle's append
    keys = torch.randn(n, 1, D, generator=torch.Generator().manual_seed(0)).half()
    pool_k = np.zeros((g["pool_blocks"], 1, bs, D), np.uint16)
    pool_v = np.zeros_like(pool_k)
    slots = np.array([oracle_mod.slot_of(table, pos, bs) for pos in range(n)], np.int64)
    kb = keys.view(torch.int16).numpy().view(np.uint16)
    oracle_mod.append(kb, kb, oracle_mod.F16, slots, pool_k, pool_v, oracle_mod.F16)
    # gather: pool[table] reshaped to tokens, first n rows
    gathered = pool_k[table][:, 0].reshape(-1, D)[:n]
    assert np.array_equal(gathered, kb[:, 0]) == g["expected_keys_intact"]
    assert bm.unused_slots(0) == g["expected_unused_slots_paged"]
    assert reserved_unused_slots(n, g["reservation_tokens"]) == g["expected_unused_slots_reserved"]
    # nothing outside the three blocks was touched
    untouched = [b for b in range(g["pool_blocks"]) if b not in table]
    assert not pool_k[untouched].any()


def test_t2_forty_one_token_table_and_next_slot(oracle_mod):
    g = golden("t2_optiverse_41_tokens.json")
    bs = g["block_size"]
    bm = RefBlockManager(64, bs, free_list=g["free_list"])
    table = bm.add_sequence(0, g["num_tokens"])
    assert table == g["expected_block_table"]
    fill = [min(bs, g["num_tokens"] - i * bs) for i in range(len(table))]
    assert fill == g["expected_fill"]
    slot, cow = bm.append_slot(0)  # token 41 (0-based)
    assert cow is None
    assert slot == g["expected_next_slot"]
    assert slot // bs == g["next_token_block"] and slot % bs + 1 == g["next_token_position_one_based"]
    # tokens 42..47 fill block 12; token 48 needs a new block from the free list
    for tok in range(42, g["last_token_filling_block"] + 1):
        s, _ = bm.append_slot(0)
        assert s // bs == 12 and s % bs == tok % bs
    assert len(bm.tables[0]) == 3
    s, _ = bm.append_slot(0)
    assert len(bm.tables[0]) == 4 and s == g["free_list"][3] * bs
    free_before = len(bm.free)
    bm.free_sequence(0)
    assert len(bm.free) - free_before == g["expected_blocks_returned"] + 1


def test_t3_eight_hundred_twenty_five_tokens():
    g = golden("t3_optiverse_825_tokens.json")
    bs, n = g["block_size"], g["num_tokens"]
    bm = RefBlockManager(100, bs)
    table = bm.add_sequence(0, n)
    assert len(table) == g["expected_blocks"]
    assert len(table) * bs == g["expected_slots"]
    assert bm.unused_slots(0) == g["expected_unused_slots"]
    assert n - (len(table) - 1) * bs == g["expected_filled_in_last_block"]
    assert reserved_unused_slots(n, g["reservation_tokens"]) == g["expected_unused_slots_reserved"]
    worst = 0
    for m in range(1, 200):
        ref = RefBlockManager(100, bs)
        ref.add_sequence(0, m)
        worst = max(worst, ref.unused_slots(0))
    assert worst == g["expected_max_unused_slots"]


def test_t4_copy_on_write_example(oracle_mod):
    g = golden("t4_ithome_copy_on_write.json")
    bs = g["block_size"]
    bm = RefBlockManager(8, bs, free_list=g["free_list"])
    prompt = bm.add_sequence("A1", len(g["prompt_tokens"]))
    assert prompt == g["expected_prompt_table"]
    bm.fork("A1", "A2")
    assert {str(b): bm.ref[b] for b in prompt} == g["expected_ref_counts_after_fork"]
    slot1, cow1 = bm.append_slot("A1")
    slot2, cow2 = bm.append_slot("A2")
    assert list(cow1) == g["expected_cow_pair_of_A1"] and cow2 is None
    assert bm.tables["A1"] == g["expected_table_A1"] and bm.tables["A2"] == g["expected_table_A2"]
    assert slot1 == g["expected_slot_A1"] and slot2 == g["expected_slot_A2"]
    counts = {str(b): bm.ref[b] for b in (7, 1, 3)}
    assert counts == g["expected_ref_counts_after_write"]

    # the device-side effect: copy the old block, then write each branch's new word
    D = 8
    k = np.zeros((8, 1, bs, D), np.uint16)
    v = np.zeros_like(k)
    words = np.arange(1, len(g["prompt_tokens"]) + 1, dtype=np.uint16)
    for pos in range(len(words)):
        s = oracle_mod.slot_of(prompt, pos, bs)
        k[s // bs, 0, s % bs, :] = words[pos]
    oracle_mod.block_copy(k, v, np.array([cow1], np.int32))
    new_a1 = np.full((1, 1, D), 100, np.uint16)  # "fathers"
    new_a2 = np.full((1, 1, D), 200, np.uint16)  # "mothers"
    oracle_mod.append(new_a1, new_a1, oracle_mod.F16, np.array([slot1]), k, v, oracle_mod.F16)
    oracle_mod.append(new_a2, new_a2, oracle_mod.F16, np.array([slot2]), k, v, oracle_mod.F16)
    assert list(k[3, 0, :, 0]) == [5, 6, 7, 100]  # copy of "years ago our" + "fathers"
    assert list(k[1, 0, :, 0]) == [5, 6, 7, 200]  # "years ago our" + "mothers"
    assert list(k[7, 0, :, 0]) == [1, 2, 3, 4]  # full shared block untouched


def test_t6_llama13b_bytes_per_sequence():
    g = golden("t6_llama13b_kv_bytes.json")
    n = kv_bytes_per_sequence(g["layers"], g["heads"], g["head_dim"], g["tokens"], g["elem_bytes"])
    assert n == 1_677_721_600
    assert round(n / 1e9, 1) == g["expected_gb_one_decimal"]


def test_full_shared_blocks_are_never_copied():
    bm = RefBlockManager(64, 16)
    bm.add_sequence(0, 32)  # two full blocks
    for c in (1, 2, 3):
        bm.fork(0, c)
    for s in (0, 1, 2, 3):
        _, cow = bm.append_slot(s)
        assert cow is None  # position 32 starts a fresh block
    assert [bm.ref[b] for b in bm.tables[0][:2]] == [4, 4]
    assert len({bm.tables[s][2] for s in range(4)}) == 4


def test_parallel_sampling_copies_n_minus_one():
    bm = RefBlockManager(64, 16)
    bm.add_sequence(0, 40)
    for c in (1, 2, 3):
        bm.fork(0, c)
    pairs = [bm.append_slot(s)[1] for s in range(4)]
    assert sum(p is not None for p in pairs) == 3 and pairs[3] is None
    last = bm.tables[3][2]
    assert bm.ref[last] == 1 and all(p[0] == last for p in pairs[:3])


def test_block_copy_whole_blocks(oracle_mod):
    rng = np.random.default_rng(0)
    k = rng.integers(0, 1 << 16, size=(6, 2, 4, 8), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(6, 2, 4, 8), dtype=np.uint16)
    k0, v0 = k.copy(), v.copy()
    oracle_mod.block_copy(k, v, np.array([[1, 4], [2, 5]], np.int32))
    assert np.array_equal(k[4], k0[1]) and np.array_equal(v[5], v0[2])
    assert np.array_equal(k[:4], k0[:4]) and np.array_equal(v[:4], v0[:4])
    with pytest.raises(ValueError):
        oracle_mod.block_copy(k, v, np.array([[1, 6]], np.int32))


def test_append_skips_negative_slots_and_quantises(oracle_mod):
    rng = np.random.default_rng(1)
    x = torch.from_numpy(rng.standard_normal((3, 2, 16)).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    kc = np.zeros((2, 2, 4, 16), np.uint8)
    vc = np.zeros_like(kc)
    oracle_mod.append(xb, xb, oracle_mod.BF16, np.array([5, -1, 2]), kc, vc, oracle_mod.E4M3,
                      k_scale=0.01, v_scale=0.02)
    want_k = torch.from_numpy((x.float() / torch.tensor(0.01, dtype=torch.float32)).numpy())
    want_k = want_k.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(kc[1, :, 1], want_k[0]) and np.array_equal(kc[0, :, 2], want_k[2])
    assert not kc[0, :, 1].any() and not kc[1, :, 0].any()
    with pytest.raises(ValueError):
        oracle_mod.append(xb, xb, oracle_mod.BF16, np.array([8, 0, 0]), kc, vc, oracle_mod.E4M3)


def test_out_of_blocks_raises():
    bm = RefBlockManager(2, 16)
    bm.add_sequence(0, 32)
    with pytest.raises(OutOfBlocks):
        bm.append_slot(0)
    with pytest.raises(OutOfBlocks):
        bm.add_sequence(1, 1)


def test_reference_swap_hand_example():
    """Preemption by swapping, worked by hand: a 10-token sequence at block
    size 4 holds 3 blocks; swapping it out returns them to the back of the free
    list (FIFO); another request then takes blocks from the front; swapping
    back in takes 3 fresh blocks from the front in order, with the length kept.
    A shared (forked) block is only released when its last holder leaves."""
    from oracle.block_manager_ref import OutOfBlocks, RefBlockManager
    ref = RefBlockManager(8, 4)                     # free list 0..7
    ref.add_sequence("a", 10)                       # blocks 0, 1, 2
    assert ref.tables["a"] == [0, 1, 2] and ref.free == [3, 4, 5, 6, 7]
    assert ref.swap_out("a") == [0, 1, 2]
    assert ref.free == [3, 4, 5, 6, 7, 0, 1, 2] and "a" not in ref.tables
    ref.add_sequence("b", 17)                       # ceil(17/4) = 5 blocks from the front
    assert ref.tables["b"] == [3, 4, 5, 6, 7] and ref.free == [0, 1, 2]
    assert ref.swap_in("a") == [0, 1, 2] and ref.lens["a"] == 10 and ref.free == []
    assert ref.swap_out("b") == [3, 4, 5, 6, 7]
    ref.add_sequence("c", 20)                       # 5 blocks: b's freed blocks
    with pytest.raises(OutOfBlocks):
        ref.swap_in("b")                            # no room: b stays swapped out
    assert set(ref.swapped) == {"b"} and ref.swapped["b"]["len"] == 17
    # a forked sequence shares its parent's blocks: swapping the child out
    # releases nothing, swapping the parent out too releases them
    ref2 = RefBlockManager(4, 4)
    ref2.add_sequence("p", 6)                       # blocks 0, 1
    ref2.fork("p", "q")
    ref2.swap_out("q")
    assert ref2.free == [2, 3] and ref2.ref[:2] == [1, 1]
    ref2.swap_out("p")
    assert ref2.free == [2, 3, 0, 1]


def test_reference_prefix_cache_multi_turn_hand_example():
    """Automatic prefix caching across the rounds of a dialogue, worked by hand
    (the PagedAttention notes page, section on automatic prefix caching: a
    block is found by its own and all earlier tokens, so the next turn reuses
    the KV of the previous turn's prompt AND answer).  Block size 4, free
    list [5, 2, 7, 0, 1, 3, 4, 6]:

    turn 1  prompt 11..16 (6 tokens): block 5 = 11..14 (full, registered),
             block 2 = 15, 16 (partial).  Decoding 17 and 18 fills block 2,
             which is registered under 11..18; 19 starts block 7 (slot 28).
             Freeing the request parks the registered blocks 5 and 2 on the
             LRU list; block 7 goes to the back of the free list.
    turn 2  prompt 11..19, 30, 31, 32 (12 tokens): 11..14 and 11..18 hit
             (blocks 5 and 2), 11..32 misses and takes block 0 -> 8 tokens
             already in the pool.
    """
    from oracle.block_manager_ref import RefBlockManager
    ref = RefBlockManager(8, 4, free_list=[5, 2, 7, 0, 1, 3, 4, 6])
    assert ref.add_sequence_cached("r1", [11, 12, 13, 14, 15, 16]) == 0
    assert ref.tables["r1"] == [5, 2] and ref.block_of_prefix == {(11, 12, 13, 14): 5}
    assert ref.append_token("r1", 17) == (2 * 4 + 2, None)
    assert ref.append_token("r1", 18) == (2 * 4 + 3, None)
    assert ref.block_of_prefix[(11, 12, 13, 14, 15, 16, 17, 18)] == 2
    assert ref.append_token("r1", 19) == (7 * 4 + 0, None)
    ref.free_sequence("r1")
    assert ref.lru == [5, 2] and ref.free == [0, 1, 3, 4, 6, 7]
    assert ref.add_sequence_cached("r2", [11, 12, 13, 14, 15, 16, 17, 18, 19, 30, 31, 32]) == 8
    assert ref.tables["r2"] == [5, 2, 0] and ref.lru == [] and ref.free == [1, 3, 4, 6, 7]
    assert ref.ref[5] == ref.ref[2] == ref.ref[0] == 1
    # a sequence appended to without token ids stops registering blocks
    ref.add_sequence_cached("r3", [40, 41, 42])
    ref.append_slot("r3")
    ref.append_token("r3", 44)
    assert all(40 not in key for key in ref.block_of_prefix)
    # the first registration of a prefix stays: a second request that decodes
    # the same tokens into its own block does not replace it
    ref.add_sequence_cached("r4", [50, 51])
    ref.add_sequence_cached("r5", [50, 51])
    for t in (52, 53):
        ref.append_token("r4", t)
        ref.append_token("r5", t)
    assert ref.block_of_prefix[(50, 51, 52, 53)] == ref.tables["r4"][0] != ref.tables["r5"][0]


def test_reference_group_swap_hand_example():
    """Swapping a forked group together keeps its sharing, worked by hand.
    Block size 4, free list 0..9.  p holds 6 tokens in blocks [0, 1]; c1 and c2
    fork p; c1 appends a token, copying the shared partial block 1 to block 2.
    Tables p = [0, 1], c1 = [0, 2], c2 = [0, 1]; counts 0:3, 1:2, 2:1.

    swap_out_group(p, c1, c2) lists the distinct blocks once, in first-use
    order: [0, 1, 2] (three stagings, not six).  Releases run member by
    member, table order: 2 reaches 0 in c1's release, then 0 and 1 in c2's,
    so the free list becomes 3..9, 2, 0, 1.

    swap_in_group takes three fresh blocks from the front, 3, 4, 5, for list
    entries 0, 1, 2: p = [3, 4], c1 = [3, 5], c2 = [3, 4], counts 3:3, 4:2,
    5:1 -- the sharing is back, so c2's next token copies block 4 again."""
    from oracle.block_manager_ref import RefBlockManager
    ref = RefBlockManager(10, 4)
    ref.add_sequence("p", 6)
    ref.fork("p", "c1")
    ref.fork("p", "c2")
    assert ref.append_slot("c1") == (2 * 4 + 2, (1, 2))
    assert (ref.tables["p"], ref.tables["c1"], ref.tables["c2"]) == ([0, 1], [0, 2], [0, 1])
    assert ref.swap_out_group(["p", "c1", "c2"]) == [0, 1, 2]
    assert ref.free == [3, 4, 5, 6, 7, 8, 9, 2, 0, 1] and ref.ref[:3] == [0, 0, 0]
    assert ref.swap_in_group(["c2", "p", "c1"]) == [3, 4, 5]
    assert (ref.tables["p"], ref.tables["c1"], ref.tables["c2"]) == ([3, 4], [3, 5], [3, 4])
    assert ref.ref[3:6] == [3, 2, 1] and ref.lens == {"p": 6, "c1": 7, "c2": 6}
    assert ref.append_slot("c2") == (6 * 4 + 2, (4, 6))
    # a member freed while swapped out: its only block is taken and released at once
    ref2 = RefBlockManager(6, 4)
    ref2.add_sequence("a", 4)                       # block 0 (full)
    ref2.fork("a", "b")
    ref2.append_slot("b")                           # b: [0, 1]
    assert ref2.swap_out_group(["a", "b"]) == [0, 1]
    ref2.free_sequence("b")
    assert ref2.swap_in_group(["a"]) == [2, 3]
    assert ref2.tables["a"] == [2] and ref2.ref[2:4] == [1, 0] and ref2.free[-1] == 3


def test_reference_block_swap_bytes(oracle_mod):
    """Swap staging by hand: every byte of K block b is b, of V block b is 100 + b;
    ids [3, 0, 2] stage entries (3, 103), (0, 100), (2, 102); swapping the
    entries back in to blocks [1, 4, 0] makes those blocks hold them."""
    NB, nbytes = 5, 32
    k = np.repeat(np.arange(NB, dtype=np.uint8), nbytes).reshape(NB, 2, 16)
    v = (k + 100).astype(np.uint8)
    st = oracle_mod.block_swap_out(k, v, [3, 0, 2])
    assert st.shape == (3, 2, nbytes)
    assert [int(x) for x in st[:, 0, 0]] == [3, 0, 2] and [int(x) for x in st[:, 1, 0]] == [103, 100, 102]
    assert all(np.all(st[i, j] == st[i, j, 0]) for i in range(3) for j in range(2))
    oracle_mod.block_swap_in(k, v, [1, 4, 0], st)
    assert [int(x) for x in k[:, 0, 0]] == [2, 3, 2, 3, 0] and [int(x) for x in v[:, 0, 0]] == [102, 103, 102, 103, 100]
