"""The C++ block manager (libpagedkv.so) against the naive oracle allocator
and the pages' worked examples."""
import numpy as np
import pytest

from oracle.block_manager_ref import OutOfBlocks as RefOutOfBlocks
from oracle.block_manager_ref import RefBlockManager
from tests.conftest import golden


def test_t1_t2_t3_tables(pkv_lib):
    g = golden("t1_ultralytics_40_tokens.json")
    bm = pkv_lib.BlockManager(g["pool_blocks"], g["block_size"], free_list=g["free_list"])
    bm.add_sequence(0, g["num_tokens"])
    t, lens = bm.tables([0])
    assert list(t[0]) == g["expected_block_table"] and lens[0] == 40
    g = golden("t2_optiverse_41_tokens.json")
    bm = pkv_lib.BlockManager(64, g["block_size"], free_list=g["free_list"])
    bm.add_sequence(7, g["num_tokens"])
    slots, pairs = bm.append_slots([7])
    assert slots[0] == g["expected_next_slot"] and len(pairs) == 0
    for _ in range(42, g["last_token_filling_block"] + 1):
        bm.append_slots([7])
    assert bm.num_seq_blocks(7) == 3
    bm.append_slots([7])
    assert bm.num_seq_blocks(7) == 4
    n0 = bm.num_free
    bm.free_sequence(7)
    assert bm.num_free - n0 == 4
    g = golden("t3_optiverse_825_tokens.json")
    bm = pkv_lib.BlockManager(100, 16)
    bm.add_sequence(0, g["num_tokens"])
    assert bm.num_seq_blocks(0) == g["expected_blocks"]


def test_t4_copy_on_write(pkv_lib):
    g = golden("t4_ithome_copy_on_write.json")
    bm = pkv_lib.BlockManager(8, g["block_size"], free_list=g["free_list"])
    bm.add_sequence(1, len(g["prompt_tokens"]))  # A1
    bm.fork(1, 2)  # A2
    assert {str(b): bm.ref_count(b) for b in g["expected_prompt_table"]} == g["expected_ref_counts_after_fork"]
    slots, pairs = bm.append_slots([1, 2])  # A1 writes first, then A2
    assert [list(p) for p in pairs] == [g["expected_cow_pair_of_A1"]]
    assert list(slots) == [g["expected_slot_A1"], g["expected_slot_A2"]]
    t, _ = bm.tables([1, 2])
    assert list(t[0]) == g["expected_table_A1"] and list(t[1]) == g["expected_table_A2"]
    assert {str(b): bm.ref_count(b) for b in (7, 1, 3)} == g["expected_ref_counts_after_write"]


def _run_random(pkv_lib, seed, n_ops=600):
    rng = np.random.default_rng(seed)
    NB, bs = int(rng.integers(8, 64)), int(rng.choice([1, 4, 16]))
    fl = rng.permutation(NB).astype(np.int32)
    ref = RefBlockManager(NB, bs, free_list=fl)
    bm = pkv_lib.BlockManager(NB, bs, free_list=fl)
    live, next_id = [], 0
    for _ in range(n_ops):
        op = rng.integers(0, 4)
        if op == 0 or not live:
            n = int(rng.integers(0, 3 * bs + 2))
            try:
                ref.add_sequence(next_id, n)
                ok = True
            except RefOutOfBlocks:
                ok = False
            if ok:
                bm.add_sequence(next_id, n)
                live.append(next_id)
            else:
                with pytest.raises(pkv_lib.OutOfBlocks):
                    bm.add_sequence(next_id, n)
            next_id += 1
        elif op == 1:
            k = int(rng.integers(1, len(live) + 1))
            batch = [int(x) for x in rng.choice(live, size=k, replace=False)]
            # the oracle handles writers one at a time; the batch call is all or nothing
            snap = (list(ref.free), list(ref.ref), {s: list(t) for s, t in ref.tables.items()}, dict(ref.lens))
            try:
                want = [ref.append_slot(s) for s in batch]
                ok = True
            except RefOutOfBlocks:
                ref.free, ref.ref, ref.tables, ref.lens = snap
                ok = False
            if ok:
                slots, pairs = bm.append_slots(batch)
                assert list(slots) == [w[0] for w in want]
                assert [tuple(p) for p in pairs] == [w[1] for w in want if w[1] is not None]
            else:
                with pytest.raises(pkv_lib.OutOfBlocks):
                    bm.append_slots(batch)
        elif op == 2:
            parent = int(rng.choice(live))
            ref.fork(parent, next_id)
            bm.fork(parent, next_id)
            live.append(next_id)
            next_id += 1
        else:
            s = live.pop(int(rng.integers(0, len(live))))
            ref.free_sequence(s)
            bm.free_sequence(s)
        assert list(bm.free_list()) == ref.free
        assert [bm.ref_count(b) for b in range(NB)] == ref.ref
    for s in live:
        t, lens = bm.tables([s])
        assert list(t[0][: len(ref.tables[s])]) == ref.tables[s] and lens[0] == ref.lens[s]


@pytest.mark.parametrize("seed", range(12))
def test_random_operations_match_oracle(pkv_lib, seed):
    _run_random(pkv_lib, seed)


def test_errors(pkv_lib):
    bm = pkv_lib.BlockManager(4, 16)
    bm.add_sequence(1, 10)
    with pytest.raises(pkv_lib.PagedKVError):
        bm.add_sequence(1, 3)  # id in use
    with pytest.raises(pkv_lib.PagedKVError):
        bm.append_slots([1, 1])  # repeated id
    with pytest.raises(pkv_lib.PagedKVError):
        bm.free_sequence(9)
    with pytest.raises(pkv_lib.OutOfBlocks):
        bm.add_sequence(2, 64)
    assert bm.num_free == 3 and bm.context_len(1) == 10 and bm.context_len(9) == -1
    with pytest.raises(pkv_lib.PagedKVError):
        pkv_lib.BlockManager(4, 16, free_list=[0, 0])
    t, lens = bm.tables([1], max_blocks_per_seq=3, pad=-1)
    assert list(t[0]) == [0, -1, -1] and lens[0] == 10


@pytest.mark.parametrize("seed", range(6))
def test_swap_out_in_matches_oracle(pkv_lib, seed):
    rng = np.random.default_rng(100 + seed)
    NB, bs = int(rng.integers(10, 40)), int(rng.choice([4, 16]))
    fl = rng.permutation(NB).astype(np.int32)
    bm = pkv_lib.BlockManager(NB, bs, free_list=fl)
    ref = RefBlockManager(NB, bs, free_list=fl)
    live, out, nid = [], [], 0
    for _ in range(250):
        op = int(rng.integers(0, 6))
        if op == 0 or not (live or out):
            n = int(rng.integers(1, 3 * bs))
            try:
                ref.add_sequence(nid, n)
                bm.add_sequence(nid, n)
                live.append(nid)
            except RefOutOfBlocks:
                with pytest.raises(pkv_lib.OutOfBlocks):
                    bm.add_sequence(nid, n)
            nid += 1
        elif op == 1 and live:
            s = int(rng.choice(live))
            try:
                want = ref.append_slot(s)
            except RefOutOfBlocks:
                continue  # (state unchanged on both sides only if the product also refuses)
            slots, _ = bm.append_slots([s])
            assert slots[0] == want[0]
        elif op == 2 and live:
            parent = int(rng.choice(live))
            ref.fork(parent, nid)
            bm.fork(parent, nid)
            live.append(nid)
            nid += 1
        elif op == 3 and live:
            s = live.pop(int(rng.integers(0, len(live))))
            assert list(bm.swap_out(s)) == ref.swap_out(s)
            out.append(s)
            with pytest.raises(pkv_lib.PagedKVError):
                bm.append_slots([s])
        elif op == 4 and out:
            s = out[int(rng.integers(0, len(out)))]
            try:
                want = ref.swap_in(s)
            except RefOutOfBlocks:
                with pytest.raises(pkv_lib.OutOfBlocks):
                    bm.swap_in(s, 64)
                continue
            assert list(bm.swap_in(s, 64)) == want
            out.remove(s)
            live.append(s)
        elif op == 5 and (live or out):
            pool = live + out
            s = pool[int(rng.integers(0, len(pool)))]
            bm.free_sequence(s)
            ref.free_sequence(s)
            (live if s in live else out).remove(s)
        assert list(bm.free_list()) == ref.free
        assert [bm.ref_count(b) for b in range(NB)] == ref.ref


def _snapshot(bm, ids, NB):
    t, lens = bm.tables(ids)
    return (t.tolist(), lens.tolist(), list(bm.free_list()), [bm.ref_count(b) for b in range(NB)])


def test_pool_exhausted_mid_step_changes_nothing(pkv_lib):
    """A batched append that runs out of blocks part-way fails as a whole: no
    slot is handed out, and tables, lengths, free list and reference counts
    stay as they were (host-side fault injection: the pool empties mid-step)."""
    NB, bs = 4, 4
    bm = pkv_lib.BlockManager(NB, bs)
    bm.add_sequence(1, 8)  # two full blocks
    bm.add_sequence(2, 4)  # one full block; one block left
    before = _snapshot(bm, [1, 2], NB)
    with pytest.raises(pkv_lib.OutOfBlocks):
        bm.append_slots([1, 2])  # each needs a fresh block, only one is free
    assert _snapshot(bm, [1, 2], NB) == before
    slots, copies = bm.append_slots([1])  # the pool still serves a step that fits
    assert len(slots) == 1 and len(copies) == 0 and bm.num_free == 0


def test_copy_on_write_without_a_free_block_changes_nothing(pkv_lib):
    """The last block of a forked sequence is shared and partly filled; the
    child's write needs a copy, the pool is empty, so the step fails and the
    shared block keeps its reference count of 2."""
    NB, bs = 3, 4
    bm = pkv_lib.BlockManager(NB, bs)
    bm.add_sequence(1, 6)  # blocks: one full, one partly filled
    bm.fork(1, 2)
    bm.add_sequence(3, 4)  # takes the last free block
    before = _snapshot(bm, [1, 2, 3], NB)
    shared = before[0][0][1]
    assert bm.ref_count(shared) == 2 and bm.num_free == 0
    with pytest.raises(pkv_lib.OutOfBlocks):
        bm.append_slots([2])
    assert _snapshot(bm, [1, 2, 3], NB) == before
    bm.free_sequence(3)  # a block comes back; now the copy succeeds
    slots, copies = bm.append_slots([2])
    assert len(copies) == 1 and copies[0][0] == shared and bm.ref_count(shared) == 1


def test_group_swap_hand_example_matches_oracle(pkv_lib):
    """The oracle's hand-worked group swap (block size 4, free list 0..9):
    three forked samples stage their 3 distinct blocks once and get them back
    shared (counts 3, 2, 1)."""
    bm = pkv_lib.BlockManager(10, 4)
    ref = RefBlockManager(10, 4)
    ids = {"p": 0, "c1": 1, "c2": 2}
    for m, key in ((bm, lambda x: ids[x]), (ref, lambda x: x)):
        m.add_sequence(key("p"), 6)
        m.fork(key("p"), key("c1"))
        m.fork(key("p"), key("c2"))
    s, pairs = bm.append_slots([1])
    assert (s[0], tuple(pairs[0])) == ref.append_slot("c1")
    assert list(bm.swap_out_group([0, 1, 2])) == ref.swap_out_group(["p", "c1", "c2"]) == [0, 1, 2]
    assert list(bm.free_list()) == ref.free
    assert list(bm.swap_in_group([2, 0, 1], 8)) == ref.swap_in_group(["c2", "p", "c1"]) == [3, 4, 5]
    t, lens = bm.tables([0, 1, 2])
    assert [list(r[:2]) for r in t] == [ref.tables["p"], ref.tables["c1"], ref.tables["c2"]]
    assert [bm.ref_count(b) for b in range(10)] == ref.ref
    s, pairs = bm.append_slots([2])
    assert (s[0], tuple(pairs[0])) == ref.append_slot("c2")
    # the single-sequence calls refuse a member of a group
    bm.swap_out_group([0, 1])
    with pytest.raises(pkv_lib.PagedKVError):
        bm.swap_in(0, 8)
    with pytest.raises(pkv_lib.PagedKVError):
        bm.swap_in_group([0], 8)
    assert len(bm.swap_in_group([1, 0], 8)) == 3


@pytest.mark.parametrize("seed", range(6))
def test_group_swap_matches_oracle(pkv_lib, seed):
    """Random forks, appends (with copy-on-write), group swaps, frees of
    resident and swapped members: lists, tables, counts and free lists equal
    the oracle allocator's after every step."""
    rng = np.random.default_rng(300 + seed)
    NB, bs = int(rng.integers(16, 48)), int(rng.choice([2, 4, 16]))
    fl = rng.permutation(NB).astype(np.int32)
    bm = pkv_lib.BlockManager(NB, bs, free_list=fl)
    ref = RefBlockManager(NB, bs, free_list=fl)
    live, groups, nid = [], [], 0

    def check():
        assert [bm.ref_count(b) for b in range(NB)] == ref.ref
        assert list(bm.free_list()) == ref.free
        if live:
            t, lens = bm.tables(live)
            for i, s in enumerate(live):
                assert list(t[i][: len(ref.tables[s])]) == ref.tables[s] and lens[i] == ref.lens[s]

    for _ in range(300):
        op = int(rng.integers(0, 7))
        if op == 0 or not (live or groups):
            n = int(rng.integers(1, 3 * bs))
            try:
                ref.add_sequence(nid, n)
                bm.add_sequence(nid, n)
                live.append(nid)
            except RefOutOfBlocks:
                with pytest.raises(pkv_lib.OutOfBlocks):
                    bm.add_sequence(nid, n)
            nid += 1
        elif op in (1, 2) and live:
            s = int(rng.choice(live))
            try:
                want = ref.append_slot(s)
            except RefOutOfBlocks:
                with pytest.raises(pkv_lib.OutOfBlocks):
                    bm.append_slots([s])
                continue
            slots, pairs = bm.append_slots([s])
            assert slots[0] == want[0] and [tuple(p) for p in pairs] == ([want[1]] if want[1] else [])
        elif op == 3 and live:
            parent = int(rng.choice(live))
            ref.fork(parent, nid)
            bm.fork(parent, nid)
            live.append(nid)
            nid += 1
        elif op == 4 and live:
            k = int(rng.integers(1, min(4, len(live)) + 1))
            members = [int(x) for x in rng.choice(live, size=k, replace=False)]
            assert list(bm.swap_out_group(members)) == ref.swap_out_group(members)
            for s in members:
                live.remove(s)
            groups.append(members)
        elif op == 5 and groups:
            g = groups[int(rng.integers(0, len(groups)))]
            order = [int(x) for x in rng.permutation(g)]
            try:
                want = ref.swap_in_group(order)
            except RefOutOfBlocks:
                with pytest.raises(pkv_lib.OutOfBlocks):
                    bm.swap_in_group(order, 4 * NB)
                continue
            assert list(bm.swap_in_group(order, 4 * NB)) == want
            groups.remove(g)
            live.extend(g)
        elif op == 6 and (live or groups):
            pool = live + [s for g in groups for s in g]
            s = pool[int(rng.integers(0, len(pool)))]
            bm.free_sequence(s)
            ref.free_sequence(s)
            if s in live:
                live.remove(s)
            else:
                for g in groups:
                    if s in g:
                        g.remove(s)
                groups = [g for g in groups if g]
        check()
