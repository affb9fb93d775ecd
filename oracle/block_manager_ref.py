"""Naive block allocator: the oracle for the host-side block manager.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Plain Python lists and
dicts, one operation at a time, written from the pages:

* Ultralytics glossary "PagedAttention", section "How paging works": a request
  of n tokens takes ceil(n / block_size) blocks popped from the front of the
  free list; a new block is taken only when the last one is full.
* OptiVerse "Paged KV cache", section "Block table and non-contiguous
  allocation": the table maps logical block i (tokens 16 i .. 16 i + 15) to a
  physical block; the token after a 41-token prompt goes to offset 9 (the
  10th position) of the third block; all blocks return to the pool when the
  request ends.
* iThome "how to store the KV cache", sections "Physical Block sharing" and
  "Copy-on-Write": forked samples point at the same blocks with a reference
  count; a writer into a shared, partly filled last block gets a fresh block
  holding a copy, and the old block's count drops by one; full shared blocks
  stay shared with unchanged counts.

* PagedAttention notes, section on automatic prefix caching: a KV block is
  looked up by all tokens up to and including it; equal keys are equal
  blocks, and the stated use is a later turn of a dialogue reusing the
  KV of the earlier turns (prompt and answer).  Here the key is the exact
  token prefix itself (a tuple), not a hash of it.  A block is registered
  when it becomes full: a prompt's full blocks when the prompt is added, and
  a block filled by decoding when its last token is appended with its id.

Readings where the pages are silent: freed blocks go to the back of the free
list; writers are processed one at a time in call order, and a writer copies
only while the block's count is above 1, so the last holder writes in place.
Prefix cache: a sequence added from its token ids keeps its token list;
appending a token with its id extends the list, and a block that becomes full
is registered under its prefix unless that prefix already names a block (the
first registration stays).  Appending without an id ends the tracking of that
sequence (its later blocks are not registered).  A registered block whose
count reaches 0 keeps its contents on a least-recently-freed list and is taken
(and forgotten) only when the free list is empty.
"""
from __future__ import annotations


class OutOfBlocks(RuntimeError):
    pass


class RefBlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_list=None):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = list(range(num_blocks)) if free_list is None else [int(b) for b in free_list]
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        self.prefix_of_block: dict[int, tuple] = {}  # registered block -> its token prefix
        self.block_of_prefix: dict[tuple, int] = {}
        self.lru: list[int] = []  # registered blocks with count 0, least recently freed first
        self.tokens: dict[int, list[int]] = {}  # token ids of sequences added from their prompt ids

    def available(self) -> int:
        return len(self.free) + len(self.lru)

    def _take(self) -> int:
        if self.free:
            b = self.free.pop(0)
        elif self.lru:
            b = self.lru.pop(0)
            del self.block_of_prefix[self.prefix_of_block.pop(b)]
        else:
            raise OutOfBlocks("no free block")
        self.ref[b] = 1
        return b

    def add_sequence(self, seq: int, num_tokens: int) -> list[int]:
        """Give a new request ceil(num_tokens / bs) blocks (its prompt)."""
        assert seq not in self.tables
        need = -(-num_tokens // self.block_size)
        if need > self.available():
            raise OutOfBlocks(f"need {need} blocks, {self.available()} free")
        self.tables[seq] = [self._take() for _ in range(need)]
        self.lens[seq] = num_tokens
        return list(self.tables[seq])

    def append_slot(self, seq: int):
        """Reserve the slot of the next token; return (slot, cow_pair or None).
        The token's id is not known, so the sequence's blocks are no longer
        registered from here on."""
        self.tokens.pop(seq, None)
        return self._reserve(seq)

    def append_token(self, seq: int, token: int):
        """Reserve the slot of the next token, whose id is `token`; return
        (slot, cow_pair or None).  If the token fills its block and the
        sequence's token ids are known, the block is registered under the
        sequence's whole token prefix (unless that prefix already names a
        block)."""
        pos = self.lens[seq]
        slot, cow = self._reserve(seq)
        toks = self.tokens.get(seq)
        if toks is not None:
            toks.append(int(token))
            if (pos + 1) % self.block_size == 0:
                key = tuple(toks[: pos + 1])
                if key not in self.block_of_prefix:
                    b = self.tables[seq][pos // self.block_size]
                    self.block_of_prefix[key] = b
                    self.prefix_of_block[b] = key
        return slot, cow

    def _reserve(self, seq: int):
        table = self.tables[seq]
        pos = self.lens[seq]
        bs = self.block_size
        cow = None
        if pos % bs == 0:
            table.append(self._take())
        else:
            last = table[pos // bs]
            if self.ref[last] > 1:
                new = self._take()
                cow = (last, new)
                self.ref[last] -= 1
                table[pos // bs] = new
        self.lens[seq] = pos + 1
        return table[pos // bs] * bs + pos % bs, cow

    def add_sequence_cached(self, seq, tokens) -> int:
        """Register a prompt by its token ids, sharing the blocks of the longest
        registered prefix of full blocks; returns the number of leading tokens
        whose blocks were shared."""
        assert seq not in self.tables
        tokens = [int(t) for t in tokens]
        bs = self.block_size
        n_full = len(tokens) // bs
        n_blocks = -(-len(tokens) // bs)
        shared = []
        for i in range(n_full):
            key = tuple(tokens[: (i + 1) * bs])
            if key not in self.block_of_prefix:
                break
            shared.append(self.block_of_prefix[key])
        revived = sum(1 for b in shared if self.ref[b] == 0)
        if n_blocks - len(shared) > self.available() - revived:
            raise OutOfBlocks("not enough free blocks")
        for b in shared:
            if self.ref[b] == 0:
                self.lru.remove(b)
            self.ref[b] += 1
        table = list(shared)
        for i in range(len(shared), n_blocks):
            b = self._take()
            key = tuple(tokens[: (i + 1) * bs])
            if i < n_full and key not in self.block_of_prefix:  # the first registration stays
                self.block_of_prefix[key] = b
                self.prefix_of_block[b] = key
            table.append(b)
        self.tables[seq] = table
        self.lens[seq] = len(tokens)
        self.tokens[seq] = tokens
        return len(shared) * bs

    def fork(self, parent: int, child: int) -> None:
        """The child shares every block of the parent (counts + 1)."""
        assert child not in self.tables
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        if parent in self.tokens:
            self.tokens[child] = list(self.tokens[parent])
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_sequence(self, seq: int) -> None:
        """Release a finished request: counts - 1, blocks at 0 go back to the pool."""
        self.tokens.pop(seq, None)
        if seq in getattr(self, "swapped", {}):
            gid = self.swapped.pop(seq)["group"]
            self.swap_groups[gid]["members"].discard(seq)
            if not self.swap_groups[gid]["members"]:
                del self.swap_groups[gid]
            return
        for b in self.tables.pop(seq):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                if b in self.prefix_of_block:
                    self.lru.append(b)
                else:
                    self.free.append(b)
        del self.lens[seq]

    def swap_out(self, seq) -> list:
        """Preemption by swapping (PagedAttention notes, section on preemption):
        release the sequence's blocks, remember its length; returns its table."""
        return self.swap_out_group([seq])

    def swap_in(self, seq) -> list:
        """Give a swapped-out sequence ceil(len / bs) fresh blocks; returns them."""
        return self.swap_in_group([seq])

    def swap_out_group(self, seqs) -> list:
        """Swap out several sequences together (the samples of one prompt):
        their distinct blocks, in first-use order (members in the given order,
        each table in logical order), are listed once -- each is staged once --
        and every member remembers its table as positions in that list.  Then
        each member releases its blocks (members in order, tables in logical
        order).  Returns the list."""
        seqs = list(seqs)
        assert len(set(seqs)) == len(seqs)
        staged, pos = [], {}
        for s in seqs:
            for b in self.tables[s]:
                if b not in pos:
                    pos[b] = len(staged)
                    staged.append(b)
        self.swapped = getattr(self, "swapped", {})
        self.swap_groups = getattr(self, "swap_groups", {})
        gid = object()
        self.swap_groups[gid] = {"members": set(seqs), "staged": len(staged)}
        for s in seqs:
            table = self.tables.pop(s)
            for b in table:
                self.ref[b] -= 1
                if self.ref[b] == 0:
                    if b in self.prefix_of_block:
                        self.lru.append(b)
                    else:
                        self.free.append(b)
            self.swapped[s] = {"len": self.lens.pop(s), "idx": [pos[b] for b in table], "group": gid}
        return staged

    def swap_in_group(self, seqs) -> list:
        """Bring a group swapped out together back (the same members, in any
        order; a member freed meanwhile is left out): one fresh block per
        listed entry, taken in list order; each member's table is rebuilt over
        them, so blocks the members shared are shared again, with counts equal
        to the number of members holding them.  An entry no member holds any
        more is released at once.  Returns the blocks, in list order."""
        seqs = list(seqs)
        gid = self.swapped[seqs[0]]["group"]
        grp = self.swap_groups[gid]
        assert set(seqs) == grp["members"], "swap in the whole group"
        n = grp["staged"]
        if n > self.available():
            raise OutOfBlocks("not enough free blocks")
        blocks = [self._take() for _ in range(n)]
        held = [0] * n
        for s in seqs:
            for i in self.swapped[s]["idx"]:
                held[i] += 1
        for i, b in enumerate(blocks):
            self.ref[b] = held[i]
            if held[i] == 0:
                self.free.append(b)
        for s in seqs:
            info = self.swapped.pop(s)
            self.tables[s] = [blocks[i] for i in info["idx"]]
            self.lens[s] = info["len"]
        del self.swap_groups[gid]
        return blocks

    def unused_slots(self, seq: int) -> int:
        """Slots allocated to the request but not yet written."""
        return len(self.tables[seq]) * self.block_size - self.lens[seq]


def reserved_unused_slots(num_tokens: int, reservation: int) -> int:
    """Slots left empty by a contiguous reservation of ``reservation`` tokens."""
    return reservation - num_tokens


def kv_bytes_per_sequence(layers: int, heads: int, head_dim: int, tokens: int, elem_bytes: int) -> int:
    """K and V bytes of one sequence across all layers."""
    return layers * heads * head_dim * 2 * elem_bytes * tokens
