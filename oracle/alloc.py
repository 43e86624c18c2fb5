"""ORACLE -- test infrastructure only.

Plain Python model of the paged KV cache's block manager: a fixed pool of
physical blocks, a free-block queue, a reference count per physical block and
one block table per sequence whose entries carry the logical->physical
mapping and the number of filled slots ("#filled").  Only ``tests/``,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may use it.

Sources, in the order the steps are taken:

* Pool and free queue: a fixed set of equal-size blocks, sized once; new
  blocks come from the head of a free queue (vLLM teardown,
  arcyou.ai/ko/teardowns/vllm-paged-attention, "PagedAttention" section;
  vLLM paper review, mz-moonzoo.tistory.com/116, §4.2 KV Cache Manager).
* Block table and #filled, allocation on demand: a prompt of n tokens takes
  ceil(n/B) blocks; a new token goes into the free slot of the last block if
  there is one, otherwise a new block is appended to the table (review §4.3
  example: 7-token prompt in P7 (4/4) + P1 (3/4), step 1 fills P1 slot 3,
  step 2 takes P3; paged KV cache tutorial,
  llm-systems-engineering.pages.dev/posts/paged-kv-cache, Fig. 1-3).
* Slot of a token: position p -> logical block p // B, offset p % B ->
  physical block table[p // B] -> slot = physical * B + offset (tutorial,
  Fig. 2; all numbering starts at 0).
* Sharing and copy-on-write: fork copies the table and increments every
  block's reference count; a write into a last block whose count is above 1
  takes a new block, records a copy of the old block into it, decrements the
  old block's count and points the writer's table at the new block; the last
  holder writes in place; a shared block that is already full is never
  copied -- the writer simply gets a fresh block (tutorial, Fig. 5-6 and the
  paragraph after them; PagedAttention notes, unpurerationalist.github.io,
  §3.4.1).
* Release: free decrements the count of every block of the sequence and
  returns a block to the free queue when its count reaches 0 (tutorial,
  "returning blocks after a request ends"; notes §3.4.2, §4.2).  Blocks are
  released from the tail of the sequence first (teardown, "when blocks run
  out": tail blocks are evicted first); freed blocks join the tail of the
  queue.
* Failure: when the pool cannot cover a request, the allocation reports
  failure and changes nothing (teardown: allocate_slots returns None).

* Prefix caching (vLLM teardown, "PagedAttention" section): every full
  block of a prompt is identified by its whole prefix (the pages hash the
  chain (parent hash, block tokens, extra keys)); a request whose leading full
  blocks are cached touches them -- count + 1, no copy, a free cached block
  leaves the free queue -- instead of allocating; the scan stops at the first
  block that is not cached; freed cached blocks stay cached at the tail of
  the free queue and are evicted (forgotten) only when the queue hands them
  out again, least recently freed first.  Here the key is the exact token
  prefix plus the extra key, so no hash is involved.

* Swapping (review §4.5 (1), notes §3.5): a preempted sequence group moves
  all its blocks to a second pool standing for swap space in host memory, and
  back later; sequences sharing blocks move together (review §4.5 (2)).
  ``move_group`` below gives each distinct block of the group a block of the
  target pool (same reference count), rewrites the tables and returns the
  source blocks to their free queue, last-used first.

Readings where the pages are silent (stated, not found on the pages): the
queue is FIFO; a multi-sequence ``alloc_slots`` handles the sequences in the
order given and is all-or-nothing as a whole; a sequence may appear only once
per ``alloc_slots`` call.
"""
from __future__ import annotations

import copy
from collections import deque


class OutOfBlocks(Exception):
    """The free queue cannot cover the request; nothing was changed."""


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order=None,
                 prefix_caching: bool = False):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("bad pool geometry")
        self.prefix_caching = prefix_caching
        self.cache = {}          # (extra_key, token prefix tuple) -> physical block
        self.block_key = {}      # physical block -> its key while cached
        self.num_blocks = int(num_blocks)
        self.B = int(block_size)
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the pool's block ids")
        self.free_queue = deque(order)
        self.ref = [0] * num_blocks
        # seq_id -> list of [physical_block, filled]
        self.tables: dict[int, list[list[int]]] = {}

    # -- queries -----------------------------------------------------------
    def block_table(self, seq_id: int) -> list[int]:
        return [e[0] for e in self.tables[seq_id]]

    def filled(self, seq_id: int) -> list[int]:
        return [e[1] for e in self.tables[seq_id]]

    def num_tokens(self, seq_id: int) -> int:
        return sum(e[1] for e in self.tables[seq_id])

    def num_free(self) -> int:
        return len(self.free_queue)

    def slot_of(self, seq_id: int, position: int) -> int:
        """Slot holding token ``position`` of the sequence (tutorial, Fig. 2)."""
        table = self.tables[seq_id]
        logical, offset = divmod(position, self.B)
        if position < 0 or logical >= len(table) or offset >= table[logical][1]:
            raise IndexError("position not stored")
        return table[logical][0] * self.B + offset

    # -- primitives --------------------------------------------------------
    def _take_block(self) -> int:
        if not self.free_queue:
            raise OutOfBlocks()
        b = self.free_queue.popleft()
        assert self.ref[b] == 0
        self.ref[b] = 1
        if b in self.block_key:               # evicted from the prefix cache
            del self.cache[self.block_key.pop(b)]
        return b

    def _release_block(self, b: int) -> None:
        self.ref[b] -= 1
        assert self.ref[b] >= 0
        if self.ref[b] == 0:
            self.free_queue.append(b)

    def add(self, seq_id: int, n_tokens: int) -> list[int]:
        """Admit a sequence with a prompt of ``n_tokens``; returns its slots."""
        if seq_id in self.tables:
            raise ValueError("sequence exists")
        if n_tokens < 0:
            raise ValueError("negative prompt length")
        need = -(-n_tokens // self.B)
        if need > len(self.free_queue):
            raise OutOfBlocks()
        table = []
        left = n_tokens
        for _ in range(need):
            table.append([self._take_block(), min(self.B, left)])
            left -= self.B
        self.tables[seq_id] = table
        return [self.slot_of(seq_id, p) for p in range(n_tokens)]

    def add_tokens(self, seq_id: int, tokens, extra_key: int = 0):
        """Admit a sequence from its prompt tokens, reusing cached full blocks.

        Returns (slots, n_cached_tokens)."""
        if seq_id in self.tables:
            raise ValueError("sequence exists")
        tokens = [int(t) for t in tokens]
        n, B = len(tokens), self.B
        total, full = -(-n // B), n // B
        hits = []
        if self.prefix_caching:
            # the block holding the last prompt token is never reused: that
            # token's query must be computed, so its K/V is written afresh
            for j in range((n - 1) // B if n else 0):
                b = self.cache.get((extra_key, tuple(tokens[:(j + 1) * B])))
                if b is None:
                    break
                hits.append(b)
        need = total - len(hits)
        if need > len(self.free_queue) - sum(1 for b in hits if self.ref[b] == 0):
            raise OutOfBlocks()
        table = []
        for b in hits:
            if self.ref[b] == 0:
                self.free_queue.remove(b)
            self.ref[b] += 1
            table.append([b, B])
        left = n - len(hits) * B
        for _ in range(need):
            table.append([self._take_block(), min(B, left)])
            left -= B
        if self.prefix_caching:
            for j in range(len(hits), full):
                key = (extra_key, tuple(tokens[:(j + 1) * B]))
                if key not in self.cache:
                    self.cache[key] = table[j][0]
                    self.block_key[table[j][0]] = key
        self.tables[seq_id] = table
        return [self.slot_of(seq_id, p) for p in range(n)], len(hits) * B

    def fork(self, parent: int, child: int) -> None:
        """Child shares every block of the parent; counts go up by one."""
        if parent not in self.tables:
            raise KeyError(parent)
        if child in self.tables:
            raise ValueError("child exists")
        self.tables[child] = [list(e) for e in self.tables[parent]]
        for b, _ in self.tables[child]:
            self.ref[b] += 1

    def free(self, seq_id: int) -> None:
        """Drop the sequence; blocks at count 0 go back, tail blocks first."""
        table = self.tables.pop(seq_id)
        for b, _ in reversed(table):
            self._release_block(b)

    def append(self, seq_id: int):
        """Store one more token of the sequence.

        Returns (slot, copy) where copy is None or (src_block, dst_block).
        """
        table = self.tables[seq_id]
        copy_pair = None
        if not table or table[-1][1] == self.B:
            # no block yet, or the last block is full (shared or not): new block
            table.append([self._take_block(), 0])
        elif self.ref[table[-1][0]] > 1:
            # partially filled and shared: copy-on-write
            old = table[-1][0]
            new = self._take_block()
            copy_pair = (old, new)
            self.ref[old] -= 1
            table[-1][0] = new
        entry = table[-1]
        slot = entry[0] * self.B + entry[1]
        entry[1] += 1
        return slot, copy_pair

    def alloc_slots(self, seq_ids):
        """One new token for each listed sequence, in the order given.

        Returns (slot_mapping, copies).  All-or-nothing: on failure the
        state is exactly what it was before the call.
        """
        seq_ids = [int(s) for s in seq_ids]
        if len(set(seq_ids)) != len(seq_ids):
            raise ValueError("a sequence may appear once per call")
        for s in seq_ids:
            if s not in self.tables:
                raise KeyError(s)
        saved = (copy.deepcopy(self.free_queue), list(self.ref), copy.deepcopy(self.tables),
                 dict(self.cache), dict(self.block_key))
        slots, copies = [], []
        try:
            for s in seq_ids:
                slot, cp = self.append(s)
                slots.append(slot)
                if cp is not None:
                    copies.append(cp)
        except OutOfBlocks:
            self.free_queue, self.ref, self.tables, self.cache, self.block_key = saved
            raise
        return slots, copies

    def alloc_slots_n(self, seq_ids, counts):
        """counts[i] new tokens for seq_ids[i]: repeated appends, sequence by
        sequence in the order given (a chunk of tokens is appended one after
        the other).  All-or-nothing; returns (slot_mapping, copies)."""
        seq_ids = [int(s) for s in seq_ids]
        if len(set(seq_ids)) != len(seq_ids) or any(int(c) < 0 for c in counts):
            raise ValueError("bad batch")
        for s in seq_ids:
            if s not in self.tables:
                raise KeyError(s)
        saved = (copy.deepcopy(self.free_queue), list(self.ref), copy.deepcopy(self.tables),
                 dict(self.cache), dict(self.block_key))
        slots, copies = [], []
        try:
            for s, n in zip(seq_ids, counts):
                for _ in range(int(n)):
                    slot, cp = self.append(s)
                    slots.append(slot)
                    if cp is not None:
                        copies.append(cp)
        except OutOfBlocks:
            self.free_queue, self.ref, self.tables, self.cache, self.block_key = saved
            raise
        return slots, copies

    # -- whole-state views (for comparisons) ---------------------------------
    def padded_tables(self, seq_ids, max_blocks: int, pad: int = -1):
        """[len(seq_ids)][max_blocks] physical ids, padded with ``pad``."""
        out = []
        for s in seq_ids:
            t = self.block_table(s)
            if len(t) > max_blocks:
                raise ValueError("table longer than max_blocks")
            out.append(t + [pad] * (max_blocks - len(t)))
        return out

    def snapshot(self):
        return copy.deepcopy((list(self.free_queue), list(self.ref), self.tables,
                              sorted(self.block_key.items())))


def move_group(src: BlockManager, dst: BlockManager, seq_ids):
    """Swap a sequence group from ``src`` to ``dst``; returns the
    (source block, target block) pairs to copy, in first-use order.

    Raises KeyError (unknown sequence), ValueError (block shared outside
    the group, sequence already in ``dst``, block sizes differ) or OutOfBlocks;
    nothing changes on failure."""
    seq_ids = [int(s) for s in seq_ids]
    if src.B != dst.B or len(set(seq_ids)) != len(seq_ids):
        raise ValueError("bad group")
    uses, blocks = {}, []
    for s in seq_ids:
        if s not in src.tables:
            raise KeyError(s)
        if s in dst.tables:
            raise ValueError("sequence already in the target pool")
        for b in src.block_table(s):
            if b not in uses:
                uses[b] = 0
                blocks.append(b)
            uses[b] += 1
    if any(src.ref[b] != uses[b] for b in blocks):
        raise ValueError("a block is shared outside the group")
    if len(blocks) > len(dst.free_queue):
        raise OutOfBlocks()
    moved, pairs = {}, []
    for b in blocks:
        nb = dst._take_block()
        dst.ref[nb] = uses[b]
        moved[b] = nb
        pairs.append((b, nb))
    for s in seq_ids:
        dst.tables[s] = [[moved[b], f] for b, f in src.tables.pop(s)]
    for b in reversed(blocks):
        src.ref[b] = 0
        src.free_queue.append(b)
    return pairs

