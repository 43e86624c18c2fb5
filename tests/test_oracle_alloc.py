"""Pins for the oracle's block-manager model (oracle/alloc.py).

* The pages' worked examples (tests/golden/*.json): the tutorial's block
  table example (Fig. 1-4), the review's 7-token decoding example (§4.3), the
  tutorial's copy-on-write example (Fig. 5-6) and its full-shared-block rule.
* A content model: every stored token gets a unique id, every write and block
  copy is applied to a slot -> id memory, and after every operation reading a
  sequence's positions through its block table must give exactly the tokens
  that sequence wrote (its own history, or its parent's up to the fork).  A
  wrong slot, a missing copy, a copy in the wrong direction or a write into a
  still-shared block breaks it.
* Invariants (reference count = number of table entries that point at the
  block; the free queue holds exactly the unreferenced blocks, once each;
  every table entry but the last is full) and all-or-nothing failure, checked
  on random and on exhaustively enumerated operation sequences.
"""
import itertools
import random

import pytest

from oracle.alloc import BlockManager, OutOfBlocks
from tests.allocator_replay import load, replay

GOLDEN = ["tutorial_fig1_4_block_table.json", "review_s4_3_decoding.json",
          "tutorial_fig5_6_cow.json", "tutorial_full_shared_block.json"]


class OracleAdapter:
    def __init__(self, doc):
        self.m = BlockManager(doc["num_blocks"], doc["block_size"], doc["free_order"])

    def add(self, s, n):
        return self.m.add(s, n)

    def fork(self, p, c):
        self.m.fork(p, c)

    def free(self, s):
        self.m.free(s)

    def alloc_slots(self, seqs):
        return self.m.alloc_slots(seqs)

    def table(self, s):
        return self.m.block_table(s)

    def filled(self, s):
        return self.m.filled(s)

    def ref(self, b):
        return self.m.ref[b]

    def free_queue(self):
        return list(self.m.free_queue)


@pytest.mark.parametrize("name", GOLDEN)
def test_golden_examples(golden_dir, name):
    replay(load(golden_dir, name), OracleAdapter(load(golden_dir, name)))


def test_tutorial_attention_context_slots(golden_dir):
    """Fig. 4: the 9 positions of request B live in P3 (4), P0 (4), P5 (1)."""
    doc = load(golden_dir, "tutorial_fig1_4_block_table.json")
    a = OracleAdapter(doc)
    for step in doc["ops"]:
        if step["op"] == "add":
            a.add(step["seq"], step["n"])
        elif step["op"] == "alloc_slots":
            a.alloc_slots(step["seqs"])
    ctx = doc["attention_context"]
    slots = [a.m.slot_of(ctx["seq"], p) for p in range(ctx["ctx_len"])]
    assert slots == ctx["expect_slots"]
    assert not set(slots) & set(ctx["excluded_slots"])


class ContentModel:
    """Independent bookkeeping of what every sequence must read back."""

    def __init__(self, mgr: BlockManager):
        self.m = mgr
        self.mem = {}
        self.hist = {}
        self.next_id = 0

    def _new_ids(self, n):
        ids = list(range(self.next_id, self.next_id + n))
        self.next_id += n
        return ids

    def add(self, s, n):
        slots = self.m.add(s, n)
        ids = self._new_ids(n)
        for slot, i in zip(slots, ids):
            self.mem[slot] = i
        self.hist[s] = ids

    def fork(self, p, c):
        self.m.fork(p, c)
        self.hist[c] = list(self.hist[p])

    def free(self, s):
        self.m.free(s)
        del self.hist[s]

    def alloc_slots(self, seqs):
        slots, copies = self.m.alloc_slots(seqs)
        B = self.m.B
        for src, dst in copies:           # copies run before the writes
            for i in range(B):
                self.mem[dst * B + i] = self.mem.get(src * B + i)
        ids = self._new_ids(len(seqs))
        for s, slot, i in zip(seqs, slots, ids):
            self.mem[slot] = i
            self.hist[s].append(i)
        return slots, copies

    def check(self):
        m = self.m
        B = m.B
        # contents
        for s, h in self.hist.items():
            assert m.num_tokens(s) == len(h)
            got = [self.mem.get(m.slot_of(s, p)) for p in range(len(h))]
            assert got == h, (s, got, h)
        # reference counts
        count = [0] * m.num_blocks
        for s in self.hist:
            for b in m.block_table(s):
                count[b] += 1
        assert count == m.ref
        # free queue = unreferenced blocks, each once
        fq = list(m.free_queue)
        assert len(fq) == len(set(fq))
        assert set(fq) == {b for b in range(m.num_blocks) if m.ref[b] == 0}
        # #filled: all entries full but the last, which holds 1..B
        for s in self.hist:
            f = m.filled(s)
            assert all(x == B for x in f[:-1])
            if f:
                assert 1 <= f[-1] <= B


def _random_ops(rng, cm, n_ops, max_seq=6):
    live = lambda: list(cm.hist)
    next_seq = [0]
    for _ in range(n_ops):
        r = rng.random()
        before = cm.m.snapshot()
        try:
            if r < 0.2 or not live():
                s = next_seq[0]
                next_seq[0] += 1
                cm.add(s, rng.randint(0, 3 * cm.m.B))
            elif r < 0.35 and len(live()) < max_seq:
                s = next_seq[0]
                next_seq[0] += 1
                cm.fork(rng.choice(live()), s)
            elif r < 0.45:
                cm.free(rng.choice(live()))
            else:
                seqs = rng.sample(live(), rng.randint(1, len(live())))
                cm.alloc_slots(seqs)
        except OutOfBlocks:
            assert cm.m.snapshot() == before, "failed allocation changed the state"
        cm.check()


@pytest.mark.parametrize("seed", range(40))
def test_random_operation_sequences(seed):
    rng = random.Random(seed)
    B = rng.choice([1, 2, 4, 16])
    nb = rng.randint(1, 24)
    order = list(range(nb))
    rng.shuffle(order)
    cm = ContentModel(BlockManager(nb, B, order))
    _random_ops(rng, cm, 300)


def test_exhaustive_small_sequences():
    """Every sequence of 4 operations (13 kinds) over a 3-block pool with block size 2."""
    ops = [("add", 0, 1), ("add", 0, 3), ("add", 1, 2), ("fork", 0, 1), ("fork", 1, 2),
           ("free", 0), ("free", 1), ("app", (0,)), ("app", (1,)), ("app", (0, 1)),
           ("app", (1, 0)), ("app", (0, 2)), ("app", (2, 1))]
    n_runs = 0
    for seq in itertools.product(range(len(ops)), repeat=4):
        cm = ContentModel(BlockManager(3, 2, [2, 0, 1]))
        for k in seq:
            op = ops[k]
            before = cm.m.snapshot()
            try:
                if op[0] == "add":
                    if op[1] in cm.hist:
                        continue
                    cm.add(op[1], op[2])
                elif op[0] == "fork":
                    if op[1] not in cm.hist or op[2] in cm.hist:
                        continue
                    cm.fork(op[1], op[2])
                elif op[0] == "free":
                    if op[1] not in cm.hist:
                        continue
                    cm.free(op[1])
                else:
                    if any(s not in cm.hist for s in op[1]):
                        continue
                    cm.alloc_slots(list(op[1]))
            except OutOfBlocks:
                assert cm.m.snapshot() == before
            cm.check()
        n_runs += 1
    assert n_runs == len(ops) ** 4


def test_out_of_blocks_is_all_or_nothing():
    m = BlockManager(3, 2, [0, 1, 2])
    m.add(0, 2)
    m.add(1, 2)
    before = m.snapshot()
    # both sequences need a new block but only one is free
    with pytest.raises(OutOfBlocks):
        m.alloc_slots([0, 1])
    assert m.snapshot() == before
    with pytest.raises(OutOfBlocks):
        m.add(2, 3)
    assert m.snapshot() == before


def test_duplicate_sequence_in_one_call_rejected():
    m = BlockManager(4, 2)
    m.add(0, 1)
    with pytest.raises(ValueError):
        m.alloc_slots([0, 0])
