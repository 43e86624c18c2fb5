"""Prefix caching in the block manager (C ABI and oracle model).

Pinned to the vLLM teardown (arcyou.ai/ko/teardowns/vllm-paged-attention,
"PagedAttention" section): every full block is keyed by a chain over
(parent key, block token ids, extra keys), so a key covers the whole prefix;
two requests that start with the same system prompt produce the same keys
and the second one touches the existing physical blocks (count + 1, no copy)
instead of allocating; a block returns to the free pool only at count 0 and
a cached free block stays at the back of the free queue, evicted last (LRU);
tail blocks are released first, so a freed request's prompt prefix tends to
stay cached and can be returned to a later request ("get_computed_blocks").

A token-content model checks that every reused block holds exactly the
tokens the new request expects at those positions.
"""
import random

import pytest

import paged_kv_cache_106_gb300 as pk
from oracle.alloc import BlockManager, OutOfBlocks

B = 4


class Both:
    def __init__(self, nb, order=None):
        order = list(range(nb)) if order is None else order
        self.m = BlockManager(nb, B, order, prefix_caching=True)
        self.d = pk.PoolDesc(nb, B, free_order=order, flags=pk.PA_POOL_PREFIX_CACHING)
        self.p = pk.pa_pool_create(self.d)
        self.nb = nb

    def add(self, s, toks, extra=0):
        try:
            so, co = self.m.add_tokens(s, toks, extra)
        except OutOfBlocks:
            with pytest.raises(pk.OutOfBlocks):
                pk.pa_seq_add_tokens(self.p, s, toks, extra)
            return None
        sg, cg = pk.pa_seq_add_tokens(self.p, s, toks, extra)
        assert sg.tolist() == so and cg == co
        return co

    def check(self):
        assert pk.pa_pool_free_queue(self.p, self.nb).tolist() == list(self.m.free_queue)
        assert pk.pa_pool_refcounts(self.p, self.nb).tolist() == self.m.ref
        assert pk.pa_pool_cached_blocks(self.p) == len(self.m.cache)
        ids = sorted(self.m.tables)
        if ids:
            mb = max(1, max(len(self.m.block_table(s)) for s in ids))
            t, ctx = pk.pa_get_block_tables(self.p, ids, mb)
            assert t.tolist() == self.m.padded_tables(ids, mb)


def test_same_system_prompt_is_touched_not_allocated():
    x = Both(16)
    system = list(range(100, 108))                 # two full blocks
    assert x.add(0, system + [1, 2, 3]) == 0
    free_before = len(x.m.free_queue)
    assert x.add(1, system + [7, 8, 9, 10, 11]) == 8
    t0, t1 = x.m.block_table(0), x.m.block_table(1)
    assert t0[:2] == t1[:2]                        # same physical prompt blocks
    assert [x.m.ref[b] for b in t0[:2]] == [2, 2]  # touched: count + 1
    assert free_before - len(x.m.free_queue) == 2  # only the request's own blocks
    x.check()


def test_all_cached_prompt_recomputes_its_last_block():
    """A prompt whose every block is cached (its length a multiple of B) does
    not reuse the block of its last token: the prefill needs that token's
    query, so the block is taken new and its B tokens are reported uncached
    (the pages do not cover this case; no write lands in a shared block)."""
    x = Both(16)
    prompt = list(range(200, 212))                 # three full blocks
    assert x.add(0, prompt) == 0
    assert x.add(1, prompt) == 8                   # blocks 0 and 1 reused, block 2 new
    t0, t1 = x.m.block_table(0), x.m.block_table(1)
    assert t0[:2] == t1[:2] and t0[2] != t1[2]
    assert [x.m.ref[b] for b in t1] == [2, 2, 1]
    x.check()
    assert x.add(2, prompt[:4]) == 0               # one full block, the last token's: new
    assert x.m.block_table(2)[0] != t0[0]
    x.check()


def test_extra_key_and_divergence_break_sharing():
    x = Both(32)
    p = list(range(12))
    x.add(0, p)
    assert x.add(1, p, extra=5) == 0               # different extra key: nothing shared
    q = p[:4] + [99, 98, 97, 96] + p[8:]           # second block differs, third coincides
    assert x.add(2, q) == 4                        # the chain stops at the first miss
    assert x.m.block_table(2)[2] != x.m.block_table(0)[2]
    x.check()


def test_freed_prefix_stays_cached_and_is_reused_lru():
    x = Both(12)
    sys_p = list(range(8))
    x.add(0, sys_p + [50, 51, 52, 53, 54])         # 4 blocks: 2 prompt + 1 full + 1 partial
    pk.pa_seq_free(x.p, 0)
    x.m.free(0)
    x.check()
    # tail blocks went back first: the cached prompt blocks sit at the very end of the queue
    q = list(x.m.free_queue)
    cached = set(x.m.cache.values())
    assert cached and all(q.index(b) >= len(q) - len(cached) for b in cached)
    assert x.add(1, sys_p + [60]) == 8            # "computed blocks" returned after the free
    x.check()


def test_eviction_forgets_the_block():
    x = Both(4)
    x.add(0, [1, 2, 3, 4, 5, 6, 7, 8])            # 2 cached full blocks, the whole pool half
    pk.pa_seq_free(x.p, 0)
    x.m.free(0)
    x.add(1, [9] * 16)                             # takes all 4 blocks: evicts both cached ones
    pk.pa_seq_free(x.p, 1)
    x.m.free(1)
    assert x.add(2, [1, 2, 3, 4, 5, 6, 7, 8]) == 0
    x.check()


def test_out_of_blocks_counts_touched_free_blocks():
    x = Both(3)
    x.add(0, [1, 2, 3, 4])
    pk.pa_seq_free(x.p, 0)
    x.m.free(0)
    # reuses the cached free block (leaves the queue) and needs 2 more: only 2 remain
    assert x.add(1, [1, 2, 3, 4, 5, 6, 7, 8, 9]) == 4
    x.check()
    assert x.add(2, [7] * 5) is None               # all-or-nothing failure on both sides
    x.check()


class ContentModel:
    """What every slot holds: the token whose K/V was written there."""

    def __init__(self):
        self.mem = {}
        self.hist = {}

    def admit(self, m, s, toks, n_cached):
        for pos in range(n_cached, len(toks)):    # the caller writes only the uncached tail
            self.mem[m.slot_of(s, pos)] = toks[pos]
        self.hist[s] = list(toks)

    def check(self, m):
        for s, h in self.hist.items():
            assert [self.mem.get(m.slot_of(s, p)) for p in range(len(h))] == h, s


@pytest.mark.parametrize("seed", range(25))
def test_random_lockstep_with_content(seed):
    rng = random.Random(seed)
    prefixes = [[rng.randrange(5) for _ in range(rng.randrange(0, 13))] for _ in range(4)]
    nb = rng.randint(4, 30)
    order = list(range(nb))
    rng.shuffle(order)
    x = Both(nb, order)
    cm = ContentModel()
    live, nxt = set(), 0
    for _ in range(250):
        r = rng.random()
        if r < 0.35 or not live:
            toks = rng.choice(prefixes) + [rng.randrange(5) for _ in range(rng.randrange(0, 9))]
            extra = rng.choice([0, 0, 0, 1])
            n_cached = x.add(nxt, toks, extra)
            if n_cached is not None:
                cm.admit(x.m, nxt, toks, n_cached)
                live.add(nxt)
            nxt += 1
        elif r < 0.45:
            p = rng.choice(sorted(live))
            pk.pa_seq_fork(x.p, p, nxt)
            x.m.fork(p, nxt)
            cm.hist[nxt] = list(cm.hist[p])
            live.add(nxt)
            nxt += 1
        elif r < 0.65:
            s = rng.choice(sorted(live))
            pk.pa_seq_free(x.p, s)
            x.m.free(s)
            del cm.hist[s]
            live.discard(s)
        else:
            seqs = rng.sample(sorted(live), rng.randint(1, len(live)))
            try:
                so, co = x.m.alloc_slots(seqs)
            except OutOfBlocks:
                with pytest.raises(pk.OutOfBlocks):
                    pk.pa_alloc_slots(x.p, seqs)
            else:
                sg, cg = pk.pa_alloc_slots(x.p, seqs)
                assert sg.tolist() == so and [tuple(c) for c in cg.tolist()] == co
                for src, dst in co:
                    for i in range(B):
                        cm.mem[dst * B + i] = cm.mem.get(src * B + i)
                for s, slot in zip(seqs, so):
                    tok = 1000 + nxt + s
                    cm.mem[slot] = tok
                    cm.hist[s].append(tok)
        x.check()
        cm.check(x.m)


def test_without_the_flag_nothing_is_cached():
    d = pk.PoolDesc(8, B)
    p = pk.pa_pool_create(d)
    _, c0 = pk.pa_seq_add_tokens(p, 0, list(range(8)))
    _, c1 = pk.pa_seq_add_tokens(p, 1, list(range(8)))
    assert (c0, c1) == (0, 0) and pk.pa_pool_cached_blocks(p) == 0
    with pytest.raises(pk.PagedKVError):
        pk.pa_pool_create(pk.PoolDesc(8, B, flags=6))
