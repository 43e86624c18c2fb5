"""Swapping sequence groups between a GPU pool and a CPU (swap space) pool:
the C ABI (pa_swap_out / pa_swap_in) against the oracle's move_group, with
a content model that follows every token across the two pools.

Pinned to the pages: a preempted request's blocks move to CPU memory and
back (vLLM paper review, mz-moonzoo.tistory.com/116, §4.5 (1);
PagedAttention notes, unpurerationalist.github.io, §3.5), sequences sharing
blocks move as one group (review §4.5 (2)), and the move is all-or-nothing."""
import random

import pytest

import paged_kv_cache_106_gb300 as pk
from oracle.alloc import BlockManager, OutOfBlocks, move_group

B = 4


class Side:
    def __init__(self, nb, order):
        self.m = BlockManager(nb, B, order)
        self.p = pk.pa_pool_create(pk.PoolDesc(nb, B, free_order=order))
        self.nb = nb

    def check(self):
        assert pk.pa_pool_free_queue(self.p, self.nb).tolist() == list(self.m.free_queue)
        assert pk.pa_pool_refcounts(self.p, self.nb).tolist() == self.m.ref
        ids = sorted(self.m.tables)
        if ids:
            mb = max(1, max(len(self.m.block_table(s)) for s in ids))
            assert pk.pa_get_block_tables(self.p, ids, mb)[0].tolist() == \
                self.m.padded_tables(ids, mb)


def _move(fn, a: Side, b: Side, ids):
    try:
        exp = move_group(a.m, b.m, ids)
    except (OutOfBlocks, ValueError, KeyError) as e:
        with pytest.raises(pk.PagedKVError):
            fn(a.p, b.p, ids)
        return None
    got = fn(a.p, b.p, ids)
    assert [tuple(x) for x in got.tolist()] == exp
    return exp


def test_group_round_trip_and_gang_rule():
    g, c = Side(8, list(range(8))), Side(6, [5, 4, 3, 2, 1, 0])
    pk.pa_seq_add(g.p, 0, 6); g.m.add(0, 6)
    pk.pa_seq_fork(g.p, 0, 1); g.m.fork(0, 1)
    pk.pa_seq_add(g.p, 2, 3); g.m.add(2, 3)
    assert _move(pk.pa_swap_out, g, c, [0]) is None          # shares blocks with 1: refused
    g.check(); c.check()
    pairs = _move(pk.pa_swap_out, g, c, [0, 1])                # the whole group moves
    assert pairs == [(0, 5), (1, 4)]                            # distinct blocks once, first-use order
    assert c.m.ref[5] == 2 and c.m.ref[4] == 2
    assert list(g.m.free_queue)[-2:] == [1, 0]                  # last-used first
    back = _move(pk.pa_swap_in, c, g, [1, 0])
    assert [a for a, _ in back] == [5, 4]                       # first use in seq 1's table
    g.check(); c.check()


def test_target_full_changes_nothing():
    g, c = Side(6, list(range(6))), Side(2, [0, 1])
    pk.pa_seq_add(g.p, 0, 12); g.m.add(0, 12)                  # 3 blocks, CPU pool has 2
    assert _move(pk.pa_swap_out, g, c, [0]) is None
    g.check(); c.check()


@pytest.mark.parametrize("seed", range(20))
def test_random_swaps_lockstep_with_content(seed):
    rng = random.Random(500 + seed)
    ng, nc = rng.randint(3, 20), rng.randint(2, 20)
    og, oc_ = list(range(ng)), list(range(nc))
    rng.shuffle(og); rng.shuffle(oc_)
    g, c = Side(ng, og), Side(nc, oc_)
    mem = {}                       # (pool name, slot) -> token
    hist = {}
    where = {}                     # seq -> "g" / "c"
    nxt = 0

    def pools(name):
        return (g, "g") if name == "g" else (c, "c")

    for _ in range(200):
        r = rng.random()
        on_gpu = [s for s in hist if where[s] == "g"]
        on_cpu = [s for s in hist if where[s] == "c"]
        if r < 0.25 or not hist:
            n = rng.randint(0, 3 * B)
            try:
                slots = g.m.add(nxt, n)
            except OutOfBlocks:
                with pytest.raises(pk.OutOfBlocks):
                    pk.pa_seq_add(g.p, nxt, n)
            else:
                assert pk.pa_seq_add(g.p, nxt, n).tolist() == slots
                hist[nxt] = [1000 * nxt + i for i in range(n)]
                for slot, t in zip(slots, hist[nxt]):
                    mem[("g", slot)] = t
                where[nxt] = "g"
            nxt += 1
        elif r < 0.35 and on_gpu:
            p = rng.choice(on_gpu)
            pk.pa_seq_fork(g.p, p, nxt); g.m.fork(p, nxt)
            hist[nxt] = list(hist[p]); where[nxt] = "g"; nxt += 1
        elif r < 0.5 and on_gpu:
            s = rng.choice(on_gpu)
            pk.pa_seq_free(g.p, s); g.m.free(s)
            del hist[s], where[s]
        elif r < 0.7 and on_gpu:
            ids = rng.sample(on_gpu, rng.randint(1, len(on_gpu)))
            pairs = _move(pk.pa_swap_out, g, c, ids)
            if pairs is not None:
                for a, b in pairs:
                    for i in range(B):
                        mem[("c", b * B + i)] = mem.get(("g", a * B + i))
                for s in ids:
                    where[s] = "c"
        elif r < 0.85 and on_cpu:
            ids = rng.sample(on_cpu, rng.randint(1, len(on_cpu)))
            pairs = _move(pk.pa_swap_in, c, g, ids)
            if pairs is not None:
                for a, b in pairs:
                    for i in range(B):
                        mem[("g", b * B + i)] = mem.get(("c", a * B + i))
                for s in ids:
                    where[s] = "g"
        elif on_gpu:
            ids = rng.sample(on_gpu, rng.randint(1, len(on_gpu)))
            try:
                so, co = g.m.alloc_slots(ids)
            except OutOfBlocks:
                with pytest.raises(pk.OutOfBlocks):
                    pk.pa_alloc_slots(g.p, ids)
            else:
                sg, cg = pk.pa_alloc_slots(g.p, ids)
                assert sg.tolist() == so and [tuple(x) for x in cg.tolist()] == co
                for a, b in co:
                    for i in range(B):
                        mem[("g", b * B + i)] = mem.get(("g", a * B + i))
                for s, slot in zip(ids, so):
                    t = 7_000_000 + len(hist[s]) + 1000 * s
                    mem[("g", slot)] = t
                    hist[s].append(t)
        g.check(); c.check()
        for s, h in hist.items():
            side, name = pools(where[s])
            assert [mem.get((name, side.m.slot_of(s, p))) for p in range(len(h))] == h
