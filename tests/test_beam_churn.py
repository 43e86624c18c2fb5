"""Beam-search churn through the C-ABI block manager, step by step against
the oracle's block manager: every step appends a token to every beam
(copy-on-write where forked beams share a partial last block), then prunes
(forks repeated survivors, frees the others).  Slots, copy pairs, tables,
reference counts and the free queue must agree at every step."""
import numpy as np
import pytest

import paged_kv_cache_106_gb300 as pk
from oracle.alloc import BlockManager
import workloads as wl
from paged_kv_cache_106_gb300.step import BeamGroups


def _oracle_groups(m, churn):
    beams, nxt = [], 0
    for n in churn.prompt_lens:
        m.add(nxt, n)
        members = [nxt]
        for j in range(1, churn.width):
            m.fork(nxt, nxt + j)
            members.append(nxt + j)
        nxt += churn.width
        beams.append(members)
    return beams, nxt


def _oracle_prune(m, beams, nxt, survivors):
    for g, keep in enumerate(survivors):
        members, new = beams[g], []
        for i in sorted(set(keep)):
            new.append(members[i])
            for _ in range(keep.count(i) - 1):
                m.fork(members[i], nxt)
                new.append(nxt)
                nxt += 1
        for i, s in enumerate(members):
            if i not in keep:
                m.free(s)
        beams[g] = new
    return nxt


@pytest.mark.parametrize("groups,width,B", [(3, 2, 4), (8, 4, 16), (5, 6, 8)])
def test_churn_lockstep(groups, width, B):
    churn = wl.beam_churn(groups=groups, width=width, seed=200 + groups)
    nb = sum(-(-n // B) for n in churn.prompt_lens) * width + groups * width * 12
    order = np.random.default_rng(groups).permutation(nb).tolist()
    p = pk.pa_pool_create(pk.PoolDesc(nb, B, free_order=order))
    m = BlockManager(nb, B, order)
    bg = BeamGroups(p, churn)
    beams, nxt = _oracle_groups(m, churn)
    rg, ro = np.random.default_rng(1), np.random.default_rng(1)
    total_copies = 0
    for step in range(40):
        ids = bg.ids()
        assert ids == [s for mb in beams for s in mb]
        sg, cg = pk.pa_alloc_slots(p, ids)
        so, co = m.alloc_slots(ids)
        assert sg.tolist() == so and [tuple(c) for c in cg.tolist()] == co
        total_copies += len(co)
        bg.prune(churn.survivors(rg))
        nxt = _oracle_prune(m, beams, nxt, churn.survivors(ro))
        assert pk.pa_pool_refcounts(p, nb).tolist() == m.ref
        assert pk.pa_pool_free_queue(p, nb).tolist() == list(m.free_queue)
        ids = bg.ids()
        mb = max(len(m.block_table(s)) for s in ids)
        assert pk.pa_get_block_tables(p, ids, mb)[0].tolist() == m.padded_tables(ids, mb)
    assert total_copies > 0


def test_beam_prune_checks_everything_before_changing_anything():
    """pa_beam_prune refuses a row that does not keep `width` beams, an
    unknown or repeated beam and a new id already in use, with the pool
    unchanged; a valid call forks and frees exactly like per-beam calls."""
    B, nb = 4, 40
    p = pk.pa_pool_create(pk.PoolDesc(nb, B))
    m = BlockManager(nb, B, list(range(nb)))
    for s, n in ((0, 6), (1, 3)):
        pk.pa_seq_add(p, s, n)
        m.add(s, n)
    pk.pa_seq_fork(p, 0, 2)
    m.fork(0, 2)
    beams = np.array([[0, 2], [1, 1]], np.int32)
    state = (pk.pa_pool_refcounts(p, nb).tolist(), pk.pa_pool_free_queue(p, nb).tolist())
    bad = [
        (np.array([[0, 2], [1, 3]], np.int32), [[2, 0], [2, 0]], 10, pk.PA_ERR_NO_SEQ),       # no 3
        (np.array([[0, 2], [1, 1]], np.int32), [[2, 0], [1, 1]], 10, pk.PA_ERR_INVALID_ARG),  # 1 twice
        (np.array([[0, 2], [1, 0]], np.int32), [[1, 0], [2, 0]], 10, pk.PA_ERR_INVALID_ARG),  # sum 1
        (np.array([[0, 2]], np.int32), [[2, 0]], 1, pk.PA_ERR_NO_SEQ),                         # id 1 in use
        (np.array([[0, 2]], np.int32), [[3, -1]], 10, pk.PA_ERR_INVALID_ARG),                  # negative
    ]
    for b, c, nid, code in bad:
        with pytest.raises(pk.PagedKVError) as e:
            pk.pa_beam_prune(p, b, c, nid)
        assert e.value.code == code
        assert (pk.pa_pool_refcounts(p, nb).tolist(), pk.pa_pool_free_queue(p, nb).tolist()) == state
    beams = np.array([[0, 2]], np.int32)
    assert pk.pa_beam_prune(p, beams, [[0, 2]], 7) == 8        # beam 2 kept twice, beam 0 freed
    assert beams.tolist() == [[2, 7]]
    m.fork(2, 7)
    m.free(0)
    assert pk.pa_pool_refcounts(p, nb).tolist() == m.ref
    assert pk.pa_pool_free_queue(p, nb).tolist() == list(m.free_queue)
    t, _ = pk.pa_get_block_tables(p, [2, 7, 1], 2)
    assert t.tolist() == m.padded_tables([2, 7, 1], 2)
    pk.pa_pool_destroy(p)
