"""The C-ABI block manager (libpagedkv.so, host calls only -- no GPU needed)
against the pages' worked examples and, operation by operation, against the
oracle's block manager: slots, copy pairs, block tables, token counts,
reference counts and the free queue must be identical (bit-exact indexing)."""
import copy
import ctypes
import random
import re
import subprocess

import numpy as np
import pytest

import paged_kv_cache_106_gb300 as pk
from oracle.alloc import BlockManager, OutOfBlocks, move_group
from tests.allocator_replay import load, replay
from tests.conftest import ROOT

GOLDEN = ["tutorial_fig1_4_block_table.json", "review_s4_3_decoding.json",
          "tutorial_fig5_6_cow.json", "tutorial_full_shared_block.json"]


def declared_functions():
    src = open(f"{ROOT}/include/pagedkv.h").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\**\s*(pa_\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 16, names
    out = subprocess.run(["nm", "-D", "--defined-only", pk.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    # and the binding binds each of them under the same name
    for n in names:
        assert callable(getattr(pk, n)), n


class AbiAdapter:
    def __init__(self, doc):
        self.nb = doc["num_blocks"]
        self.desc = pk.PoolDesc(doc["num_blocks"], doc["block_size"], free_order=doc["free_order"])
        self.p = pk.pa_pool_create(self.desc)

    def add(self, s, n):
        return pk.pa_seq_add(self.p, s, n).tolist()

    def fork(self, a, b):
        pk.pa_seq_fork(self.p, a, b)

    def free(self, s):
        pk.pa_seq_free(self.p, s)

    def alloc_slots(self, seqs):
        slots, copies = pk.pa_alloc_slots(self.p, seqs)
        return slots.tolist(), copies.tolist()

    def table(self, s):
        nt, nb = pk.pa_seq_info(self.p, s)
        t, _ = pk.pa_get_block_tables(self.p, [s], max(nb, 1))
        return t[0, :nb].tolist()

    def filled(self, s):
        nt, nb = pk.pa_seq_info(self.p, s)
        B = self.desc.block_size
        return [B] * (nb - 1) + [nt - (nb - 1) * B] if nb else []

    def ref(self, b):
        return int(pk.pa_pool_refcounts(self.p, self.nb)[b])

    def free_queue(self):
        return pk.pa_pool_free_queue(self.p, self.nb).tolist()


def test_bounded_wait_selftest_refuses_a_null_status_before_any_launch():
    """Argument checks of a device call run on the host: a NULL status is
    refused with PA_ERR_INVALID_ARG and nothing is launched (no GPU needed)."""
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_selftest_bounded_wait(None, stream=0)
    assert e.value.code == pk.PA_ERR_INVALID_ARG
    assert "status is NULL" in pk.pa_last_error_string()


def test_one_call_step_bindings_refuse_short_new_rows_before_any_device_call():
    """The bindings of the one-call steps check that the new rows (and, for
    decode, the slot mapping) hold what the library will read, before any
    pointer reaches the library: host tensors suffice to see the refusal."""
    import torch
    H, D = 2, 64
    d = pk.PoolDesc(8, 16, num_heads=H, head_dim=D)
    q = torch.empty((3, H, D), dtype=torch.float16)
    short = torch.empty((2, H, D), dtype=torch.float16)
    slots = torch.zeros(3, dtype=torch.int64)
    t = torch.empty(1)
    tables = torch.zeros((3, 4), dtype=torch.int32)
    ctx = torch.ones(3, dtype=torch.int32)
    with pytest.raises(ValueError, match="k_new"):
        pk.pa_decode_step_attention(q, q, short, q, slots, t, t, tables, ctx, 0.1, d)
    with pytest.raises(ValueError, match="slot_mapping"):
        pk.pa_decode_step_attention(q, q, q, q, slots[:2], t, t, tables, ctx, 0.1, d)
    with pytest.raises(ValueError, match="v_new"):
        pk.pa_prefill_step_attention(q, q, q, short, t, t, tables, ctx, t, 0.1, d, max_q_len=3)


@pytest.mark.parametrize("name", GOLDEN)
def test_golden_examples_through_abi(golden_dir, name):
    doc = load(golden_dir, name)
    replay(doc, AbiAdapter(doc))


def _compare(abi: AbiAdapter, m: BlockManager, live):
    assert abi.free_queue() == list(m.free_queue)
    assert pk.pa_pool_refcounts(abi.p, abi.nb).tolist() == m.ref
    assert pk.pa_pool_num_free(abi.p) == len(m.free_queue)
    if live:
        ids = sorted(live)
        mb = max(1, max(len(m.block_table(s)) for s in ids))
        t, ctx = pk.pa_get_block_tables(abi.p, ids, mb)
        assert t.tolist() == m.padded_tables(ids, mb)
        assert ctx.tolist() == [m.num_tokens(s) for s in ids]


@pytest.mark.parametrize("seed", range(30))
def test_lockstep_with_oracle(seed):
    rng = random.Random(1000 + seed)
    B = rng.choice([1, 2, 3, 4, 16])
    nb = rng.randint(0, 40)
    order = list(range(nb))
    rng.shuffle(order)
    doc = {"num_blocks": nb, "block_size": B, "free_order": order}
    abi = AbiAdapter(doc)
    m = BlockManager(nb, B, order)
    live, nxt = set(), 0
    for _ in range(400):
        r = rng.random()
        if r < 0.2 or not live:
            n = rng.randint(0, 4 * B)
            try:
                exp = m.add(nxt, n)
            except OutOfBlocks:
                with pytest.raises(pk.OutOfBlocks):
                    abi.add(nxt, n)
            else:
                assert abi.add(nxt, n) == exp
                live.add(nxt)
            nxt += 1
        elif r < 0.35:
            p = rng.choice(sorted(live))
            m.fork(p, nxt)
            abi.fork(p, nxt)
            live.add(nxt)
            nxt += 1
        elif r < 0.45:
            s = rng.choice(sorted(live))
            m.free(s)
            abi.free(s)
            live.discard(s)
        else:
            seqs = rng.sample(sorted(live), rng.randint(1, len(live)))
            try:
                exp = m.alloc_slots(seqs)
            except OutOfBlocks:
                with pytest.raises(pk.OutOfBlocks):
                    abi.alloc_slots(seqs)
            else:
                got = abi.alloc_slots(seqs)
                assert got[0] == exp[0]
                assert [tuple(c) for c in got[1]] == exp[1]
        _compare(abi, m, live)


class FusedStepAdapter(AbiAdapter):
    """The same block manager, appending through pa_decode_step_prepare."""

    def alloc_slots(self, seqs):
        nb = max([pk.pa_seq_info(self.p, s)[1] for s in seqs] + [0]) + 1
        slots, ctx, tables, copies = pk.pa_decode_step_prepare(self.p, seqs, nb)
        for i, s in enumerate(seqs):
            nt, n = pk.pa_seq_info(self.p, s)
            assert ctx[i] == nt
            assert tables[i, n:].tolist() == [-1] * (nb - n)
        return slots.tolist(), copies.tolist()


@pytest.mark.parametrize("name", GOLDEN)
def test_golden_examples_through_the_fused_step_call(golden_dir, name):
    doc = load(golden_dir, name)
    replay(doc, FusedStepAdapter(doc))


@pytest.mark.parametrize("seed", range(20))
def test_fused_step_call_lockstep_with_oracle(seed):
    """pa_decode_step_prepare = pa_alloc_slots followed by the table export:
    slots, copies, padded tables and token counts against the oracle, and
    the same all-or-nothing failures (out of blocks, a table that would
    outgrow max_blocks, a sequence listed twice, an unknown sequence)."""
    rng = random.Random(5000 + seed)
    B = rng.choice([1, 2, 4, 16])
    nb = rng.randint(0, 48)
    order = list(range(nb))
    rng.shuffle(order)
    abi = AbiAdapter({"num_blocks": nb, "block_size": B, "free_order": order})
    m = BlockManager(nb, B, order)
    live, nxt = set(), 0
    for _ in range(300):
        r = rng.random()
        if r < 0.2 or not live:
            n = rng.randint(0, 3 * B)
            try:
                exp = m.add(nxt, n)
            except OutOfBlocks:
                with pytest.raises(pk.OutOfBlocks):
                    abi.add(nxt, n)
            else:
                assert abi.add(nxt, n) == exp
                live.add(nxt)
            nxt += 1
        elif r < 0.35:
            p = rng.choice(sorted(live))
            m.fork(p, nxt)
            abi.fork(p, nxt)
            live.add(nxt)
            nxt += 1
        elif r < 0.45:
            s = rng.choice(sorted(live))
            m.free(s)
            abi.free(s)
            live.discard(s)
        else:
            seqs = rng.sample(sorted(live), rng.randint(1, len(live)))
            longest = max(len(m.block_table(s)) for s in seqs)
            mb = longest + rng.choice([0, 1, 1, 2])      # 0: may be one short after the append
            probe = rng.random()
            if probe < 0.1:                              # a sequence listed twice
                with pytest.raises(pk.PagedKVError) as e:
                    pk.pa_decode_step_prepare(abi.p, seqs + seqs[:1], mb + 1)
                assert e.value.code == pk.PA_ERR_INVALID_ARG
            elif probe < 0.15:                           # an unknown sequence
                with pytest.raises(pk.PagedKVError) as e:
                    pk.pa_decode_step_prepare(abi.p, seqs + [10 ** 6], mb + 1)
                assert e.value.code == pk.PA_ERR_NO_SEQ
            else:
                saved = copy.deepcopy(m)
                try:
                    exp_slots, exp_copies = m.alloc_slots(seqs)
                except OutOfBlocks:
                    # either failure may be the one reported when both apply
                    with pytest.raises(pk.PagedKVError) as e:
                        pk.pa_decode_step_prepare(abi.p, seqs, mb)
                    assert e.value.code in (pk.PA_ERR_OUT_OF_BLOCKS, pk.PA_ERR_INVALID_ARG)
                else:
                    if max(len(m.block_table(s)) for s in seqs) > mb:
                        m = saved                        # the call must change nothing
                        with pytest.raises(pk.PagedKVError) as e:
                            pk.pa_decode_step_prepare(abi.p, seqs, mb)
                        assert e.value.code == pk.PA_ERR_INVALID_ARG
                    else:
                        slots, ctx, tables, copies = pk.pa_decode_step_prepare(abi.p, seqs, mb)
                        assert slots.tolist() == exp_slots
                        assert [tuple(c) for c in copies.tolist()] == exp_copies
                        assert tables.tolist() == m.padded_tables(seqs, mb)
                        assert ctx.tolist() == [m.num_tokens(s) for s in seqs]
        _compare(abi, m, live)


@pytest.mark.parametrize("seed", range(12))
def test_row_skipping_step_call_keeps_every_row_current(seed):
    """pa_decode_step_prepare_rows into two staging buffers used in turn, as a
    serving loop uses them, while the batch's rows are replaced (free + add,
    sometimes under the freed id again), forked into, and swapped out and back
    in: after every call every row of the buffer it wrote equals the oracle's
    padded table (rows it skipped included), and slots, copy pairs and
    lengths match the oracle's append."""
    rng = random.Random(7000 + seed)
    B = rng.choice([1, 2, 4, 16])
    S = rng.randint(1, 10)
    MB = 10
    nb = S * (MB + 4)
    order = list(range(nb))
    rng.shuffle(order)
    gpu = pk.pa_pool_create(pk.PoolDesc(nb, B, free_order=order))
    cpu = pk.pa_pool_create(pk.PoolDesc(nb, B, free_order=list(range(nb))))
    m, mc = BlockManager(nb, B, order), BlockManager(nb, B, list(range(nb)))
    ids = np.arange(S, dtype=np.int32)
    nxt = S
    for s in ids.tolist():
        n = rng.randint(1, 3 * B)
        m.add(s, n)
        pk.pa_seq_add(gpu, s, n, want_slots=False)
    bufs = [np.full((S, MB), -7, np.int32) for _ in range(2)]
    vers = [np.zeros(S, np.uint64) for _ in range(2)]
    slots = np.empty(S, np.int64)
    ctx = np.empty(S, np.int32)
    copies = np.empty((S, 2), np.int32)
    ncp = ctypes.c_int32()

    def replace(i, same_id):
        nonlocal nxt
        old = int(ids[i])
        m.free(old)
        pk.pa_seq_free(gpu, old)
        new = old if same_id else nxt
        nxt += 0 if same_id else 1
        n = rng.randint(1, 3 * B)
        m.add(new, n)
        pk.pa_seq_add(gpu, new, n, want_slots=False)
        ids[i] = new

    for step in range(160):
        i = rng.randrange(S)
        r = rng.random()
        if r < 0.15:
            replace(i, rng.random() < 0.3)
        elif r < 0.25 and S > 1:
            j = rng.randrange(S)
            if j != i:
                old = int(ids[i])
                m.free(old)
                pk.pa_seq_free(gpu, old)
                m.fork(int(ids[j]), nxt)
                pk.pa_seq_fork(gpu, int(ids[j]), nxt)
                ids[i] = nxt
                nxt += 1
        elif r < 0.35:
            s = int(ids[i])
            try:
                exp_out = move_group(m, mc, [s])
            except ValueError:                       # a block shared outside the row
                pass
            else:
                assert [tuple(p) for p in pk.pa_swap_out(gpu, cpu, [s]).tolist()] == exp_out
                exp_in = move_group(mc, m, [s])
                assert [tuple(p) for p in pk.pa_swap_in(cpu, gpu, [s]).tolist()] == exp_in
        for i2 in range(S):                          # keep every table inside the rows
            if len(m.block_table(int(ids[i2]))) >= MB:
                replace(i2, False)
        k = step & 1
        exp_slots, exp_copies = m.alloc_slots(ids.tolist())
        n_cp = pk.pa_decode_step_prepare_rows_into(
            gpu, S, ids.ctypes.data, MB, slots.ctypes.data, ctx.ctypes.data, bufs[k].ctypes.data,
            vers[k].ctypes.data, copies.ctypes.data, S, ncp)
        assert slots.tolist() == exp_slots, step
        assert [tuple(c) for c in copies[:n_cp].tolist()] == exp_copies, step
        assert ctx.tolist() == [m.num_tokens(int(s)) for s in ids], step
        assert bufs[k].tolist() == m.padded_tables(ids.tolist(), MB), step
    pk.pa_pool_destroy(gpu)
    pk.pa_pool_destroy(cpu)


def test_row_skipping_step_call_refuses_a_null_versions_array():
    p = pk.pa_pool_create(pk.PoolDesc(8, 4))
    pk.pa_seq_add(p, 0, 3, want_slots=False)
    ids = np.zeros(1, np.int32)
    slots, ctx, tab, cps = np.empty(1, np.int64), np.empty(1, np.int32), np.empty(4, np.int32), np.empty(2, np.int32)
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_decode_step_prepare_rows_into(p, 1, ids.ctypes.data, 4, slots.ctypes.data, ctx.ctypes.data,
                                            tab.ctypes.data, 0, cps.ctypes.data, 1, ctypes.c_int32())
    assert e.value.code == pk.PA_ERR_INVALID_ARG
    assert pk.pa_seq_info(p, 0) == (3, 1)                  # nothing appended
    pk.pa_pool_destroy(p)


def test_abi_error_codes_and_no_partial_change():
    d = pk.PoolDesc(3, 2, free_order=[0, 1, 2])
    p = pk.pa_pool_create(d)
    pk.pa_seq_add(p, 0, 2)
    pk.pa_seq_add(p, 1, 2)
    q0, r0 = pk.pa_pool_free_queue(p, 3).tolist(), pk.pa_pool_refcounts(p, 3).tolist()
    with pytest.raises(pk.OutOfBlocks):
        pk.pa_alloc_slots(p, [0, 1])
    assert pk.pa_pool_free_queue(p, 3).tolist() == q0
    assert pk.pa_pool_refcounts(p, 3).tolist() == r0
    assert pk.pa_seq_info(p, 0) == (2, 1)
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_alloc_slots(p, [0, 0])
    assert e.value.code == pk.PA_ERR_INVALID_ARG
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_alloc_slots(p, [7])
    assert e.value.code == pk.PA_ERR_NO_SEQ
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_seq_add(p, 0, 1)
    assert e.value.code == pk.PA_ERR_NO_SEQ
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_seq_fork(p, 5, 6)
    assert e.value.code == pk.PA_ERR_NO_SEQ
    # copies_cap too small: copy-on-write needs one copy
    pk.pa_seq_free(p, 1)
    pk.pa_seq_add(p, 2, 1)
    pk.pa_seq_fork(p, 2, 3)
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_alloc_slots(p, [2], copies_cap=0)
    assert e.value.code == pk.PA_ERR_INVALID_ARG
    slots, copies = pk.pa_alloc_slots(p, [2], copies_cap=1)
    assert copies.shape == (1, 2)
    # table longer than max_blocks
    with pytest.raises(pk.PagedKVError):
        pk.pa_get_block_tables(p, [0], 0)
    with pytest.raises(pk.PagedKVError):
        pk.pa_pool_create(pk.PoolDesc(3, 2, free_order=[0, 0, 1]))
    pk.pa_pool_destroy(p)


def test_device_calls_reject_bad_geometry_before_any_cuda_work():
    bad = pk.PoolDesc(4, 5, num_heads=2, head_dim=8)        # block size 5 unsupported
    assert pk.pa_decode_workspace_bytes(2, 4, bad) == 0
    for call in (
        lambda: pk._lib.pa_write_kv(None, None, None, 1, None, None, bad.ref, None, None),
        lambda: pk._lib.pa_decode_attention(None, None, None, None, None, None, 1, 4,
                                            pk.ctypes.c_float(1.0), None, 0, None, bad.ref, None),
        lambda: pk._lib.pa_copy_blocks(None, None, 1, None, 1, bad.ref, None, None),
    ):
        assert call() == pk.PA_ERR_INVALID_ARG
        assert "block_size" in pk.pa_last_error_string()
    d = pk.PoolDesc(4, 16, num_heads=40, head_dim=128)
    # splitting at 512 tokens: 128 blocks -> 4 partitions, workspace (2 + D) floats per partition
    ws = pk.pa_decode_workspace_bytes(3, 128, d)
    rows = 3 * 40 * 4
    assert ws >= rows * (128 + 2) * 4
    assert pk.pa_decode_workspace_bytes(3, 32, d) == 256   # one partition: scheduling word only
    assert pk.pa_decode_workspace_bytes(0, 32, d) == 0
    # NULL pointers with a valid geometry are refused on the host
    assert pk._lib.pa_write_kv(None, None, None, 1, None, None, d.ref, None, None) == \
        pk.PA_ERR_INVALID_ARG


def test_noalloc_rejects_every_bad_argument_before_any_cuda_call():
    """The workspace-free decode call checks its arguments first: with no GPU
    in the process, a CUDA call would fail with PA_ERR_CUDA instead."""
    noalloc = lambda desc, n, mb, ptrs=None: pk._lib.pa_decode_attention_noalloc(
        *(ptrs or (None,) * 6), n, mb, pk.ctypes.c_float(1.0), None, desc, None)
    bad = pk.PoolDesc(4, 5, num_heads=2, head_dim=8)
    assert noalloc(bad.ref, 1, 4) == pk.PA_ERR_INVALID_ARG
    assert "block_size" in pk.pa_last_error_string()
    assert noalloc(None, 1, 4) == pk.PA_ERR_INVALID_ARG
    d = pk.PoolDesc(4, 16, num_heads=40, head_dim=128)
    assert noalloc(d.ref, -1, 4) == pk.PA_ERR_INVALID_ARG
    assert noalloc(d.ref, 1, -4) == pk.PA_ERR_INVALID_ARG
    assert noalloc(d.ref, 0, 4) == pk.PA_OK                   # empty batch: nothing to do
    assert noalloc(d.ref, 2048, 128) == pk.PA_ERR_INVALID_ARG  # workspace beyond the scratch
    assert "scratch" in pk.pa_last_error_string()
    assert noalloc(d.ref, 2, 4) == pk.PA_ERR_INVALID_ARG       # NULL pointers
    assert "NULL" in pk.pa_last_error_string()
    odd = (8, 16, 16, 16, 16, 16)                              # out not 16-byte aligned
    assert noalloc(d.ref, 2, 4, odd) == pk.PA_ERR_INVALID_ARG
    assert "aligned" in pk.pa_last_error_string()


@pytest.mark.parametrize("seed", range(25))
def test_multi_token_append_lockstep(seed):
    """pa_alloc_slots_n against repeated single appends in the oracle."""
    rng = random.Random(7000 + seed)
    B = rng.choice([1, 2, 4, 16])
    nb = rng.randint(0, 48)
    order = list(range(nb))
    rng.shuffle(order)
    abi = AbiAdapter({"num_blocks": nb, "block_size": B, "free_order": order})
    m = BlockManager(nb, B, order)
    live, nxt = set(), 0
    for _ in range(200):
        r = rng.random()
        if r < 0.2 or not live:
            n = rng.randint(0, 3 * B)
            try:
                exp = m.add(nxt, n)
            except OutOfBlocks:
                with pytest.raises(pk.OutOfBlocks):
                    abi.add(nxt, n)
            else:
                assert abi.add(nxt, n) == exp
                live.add(nxt)
            nxt += 1
        elif r < 0.35:
            p = rng.choice(sorted(live))
            m.fork(p, nxt)
            abi.fork(p, nxt)
            live.add(nxt)
            nxt += 1
        elif r < 0.45:
            s = rng.choice(sorted(live))
            m.free(s)
            abi.free(s)
            live.discard(s)
        else:
            seqs = rng.sample(sorted(live), rng.randint(1, len(live)))
            counts = [rng.randint(0, 2 * B + 1) for _ in seqs]
            try:
                exp = m.alloc_slots_n(seqs, counts)
            except OutOfBlocks:
                with pytest.raises(pk.OutOfBlocks):
                    pk.pa_alloc_slots_n(abi.p, seqs, counts)
            else:
                slots, copies = pk.pa_alloc_slots_n(abi.p, seqs, counts)
                assert slots.tolist() == exp[0]
                assert [tuple(c) for c in copies.tolist()] == exp[1]
        _compare(abi, m, live)
