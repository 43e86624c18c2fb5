"""End-to-end decode steps of the seeded workloads on the GPU, against the
oracle run on the same seeded inputs.

For every workload the block manager (C ABI) and the oracle's model must
produce identical prompt slots, decode slots, copy-on-write pairs and block
tables; the cache byte image after the prompt writes, the copies and the
decode write must be identical; the attention outputs must be within 2e-3 of
the fp64 oracle -- every output of every workload, the full-size ones in the
launch configuration the benchmark times; the benchmark's own steady-state
batch (finished sequences freed and replaced between steps) is driven for 60
steps in lockstep with the oracle's block manager; the 40-layer pool-filling
step is checked on sampled sequences in four layers spread over the 40.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_106_gb300 as pk
import workloads as wl
from paged_kv_cache_106_gb300.step import DecodeStepRunner
from oracle import attention as oa
from oracle import cache_ops as oc
from oracle.alloc import BlockManager

pytestmark = pytest.mark.gpu
TOL = 2e-3


class Both:
    """The same workload driven through the library and through the oracle."""

    def __init__(self, w: wl.DecodeWorkload, max_extra_steps: int = 1):
        self.w = w
        H, D, B, NB = w.num_heads, w.head_dim, w.block_size, w.num_blocks
        self.m = BlockManager(NB, B, w.free_order)
        self.desc = pk.PoolDesc(NB, B, num_layers=1, num_heads=H, head_dim=D,
                                partition_tokens=w.split_tokens, free_order=w.free_order)
        self.pool = pk.pa_pool_create(self.desc)
        rng = wl.value_rng(w, 0)
        ks, vs, slots = [], [], []
        for i, n in enumerate(w.prompt_lens):
            so = self.m.add(i, n)
            sg = pk.pa_seq_add(self.pool, i, n)
            assert sg.tolist() == so
            slots.append(sg)
            ks.append(wl.normal_f16(rng, (n, H, D)))
            vs.append(wl.normal_f16(rng, (n, H, D)))
        self.ids = list(range(len(w.prompt_lens)))
        nxt = len(self.ids)
        for root, extra in w.forks:
            for _ in range(extra):
                self.m.fork(root, nxt)
                pk.pa_seq_fork(self.pool, root, nxt)
                self.ids.append(nxt)
                nxt += 1
        K = np.concatenate(ks) if ks else np.zeros((0, H, D), np.float16)
        V = np.concatenate(vs) if vs else np.zeros((0, H, D), np.float16)
        S = np.concatenate(slots).astype(np.int64) if slots else np.zeros(0, np.int64)
        # device cache, zero-filled, prompt written by the slot-write kernel
        self.kc = torch.zeros((NB, H, B, D), dtype=torch.float16, device="cuda")
        self.vc = torch.zeros_like(self.kc)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        if len(S):
            pk.pa_write_kv(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda(),
                           torch.from_numpy(S).cuda(), self.kc, self.vc, self.desc,
                           status=self.status)
        # oracle cache image
        self.okc = np.zeros((NB, H, B, D), np.float16)
        self.ovc = np.zeros_like(self.okc)
        oc.write_kv(self.okc, self.ovc, K, V, S)
        del K, V
        longest = max(m + max_extra_steps for m in w.prompt_lens)
        self.max_blocks = -(-longest // B) + 1
        self.runner = DecodeStepRunner(self.pool, self.desc, self.ids, self.max_blocks)
        self.vrng = wl.value_rng(w, 1)

    def check_cache(self):
        torch.cuda.synchronize()
        assert self.status.item() == 0
        assert torch.equal(self.kc, torch.from_numpy(self.okc).cuda())
        assert torch.equal(self.vc, torch.from_numpy(self.ovc).cuda())

    def decode_step(self):
        """One step on both sides; returns (gpu out [S,H,D] fp16 tensor, oracle inputs)."""
        w = self.w
        S, H, D = len(self.ids), w.num_heads, w.head_dim
        q = wl.normal_f16(self.vrng, (S, H, D))
        k = wl.normal_f16(self.vrng, (S, H, D))
        v = wl.normal_f16(self.vrng, (S, H, D))
        r = self.runner
        r.prepare()
        slots_o, copies_o = self.m.alloc_slots(self.ids)
        _, _, tables_g, copies_g = r._views(r.host[(r.i - 1) & 1])
        slots_g = r._views(r.host[(r.i - 1) & 1])[0]
        assert slots_g.tolist() == slots_o
        assert [tuple(c) for c in copies_g[: r.n_copies].tolist()] == copies_o
        tables_o = np.array(self.m.padded_tables(self.ids, self.max_blocks), np.int32)
        assert np.array_equal(tables_g, tables_o)
        ctx_o = np.array([self.m.num_tokens(s) for s in self.ids], np.int32)
        assert np.array_equal(r.ctx_host, ctx_o)
        out = torch.empty((S, H, D), dtype=torch.float16, device="cuda")
        r.copy_blocks([self.kc], [self.vc])
        r.write_kv(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), self.kc, self.vc)
        r.attention(out, torch.from_numpy(q).cuda(), self.kc, self.vc, w.scale)
        oc.copy_blocks([self.okc], [self.ovc], copies_o)
        oc.write_kv(self.okc, self.ovc, k, v, slots_o)
        torch.cuda.synchronize()
        assert r.status.item() == 0
        return out, q, tables_o, ctx_o

    def oracle_attention(self, q, tables, ctx, rows=None):
        if rows is not None:
            q, tables, ctx = q[rows], tables[rows], ctx[rows]
        return oa.paged_attention(q, self.okc, self.ovc, tables, ctx, self.w.scale)


def _err(gpu, ref):
    return float(np.abs(gpu.astype(np.float64) - ref).max())


def test_tiny_workload_everything_exact_and_attention_within_tolerance():
    w = wl.tiny()
    b = Both(w)
    b.check_cache()
    out, q, tables, ctx = b.decode_step()
    assert ctx.tolist() == [9, 6]
    b.check_cache()
    ref = b.oracle_attention(q, tables, ctx)
    assert _err(out.cpu().numpy(), ref) <= TOL


def test_tiny_workload_with_the_tutorial_fixed_table():
    """Same shapes, free order of the tutorial's Fig. 1-4: seq 0 ends on P5."""
    w = wl.tiny()
    w.free_order = np.array([3, 0, 1, 4, 5, 2], np.int32)
    w.prompt_lens = [8, 5]
    b = Both(w)
    out, q, tables, ctx = b.decode_step()
    assert tables[0].tolist()[:3] == [3, 0, 5]
    ref = b.oracle_attention(q, tables, ctx)
    assert _err(out.cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("name", ["opt13b_b64", "mixed_b256"])
def test_full_size_workloads_every_row(name):
    w = wl.WORKLOADS[name]()
    b = Both(w)
    b.check_cache()
    out, q, tables, ctx = b.decode_step()
    b.check_cache()
    ref = b.oracle_attention(q, tables, ctx)
    assert _err(out.cpu().numpy(), ref) <= TOL
    # a second step (contexts grow by one, some sequences take a new block)
    out2, q2, tables2, ctx2 = b.decode_step()
    assert np.array_equal(ctx2, ctx + 1)
    ref2 = b.oracle_attention(q2, tables2, ctx2)
    assert _err(out2.cpu().numpy(), ref2) <= TOL


def test_parallel_sampling_copy_on_write_64_steps():
    w = wl.parallel_sampling()
    b = Both(w, max_extra_steps=w.decode_steps)
    b.check_cache()
    total_copies = 0
    for step in range(w.decode_steps):
        out, q, tables, ctx = b.decode_step()
        total_copies += b.runner.n_copies
        if step in (0, 1, 15, 16, 17, w.decode_steps - 1):
            b.check_cache()
        ref = b.oracle_attention(q, tables, ctx)
        assert _err(out.cpu().numpy(), ref) <= TOL, step
    # every prompt whose last block is partial is copied for 3 of its 4 samples
    partial = sum(1 for p in w.prompt_lens if p % w.block_size)
    assert total_copies == 3 * partial


def _oracle_admit(m: BlockManager, w):
    """The workload's admission on the oracle's block manager (own loop)."""
    groups = {root: (extra, shared) for (root, extra), shared in zip(w.forks, w.shared_prefix)}
    ids, nxt, growing = [], len(w.prompt_lens), []
    for i, n in enumerate(w.prompt_lens):
        if i not in groups:
            m.add(i, n)
            ids.append(i)
            continue
        extra, shared = groups[i]
        m.add(i, shared)
        members = [i]
        for _ in range(extra):
            m.fork(i, nxt)
            members.append(nxt)
            nxt += 1
        ids.extend(members)
        growing.append((members, n - shared))
    for t in range(max((g[1] for g in growing), default=0)):
        batch = [s for members, own in growing if own > t for s in members]
        if batch:
            m.alloc_slots(batch)
    return ids


@pytest.mark.parametrize("beam", [False, True])
def test_full_40_layer_pool_filling_step_sampled(beam):
    """40 layers over a pool of min(120 GB, half the free memory), as the
    benchmark's 40-layer mode runs it; layers 0, 13, 26 and 39, each with
    its own cache values and new q / k / v, checked on a sample of sequences
    (a whole beam group in the beam variant)."""
    from paged_kv_cache_106_gb300.step import admit_workload

    free = torch.cuda.mem_get_info()[0]
    w = wl.full_40l(int(min(120e9, 0.5 * free)), beam=beam)
    L, H, D, B, NB = w.num_layers, w.num_heads, w.head_dim, w.block_size, w.num_blocks
    desc = pk.PoolDesc(NB, B, num_layers=L, num_heads=H, head_dim=D,
                       partition_tokens=w.split_tokens, free_order=w.free_order)
    pool = pk.pa_pool_create(desc)
    ids = admit_workload(pool, w)
    m = BlockManager(NB, B, w.free_order)
    assert _oracle_admit(m, w) == ids
    max_blocks = -(-(wl.CTX_CAP + 16) // B)
    t_gpu, ctx_gpu = pk.pa_get_block_tables(pool, ids, max_blocks)
    assert t_gpu.tolist() == m.padded_tables(ids, max_blocks)

    rng = np.random.default_rng(77)
    rows = sorted(set(rng.choice(len(ids), 6, replace=False).tolist()) | {int(np.argmax(ctx_gpu))})
    if beam:
        rows = sorted(set(rows) | set(range(4)))           # the first beam group
    layers = [0, 13, 26, L - 1]
    kc_all = torch.empty((L, NB, H, B, D), dtype=torch.float16, device="cuda")
    vc_all = torch.empty_like(kc_all)
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    kc_all.normal_(generator=g)
    vc_all.normal_(generator=g)
    vr = wl.value_rng(w, 3)
    blocks = sorted({b for r in rows for b in m.block_table(ids[r])})
    okc = {l: np.zeros((NB, H, B, D), np.float16) for l in layers}
    ovc = {l: np.zeros((NB, H, B, D), np.float16) for l in layers}
    bidx = torch.tensor(blocks, device="cuda")
    for l in layers:
        okc[l][blocks] = wl.normal_f16(vr, (len(blocks), H, B, D))
        ovc[l][blocks] = wl.normal_f16(vr, (len(blocks), H, B, D))
        kc_all[l][bidx] = torch.from_numpy(okc[l][blocks]).cuda()
        vc_all[l][bidx] = torch.from_numpy(ovc[l][blocks]).cuda()
    S = len(ids)
    q = {l: wl.normal_f16(vr, (S, H, D)) for l in layers}
    kn = {l: wl.normal_f16(vr, (S, H, D)) for l in layers}
    vn = {l: wl.normal_f16(vr, (S, H, D)) for l in layers}

    runner = DecodeStepRunner(pool, desc, ids, max_blocks)
    runner.prepare()
    slots_o, copies_o = m.alloc_slots(ids)
    slots_g = runner._views(runner.host[0])[0]
    assert slots_g.tolist() == slots_o
    kcs, vcs = list(kc_all.unbind(0)), list(vc_all.unbind(0))
    runner.copy_blocks(kcs, vcs)
    assert [tuple(c) for c in runner._views(runner.host[0])[3][: runner.n_copies].tolist()] == copies_o
    outs = {}
    dev_rand = torch.randn((S, H, D), dtype=torch.float16, device="cuda", generator=g)
    for l in range(L):
        if l in layers:
            qd, kd, vd = (torch.from_numpy(x[l]).cuda() for x in (q, kn, vn))
        else:
            qd = kd = vd = dev_rand
        out = torch.empty((S, H, D), dtype=torch.float16, device="cuda")
        runner.write_kv(kd, vd, kcs[l], vcs[l])
        runner.attention(out, qd, kcs[l], vcs[l], w.scale)
        if l in layers:
            outs[l] = out
    torch.cuda.synchronize()
    assert runner.status.item() == 0
    tables = np.array(m.padded_tables(ids, max_blocks), np.int32)
    ctx = np.array([m.num_tokens(s) for s in ids], np.int32)
    for l in layers:
        oc.copy_blocks([okc[l]], [ovc[l]], copies_o)
        oc.write_kv(okc[l], ovc[l], kn[l], vn[l], slots_o)
        ref = oa.paged_attention(q[l][rows], okc[l], ovc[l], tables[rows], ctx[rows], w.scale)
        assert _err(outs[l].cpu().numpy()[rows], ref) <= TOL, l
    pk.pa_pool_destroy(pool)


def test_prefix_cached_prompts_write_only_their_tails():
    """Requests sharing system prompts through the prefix cache: each writes
    the K/V of its uncached tail only, yet attends over its whole prompt."""
    H, D, B, NB = 4, 128, 16, 96
    rng = np.random.default_rng(41)
    vocab = 50
    systems = [list(rng.integers(0, vocab, n)) for n in (64, 40, 200)]
    reqs = [(systems[i % 3] + list(rng.integers(0, vocab, int(rng.integers(1, 60)))), i % 2)
            for i in range(9)]
    desc = pk.PoolDesc(NB, B, num_heads=H, head_dim=D, flags=pk.PA_POOL_PREFIX_CACHING)
    pool = pk.pa_pool_create(desc)
    m = BlockManager(NB, B, prefix_caching=True)
    kc = torch.zeros((NB, H, B, D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    okc, ovc = np.zeros((NB, H, B, D), np.float16), np.zeros((NB, H, B, D), np.float16)
    # the K/V of a token depend only on its prefix: derive them from a per-prefix seed
    def kv_of(toks, extra):
        r = np.random.default_rng(abs(hash((extra, tuple(toks)))) % (2**32))
        return wl.normal_f16(r, (2, H, D))
    written = 0
    for s, (toks, extra) in enumerate(reqs):
        slots_g, n_cached = pk.pa_seq_add_tokens(pool, s, toks, extra)
        slots_o, n_cached_o = m.add_tokens(s, toks, extra)
        assert slots_g.tolist() == slots_o and n_cached == n_cached_o
        tail = range(n_cached, len(toks))
        kv = np.stack([kv_of(toks[:p + 1], extra) for p in tail]) if len(tail) else \
            np.zeros((0, 2, H, D), np.float16)
        k, v = np.ascontiguousarray(kv[:, 0]), np.ascontiguousarray(kv[:, 1])
        sl = np.array(slots_o[n_cached:], np.int64)
        if len(sl):
            pk.pa_write_kv(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                           torch.from_numpy(sl).cuda(), kc, vc, desc)
            oc.write_kv(okc, ovc, k, v, sl)
        written += len(sl)
    assert written < sum(len(t) for t, _ in reqs)          # the cache saved writes
    ids = list(range(len(reqs)))
    mb = max(len(m.block_table(s)) for s in ids)
    tables = np.array(m.padded_tables(ids, mb), np.int32)
    ctx = np.array([len(t) for t, _ in reqs], np.int32)
    q = wl.normal_f16(rng, (len(ids), H, D))
    out = torch.empty((len(ids), H, D), dtype=torch.float16, device="cuda")
    ws = torch.empty(pk.pa_decode_workspace_bytes(len(ids), mb, desc), dtype=torch.uint8,
                     device="cuda")
    pk.pa_decode_attention(out, torch.from_numpy(q).cuda(), kc, vc, torch.from_numpy(tables).cuda(),
                           torch.from_numpy(ctx).cuda(), 0.088, desc, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(kc.cpu(), torch.from_numpy(okc))
    # every request reads the K/V its own full prompt defines, shared blocks included
    for s, (toks, extra) in enumerate(reqs):
        for p in range(len(toks)):
            kv = kv_of(toks[:p + 1], extra)
            blk = m.block_table(s)[p // B]
            assert np.array_equal(okc[blk, :, p % B], kv[0])
    ref = oa.paged_attention(q, okc, ovc, tables, ctx, 0.088)
    assert _err(out.cpu().numpy(), ref) <= TOL


def test_beam_search_churn_on_the_gpu():
    """Beam groups decode 24 steps with pruning between steps: copy-on-write
    copies, slot writes and attention of every beam against the oracle."""
    from paged_kv_cache_106_gb300.step import BeamGroups
    from tests.test_beam_churn import _oracle_groups, _oracle_prune

    H, D, B = 8, 128, 16
    churn = wl.beam_churn(groups=6, width=4, seed=321)
    nb = sum(-(-n // B) for n in churn.prompt_lens) * churn.width + 6 * 4 * 6
    order = np.random.default_rng(9).permutation(nb)
    desc = pk.PoolDesc(nb, B, num_heads=H, head_dim=D, free_order=order)
    pool = pk.pa_pool_create(desc)
    m = BlockManager(nb, B, order)
    # prompts written once by the root, shared by its beams
    rng = wl.value_rng(wl.mixed_b256(), 9)
    kc = torch.zeros((nb, H, B, D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    okc, ovc = np.zeros((nb, H, B, D), np.float16), np.zeros((nb, H, B, D), np.float16)
    bg = BeamGroups(pool, churn)
    beams, nxt = _oracle_groups(m, churn)
    for g, n in enumerate(churn.prompt_lens):
        root = beams[g][0]
        slots = np.array([m.slot_of(root, p) for p in range(n)], np.int64)
        k, v = wl.normal_f16(rng, (n, H, D)), wl.normal_f16(rng, (n, H, D))
        pk.pa_write_kv(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                       torch.from_numpy(slots).cuda(), kc, vc, desc)
        oc.write_kv(okc, ovc, k, v, slots)
    S = len(bg.ids())
    mb = -(-max(churn.prompt_lens) // B) + 3
    runner = DecodeStepRunner(pool, desc, bg.ids(), mb)
    rg, ro = np.random.default_rng(2), np.random.default_rng(2)
    copies = 0
    for step in range(24):
        runner.ids = np.array(bg.ids(), np.int32)
        q, k, v = (wl.normal_f16(rng, (S, H, D)) for _ in range(3))
        runner.prepare()
        so, co = m.alloc_slots(list(runner.ids))
        assert runner._views(runner.host[(runner.i - 1) & 1])[0].tolist() == so
        copies += len(co)
        out = torch.empty((S, H, D), dtype=torch.float16, device="cuda")
        runner.copy_blocks([kc], [vc])
        runner.write_kv(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), kc, vc)
        runner.attention(out, torch.from_numpy(q).cuda(), kc, vc, 0.088)
        oc.copy_blocks([okc], [ovc], co)
        oc.write_kv(okc, ovc, k, v, so)
        torch.cuda.synchronize()
        assert runner.status.item() == 0
        ids = list(runner.ids)
        tables = np.array(m.padded_tables(ids, mb), np.int32)
        ctx = np.array([m.num_tokens(s) for s in ids], np.int32)
        ref = oa.paged_attention(q, okc, ovc, tables, ctx, 0.088)
        assert _err(out.cpu().numpy(), ref) <= TOL, step
        if step % 8 == 7:
            assert torch.equal(kc.cpu(), torch.from_numpy(okc))
        bg.prune(churn.survivors(rg))
        nxt = _oracle_prune(m, beams, nxt, churn.survivors(ro))
    assert copies > 0
