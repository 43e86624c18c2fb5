"""GPU parity of causal paged prefill attention (pa_prefill_attention) and of
the prefill step it belongs to (pa_seq_add / pa_alloc_slots_n -> pa_write_kv
with many tokens per sequence -> pa_prefill_attention), against the fp64
oracle.

* max |gpu - oracle| <= 2e-3 (fp16 output, fp32 accumulation), over both
  supported head dimensions, every block size, whole prompts and chunks
  continuing a cached prefix, query counts that fill several 64-query tiles
  and leave a ragged tail, one-query sequences and empty ones;
* the output is bitwise independent of where the blocks sit in the pool;
* a one-query sequence agrees with pa_decode_attention on the same context;
* kernel-side checks: q_len > ctx and table entries outside the pool are
  reported through the status word; unsupported geometry is refused on the
  host.
"""
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_106_gb300 as pk
from oracle import attention as oa
from oracle import cache_ops as oc
import workloads as wl

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _f16(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _batch(rng, ctx, qlen, H, D, B, extra_blocks=3):
    nblk = [-(-c // B) for c in ctx]
    NB = sum(nblk) + extra_blocks
    perm = rng.permutation(NB).astype(np.int32)
    MB = max(1, max(nblk))
    tables = np.full((len(ctx), MB), -1, np.int32)
    pos = 0
    for i, n in enumerate(nblk):
        tables[i, :n] = perm[pos:pos + n]
        pos += n
    kc = _f16(rng, (NB, H, B, D))
    vc = _f16(rng, (NB, H, B, D))
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    q = _f16(rng, (int(qs[-1]), H, D))
    return q, kc, vc, tables, np.array(ctx, np.int32), qs


def _gpu_prefill(q, kc, vc, tables, ctx, qs, scale, B, status=None, max_q_len=None):
    T, H, D = q.shape
    desc = pk.PoolDesc(kc.shape[0], B, num_heads=H, head_dim=D)
    out = torch.full((max(T, 1), H, D), float("nan"), dtype=torch.float16, device="cuda")
    st = _status() if status is None else status
    mql = int(np.max(np.diff(qs))) if max_q_len is None and len(ctx) else (max_q_len or 0)
    pk.pa_prefill_attention(out, _dev(q) if T else out, _dev(kc), _dev(vc), _dev(tables),
                            _dev(ctx), _dev(qs), scale, desc, max_q_len=mql, status=st)
    torch.cuda.synchronize()
    if status is None:
        assert st.item() == 0, pk.pa_last_error_string()
    return out[:T].cpu().numpy()


def _check(got, ref):
    assert np.all(np.isfinite(got))
    err = np.abs(got.astype(np.float64) - ref).max() if got.size else 0.0
    assert err <= TOL, err


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [4, 8, 16, 32])
def test_prefill_matches_oracle(D, B):
    rng = np.random.default_rng(1000 + D + B)
    H = 3
    # (ctx, q_len): whole prompts of 1, 63, 64, 65, 200 tokens; chunks after
    # a cached prefix (q_len < ctx), one-query sequences, an empty query set,
    # and prompts spanning several 128-query tiles
    pairs = [(1, 1), (63, 63), (64, 64), (65, 65), (200, 200), (150, 37), (300, 129),
             (77, 1), (5, 0), (129, 128), (2 * B + 1, 2),
             # several query tiles: two pairs; two pairs and a lone first tile;
             # a chunk of 4 tiles after a prefix that is not tile-aligned
             (400, 400), (520, 520), (700, 450)]
    ctx = [c for c, _ in pairs]
    ql = [x for _, x in pairs]
    q, kc, vc, tables, ctxa, qs = _batch(rng, ctx, ql, H, D, B)
    scale = float(np.float32(1 / math.sqrt(D)))
    got = _gpu_prefill(q, kc, vc, tables, ctxa, qs, scale, B)
    ref = oa.paged_prefill(q, kc, vc, tables, ctxa, qs, scale)
    _check(got, ref)


@pytest.mark.parametrize("factor,lo,hi", [(4.0, 256, 384), (0.25, 256, 384), (8.0, 256, 384),
                                          (8.0, 288, 320), (16.0, 330, 340)])
def test_prefill_scores_that_jump_on_a_later_tile(factor, lo, hi):
    """Keys at positions lo..hi-1 (inside the third key tile) scaled by
    `factor`.  With 4 the rows that reach them see their maximum jump past
    the running one by about 2^11 on a later, unmasked key tile (the lazy
    rescale of O); with 1/4 the maximum stays where it was.  With 8 and 16
    the jump passes 2^15, what fp16 probabilities computed against the
    running maximum could hold: over the whole tile a chunk's maximum is past
    it before any of the tile's P is written, and the two halves of a row end
    with different references; over keys 288-319 only the second 32-key
    chunk of the first half jumps, after the first chunk's P is written, and
    the second half must take its partner's higher reference; over keys
    330-339 the jump is inside one chunk of the second half."""
    rng = np.random.default_rng(77)
    H, D, B = 2, 128, 16
    ctx = [520, 400]
    q, kc, vc, tables, ctxa, qs = _batch(rng, ctx, ctx, H, D, B)
    for s in range(len(ctx)):
        for p in range(lo, min(hi, ctx[s])):
            kc[tables[s][p // B], :, p % B, :] = (kc[tables[s][p // B], :, p % B, :].astype(np.float32)
                                                 * factor).astype(np.float16)
    scale = float(np.float32(1 / math.sqrt(D)))
    got = _gpu_prefill(q, kc, vc, tables, ctxa, qs, scale, B)
    ref = oa.paged_prefill(q, kc, vc, tables, ctxa, qs, scale)
    _check(got, ref)


def test_prefill_block_placement_is_bitwise_irrelevant():
    rng = np.random.default_rng(7)
    H, D, B = 2, 128, 16
    ctx, ql = [300, 90, 17], [300, 50, 17]
    q, kc, vc, tables, ctxa, qs = _batch(rng, ctx, ql, H, D, B, extra_blocks=0)
    scale = 1 / math.sqrt(D)
    a = _gpu_prefill(q, kc, vc, tables, ctxa, qs, scale, B)
    # move every block to a new physical id, carrying its contents along
    NB = kc.shape[0]
    new = rng.permutation(NB).astype(np.int32)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[new] = kc
    vc2[new] = vc
    t2 = np.where(tables >= 0, new[np.maximum(tables, 0)], -1).astype(np.int32)
    b = _gpu_prefill(q, kc2, vc2, t2, ctxa, qs, scale, B)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_one_query_prefill_agrees_with_decode():
    rng = np.random.default_rng(9)
    H, D, B = 4, 128, 16
    ctx = [1, 17, 300, 511]
    q, kc, vc, tables, ctxa, qs = _batch(rng, ctx, [1] * len(ctx), H, D, B)
    scale = 1 / math.sqrt(D)
    pre = _gpu_prefill(q, kc, vc, tables, ctxa, qs, scale, B)
    desc = pk.PoolDesc(kc.shape[0], B, num_heads=H, head_dim=D)
    out = torch.empty((len(ctx), H, D), dtype=torch.float16, device="cuda")
    ws_bytes = pk.pa_decode_workspace_bytes(len(ctx), tables.shape[1], desc)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = _status()
    pk.pa_decode_attention(out, _dev(q), _dev(kc), _dev(vc), _dev(tables), _dev(ctxa), scale,
                           desc, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    dec = out.cpu().numpy().astype(np.float64)
    ref = oa.paged_attention(q, kc, vc, tables, ctxa, scale)
    _check(pre, ref)
    assert np.abs(dec - pre.astype(np.float64)).max() <= 2 * TOL


def _prefill_step(pool, desc, kc, vc, seq_ids, chunks, rng, H, D, MB, known):
    """One prefill step through the pool: allocate slots for each sequence's
    chunk (pa_alloc_slots_n for known sequences, pa_seq_add for new ones),
    write the chunk's K/V, run prefill attention; returns what the oracle
    needs."""
    slots = []
    for sid, n in zip(seq_ids, chunks):
        if sid not in known:
            slots.append(pk.pa_seq_add(pool, sid, n))
            known.add(sid)
        else:
            s, copies = pk.pa_alloc_slots_n(pool, [sid], [n])
            assert len(copies) == 0
            slots.append(s)
    slot_mapping = np.concatenate(slots).astype(np.int64)
    T = slot_mapping.shape[0]
    k_new, v_new, q = _f16(rng, (T, H, D)), _f16(rng, (T, H, D)), _f16(rng, (T, H, D))
    st = _status()
    pk.pa_write_kv(_dev(k_new), _dev(v_new), _dev(slot_mapping), kc, vc, desc, status=st)
    tables, ctx = pk.pa_get_block_tables(pool, seq_ids, MB)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    out = torch.empty((T, H, D), dtype=torch.float16, device="cuda")
    pk.pa_prefill_attention(out, _dev(q), kc, vc, _dev(tables), _dev(ctx), _dev(qs),
                            1 / math.sqrt(D), desc, max_q_len=int(max(chunks)), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return q, tables, ctx, qs, out.cpu().numpy()


def test_prefill_step_through_the_pool_whole_prompts_then_chunks():
    rng = np.random.default_rng(11)
    H, D, B, NB, MB = 2, 64, 16, 256, 64
    order = rng.permutation(NB).astype(np.int32)
    desc = pk.PoolDesc(NB, B, num_heads=H, head_dim=D, free_order=order)
    pool = pk.pa_pool_create(desc)
    try:
        kc = torch.zeros((NB, H, B, D), dtype=torch.float16, device="cuda")
        vc = torch.zeros_like(kc)
        ids, known = [3, 8, 21, 40], set()
        for chunks in ([70, 16, 1, 130], [64, 9, 33, 1], [1, 100, 15, 64]):
            q, tables, ctx, qs, got = _prefill_step(pool, desc, kc, vc, ids, chunks, rng, H, D, MB, known)
            ref = oa.paged_prefill(q, kc.cpu().numpy(), vc.cpu().numpy(), tables, ctx, qs,
                                   1 / math.sqrt(D))
            _check(got, ref)
        assert list(ctx) == [135, 125, 49, 195]
    finally:
        pk.pa_pool_destroy(pool)


def test_prefill_writes_land_where_the_oracle_byte_model_puts_them():
    """The K1 write with N >> S tokens (a whole prompt per sequence) gives the
    oracle's byte image, and prefill then reads exactly those bytes."""
    rng = np.random.default_rng(12)
    H, D, B, NB = 2, 128, 8, 96
    desc = pk.PoolDesc(NB, B, num_heads=H, head_dim=D, free_order=rng.permutation(NB).astype(np.int32))
    pool = pk.pa_pool_create(desc)
    try:
        lens = [200, 3, 97, 64]
        slots = np.concatenate([pk.pa_seq_add(pool, i, n) for i, n in enumerate(lens)])
        T = slots.shape[0]
        k_new, v_new = _f16(rng, (T, H, D)), _f16(rng, (T, H, D))
        kc0, vc0 = _f16(rng, (NB, H, B, D)), _f16(rng, (NB, H, B, D))
        kc, vc = _dev(kc0), _dev(vc0)
        st = _status()
        pk.pa_write_kv(_dev(k_new), _dev(v_new), _dev(slots), kc, vc, desc, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        ek, ev = kc0.copy(), vc0.copy()
        oc.write_kv(ek, ev, k_new, v_new, slots)
        assert np.array_equal(kc.cpu().numpy().view(np.uint16), ek.view(np.uint16))
        assert np.array_equal(vc.cpu().numpy().view(np.uint16), ev.view(np.uint16))
        tables, ctx = pk.pa_get_block_tables(pool, list(range(len(lens))), 32)
        qs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        q = _f16(rng, (T, H, D))
        got = _gpu_prefill(q, ek, ev, tables, ctx, qs, 0.08, B)
        _check(got, oa.paged_prefill(q, ek, ev, tables, ctx, qs, 0.08))
    finally:
        pk.pa_pool_destroy(pool)


def test_prefill_full_size_batch_every_row():
    """The bench's prefill batch (256 prompts, 81 539 tokens, 40 heads x 128,
    block 16) in the launch configuration the bench times; every output row
    against the oracle (about 1.1 G query-key pairs in fp64 on the host)."""
    w = wl.prefill_b256()
    H, D, B = w.num_heads, w.head_dim, w.block_size
    lens = np.array(w.prompt_lens)
    desc = pk.PoolDesc(w.num_blocks, B, num_heads=H, head_dim=D, free_order=w.free_order)
    pool = pk.pa_pool_create(desc)
    try:
        slots = np.concatenate([pk.pa_seq_add(pool, i, int(n)) for i, n in enumerate(lens)])
        MB = -(-int(lens.max()) // B)
        tables, ctx = pk.pa_get_block_tables(pool, list(range(len(lens))), MB)
    finally:
        pk.pa_pool_destroy(pool)
    T = int(lens.sum())
    g = torch.Generator(device="cuda").manual_seed(5)
    kc = torch.randn((w.num_blocks, H, B, D), generator=g, device="cuda", dtype=torch.float16)
    vc = torch.randn((w.num_blocks, H, B, D), generator=g, device="cuda", dtype=torch.float16)
    q = torch.randn((T, H, D), generator=g, device="cuda", dtype=torch.float16)
    qs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out = torch.empty_like(q)
    st = _status()
    pk.pa_prefill_attention(out, q, kc, vc, _dev(tables), _dev(ctx), _dev(qs), w.scale, desc,
                            max_q_len=int(lens.max()), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert slots.shape == (T,)
    ref = oa.paged_prefill(q.cpu().numpy(), kc.cpu().numpy(), vc.cpu().numpy(), tables, ctx, qs,
                           w.scale)
    _check(out.cpu().numpy(), ref)


def test_prefill_is_bitwise_repeatable():
    """The first 64 prompts of the bench batch (40 heads x 128, block 16),
    launched ten times on the same inputs, give bitwise the same output: the
    kernel's orderings (a slot's next Q K^T overwriting the P that the
    preceding P V reads, issued by one thread; the output of a job read from
    tensor memory before the next job's first product) leave no race that
    could change a value from run to run."""
    w = wl.prefill_b256()
    H, D, B = w.num_heads, w.head_dim, w.block_size
    lens = np.array(w.prompt_lens[:64])
    desc = pk.PoolDesc(w.num_blocks, B, num_heads=H, head_dim=D, free_order=w.free_order)
    pool = pk.pa_pool_create(desc)
    try:
        for i, n in enumerate(lens):
            pk.pa_seq_add(pool, i, int(n))
        tables, ctx = pk.pa_get_block_tables(pool, list(range(len(lens))), -(-int(lens.max()) // B))
    finally:
        pk.pa_pool_destroy(pool)
    T = int(lens.sum())
    g = torch.Generator(device="cuda").manual_seed(9)
    kc = torch.randn((w.num_blocks, H, B, D), generator=g, device="cuda", dtype=torch.float16)
    vc = torch.randn((w.num_blocks, H, B, D), generator=g, device="cuda", dtype=torch.float16)
    q = torch.randn((T, H, D), generator=g, device="cuda", dtype=torch.float16)
    qs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    d_tab, d_ctx, d_qs = _dev(tables), _dev(ctx), _dev(qs)
    st = _status()
    first = None
    for _ in range(10):
        out = torch.full_like(q, float("nan"))
        pk.pa_prefill_attention(out, q, kc, vc, d_tab, d_ctx, d_qs, w.scale, desc,
                                max_q_len=int(lens.max()), status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        if first is None:
            first = out
            assert bool(torch.isfinite(first).all())
        else:
            assert torch.equal(out.view(torch.int16), first.view(torch.int16))


def test_prefill_replayed_from_a_graph_repeated_and_on_two_streams():
    """A launch takes its (sequence, query-tile pair, head) units one at a
    time from a counter that the launch sets back to zero when it ends, one of
    64 counters picked per call.  A launch captured in a CUDA graph and
    replayed five times, 70 launches in a row (more calls than counters) and
    two launches in flight at once on two streams each give bitwise the
    output of a single launch, which matches the oracle."""
    rng = np.random.default_rng(31)
    H, D, B = 4, 128, 16
    ctx = [300, 129, 1, 520, 77, 256]
    q, kc, vc, tables, ctxa, qs = _batch(rng, ctx, ctx, H, D, B)
    scale = 1.0 / math.sqrt(D)
    desc = pk.PoolDesc(kc.shape[0], B, num_heads=H, head_dim=D)
    dq, dk, dv, dt, dc, dqs = (_dev(a) for a in (q, kc, vc, tables, ctxa, qs))
    mql = max(ctx)
    st = _status()

    def launch(out, stream=None):
        pk.pa_prefill_attention(out, dq, dk, dv, dt, dc, dqs, scale, desc, max_q_len=mql,
                                status=st, stream=stream)

    ref = torch.full_like(dq, float("nan"))
    launch(ref)
    torch.cuda.synchronize()
    assert st.item() == 0
    _check(ref.cpu().numpy(), oa.paged_prefill(q, kc, vc, tables, ctxa, qs, scale))
    bits = ref.view(torch.int16)

    s = torch.cuda.Stream()
    out_g = torch.full_like(dq, float("nan"))
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        launch(out_g, s)   # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        launch(out_g, s)
    for _ in range(5):
        out_g.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g.view(torch.int16), bits)

    outs = [torch.full_like(dq, float("nan")) for _ in range(70)]
    for o in outs:
        launch(o)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), bits)

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    o1, o2 = torch.full_like(dq, float("nan")), torch.full_like(dq, float("nan"))
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        launch(o1, s1)
    with torch.cuda.stream(s2):
        launch(o2, s2)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(o1.view(torch.int16), bits) and torch.equal(o2.view(torch.int16), bits)


def _fused_vs_separate(q, kn, vn, kc, vc, tables, ctxa, qs, scale, B, mql):
    """Runs pa_write_kv + pa_prefill_attention and pa_prefill_step_attention
    from the same caches; returns both outputs and cache images."""
    T, H, D = q.shape
    desc = pk.PoolDesc(kc.shape[0], B, num_heads=H, head_dim=D)
    slots = np.concatenate([[tables[s][p // B] * B + p % B for p in range(int(ctxa[s]))]
                            for s in range(len(ctxa))]).astype(np.int64)
    res = []
    for fused in (False, True):
        dk, dv = _dev(kc), _dev(vc)
        out = torch.full((T, H, D), float("nan"), dtype=torch.float16, device="cuda")
        st = _status()
        if fused:
            pk.pa_prefill_step_attention(out, _dev(q), _dev(kn), _dev(vn), dk, dv, _dev(tables),
                                         _dev(ctxa), _dev(qs), scale, desc, max_q_len=mql, status=st)
        else:
            pk.pa_write_kv(_dev(kn), _dev(vn), _dev(slots), dk, dv, desc, status=st)
            pk.pa_prefill_attention(out, _dev(q), dk, dv, _dev(tables), _dev(ctxa), _dev(qs), scale,
                                    desc, max_q_len=mql, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0, (fused, st.item())
        res.append((out.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy()))
    return res, slots


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_fused_prefill_step_equals_write_then_prefill_and_the_oracle(D, B):
    """pa_prefill_step_attention on whole prompts (keys and values read from
    the new rows, written into the cache by the unit that reaches each
    prompt's last key): the cache image and the output bitwise those of
    pa_write_kv followed by pa_prefill_attention, the image that of the
    oracle's slot write, the output within 2e-3 of the oracle.  Prompt
    lengths cover one token, partial and full 128-query tiles, odd and even
    tile counts, and blocks cut by tile edges."""
    rng = np.random.default_rng(10 * D + B)
    H = 3
    ctx = [1, 7, B, 127, 128, 129, 300, 520, 64 + B // 2]
    q, kc, vc, tables, ctxa, qs = _batch(rng, ctx, ctx, H, D, B)
    T = int(qs[-1])
    kn, vn = _f16(rng, (T, H, D)), _f16(rng, (T, H, D))
    scale = 1.0 / math.sqrt(D)
    (sep, fus), slots = _fused_vs_separate(q, kn, vn, kc, vc, tables, ctxa, qs, scale, B, max(ctx))
    for a, b in zip(sep, fus):
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    okc, ovc = kc.copy(), vc.copy()
    oc.write_kv(okc, ovc, kn, vn, slots)
    assert np.array_equal(fus[1].view(np.uint16), okc.view(np.uint16))
    assert np.array_equal(fus[2].view(np.uint16), ovc.view(np.uint16))
    _check(fus[0], oa.paged_prefill(q, okc, ovc, tables, ctxa, qs, scale))


def test_fused_prefill_step_full_size_batch():
    """The benchmark's 256 prompts (81 539 tokens, 40 heads x 128, block 16):
    fused and separate give bitwise the same output and cache."""
    w = wl.prefill_b256()
    H, D, B = w.num_heads, w.head_dim, w.block_size
    lens = np.array(w.prompt_lens)
    desc = pk.PoolDesc(w.num_blocks, B, num_heads=H, head_dim=D, free_order=w.free_order)
    pool = pk.pa_pool_create(desc)
    try:
        slots = np.concatenate([pk.pa_seq_add(pool, i, int(n)) for i, n in enumerate(lens)])
        tables, ctx = pk.pa_get_block_tables(pool, list(range(len(lens))), -(-int(lens.max()) // B))
    finally:
        pk.pa_pool_destroy(pool)
    T = int(lens.sum())
    g = torch.Generator(device="cuda").manual_seed(3)
    q, kn, vn = (torch.randn((T, H, D), generator=g, device="cuda", dtype=torch.float16) for _ in range(3))
    kc0 = torch.randn((w.num_blocks, H, B, D), generator=g, device="cuda", dtype=torch.float16)
    vc0 = torch.randn_like(kc0)
    qs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    d_tab, d_ctx, d_qs = _dev(tables), _dev(ctx), _dev(qs)
    outs, caches = [], []
    for fused in (False, True):
        kc, vc = kc0.clone(), vc0.clone()
        out = torch.full_like(q, float("nan"))
        st = _status()
        if fused:
            pk.pa_prefill_step_attention(out, q, kn, vn, kc, vc, d_tab, d_ctx, d_qs, w.scale, desc,
                                         max_q_len=int(lens.max()), status=st)
        else:
            pk.pa_write_kv(kn, vn, _dev(slots), kc, vc, desc, status=st)
            pk.pa_prefill_attention(out, q, kc, vc, d_tab, d_ctx, d_qs, w.scale, desc,
                                    max_q_len=int(lens.max()), status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        outs.append(out)
        caches.append((kc, vc))
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(caches[0][0].view(torch.int16), caches[1][0].view(torch.int16))
    assert torch.equal(caches[0][1].view(torch.int16), caches[1][1].view(torch.int16))


def test_fused_prefill_step_refusals():
    """A sequence that is not a whole prompt (q_len < ctx) is reported in the
    status word; block size 4 and a NULL k_new are refused on the host."""
    rng = np.random.default_rng(43)
    H, D, B = 2, 128, 16
    q, kc, vc, tables, ctxa, qs = _batch(rng, [40, 90], [40, 60], H, D, B)
    T = int(qs[-1])
    kn, vn = _f16(rng, (T, H, D)), _f16(rng, (T, H, D))
    desc = pk.PoolDesc(kc.shape[0], B, num_heads=H, head_dim=D)
    out = torch.empty((T, H, D), dtype=torch.float16, device="cuda")
    st = _status()
    pk.pa_prefill_step_attention(out, _dev(q), _dev(kn), _dev(vn), _dev(kc), _dev(vc), _dev(tables),
                                 _dev(ctxa), _dev(qs), 0.1, desc, max_q_len=60, status=st)
    torch.cuda.synchronize()
    assert st.item() == pk.PA_ERR_INVALID_ARG
    desc4 = pk.PoolDesc(kc.shape[0], 4, num_heads=H, head_dim=D)
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_prefill_step_attention(out, _dev(q), _dev(kn), _dev(vn), _dev(kc), _dev(vc),
                                     _dev(tables), _dev(ctxa), _dev(qs), 0.1, desc4, max_q_len=60)
    assert e.value.code == pk.PA_ERR_INVALID_ARG
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_prefill_step_attention(out, _dev(q), None, _dev(vn), _dev(kc), _dev(vc),
                                     _dev(tables), _dev(ctxa), _dev(qs), 0.1, desc, max_q_len=60)
    assert e.value.code == pk.PA_ERR_INVALID_ARG


def test_prefill_status_reports_bad_lengths_and_blocks():
    rng = np.random.default_rng(13)
    H, D, B = 2, 64, 4
    q, kc, vc, tables, ctxa, qs = _batch(rng, [10, 10], [10, 4], H, D, B)
    # q_len > ctx for sequence 1: its rows stay unwritten, the status says why
    bad_ctx = ctxa.copy()
    bad_ctx[1] = 3
    st = _status()
    got = _gpu_prefill(q, kc, vc, tables, bad_ctx, qs, 0.1, B, status=st)
    assert st.item() == pk.PA_ERR_INVALID_ARG
    assert np.all(np.isnan(got[qs[1]:qs[2]].astype(np.float32)))
    _check(got[:qs[1]], oa.paged_prefill(q[:qs[1]], kc, vc, tables[:1], ctxa[:1], qs[:2], 0.1))
    # a table entry outside the pool is skipped and reported
    t2 = tables.copy()
    t2[0, 1] = kc.shape[0] + 5
    st = _status()
    _gpu_prefill(q, kc, vc, t2, ctxa, qs, 0.1, B, status=st)
    assert st.item() == pk.PA_ERR_BAD_BLOCK
    # a context longer than the table
    st = _status()
    c3 = ctxa.copy()
    c3[0] = tables.shape[1] * B + 1
    _gpu_prefill(q, kc, vc, tables, c3, qs, 0.1, B, status=st)
    assert st.item() == pk.PA_ERR_BAD_BLOCK
    # rows past q_rows: that sequence is refused, the other one computed
    desc = pk.PoolDesc(kc.shape[0], B, num_heads=H, head_dim=D)
    out = torch.full((int(qs[-1]), H, D), float("nan"), dtype=torch.float16, device="cuda")
    st = _status()
    pk.pa_prefill_attention(out, _dev(q), _dev(kc), _dev(vc), _dev(tables), _dev(ctxa), _dev(qs),
                            0.1, desc, max_q_len=10, status=st, q_rows=int(qs[-1]) - 1)
    torch.cuda.synchronize()
    assert st.item() == pk.PA_ERR_INVALID_ARG
    got = out.cpu().numpy()
    assert np.all(np.isnan(got[qs[1]:].astype(np.float32)))
    _check(got[:qs[1]], oa.paged_prefill(q[:qs[1]], kc, vc, tables[:1], ctxa[:1], qs[:2], 0.1))


def test_prefill_host_side_refusals():
    rng = np.random.default_rng(14)
    q, kc, vc, tables, ctxa, qs = _batch(rng, [8], [8], 2, 32, 4)
    desc = pk.PoolDesc(kc.shape[0], 4, num_heads=2, head_dim=32)
    out = torch.empty((8, 2, 32), dtype=torch.float16, device="cuda")
    with pytest.raises(pk.PagedKVError):
        pk.pa_prefill_attention(out, _dev(q), _dev(kc), _dev(vc), _dev(tables), _dev(ctxa),
                                _dev(qs), 0.1, desc, max_q_len=8)
    # misaligned q
    q2, kc2, vc2, t2, c2, qs2 = _batch(rng, [8], [8], 2, 64, 4)
    desc2 = pk.PoolDesc(kc2.shape[0], 4, num_heads=2, head_dim=64)
    qbuf = torch.empty(8 * 2 * 64 + 1, dtype=torch.float16, device="cuda")
    out2 = torch.empty((8, 2, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(pk.PagedKVError):
        pk.pa_prefill_attention(out2, qbuf[1:].view(8, 2, 64), _dev(kc2), _dev(vc2), _dev(t2),
                                _dev(c2), _dev(qs2), 0.1, desc2, max_q_len=8)
    # the scale must be finite and positive
    for bad in (0.0, -0.1, float("inf"), float("nan")):
        with pytest.raises(pk.PagedKVError):
            pk.pa_prefill_attention(out2, _dev(q2), _dev(kc2), _dev(vc2), _dev(t2), _dev(c2),
                                    _dev(qs2), bad, desc2, max_q_len=8)


def test_prefill_after_a_prefix_cache_hit_computes_only_the_new_tokens():
    """Two prompts share a 48-token system prompt in a pool with prefix
    caching: the second finds those three blocks cached, writes K/V for its
    own tokens only and prefills only them (q_len < ctx).  Its rows agree
    with the oracle and bitwise with prefilling the whole prompt in a fresh
    pool (each query row is computed on its own)."""
    H, D, B = 2, 64, 16
    rng = np.random.default_rng(21)
    system = rng.integers(0, 50000, 48).tolist()
    toks_a = system + rng.integers(0, 50000, 20).tolist()
    toks_b = system + rng.integers(0, 50000, 30).tolist()

    def kv_of(tokens):   # K/V of a position: a function of (position, token) only
        out_k, out_v = [], []
        for p_, t_ in enumerate(tokens):
            g = np.random.default_rng(1_000_003 * p_ + t_)
            out_k.append(_f16(g, (H, D)))
            out_v.append(_f16(g, (H, D)))
        return np.stack(out_k), np.stack(out_v)

    def prefill(pool, desc, kc, vc, sid, tokens, q_all):
        slots, n_cached = pk.pa_seq_add_tokens(pool, sid, tokens)
        k_all, v_all = kv_of(tokens)
        new = slice(n_cached, len(tokens))
        st = _status()
        pk.pa_write_kv(_dev(k_all[new]), _dev(v_all[new]), _dev(slots[new]), kc, vc, desc, status=st)
        tables, ctx = pk.pa_get_block_tables(pool, [sid], 8)
        q = q_all[new]
        qs = np.array([0, q.shape[0]], np.int32)
        out = torch.empty((q.shape[0], H, D), dtype=torch.float16, device="cuda")
        pk.pa_prefill_attention(out, _dev(q), kc, vc, _dev(tables), _dev(ctx), _dev(qs), 0.125,
                                desc, max_q_len=q.shape[0], status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        return n_cached, out.cpu().numpy(), tables, ctx, q, qs

    q_b = _f16(rng, (len(toks_b), H, D))
    q_a = _f16(rng, (len(toks_a), H, D))
    NB = 32
    desc = pk.PoolDesc(NB, B, num_heads=H, head_dim=D, flags=pk.PA_POOL_PREFIX_CACHING)
    pool = pk.pa_pool_create(desc)
    kc = torch.zeros((NB, H, B, D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    try:
        n0, _, _, _, _, _ = prefill(pool, desc, kc, vc, 0, toks_a, q_a)
        assert n0 == 0
        n1, got, tables, ctx, q, qs = prefill(pool, desc, kc, vc, 1, toks_b, q_b)
        assert n1 == 48 and list(ctx) == [len(toks_b)] and q.shape[0] == 30
        ref = oa.paged_prefill(q, kc.cpu().numpy(), vc.cpu().numpy(), tables, ctx, qs, 0.125)
        _check(got, ref)
    finally:
        pk.pa_pool_destroy(pool)
    # the same prompt prefilled whole in a fresh pool
    desc2 = pk.PoolDesc(NB, B, num_heads=H, head_dim=D)
    pool2 = pk.pa_pool_create(desc2)
    kc2 = torch.zeros((NB, H, B, D), dtype=torch.float16, device="cuda")
    vc2 = torch.zeros_like(kc2)
    try:
        n2, whole, _, _, _, _ = prefill(pool2, desc2, kc2, vc2, 7, toks_b, q_b)
        assert n2 == 0
        assert np.array_equal(whole[48:].view(np.uint16), got.view(np.uint16))
    finally:
        pk.pa_pool_destroy(pool2)
