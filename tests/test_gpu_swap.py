"""Swapping on the GPU: a sequence group goes to swap space in pinned host
memory (pa_swap_out + pa_swap_blocks), its GPU blocks are reused and
overwritten, and it comes back (pa_swap_in + pa_swap_blocks) to other
physical blocks.  The cache bytes must equal the oracle's byte model, and
the attention of the swapped sequences must be bitwise what it was before
(the result does not depend on where blocks sit)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_106_gb300 as pk
from oracle import attention as oa
from oracle import cache_ops as oc
from oracle.alloc import BlockManager, move_group
import workloads as wl

pytestmark = pytest.mark.gpu
H, D, B = 8, 128, 16


def _attend(desc, kc, vc, m_tables, ctx, q):
    S = len(ctx)
    out = torch.empty((S, H, D), dtype=torch.float16, device="cuda")
    mb = max(len(t) for t in m_tables)
    tables = np.array([t + [-1] * (mb - len(t)) for t in m_tables], np.int32)
    ws = torch.empty(pk.pa_decode_workspace_bytes(S, mb, desc), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.pa_decode_attention(out, torch.from_numpy(q).cuda(), kc, vc, torch.from_numpy(tables).cuda(),
                           torch.from_numpy(np.array(ctx, np.int32)).cuda(), 0.088, desc,
                           workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out.cpu().numpy(), tables


def test_swap_out_reuse_swap_in_round_trip():
    NG, NC = 64, 40
    rng = np.random.default_rng(3)
    dg = pk.PoolDesc(NG, B, num_heads=H, head_dim=D, free_order=rng.permutation(NG))
    dc = pk.PoolDesc(NC, B, num_heads=H, head_dim=D, free_order=rng.permutation(NC))
    gp, cp = pk.pa_pool_create(dg), pk.pa_pool_create(dc)
    gm = BlockManager(NG, B, dg._free)
    cm = BlockManager(NC, B, dc._free)
    kc = torch.zeros((NG, H, B, D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    hk = torch.zeros((NC, H, B, D), dtype=torch.float16).pin_memory()   # swap space
    hv = torch.zeros_like(hk).pin_memory()
    okc, ovc = np.zeros((NG, H, B, D), np.float16), np.zeros((NG, H, B, D), np.float16)
    ohk, ohv = np.zeros((NC, H, B, D), np.float16), np.zeros((NC, H, B, D), np.float16)

    def write(seq, n):
        slots = pk.pa_seq_add(gp, seq, n)
        assert slots.tolist() == gm.add(seq, n)
        k, v = wl.normal_f16(rng, (n, H, D)), wl.normal_f16(rng, (n, H, D))
        pk.pa_write_kv(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                       torch.from_numpy(slots).cuda(), kc, vc, dg)
        oc.write_kv(okc, ovc, k, v, slots)

    for s, n in enumerate([70, 33, 150, 16, 9]):
        write(s, n)
    pk.pa_seq_fork(gp, 2, 5)
    gm.fork(2, 5)
    group = [2, 5, 1]
    ctx = [gm.num_tokens(s) for s in group]
    q = wl.normal_f16(rng, (len(group), H, D))
    before, _ = _attend(dg, kc, vc, [gm.block_table(s) for s in group], ctx, q)

    # swap out to pinned host memory
    pairs = pk.pa_swap_out(gp, cp, group)
    assert [tuple(p) for p in pairs.tolist()] == move_group(gm, cm, group)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.pa_swap_blocks([kc], [vc], NG, [hk], [hv], NC, torch.from_numpy(pairs).cuda(), dg, status=st)
    oc.swap_blocks([okc], [ovc], [ohk], [ohv], pairs.tolist())
    torch.cuda.synchronize()
    assert st.item() == 0
    assert hk.numpy().tobytes() == ohk.tobytes() and hv.numpy().tobytes() == ohv.tobytes()

    # the freed GPU blocks go to new sequences whose K/V overwrite them
    for s, n in ((10, 200), (11, 230)):
        write(s, n)

    # swap back in (pairs array in pinned host memory this time)
    back = pk.pa_swap_in(cp, gp, group)
    assert [tuple(p) for p in back.tolist()] == move_group(cm, gm, group)
    hpairs = torch.from_numpy(back).pin_memory()
    pk.pa_swap_blocks([hk], [hv], NC, [kc], [vc], NG, hpairs, dg, status=st)
    oc.swap_blocks([ohk], [ohv], [okc], [ovc], back.tolist())
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(kc.cpu(), torch.from_numpy(okc)) and torch.equal(vc.cpu(), torch.from_numpy(ovc))
    after, tables = _attend(dg, kc, vc, [gm.block_table(s) for s in group], ctx, q)
    assert after.tobytes() == before.tobytes()
    ref = oa.paged_attention(q, okc, ovc, tables, np.array(ctx, np.int32), 0.088)
    assert np.abs(after.astype(np.float64) - ref).max() <= 2e-3

    # a pair outside either pool is skipped and reported
    bad = torch.tensor([[0, NC + 3]], dtype=torch.int32, device="cuda")
    st.zero_()
    pk.pa_swap_blocks([kc], [vc], NG, [hk], [hv], NC, bad, dg, status=st)
    torch.cuda.synchronize()
    assert st.item() == pk.PA_ERR_BAD_BLOCK
