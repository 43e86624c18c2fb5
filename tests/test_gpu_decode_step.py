"""GPU parity of pa_decode_step_attention, the decode step's slot write and
attention in one call, through the C ABI.

* Against pa_write_kv followed by pa_decode_attention on the same inputs:
  both caches and the output bitwise equal, for shapes whose write happens
  inside the persistent kernel and shapes where the library runs the slot
  write as its own launch first (more vectors per lane, or a batch too large
  for the persistent kernel's plan).
* Against the oracle: the cache byte image after the write equals the
  oracle's write_kv model, and attention is within 2e-3.
* A slot that is not position ctx - 1 of its sequence is reported
  (PA_ERR_INVALID_ARG) and not written; a negative slot is skipped.
"""
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_106_gb300 as pk
from oracle import attention as oa
from oracle import cache_ops as oc

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _f16(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def _batch(rng, ctx, H, D, B, extra_blocks=3):
    nblk = [-(-c // B) for c in ctx]
    NB = sum(nblk) + extra_blocks
    perm = rng.permutation(NB).astype(np.int32)
    MB = max(1, max(nblk))
    tables = np.full((len(ctx), MB), -1, np.int32)
    pos = 0
    for i, n in enumerate(nblk):
        tables[i, :n] = perm[pos:pos + n]
        pos += n
    kc, vc = _f16(rng, (NB, H, B, D)), _f16(rng, (NB, H, B, D))
    q, kn, vn = (_f16(rng, (len(ctx), H, D)) for _ in range(3))
    ctxa = np.array(ctx, np.int32)
    # the slot of each sequence's last position: its new token
    slots = np.array([tables[s][(c - 1) // B] * B + (c - 1) % B if c > 0 else -1
                      for s, c in enumerate(ctx)], np.int64)
    return q, kc, vc, kn, vn, tables, ctxa, slots


def _run(q, kc, vc, kn, vn, tables, ctxa, slots, scale, B, fused, part=0):
    S, H, D = q.shape
    desc = pk.PoolDesc(kc.shape[0], B, num_heads=H, head_dim=D, partition_tokens=part)
    dk, dv = _dev(kc), _dev(vc)
    out = torch.full((S, H, D), float("nan"), dtype=torch.float16, device="cuda")
    ws_bytes = pk.pa_decode_workspace_bytes(S, tables.shape[1], desc)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda") if ws_bytes else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_slots = _dev(slots)
    if fused:
        pk.pa_decode_step_attention(out, _dev(q), _dev(kn), _dev(vn), d_slots, dk, dv, _dev(tables),
                                    _dev(ctxa), scale, desc, workspace=ws, status=st)
    else:
        pk.pa_write_kv(_dev(kn), _dev(vn), d_slots, dk, dv, desc, status=st)
        pk.pa_decode_attention(out, _dev(q), dk, dv, _dev(tables), _dev(ctxa), scale, desc,
                               workspace=ws, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy(), st.item()


def _contexts(B, part):
    c = [1, B - 1, B, B + 1, 2 * B + 3, part - B, part - 1, part, part + 1, 2 * part + B // 2,
         3 * part + 5, 7]
    return [x for x in c if x >= 1]


@pytest.mark.parametrize("D,B", [(8, 16), (64, 4), (64, 16), (128, 16), (128, 32), (256, 16),
                                 (128, 4), (128, 8), (256, 4)])
def test_fused_step_equals_write_then_attention_and_the_oracle(D, B):
    """(128, 16), (128, 32), (64, *), (256, 16), (8, 16): the persistent
    kernel writes the new rows; (128, 4), (128, 8), (256, 4): the library's
    separate slot write runs first.  Contexts across partitions of 4 blocks."""
    rng = np.random.default_rng(100 * D + B)
    H = 3
    part = 4 * B
    ctx = _contexts(B, part)
    q, kc, vc, kn, vn, tables, ctxa, slots = _batch(rng, ctx, H, D, B)
    scale = float(np.float32(1 / math.sqrt(D)))
    for pt in (part, 0):
        oa_, ka, va, sa = _run(q, kc, vc, kn, vn, tables, ctxa, slots, scale, B, False, pt)
        ob, kb, vb, sb = _run(q, kc, vc, kn, vn, tables, ctxa, slots, scale, B, True, pt)
        assert sa == 0 and sb == 0
        assert np.array_equal(ka.view(np.uint16), kb.view(np.uint16))
        assert np.array_equal(va.view(np.uint16), vb.view(np.uint16))
        assert np.array_equal(oa_.view(np.uint16), ob.view(np.uint16))
        okc, ovc = kc.copy(), vc.copy()
        oc.write_kv(okc, ovc, kn, vn, slots)
        assert np.array_equal(kb.view(np.uint16), okc.view(np.uint16))
        assert np.array_equal(vb.view(np.uint16), ovc.view(np.uint16))
        ref = oa.paged_attention(q, okc, ovc, tables, ctxa, scale)
        assert np.abs(ob.astype(np.float64) - ref).max() <= TOL


def test_fused_step_opt13b_shape_long_contexts():
    """The benchmark's layer shape (40 heads x 128, block 16, 512-token
    partitions) with contexts on both sides of partition and block edges."""
    rng = np.random.default_rng(5)
    H, D, B = 40, 128, 16
    ctx = [1, 15, 16, 17, 511, 512, 513, 1024, 1500, 2047, 2048, 300]
    q, kc, vc, kn, vn, tables, ctxa, slots = _batch(rng, ctx, H, D, B)
    scale = float(np.float32(1 / math.sqrt(D)))
    oa_, ka, va, _ = _run(q, kc, vc, kn, vn, tables, ctxa, slots, scale, B, False)
    ob, kb, vb, st = _run(q, kc, vc, kn, vn, tables, ctxa, slots, scale, B, True)
    assert st == 0
    assert np.array_equal(ka.view(np.uint16), kb.view(np.uint16))
    assert np.array_equal(va.view(np.uint16), vb.view(np.uint16))
    assert np.array_equal(oa_.view(np.uint16), ob.view(np.uint16))
    okc, ovc = kc.copy(), vc.copy()
    oc.write_kv(okc, ovc, kn, vn, slots)
    ref = oa.paged_attention(q, okc, ovc, tables, ctxa, scale)
    assert np.abs(ob.astype(np.float64) - ref).max() <= TOL


def test_fused_step_large_batch_takes_the_separate_write():
    """More sequences than the persistent kernel plans: the grid kernel runs
    and the slot write is its own launch; results as the two calls give."""
    rng = np.random.default_rng(25)
    ctx = [int(c) for c in rng.integers(1, 120, size=2100)]
    q, kc, vc, kn, vn, tables, ctxa, slots = _batch(rng, ctx, 2, 64, 8)
    oa_, ka, va, _ = _run(q, kc, vc, kn, vn, tables, ctxa, slots, 0.125, 8, False)
    ob, kb, vb, st = _run(q, kc, vc, kn, vn, tables, ctxa, slots, 0.125, 8, True)
    assert st == 0
    assert np.array_equal(kb.view(np.uint16), ka.view(np.uint16))
    assert np.array_equal(vb.view(np.uint16), va.view(np.uint16))
    assert np.array_equal(ob.view(np.uint16), oa_.view(np.uint16))


def test_fused_step_refuses_a_slot_that_is_not_the_last_position():
    """In the persistent kernel's write: a slot other than position ctx - 1
    is reported and not written (the rest of the batch is written); a
    negative slot is skipped without a report."""
    rng = np.random.default_rng(31)
    H, D, B = 4, 128, 16
    ctx = [40, 17, 300, 5]
    q, kc, vc, kn, vn, tables, ctxa, slots = _batch(rng, ctx, H, D, B)
    bad = slots.copy()
    bad[0] -= 1                    # position ctx - 2 of sequence 0
    bad[3] = -1                    # sequence 3: nothing to write
    _, kb, vb, st = _run(q, kc, vc, kn, vn, tables, ctxa, bad, 0.09, B, True)
    assert st == pk.PA_ERR_INVALID_ARG
    okc, ovc = kc.copy(), vc.copy()
    oc.write_kv(okc, ovc, kn[1:3], vn[1:3], slots[1:3])   # only sequences 1 and 2
    assert np.array_equal(kb.view(np.uint16), okc.view(np.uint16))
    assert np.array_equal(vb.view(np.uint16), ovc.view(np.uint16))
    good = slots.copy()
    good[3] = -1
    _, kg, vg, st = _run(q, kc, vc, kn, vn, tables, ctxa, good, 0.09, B, True)
    assert st == 0
    okc, ovc = kc.copy(), vc.copy()
    oc.write_kv(okc, ovc, kn[:3], vn[:3], slots[:3])
    assert np.array_equal(kg.view(np.uint16), okc.view(np.uint16))
