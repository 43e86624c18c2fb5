"""GPU parity of each kernel through the C ABI against the CPU oracle.

* pa_write_kv / pa_copy_blocks: the whole cache byte image must equal the
  oracle's byte model (bit-exact), including skipped (negative) slots.
* pa_decode_attention: max |gpu - oracle| <= 2e-3 (fp16 output, fp32
  accumulation, oracle in fp64) over every head dimension / block size the
  library supports, contexts that cover 1 token, partial and full blocks,
  one block short of / past a partition, several partitions (split path) and
  empty contexts; the output is bitwise independent of where the blocks sit
  in the pool; split and unsplit results agree to the same tolerance.
* Kernel-side checks: a block id or slot outside the pool is skipped and
  reported in the status word instead of being dereferenced.
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


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _random_paged_batch(rng, ctx_lens, H, D, B, extra_blocks=3):
    """Caches filled with N(0,1) fp16, every sequence's blocks at random
    physical ids (a shuffled pool), tables padded with -1."""
    nblk = [-(-c // B) for c in ctx_lens]
    NB = sum(nblk) + extra_blocks
    perm = rng.permutation(NB).astype(np.int32)
    MB = max(1, max(nblk))
    tables = np.full((len(ctx_lens), MB), -1, np.int32)
    pos = 0
    for i, n in enumerate(nblk):
        tables[i, :n] = perm[pos:pos + n]
        pos += n
    kc = _f16(rng, (NB, H, B, D))
    vc = _f16(rng, (NB, H, B, D))
    q = _f16(rng, (len(ctx_lens), H, D))
    return q, kc, vc, tables, np.array(ctx_lens, np.int32)


def _gpu_attention(q, kc, vc, tables, ctx, scale, B, partition_tokens=0, status=None):
    S, H, D = q.shape
    desc = pk.PoolDesc(kc.shape[0], B, num_heads=H, head_dim=D, partition_tokens=partition_tokens)
    out = torch.empty((S, H, D), dtype=torch.float16, device="cuda")
    ws_bytes = pk.pa_decode_workspace_bytes(S, tables.shape[1], desc)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda") if ws_bytes else None
    st = _status() if status is None else status
    pk.pa_decode_attention(out, _dev(q), _dev(kc), _dev(vc), _dev(tables), _dev(ctx), scale, desc,
                           workspace=ws, status=st)
    torch.cuda.synchronize()
    if status is None:
        assert st.item() == 0
    return out.cpu().numpy()


def _contexts(B, part):
    c = [1, B - 1, B, B + 1, 2 * B + 3, part - B, part - 1, part, part + 1, 2 * part + B // 2,
         3 * part + 5, 7]
    return [x for x in c if x >= 1]


@pytest.mark.parametrize("D", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("B", [4, 8, 16, 32])
def test_attention_matches_oracle_all_shapes(D, B):
    rng = np.random.default_rng(1000 * D + B)
    H = 3
    part = 4 * B
    ctx = _contexts(B, part)
    q, kc, vc, tables, ctxa = _random_paged_batch(rng, ctx, H, D, B)
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oa.paged_attention(q, kc, vc, tables, ctxa, scale)
    for pt in (part, 0):   # split every 4 blocks, and the default partition
        got = _gpu_attention(q, kc, vc, tables, ctxa, scale, B, partition_tokens=pt)
        err = np.abs(got.astype(np.float64) - ref).max()
        assert err <= TOL, (D, B, pt, err)


def test_attention_opt13b_shape_long_contexts_split_and_unsplit():
    rng = np.random.default_rng(7)
    H, D, B = 40, 128, 16
    ctx = [1, 15, 16, 17, 511, 512, 513, 1024, 1500, 2047, 2048, 300]
    q, kc, vc, tables, ctxa = _random_paged_batch(rng, ctx, H, D, B)
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oa.paged_attention(q, kc, vc, tables, ctxa, scale)
    split = _gpu_attention(q, kc, vc, tables, ctxa, scale, B)                   # 512-token partitions
    whole = _gpu_attention(q, kc, vc, tables, ctxa, scale, B, partition_tokens=4096)
    assert np.abs(split.astype(np.float64) - ref).max() <= TOL
    assert np.abs(whole.astype(np.float64) - ref).max() <= TOL
    assert np.abs(split.astype(np.float64) - whole.astype(np.float64)).max() <= TOL


def test_attention_is_bitwise_independent_of_block_placement():
    rng = np.random.default_rng(9)
    H, D, B = 4, 128, 16
    ctx = [700, 33, 16, 1, 1300]
    q, kc, vc, tables, ctxa = _random_paged_batch(rng, ctx, H, D, B)
    # move every block to another physical id
    NB = kc.shape[0]
    perm = rng.permutation(NB)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    tables2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    a = _gpu_attention(q, kc, vc, tables, ctxa, 0.088, B)
    b = _gpu_attention(q, kc2, vc2, tables2, ctxa, 0.088, B)
    assert a.tobytes() == b.tobytes()


def test_attention_empty_context_and_empty_batch():
    rng = np.random.default_rng(11)
    q, kc, vc, tables, ctxa = _random_paged_batch(rng, [0, 5, 0], 2, 64, 8)
    got = _gpu_attention(q, kc, vc, tables, ctxa, 0.125, 8)
    ref = oa.paged_attention(q, kc, vc, tables, ctxa, 0.125)
    assert not np.any(got[0]) and not np.any(got[2])
    assert np.abs(got.astype(np.float64) - ref).max() <= TOL
    desc = pk.PoolDesc(4, 8, num_heads=2, head_dim=64)
    e = torch.empty((0, 2, 64), dtype=torch.float16, device="cuda")
    pk.pa_decode_attention(e, e, _dev(kc), _dev(vc), _dev(tables[:0]), _dev(ctxa[:0]), 0.1, desc,
                           n_seqs=0)


def test_attention_nan_in_unwritten_slots_is_never_used():
    """Slots past ctx hold NaN: the result must be finite and match the oracle."""
    rng = np.random.default_rng(13)
    H, D, B = 2, 128, 16
    ctx = [5, 16, 17, 530, 1]
    q, kc, vc, tables, ctxa = _random_paged_batch(rng, ctx, H, D, B)
    for i, c in enumerate(ctx):
        last = tables[i, (c - 1) // B]
        kc[last, :, c % B if c % B else B:, :] = np.nan
        vc[last, :, c % B if c % B else B:, :] = np.nan
    got = _gpu_attention(q, kc, vc, tables, ctxa, 0.088, B)
    assert np.all(np.isfinite(got))
    ref = oa.paged_attention(q, kc, vc, tables, ctxa, 0.088)
    assert np.abs(got.astype(np.float64) - ref).max() <= TOL


def test_attention_bad_block_id_is_reported_not_dereferenced():
    rng = np.random.default_rng(15)
    q, kc, vc, tables, ctxa = _random_paged_batch(rng, [40, 20], 2, 64, 8)
    tables[1, 1] = kc.shape[0] + 1000          # outside the pool
    st = _status()
    _gpu_attention(q, kc, vc, tables, ctxa, 0.1, 8, status=st)
    assert st.item() == pk.PA_ERR_BAD_BLOCK
    tables[1, 1] = -1
    st = _status()
    _gpu_attention(q, kc, vc, tables, ctxa, 0.1, 8, status=st)
    assert st.item() == pk.PA_ERR_BAD_BLOCK


@pytest.mark.parametrize("T,H,NB", [(300, 40, 37), (5000, 8, 400)])
def test_write_kv_is_bit_exact(T, H, NB):
    # 300 tokens: a thread per vector; 5000: the token-major grid-stride launch
    rng = np.random.default_rng(17 + T)
    B, D = 16, 128
    kc = _f16(rng, (NB, H, B, D))
    vc = _f16(rng, (NB, H, B, D))
    slots = rng.choice(NB * B, size=T, replace=False).astype(np.int64)
    slots[::17] = -1                           # tokens that are not stored
    k = _f16(rng, (T, H, D))
    v = _f16(rng, (T, H, D))
    dk, dv = _dev(kc), _dev(vc)
    desc = pk.PoolDesc(NB, B, num_heads=H, head_dim=D)
    st = _status()
    pk.pa_write_kv(_dev(k), _dev(v), _dev(slots), dk, dv, desc, status=st)
    torch.cuda.synchronize()
    oc.write_kv(kc, vc, k, v, slots)
    assert st.item() == 0
    assert dk.cpu().numpy().tobytes() == kc.tobytes()
    assert dv.cpu().numpy().tobytes() == vc.tobytes()


@pytest.mark.parametrize("H,D,B", [(2, 8, 4), (3, 64, 8), (40, 128, 16), (1, 256, 32)])
def test_write_kv_shapes_and_bad_slot(H, D, B):
    rng = np.random.default_rng(H * D + B)
    NB, T = 9, 2 * B + 3
    kc = np.zeros((NB, H, B, D), np.float16)
    vc = np.zeros_like(kc)
    slots = rng.choice(NB * B, size=T, replace=False).astype(np.int64)
    k, v = _f16(rng, (T, H, D)), _f16(rng, (T, H, D))
    dk, dv = _dev(kc), _dev(vc)
    desc = pk.PoolDesc(NB, B, num_heads=H, head_dim=D)
    bad = slots.copy()
    bad[3] = NB * B + 5                        # outside the pool: skipped, reported
    st = _status()
    pk.pa_write_kv(_dev(k), _dev(v), _dev(bad), dk, dv, desc, status=st)
    torch.cuda.synchronize()
    assert st.item() == pk.PA_ERR_BAD_BLOCK
    bad[3] = -1
    oc.write_kv(kc, vc, k, v, bad)
    assert dk.cpu().numpy().tobytes() == kc.tobytes()
    assert dv.cpu().numpy().tobytes() == vc.tobytes()


def test_copy_blocks_bit_exact_all_layers():
    rng = np.random.default_rng(19)
    L, NB, H, B, D = 5, 23, 40, 16, 128
    ks = [_f16(rng, (NB, H, B, D)) for _ in range(L)]
    vs = [_f16(rng, (NB, H, B, D)) for _ in range(L)]
    dks, dvs = [_dev(x) for x in ks], [_dev(x) for x in vs]
    pairs = np.array([[3, 10], [4, 0], [22, 7], [3, 15]], np.int32)
    desc = pk.PoolDesc(NB, B, num_layers=L, num_heads=H, head_dim=D)
    st = _status()
    pk.pa_copy_blocks(dks, dvs, _dev(pairs), desc, status=st)
    torch.cuda.synchronize()
    oc.copy_blocks(ks, vs, pairs.tolist())
    assert st.item() == 0
    for l in range(L):
        assert dks[l].cpu().numpy().tobytes() == ks[l].tobytes()
        assert dvs[l].cpu().numpy().tobytes() == vs[l].tobytes()
    bad = np.array([[1, NB], [2, 5]], np.int32)
    st = _status()
    pk.pa_copy_blocks(dks, dvs, _dev(bad), desc, status=st)
    torch.cuda.synchronize()
    assert st.item() == pk.PA_ERR_BAD_BLOCK
    oc.copy_blocks(ks, vs, [(2, 5)])
    for l in range(L):
        assert dks[l].cpu().numpy().tobytes() == ks[l].tobytes()


def test_context_longer_than_table_is_reported():
    rng = np.random.default_rng(21)
    q, kc, vc, tables, ctxa = _random_paged_batch(rng, [20, 8], 2, 64, 8)
    ctxa[0] = tables.shape[1] * 8 + 1
    st = _status()
    _gpu_attention(q, kc, vc, tables, ctxa, 0.1, 8, status=st)
    assert st.item() == pk.PA_ERR_BAD_BLOCK


def test_attention_many_short_units_persistent_path():
    """Hundreds of 1-3 block contexts: more units in flight than unit slots."""
    rng = np.random.default_rng(23)
    ctx = list(rng.integers(1, 41, size=500)) + [0, 1, 16, 17]
    q, kc, vc, tables, ctxa = _random_paged_batch(rng, ctx, 3, 128, 16)
    ref = oa.paged_attention(q, kc, vc, tables, ctxa, 0.088)
    got = _gpu_attention(q, kc, vc, tables, ctxa, 0.088, 16)
    assert np.abs(got.astype(np.float64) - ref).max() <= TOL


def test_attention_large_batch_grid_fallback_path():
    """More sequences than the persistent kernel plans in shared memory."""
    rng = np.random.default_rng(25)
    ctx = list(rng.integers(0, 120, size=2100))
    q, kc, vc, tables, ctxa = _random_paged_batch(rng, ctx, 2, 64, 8)
    ref = oa.paged_attention(q, kc, vc, tables, ctxa, 0.125)
    for pt in (0, 32):
        got = _gpu_attention(q, kc, vc, tables, ctxa, 0.125, 8, partition_tokens=pt)
        assert np.abs(got.astype(np.float64) - ref).max() <= TOL


def test_attention_repeated_calls_reuse_workspace():
    """The workspace needs no initialisation and may be reused: every call
    clears its scheduling word itself, and partial results are written
    before they are read.  A workspace of all-ones bytes, used three times,
    gives the oracle's result each time."""
    rng = np.random.default_rng(27)
    q, kc, vc, tables, ctxa = _random_paged_batch(rng, [600, 5, 1300, 64], 4, 128, 16)
    desc = pk.PoolDesc(kc.shape[0], 16, num_heads=4, head_dim=128)
    ws = torch.full((pk.pa_decode_workspace_bytes(4, tables.shape[1], desc),), 255, dtype=torch.uint8,
                    device="cuda")
    ref = oa.paged_attention(q, kc, vc, tables, ctxa, 0.1)
    dq, dk, dv, dt, dc = _dev(q), _dev(kc), _dev(vc), _dev(tables), _dev(ctxa)
    st = _status()
    for _ in range(3):
        out = torch.full((4, 4, 128), float("nan"), dtype=torch.float16, device="cuda")
        pk.pa_decode_attention(out, dq, dk, dv, dt, dc, 0.1, desc, workspace=ws, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        assert np.abs(out.cpu().numpy().astype(np.float64) - ref).max() <= TOL
