"""Pins for the fp64 paged-attention oracle (oracle/paged_attention.c).

Each pin fixes the oracle against something other than itself:

* its binary16 decoder against numpy's float16 -> float64 conversion, for
  all 65536 bit patterns;
* the special case of contiguous storage against a library routine
  (torch's scaled_dot_product_attention in float64), with the blocks laid
  out in order and in a random physical order (block table as in the paged
  KV cache tutorial, llm-systems-engineering.pages.dev/posts/paged-kv-cache,
  Fig. 2);
* closed forms: one token gives o = v_0; equal keys, q = 0 or scale = 0 give
  the mean of the values; two tokens give v0 + sigmoid(s1 - s0) (v1 - v0);
* invariants: the result does not depend on where blocks sit in the pool
  (bitwise) nor on the block size (bitwise: the same positions are summed in
  the same order); outputs lie in the convex hull of the values; huge scores
  do not overflow;
* the tutorial's Fig. 4 context: the query of position 8 reads exactly the
  9 stored positions -- values planted as NaN in every other slot of the pool
  leave the result finite and equal to attention over those 9 tokens.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle.alloc import BlockManager
from tests.allocator_replay import load


def _rng(seed):
    return np.random.default_rng(seed)


def _paged_from_contiguous(K, V, B, perm):
    """Lay out contiguous [H, T, D] keys/values as a paged cache.

    Logical block j goes to physical block perm[j]; returns caches
    [NB, H, B, D] and the table.  Pure numpy reshapes, no oracle code."""
    H, T, D = K.shape
    nblk = -(-T // B)
    pad = nblk * B - T
    Kp = np.concatenate([K, np.zeros((H, pad, D), K.dtype)], axis=1)
    Vp = np.concatenate([V, np.zeros((H, pad, D), V.dtype)], axis=1)
    # [H, nblk, B, D] -> [nblk, H, B, D]
    Kb = Kp.reshape(H, nblk, B, D).transpose(1, 0, 2, 3)
    Vb = Vp.reshape(H, nblk, B, D).transpose(1, 0, 2, 3)
    NB = max(perm) + 1 if len(perm) else 0
    kc = np.zeros((NB, H, B, D), np.float16)
    vc = np.zeros((NB, H, B, D), np.float16)
    kc[perm] = Kb
    vc[perm] = Vb
    return kc, vc, np.array(perm, np.int32)


def _sdpa64(q, K, V, scale):
    """torch SDPA in float64: q [H, D], K/V [H, T, D] -> [H, D]."""
    qt = torch.from_numpy(q.astype(np.float64))[:, None, :]
    Kt = torch.from_numpy(K.astype(np.float64))
    Vt = torch.from_numpy(V.astype(np.float64))
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)
    return o[:, 0, :].numpy()


def test_half_decoder_matches_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oa.half_bits_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("T,B,H,D,seed", [(1, 4, 1, 8, 0), (9, 4, 2, 8, 1), (37, 16, 3, 64, 2),
                                          (128, 16, 2, 128, 3), (257, 8, 1, 32, 4),
                                          (600, 32, 2, 128, 5)])
@pytest.mark.parametrize("layout", ["in_order", "shuffled"])
def test_matches_sdpa_on_contiguous_special_case(T, B, H, D, seed, layout):
    rng = _rng(seed)
    q = rng.standard_normal((H, D)).astype(np.float16)
    K = rng.standard_normal((H, T, D)).astype(np.float16)
    V = rng.standard_normal((H, T, D)).astype(np.float16)
    scale = float(np.float32(1 / math.sqrt(D)))
    nblk = -(-T // B)
    perm = list(range(nblk)) if layout == "in_order" else list(rng.permutation(nblk + 3)[:nblk])
    kc, vc, table = _paged_from_contiguous(K, V, B, perm)
    out = oa.paged_attention(q[None], kc, vc, table[None], np.array([T], np.int32), scale)
    ref = _sdpa64(q, K, V, scale)
    np.testing.assert_allclose(out[0], ref, rtol=0, atol=1e-12)


def test_single_token_returns_its_value_exactly():
    rng = _rng(7)
    H, D, B = 3, 16, 4
    kc = rng.standard_normal((5, H, B, D)).astype(np.float16)
    vc = rng.standard_normal((5, H, B, D)).astype(np.float16)
    q = rng.standard_normal((1, H, D)).astype(np.float16)
    out = oa.paged_attention(q, kc, vc, np.array([[3, -1]], np.int32), np.array([1], np.int32), 0.3)
    assert np.array_equal(out[0], vc[3, :, 0, :].astype(np.float64))


@pytest.mark.parametrize("case", ["equal_keys", "zero_query", "zero_scale"])
def test_uniform_weights_give_mean_of_values(case):
    rng = _rng(11)
    H, D, B, T = 2, 32, 4, 11
    K = rng.standard_normal((H, T, D)).astype(np.float16)
    if case == "equal_keys":
        K[:] = K[:, :1, :]
    V = rng.standard_normal((H, T, D)).astype(np.float16)
    q = rng.standard_normal((H, D)).astype(np.float16)
    if case == "zero_query":
        q[:] = 0
    scale = 0.0 if case == "zero_scale" else 0.25
    kc, vc, table = _paged_from_contiguous(K, V, B, [2, 0, 1])
    out = oa.paged_attention(q[None], kc, vc, table[None], np.array([T], np.int32), scale)
    np.testing.assert_allclose(out[0], V.astype(np.float64).mean(axis=1), rtol=0, atol=1e-14)


def test_two_tokens_closed_form():
    rng = _rng(13)
    H, D, B = 4, 8, 4
    K = rng.standard_normal((H, 2, D)).astype(np.float16)
    V = rng.standard_normal((H, 2, D)).astype(np.float16)
    q = rng.standard_normal((H, D)).astype(np.float16)
    scale = 0.5
    kc, vc, table = _paged_from_contiguous(K, V, B, [1])
    out = oa.paged_attention(q[None], kc, vc, table[None], np.array([2], np.int32), scale)
    K64, V64, q64 = K.astype(np.float64), V.astype(np.float64), q.astype(np.float64)
    for h in range(H):
        s0 = scale * float(q64[h] @ K64[h, 0])
        s1 = scale * float(q64[h] @ K64[h, 1])
        w1 = 1.0 / (1.0 + math.exp(-(s1 - s0)))
        ref = V64[h, 0] + w1 * (V64[h, 1] - V64[h, 0])
        np.testing.assert_allclose(out[0, h], ref, rtol=0, atol=1e-14)


def test_block_placement_and_block_size_do_not_change_the_result():
    rng = _rng(17)
    H, D, T = 2, 64, 45
    K = rng.standard_normal((H, T, D)).astype(np.float16)
    V = rng.standard_normal((H, T, D)).astype(np.float16)
    q = rng.standard_normal((1, H, D)).astype(np.float16)
    outs = []
    for B in (1, 3, 4, 16, 64):
        nblk = -(-T // B)
        for perm in (list(range(nblk)), list(rng.permutation(nblk))):
            kc, vc, table = _paged_from_contiguous(K, V, B, perm)
            outs.append(oa.paged_attention(q, kc, vc, table[None], np.array([T], np.int32), 0.125))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_convex_hull_and_large_scores():
    rng = _rng(19)
    H, D, B, T = 2, 16, 4, 13
    K = (rng.standard_normal((H, T, D)) * 40).astype(np.float16)
    V = rng.standard_normal((H, T, D)).astype(np.float16)
    q = (rng.standard_normal((1, H, D)) * 40).astype(np.float16)
    kc, vc, table = _paged_from_contiguous(K, V, B, [3, 1, 0, 2])
    # scores of order 1e4: exp would overflow without the max shift
    out = oa.paged_attention(q, kc, vc, table[None], np.array([T], np.int32), 1.0)
    assert np.all(np.isfinite(out))
    V64 = V.astype(np.float64)
    assert np.all(out[0] >= V64.min(axis=1) - 1e-12)
    assert np.all(out[0] <= V64.max(axis=1) + 1e-12)
    # with such a gap the softmax is one-hot on the best key
    s = np.einsum("hd,htd->ht", q[0].astype(np.float64), K.astype(np.float64))
    best = s.argmax(axis=1)
    for h in range(H):
        gap = np.sort(s[h])[-1] - np.sort(s[h])[-2]
        if gap > 50:
            np.testing.assert_allclose(out[0, h], V64[h, best[h]], atol=1e-12)


def test_tutorial_fig4_reads_only_the_context(golden_dir):
    doc = load(golden_dir, "tutorial_fig1_4_block_table.json")
    B, NB = doc["block_size"], doc["num_blocks"]
    m = BlockManager(NB, B, doc["free_order"])
    m.add(1, 6)
    m.add(2, 6)
    for _ in range(3):
        m.alloc_slots([1])
    ctx = doc["attention_context"]
    H, D = 2, 8
    rng = _rng(23)
    kc = np.full((NB, H, B, D), np.nan, np.float16)
    vc = np.full((NB, H, B, D), np.nan, np.float16)
    K = rng.standard_normal((H, ctx["ctx_len"], D)).astype(np.float16)
    V = rng.standard_normal((H, ctx["ctx_len"], D)).astype(np.float16)
    for p, slot in enumerate(ctx["expect_slots"]):
        kc[slot // B, :, slot % B, :] = K[:, p, :]
        vc[slot // B, :, slot % B, :] = V[:, p, :]
    table = np.array([m.padded_tables([1], 4)[0]], np.int32)
    q = rng.standard_normal((1, H, D)).astype(np.float16)
    out = oa.paged_attention(q, kc, vc, table, np.array([ctx["ctx_len"]], np.int32), 1 / math.sqrt(D))
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0], _sdpa64(q[0], K, V, 1 / math.sqrt(D)), atol=1e-12)


def test_zero_context_gives_zero_and_bad_table_is_rejected():
    kc = np.zeros((2, 1, 4, 8), np.float16)
    q = np.ones((2, 1, 8), np.float16)
    out = oa.paged_attention(q, kc, kc, np.array([[0], [5]], np.int32), np.array([0, 0], np.int32), 1.0)
    assert np.array_equal(out, np.zeros_like(out))
    with pytest.raises(IndexError):
        oa.paged_attention(q, kc, kc, np.array([[0], [5]], np.int32), np.array([1, 1], np.int32), 1.0)


# ---- causal paged prefill --------------------------------------------------

def _prefill_batch(rng, ctx, qlen, H, D, B):
    nblk = [-(-c // B) for c in ctx]
    NB = sum(nblk) + 2
    perm = rng.permutation(NB)
    MB = max(nblk)
    tables = np.full((len(ctx), MB), -1, np.int32)
    pos = 0
    for i, n in enumerate(nblk):
        tables[i, :n] = perm[pos:pos + n]
        pos += n
    kc = rng.standard_normal((NB, H, B, D)).astype(np.float16)
    vc = rng.standard_normal((NB, H, B, D)).astype(np.float16)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    q = rng.standard_normal((int(qs[-1]), H, D)).astype(np.float16)
    return q, kc, vc, tables, np.array(ctx, np.int32), qs


def test_prefill_matches_sdpa_with_an_explicit_causal_mask():
    rng = _rng(101)
    H, D, B = 3, 32, 4
    ctx, qlen = [13, 7, 20], [13, 3, 6]          # whole prompt, a chunk, a chunk
    q, kc, vc, tables, ctxa, qs = _prefill_batch(rng, ctx, qlen, H, D, B)
    out = oa.paged_prefill(q, kc, vc, tables, ctxa, qs, 0.2)
    for s, (n, ql) in enumerate(zip(ctx, qlen)):
        # contiguous K/V of the sequence, gathered with numpy indexing only
        t = tables[s, : -(-n // B)]
        K = kc[t].transpose(1, 0, 2, 3).reshape(H, -1, D)[:, :n].astype(np.float64)
        V = vc[t].transpose(1, 0, 2, 3).reshape(H, -1, D)[:, :n].astype(np.float64)
        Q = q[qs[s]:qs[s + 1]].transpose(1, 0, 2).astype(np.float64)       # [H, ql, D]
        mask = np.arange(n)[None, :] <= (n - ql + np.arange(ql))[:, None]   # bottom-right causal
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V),
            attn_mask=torch.from_numpy(mask), scale=0.2).numpy()
        np.testing.assert_allclose(out[qs[s]:qs[s + 1]].transpose(1, 0, 2), ref, atol=1e-12)


def test_prefill_first_token_and_decode_special_case():
    rng = _rng(103)
    H, D, B = 2, 16, 4
    q, kc, vc, tables, ctxa, qs = _prefill_batch(rng, [9, 5], [9, 1], H, D, B)
    out = oa.paged_prefill(q, kc, vc, tables, ctxa, qs, 0.3)
    # the first prompt token attends only to itself: o = v_0 exactly
    assert np.array_equal(out[0], vc[tables[0, 0], :, 0, :].astype(np.float64))
    # one query at the end of its context is a decode query
    dec = oa.paged_attention(q[qs[1]:qs[2]], kc, vc, tables[1:2], ctxa[1:2], 0.3)
    assert np.array_equal(out[qs[1]:qs[2]], dec)


def test_prefill_never_reads_future_or_unwritten_positions():
    rng = _rng(105)
    H, D, B = 2, 8, 4
    q, kc, vc, tables, ctxa, qs = _prefill_batch(rng, [10], [4], H, D, B)
    ref = oa.paged_prefill(q, kc, vc, tables, ctxa, qs, 0.5)
    kc2, vc2 = kc.copy(), vc.copy()
    last = tables[0, 2]
    kc2[last, :, 2:, :] = np.nan                 # slots past ctx 10
    vc2[last, :, 2:, :] = np.nan
    out = oa.paged_prefill(q, kc2, vc2, tables, ctxa, qs, 0.5)
    assert np.array_equal(out, ref)
    # changing position 9 (the last query's own token) leaves the earlier queries alone
    kc2[last, :, 1, :] += np.float16(1.0)
    out2 = oa.paged_prefill(q, kc2, vc2, tables, ctxa, qs, 0.5)
    assert np.array_equal(out2[:3], ref[:3]) and not np.array_equal(out2[3], ref[3])
