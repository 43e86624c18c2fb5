"""Pins for the oracle's slot-write and block-copy models (oracle/cache_ops.py).

* Slot arithmetic from the paged KV cache tutorial
  (llm-systems-engineering.pages.dev/posts/paged-kv-cache, Fig. 2-3): slot 2
  is P0 offset 2, slot 20 is P5 offset 0 (block size 4); a write touches only
  that (block, offset) row of every head and nothing else, byte for byte.
* A round trip: tokens written through a random slot mapping and read back
  with numpy fancy indexing on the flattened [block*B + offset] axis are the
  tokens written.
* The block copy duplicates every layer's keys and values of the source block
  into the destination block and changes no other byte; pairs run in order.
"""
import numpy as np

from oracle.cache_ops import copy_blocks, write_kv


def test_tutorial_slots_land_in_the_right_rows():
    NB, H, B, D = 6, 2, 4, 8
    kc = np.zeros((NB, H, B, D), np.float16)
    vc = np.zeros((NB, H, B, D), np.float16)
    k = np.arange(2 * H * D, dtype=np.float16).reshape(2, H, D) + 1
    v = -k
    write_kv(kc, vc, k, v, [2, 20])
    expect_k = np.zeros_like(kc)
    expect_k[0, :, 2, :] = k[0]     # slot 2  -> P0 offset 2
    expect_k[5, :, 0, :] = k[1]     # slot 20 -> P5 offset 0
    expect_v = np.zeros_like(vc)
    expect_v[0, :, 2, :] = v[0]
    expect_v[5, :, 0, :] = v[1]
    assert kc.tobytes() == expect_k.tobytes()
    assert vc.tobytes() == expect_v.tobytes()


def test_negative_slot_is_skipped():
    kc = np.zeros((2, 1, 2, 8), np.float16)
    k = np.ones((2, 1, 8), np.float16)
    write_kv(kc, kc.copy(), k, k, [-1, 3])
    assert kc[1, 0, 1].tolist() == [1.0] * 8
    assert np.count_nonzero(kc) == 8


def test_write_round_trip_through_flat_slots():
    rng = np.random.default_rng(3)
    NB, H, B, D, T = 9, 3, 4, 16, 20
    kc = np.zeros((NB, H, B, D), np.float16)
    vc = np.zeros((NB, H, B, D), np.float16)
    slots = rng.choice(NB * B, size=T, replace=False)
    k = rng.standard_normal((T, H, D)).astype(np.float16)
    v = rng.standard_normal((T, H, D)).astype(np.float16)
    write_kv(kc, vc, k, v, slots)
    flat_k = kc.transpose(0, 2, 1, 3).reshape(NB * B, H, D)
    flat_v = vc.transpose(0, 2, 1, 3).reshape(NB * B, H, D)
    assert flat_k[slots].tobytes() == k.tobytes()
    assert flat_v[slots].tobytes() == v.tobytes()
    untouched = np.setdiff1d(np.arange(NB * B), slots)
    assert not np.any(flat_k[untouched])


def test_copy_blocks_all_layers_keys_and_values():
    rng = np.random.default_rng(5)
    L, NB, H, B, D = 3, 7, 2, 4, 8
    ks = [rng.standard_normal((NB, H, B, D)).astype(np.float16) for _ in range(L)]
    vs = [rng.standard_normal((NB, H, B, D)).astype(np.float16) for _ in range(L)]
    before_k = [x.copy() for x in ks]
    before_v = [x.copy() for x in vs]
    copy_blocks(ks, vs, [(1, 4), (6, 2)])
    for l in range(L):
        for c, b in ((ks[l], before_k[l]), (vs[l], before_v[l])):
            exp = b.copy()
            exp[4] = b[1]
            exp[2] = b[6]
            assert c.tobytes() == exp.tobytes()


def test_copy_pairs_apply_in_order():
    kc = np.arange(3 * 1 * 1 * 8, dtype=np.float16).reshape(3, 1, 1, 8)
    b0 = kc[0].copy()
    copy_blocks([kc], [], [(0, 1), (1, 2)])
    assert kc[2].tobytes() == b0.tobytes()
