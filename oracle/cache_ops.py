"""ORACLE -- test infrastructure only.

Byte-image models of the two cache-mutating operations of a decode step.
Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may use this module.

Cache layout (a data format): ``cache[num_blocks][num_heads][block_size][head_dim]``
per layer, keys and values in separate arrays.

* ``write_kv`` -- the fused reshape-and-block-write: the new key/value of
  token t (all heads) goes to the slot ``slot_mapping[t]``, i.e. physical
  block ``slot // B`` at offset ``slot % B`` (vLLM paper review,
  mz-moonzoo.tistory.com/116, §5.1 (1) fused reshape and block write;
  PagedAttention notes, unpurerationalist.github.io, §4.1; slot arithmetic
  from the paged KV cache tutorial,
  llm-systems-engineering.pages.dev/posts/paged-kv-cache, Fig. 2).  A
  negative slot marks a token that is not stored (a reading: padding).
* ``copy_blocks`` -- the fused block copy used by copy-on-write: every
  listed (src, dst) pair copies the whole physical block, every layer, keys
  and values (review §5.1 (3); notes §4.1).  Pairs are applied in order.
"""
from __future__ import annotations

import numpy as np


def write_kv(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
             slot_mapping) -> None:
    """In-place: cache[slot // B, h, slot % B, :] = new[t, h, :] for every head."""
    num_blocks, H, B, D = k_cache.shape
    if k.shape != (len(slot_mapping), H, D) or v.shape != k.shape:
        raise ValueError("new k/v shape must be [n_tokens, H, D]")
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = divmod(slot, B)
        if blk >= num_blocks:
            raise IndexError("slot outside the pool")
        k_cache[blk, :, off, :] = k[t]
        v_cache[blk, :, off, :] = v[t]


def copy_blocks(k_caches, v_caches, pairs) -> None:
    """In-place: for each (src, dst) and each layer, block dst <- block src."""
    for src, dst in pairs:
        for cache in list(k_caches) + list(v_caches):
            cache[int(dst)] = cache[int(src)]


def swap_blocks(src_k, src_v, dst_k, dst_v, pairs) -> None:
    """In-place: for each (a, b) and each layer, dst block b <- src block a
    (swap out / swap in between two cache sets)."""
    for a, b in pairs:
        for s, d in list(zip(src_k, dst_k)) + list(zip(src_v, dst_v)):
            d[int(b)] = s[int(a)]

