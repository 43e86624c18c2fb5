"""The seeded workload generator and the benchmark's byte accounting.

* The notes' closed form (PagedAttention notes, unpurerationalist.github.io,
  §2): one OPT-13B token holds 2 x 5120 x 40 x 2 B = 800 KB of K/V, about
  1.6 GB for 2048 tokens -- the per-layer bytes the benchmark counts per
  attended token (K + V of 40 heads x 128) must add up to it.
* Structure: free orders are permutations, lengths respect their caps, the
  generator is deterministic per seed, and the steady-state batch starts from
  its own stationary length mix (the mean context does not drift when the
  continuous batch runs).
"""
import json
import os

import numpy as np

import workloads as wl
from tests.conftest import GOLDEN


def test_kv_bytes_per_token_matches_the_notes_closed_form():
    g = json.load(open(os.path.join(GOLDEN, "notes_s2_kv_bytes_per_token.json")))
    w = wl.mixed_b256()
    assert w.num_heads * w.head_dim == g["hidden"]
    per_layer = w.kv_bytes_per_token()
    assert per_layer == 20480
    assert per_layer * wl.OPT13B_LAYERS == g["expect_bytes_per_token"]
    gb_2048 = 2048 * per_layer * wl.OPT13B_LAYERS / 1e9
    assert abs(gb_2048 - g["expect_bytes_2048_tokens_gb_approx"]) / 1.6 < 0.06


def test_structures_are_valid_and_deterministic():
    for make in wl.WORKLOADS.values():
        a, b = make(), make()
        assert sorted(a.free_order.tolist()) == list(range(a.num_blocks))
        assert a.free_order.tolist() == b.free_order.tolist()
        assert a.prompt_lens == b.prompt_lens
        assert all(n >= 0 for n in a.prompt_lens)
    w = wl.mixed_b256()
    assert max(w.prompt_lens) + 1 <= wl.CTX_CAP
    assert all(t >= n + 1 for t, n in zip(w.targets, w.prompt_lens))
    t = wl.tiny()
    assert [n + 1 for n in t.prompt_lens] == [9, 6] and t.num_blocks == 6


def test_values_are_seeded_normal_fp16():
    w = wl.opt13b_b64()
    x = wl.normal_f16(wl.value_rng(w, 0), (4096, 8))
    y = wl.normal_f16(wl.value_rng(w, 0), (4096, 8))
    assert x.dtype == np.float16 and np.array_equal(x, y)
    assert abs(float(x.astype(np.float64).mean())) < 0.05
    assert abs(float(x.astype(np.float64).std()) - 1.0) < 0.05


def test_steady_state_batch_does_not_drift():
    w = wl.mixed_b256(steady_state=True)
    held = np.array(w.prompt_lens, np.int64)
    target = np.array(w.targets, np.int64)
    rng = np.random.default_rng(3)
    prompts, targets = wl.draw_mixed_sequences(rng, 20000)
    nxt = 0
    means = []
    for _ in range(1500):
        for i in np.nonzero(held >= target)[0]:
            held[i], target[i] = prompts[nxt], targets[nxt]
            nxt += 1
        held += 1
        means.append(held.mean())
    first, last = np.mean(means[:300]), np.mean(means[-300:])
    assert abs(last - first) / first < 0.12
    assert held.max() <= wl.CTX_CAP


def test_generators_and_oracle_load_without_the_product_library():
    """The seeded generators and the oracle import nothing from the product
    package: a process that uses only them (the oracle's timed runs) maps no
    libpagedkv.so."""
    import subprocess
    import sys

    from tests.conftest import ROOT
    code = ("import sys; sys.path.insert(0, %r)\n"
            "import workloads, oracle.alloc, oracle.cache_ops\n"
            "from oracle import attention\n"
            "attention.max_threads()\n"
            "maps = open('/proc/self/maps').read()\n"
            "print('libpagedkv' in maps, 'liboracle_attention' in maps)\n" % ROOT)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, check=True)
    assert out.stdout.split() == ["False", "True"], out.stdout + out.stderr
