"""The benchmark's own decode loop -- the steady-state continuous batch of the
mixed-length serving workload -- against the oracle, step by step (GPU).

Per step, as ``bench.py`` runs it: finished sequences are freed and
replaced by newly drawn ones (``bench.SteadyBatch``), the block manager
appends one token to each of the 256 sequences and exports the batch's
tables into the pinned staging buffer (``DecodeStepRunner``), one upload,
then the slot write and split-context decode attention.  The oracle's block
manager replays every free, admission and append in the same order: slots,
copy pairs, tables and context lengths must be identical every step.  The
cache image of every block in use must equal the oracle's byte for byte, and
every output row must be within 2e-3 of the fp64 oracle at the first steps,
at steps that replaced sequences, and at the last one (vLLM paper review,
mz-moonzoo.tistory.com/116, §4.3: the decode loop, one new token per
sequence per step; KV cache tutorial, llm-systems-engineering.pages.dev,
Fig. 4: attention over exactly the stored context).

Unlike the benchmark, which times attention only, the test also writes each
newcomer's prompt K/V (on both sides), so that every position a query reads
holds a seeded value.  The oracle keeps its cache image only for the blocks
that sequences use (a block id is mapped to a row of a compact array), which
leaves attention unchanged: the result does not depend on where blocks sit.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_106_gb300 as pk
import workloads as wl
from bench import SteadyBatch, _pool_setup
from oracle import attention as oa
from oracle import cache_ops as oc
from oracle.alloc import BlockManager
from paged_kv_cache_106_gb300.step import DecodeStepRunner

pytestmark = pytest.mark.gpu
TOL = 2e-3
STEPS = 60


class CompactImage:
    """The oracle's cache image of the blocks in use, one compact row each."""

    def __init__(self, num_blocks, cap, H, B, D):
        self.B = B
        self.k = np.zeros((cap, H, B, D), np.float16)
        self.v = np.zeros_like(self.k)
        self.row = np.full(num_blocks, -1, np.int64)
        self.blocks = []

    def touch(self, blocks):
        for b in blocks:
            if b >= 0 and self.row[b] < 0:
                assert len(self.blocks) < self.k.shape[0], "compact image full"
                self.row[b] = len(self.blocks)
                self.blocks.append(int(b))

    def slots(self, slots):
        slots = np.asarray(slots, np.int64)
        return self.row[slots // self.B] * self.B + slots % self.B

    def tables(self, tables):
        t = np.asarray(tables, np.int64)
        return np.where(t >= 0, self.row[np.maximum(t, 0)], -1).astype(np.int32)


def test_steady_state_benchmark_loop_60_steps_against_the_oracle():
    w = wl.mixed_b256(steady_state=True)
    H, D, B, NB = w.num_heads, w.head_dim, w.block_size, w.num_blocks
    S = len(w.prompt_lens)
    max_blocks = -(-wl.CTX_CAP // B)
    desc, pool = _pool_setup(pk, w)                 # the benchmark's own admission
    m = BlockManager(NB, B, w.free_order)
    for i, n in enumerate(w.prompt_lens):
        m.add(i, n)
    ids = np.arange(S, dtype=np.int32)
    used0 = sum(len(m.block_table(s)) for s in range(S))
    img = CompactImage(NB, used0 + 4096, H, B, D)
    kc = torch.zeros((NB, H, B, D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    vr = wl.value_rng(w, 5)

    def write_prompt(s, n):
        """A sequence's prompt K/V, the same values on both sides."""
        slots = np.array([m.slot_of(s, p) for p in range(n)], np.int64)
        img.touch(m.block_table(s))
        k, v = wl.normal_f16(vr, (n, H, D)), wl.normal_f16(vr, (n, H, D))
        pk.pa_write_kv(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                       torch.from_numpy(slots).cuda(), kc, vc, desc, status=status)
        oc.write_kv(img.k, img.v, k, v, img.slots(slots))

    for s, n in enumerate(w.prompt_lens):
        write_prompt(s, n)
    stream = torch.cuda.Stream()
    runner = DecodeStepRunner(pool, desc, ids, max_blocks, stream=stream)
    runner.ids = ids                                 # replaced in place, as in the benchmark
    batch = SteadyBatch(pk, pool, w, np.random.default_rng(w.seed + 7))
    out = torch.empty((S, H, D), dtype=torch.float16, device="cuda")
    replaced_steps, checked = [], []
    for step in range(STEPS):
        old = ids.copy()
        batch.admit(ids)
        changed = np.nonzero(ids != old)[0]
        for i in changed:                            # SteadyBatch's order: ascending index
            m.free(int(old[i]))
            m.add(int(ids[i]), int(batch.held[i]))
            write_prompt(int(ids[i]), int(batch.held[i]))
        if len(changed):
            replaced_steps.append(step)
        q, k, v = (wl.normal_f16(vr, (S, H, D)) for _ in range(3))
        runner.prepare()
        batch.appended()
        slots_o, copies_o = m.alloc_slots([int(s) for s in ids])
        slots_g, ctx_g, tables_g, copies_g = runner._views(runner.host[(runner.i - 1) & 1])
        assert slots_g.tolist() == slots_o, step
        assert [tuple(c) for c in copies_g[: runner.n_copies].tolist()] == copies_o, step
        tables_o = np.array(m.padded_tables([int(s) for s in ids], max_blocks), np.int32)
        assert np.array_equal(tables_g, tables_o), step
        ctx_o = np.array([m.num_tokens(int(s)) for s in ids], np.int32)
        assert np.array_equal(ctx_g, ctx_o), step
        for s in ids:
            img.touch(m.block_table(int(s)))
        with torch.cuda.stream(stream):
            runner.copy_blocks([kc], [vc])
            runner.write_kv(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), kc, vc)
            runner.attention(out, torch.from_numpy(q).cuda(), kc, vc, w.scale)
        oc.copy_blocks([img.k], [img.v],
                       [(int(img.row[a]), int(img.row[b])) for a, b in copies_o])
        oc.write_kv(img.k, img.v, k, v, img.slots(slots_o))
        torch.cuda.synchronize()
        assert runner.status.item() == 0 and status.item() == 0, step
        first_replacements = replaced_steps[:4]
        if step in (0, 1, STEPS - 1) or (replaced_steps and replaced_steps[-1] == step
                                          and step in first_replacements):
            ref = oa.paged_attention(q, img.k, img.v, img.tables(tables_o), ctx_o, w.scale)
            err = float(np.abs(out.cpu().numpy().astype(np.float64) - ref).max())
            assert err <= TOL, (step, err)
            checked.append(step)
    assert batch.replaced > 0 and len(replaced_steps) >= 2, replaced_steps
    assert any(s in replaced_steps for s in checked), (checked, replaced_steps)
    # every block in use: the GPU cache equals the oracle's image byte for byte
    idx = torch.tensor(img.blocks, dtype=torch.int64, device="cuda")
    n = len(img.blocks)
    assert np.array_equal(kc[idx].cpu().numpy().view(np.uint16), img.k[:n].view(np.uint16))
    assert np.array_equal(vc[idx].cpu().numpy().view(np.uint16), img.v[:n].view(np.uint16))
    pk.pa_pool_destroy(pool)
