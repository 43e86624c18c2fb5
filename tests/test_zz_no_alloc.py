"""pa_decode_attention_noalloc against pa_decode_attention and the oracle
(GPU, through the C ABI).

The workspace-free entry point serves callers that cannot allocate device
memory when they run attention (a runtime that owns all device memory, a
plugin host that forbids cudaMalloc once serving has started).  It takes its
scratch from a fixed array inside the library, shared by every call, so this
checks two calls in a row -- the second one starts from whatever the first
left in the scratch.  It runs the same kernels with the same work plan as the
entry point that takes a caller-allocated workspace, so its output must equal
that entry point's bit for bit; both are also compared with the fp64 oracle
within the attention tolerance of the other GPU tests (2e-3).  A batch of
more than 2048 sequences takes the grid kernel instead of the persistent one
and is covered too.  Free device memory is read before and after repeated
calls: the entry point must not allocate.  Collected last, so a run that
stops at the first failure has already run every other test; it also passes
on its own in a fresh process.
"""
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_106_gb300 as pk
from oracle import attention as oa

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _batch(seed, ctx, H=8, D=128, B=16):
    """Host inputs: fp16 q and caches, a fragmented block table per sequence."""
    rng = np.random.default_rng(seed)
    nblk = [-(-c // B) for c in ctx]
    NB = sum(nblk) + 5
    perm = rng.permutation(NB).astype(np.int32)
    MB = max(nblk)
    tables = np.full((len(ctx), MB), -1, np.int32)
    pos = 0
    for i, n in enumerate(nblk):
        tables[i, :n] = perm[pos:pos + n]
        pos += n
    f16 = lambda shape: rng.standard_normal(shape, dtype=np.float32).astype(np.float16)
    return dict(q=f16((len(ctx), H, D)), kc=f16((NB, H, B, D)), vc=f16((NB, H, B, D)),
                tables=tables, ctx=np.array(ctx, np.int32), desc=pk.PoolDesc(NB, B, num_heads=H, head_dim=D),
                scale=float(np.float32(1 / math.sqrt(D))))


class _OnDevice:
    """The batch's device buffers and the two entry points' outputs, all
    allocated up front so that nothing is allocated between the calls."""

    def __init__(self, b):
        self.b = b
        dev = lambda a: torch.from_numpy(a).cuda()
        self.q, self.kc, self.vc = dev(b["q"]), dev(b["kc"]), dev(b["vc"])
        self.tables, self.ctx = dev(b["tables"]), dev(b["ctx"])
        S, H, D = b["q"].shape
        nbytes = pk.pa_decode_workspace_bytes(S, b["tables"].shape[1], b["desc"])
        self.ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        self.ref = torch.empty((S, H, D), dtype=torch.float16, device="cuda")
        self.got = torch.empty((S, H, D), dtype=torch.float16, device="cuda")
        self.st = torch.zeros(2, dtype=torch.int32, device="cuda")

    def run_workspace(self):
        pk.pa_decode_attention(self.ref, self.q, self.kc, self.vc, self.tables, self.ctx,
                               self.b["scale"], self.b["desc"], workspace=self.ws,
                               status=self.st[0:1])

    def run_noalloc(self):
        pk.pa_decode_attention_noalloc(self.got, self.q, self.kc, self.vc, self.tables, self.ctx,
                                       self.b["scale"], self.b["desc"], status=self.st[1:2])


CASES = [
    # contexts over one 512-token partition use the scratch for partial results
    (31, [1300, 17, 600, 2048, 5, 512, 513]),
    (32, [700, 1, 1030, 64, 1600]),
]


def _grid_case():
    # more sequences than the persistent kernel's work plan holds: the grid
    # kernel and the merge take their partials from the scratch
    rng = np.random.default_rng(33)
    return _batch(34, rng.integers(1, 640, size=2100).tolist(), H=4, D=64)


def test_noalloc_is_bitwise_the_workspace_entry_point_and_matches_the_oracle():
    for call, (seed, ctx) in enumerate(CASES):
        b = _batch(seed, ctx)
        d = _OnDevice(b)
        d.got.fill_(float("nan"))
        d.run_workspace()
        d.run_noalloc()
        torch.cuda.synchronize()
        assert d.st.tolist() == [0, 0], call
        got, ref = d.got.cpu().numpy(), d.ref.cpu().numpy()
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), call
        want = oa.paged_attention(b["q"], b["kc"], b["vc"], b["tables"], b["ctx"], b["scale"])
        for name, out in (("noalloc", got), ("workspace", ref)):
            err = np.abs(out.astype(np.float64) - want).max()
            assert err <= TOL, (call, name, err)


def test_noalloc_grid_path_beyond_2048_sequences():
    b = _grid_case()
    d = _OnDevice(b)
    for _ in range(2):                      # two calls in a row on the shared scratch
        d.got.fill_(float("nan"))
        d.run_workspace()
        d.run_noalloc()
        torch.cuda.synchronize()
        assert d.st.tolist() == [0, 0]
        got, ref = d.got.cpu().numpy(), d.ref.cpu().numpy()
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
    want = oa.paged_attention(b["q"], b["kc"], b["vc"], b["tables"], b["ctx"], b["scale"])
    assert np.abs(got.astype(np.float64) - want).max() <= TOL


def test_noalloc_allocates_no_device_memory():
    ds = [_OnDevice(_batch(seed, ctx)) for seed, ctx in CASES] + [_OnDevice(_grid_case())]
    for d in ds:                            # the first calls may load device code once
        d.run_noalloc()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        for d in ds:
            d.run_noalloc()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert all(d.st[1].item() == 0 for d in ds)


def test_noalloc_rejects_a_batch_larger_than_its_scratch():
    desc = pk.PoolDesc(16, 16, num_heads=40, head_dim=128)
    n_seqs, max_blocks = 2048, 128            # ~170 MB of partial results
    assert pk.pa_decode_workspace_bytes(n_seqs, max_blocks, desc) > pk.PA_NOALLOC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.float16, device="cuda")
    tables = torch.zeros((n_seqs, max_blocks), dtype=torch.int32, device="cuda")
    ctx = torch.zeros(n_seqs, dtype=torch.int32, device="cuda")
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_decode_attention_noalloc(t, t, t, t, tables, ctx, 0.1, desc, n_seqs=n_seqs)
    assert e.value.code == pk.PA_ERR_INVALID_ARG
    assert "scratch" in str(e.value)
