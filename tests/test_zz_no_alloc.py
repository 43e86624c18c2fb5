"""pa_decode_attention_noalloc against pa_decode_attention (GPU, through the C ABI).

The workspace-free entry point serves callers that cannot allocate device
memory when they run attention (a runtime that owns all device memory, a
plugin host that forbids cudaMalloc once serving has started).  It takes its
scratch from a fixed array inside the library, shared by every call, so this
checks two calls in a row -- the second one starts from whatever the first
left in the scratch -- each against the entry point that takes a
caller-allocated workspace, within the attention tolerance of the other GPU
tests.  Collected last, so a run that stops at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_106_gb300 as pk

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _batch(seed, ctx, H=8, D=128, B=16):
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
    f16 = lambda shape: torch.from_numpy(
        rng.standard_normal(shape, dtype=np.float32).astype(np.float16)).cuda()
    q, kc, vc = f16((len(ctx), H, D)), f16((NB, H, B, D)), f16((NB, H, B, D))
    desc = pk.PoolDesc(NB, B, num_heads=H, head_dim=D)
    return q, kc, vc, torch.from_numpy(tables).cuda(), torch.tensor(ctx, dtype=torch.int32).cuda(), desc


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    # contexts over one 512-token partition use the scratch for partial results
    for call, (seed, ctx) in enumerate([(31, [1300, 17, 600, 2048, 5, 512, 513]),
                                        (32, [700, 1, 1030, 64, 1600])]):
        q, kc, vc, tables, ctx_d, desc = _batch(seed, ctx)
        S, H, D = q.shape
        ws = torch.empty(pk.pa_decode_workspace_bytes(S, tables.shape[1], desc),
                         dtype=torch.uint8, device="cuda")
        ref = torch.empty((S, H, D), dtype=torch.float16, device="cuda")
        got = torch.full((S, H, D), float("nan"), dtype=torch.float16, device="cuda")
        st = torch.zeros(2, dtype=torch.int32, device="cuda")
        pk.pa_decode_attention(ref, q, kc, vc, tables, ctx_d, 0.088, desc, workspace=ws,
                               status=st[0:1])
        pk.pa_decode_attention_noalloc(got, q, kc, vc, tables, ctx_d, 0.088, desc,
                                       status=st[1:2])
        torch.cuda.synchronize()
        assert st.tolist() == [0, 0], call
        err = (got.double() - ref.double()).abs().max().item()
        assert err <= TOL, (call, err)


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
