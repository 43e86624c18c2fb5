"""The bounded waits of every kernel end on their own: a wait for an
mbarrier phase that nothing completes gives up after its limit (200 ms) and
reports PA_ERR_TIMEOUT through the status word, without a fault; the same
context then runs a normal call correctly.  (No GPU fault is provoked: the
wait is bounded by construction.)"""
import time

import numpy as np
import pytest
import torch

import paged_kv_cache_106_gb300 as pk
from oracle import cache_ops as oc

pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_reports_timeout_and_leaves_the_context_usable():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pk.pa_selftest_bounded_wait(status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert status.item() == pk.PA_ERR_TIMEOUT
    assert elapsed >= 0.2   # the wait ran to its limit
    assert elapsed < 10.0   # ... and no longer

    # the context still works: a slot write matches the oracle's byte model
    rng = np.random.default_rng(3)
    H, D, B, NB, T = 2, 64, 16, 8, 20
    desc = pk.PoolDesc(NB, B, num_heads=H, head_dim=D)
    k = rng.standard_normal((T, H, D)).astype(np.float16)
    v = rng.standard_normal((T, H, D)).astype(np.float16)
    slots = rng.permutation(NB * B)[:T].astype(np.int64)
    kc = torch.zeros((NB, H, B, D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.pa_write_kv(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                   torch.from_numpy(slots).cuda(), kc, vc, desc, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref_k = np.zeros((NB, H, B, D), np.float16)
    ref_v = np.zeros_like(ref_k)
    oc.write_kv(ref_k, ref_v, k, v, slots)
    assert np.array_equal(kc.cpu().numpy().view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(vc.cpu().numpy().view(np.uint16), ref_v.view(np.uint16))
