"""One decode step of a batch through the library, as a serving loop runs it.

Per step (vLLM paper review, mz-moonzoo.tistory.com/116, §4.3 global
execution loop; §4.6: the scheduler hands block tables to the worker):

1. ``pa_decode_step_prepare_rows`` host block manager, one call: one slot
                           per sequence, the copy-on-write pairs, then the
                           batch's context lengths and the table rows that
                           changed since that staging buffer last held them,
                           written straight into the pinned staging buffer;
2. one pinned host -> device copy carrying slot mapping, context lengths,
   block tables and copy pairs (double-buffered staging, so the host can
   prepare step t+1 while the GPU still runs step t);
3. ``pa_copy_blocks``      copy-on-write copies, every layer (only if any);
4. per layer ``pa_decode_step_attention``: the new token's slot write and
   decode attention in one call (one launch where the persistent kernel
   writes the rows itself).

Everything is enqueued on one stream.  This module only sequences library
calls and owns the staging buffers; the work runs in libpagedkv.so.
"""
from __future__ import annotations

import ctypes
import time

import numpy as np
import torch

from . import (PoolDesc, pa_copy_blocks, pa_decode_attention, pa_decode_step_attention,
               pa_decode_step_prepare_rows_into, pa_decode_workspace_bytes, pa_write_kv)


def _align(x, a=256):
    return (x + a - 1) // a * a


class DecodeStepRunner:
    def __init__(self, pool, desc: PoolDesc, seq_ids, max_blocks: int, device="cuda",
                 stream: torch.cuda.Stream | None = None):
        self.pool = pool
        self.desc = desc
        self.ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        self.S = int(self.ids.shape[0])
        self.max_blocks = int(max_blocks)
        self.device = torch.device(device)
        self.stream = stream or torch.cuda.current_stream(self.device)
        S, MB = self.S, self.max_blocks
        # packed metadata: slots int64[S] | ctx int32[S] | tables int32[S, MB] | copies int32[S, 2]
        self.off_slots = 0
        self.off_ctx = _align(8 * S)
        self.off_tab = self.off_ctx + _align(4 * S)
        self.off_cp = self.off_tab + _align(4 * S * MB)
        self.nbytes = self.off_cp + _align(8 * S)
        self.host = [torch.empty(self.nbytes, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
        self.host_addr = [h.data_ptr() for h in self.host]
        self.host_ctx = [self._views(h)[1] for h in self.host]
        # per staging buffer: the table version each of its rows holds (0: none)
        self.row_versions = [np.zeros(S, np.uint64) for _ in range(2)]
        self.row_versions_addr = [v.ctypes.data for v in self.row_versions]
        self._n_copies = ctypes.c_int32(0)
        self.events = [None, None]
        self.dev = torch.empty(self.nbytes, dtype=torch.uint8, device=self.device)
        self.d_slots = self.dev[self.off_slots:self.off_slots + 8 * S].view(torch.int64)
        self.d_ctx = self.dev[self.off_ctx:self.off_ctx + 4 * S].view(torch.int32)
        self.d_tables = self.dev[self.off_tab:self.off_tab + 4 * S * MB].view(torch.int32).view(S, MB)
        self.d_copies = self.dev[self.off_cp:self.off_cp + 8 * S].view(torch.int32).view(S, 2)
        ws = pa_decode_workspace_bytes(S, MB, desc)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=self.device) if ws else None
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.n_copies = 0
        self.ctx_host = None
        self.host_seconds = 0.0
        self.i = 0

    def _views(self, buf):
        a = buf.numpy()
        S, MB = self.S, self.max_blocks
        return (a[self.off_slots:self.off_slots + 8 * S].view(np.int64),
                a[self.off_ctx:self.off_ctx + 4 * S].view(np.int32),
                a[self.off_tab:self.off_tab + 4 * S * MB].view(np.int32).reshape(S, MB),
                a[self.off_cp:self.off_cp + 8 * S].view(np.int32).reshape(S, 2))

    def prepare_host(self) -> None:
        """Host bookkeeping of the next step (block manager) into a pinned
        staging buffer; no device work.  May run while the previous step's
        kernels are in flight."""
        k = self.i & 1
        self.i += 1
        if self.events[k] is not None:
            self.events[k].synchronize()     # staging buffer k no longer in flight
        t0 = time.perf_counter()
        if self.ids.dtype != np.int32 or not self.ids.flags.c_contiguous or \
                self.ids.shape[0] != self.S:
            raise ValueError("ids must be a contiguous int32 array of the batch size")
        base = self.host_addr[k]
        n_cp = pa_decode_step_prepare_rows_into(
            self.pool, self.S, self.ids.ctypes.data, self.max_blocks, base + self.off_slots,
            base + self.off_ctx, base + self.off_tab, self.row_versions_addr[k], base + self.off_cp,
            self.S, self._n_copies)
        self.host_seconds = time.perf_counter() - t0   # block manager work of this step
        self._pending = (k, n_cp, self.host_ctx[k])

    def upload(self) -> int:
        """Enqueue the prepared step's metadata upload on the stream."""
        k, n_copies, ctx = self._pending
        with torch.cuda.stream(self.stream):
            self.dev.copy_(self.host[k], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(self.stream)
        self.events[k] = ev
        self.n_copies, self.ctx_host = n_copies, ctx
        return n_copies

    def prepare(self) -> int:
        """Host bookkeeping for one step and the upload of its metadata."""
        self.prepare_host()
        return self.upload()

    def copy_blocks(self, k_caches, v_caches):
        if self.n_copies:
            pa_copy_blocks(k_caches, v_caches, self.d_copies, self.desc, status=self.status,
                           stream=self.stream, n_pairs=self.n_copies)

    def write_kv(self, k_new, v_new, k_cache, v_cache):
        pa_write_kv(k_new, v_new, self.d_slots, k_cache, v_cache, self.desc, status=self.status,
                    stream=self.stream)

    def attention(self, out, q, k_cache, v_cache, scale: float):
        pa_decode_attention(out, q, k_cache, v_cache, self.d_tables, self.d_ctx, scale, self.desc,
                            workspace=self.workspace, status=self.status, stream=self.stream)

    def step_attention(self, out, q, k_new, v_new, k_cache, v_cache, scale: float):
        """The new tokens' slot write and attention of one layer, one call."""
        pa_decode_step_attention(out, q, k_new, v_new, self.d_slots, k_cache, v_cache,
                                 self.d_tables, self.d_ctx, scale, self.desc,
                                 workspace=self.workspace, status=self.status, stream=self.stream)

    def step(self, q, k_new, v_new, out, k_caches, v_caches, scale: float):
        """A whole decode step over all layers (lists of per-layer tensors)."""
        self.prepare()
        self.copy_blocks(k_caches, v_caches)
        for l in range(len(k_caches)):
            self.step_attention(out[l], q[l], k_new[l], v_new[l], k_caches[l], v_caches[l], scale)


def admit_workload(pool, w) -> list:
    """Admit a workload's sequences into a pool through the block manager.

    A plain sequence is added with its prompt.  A beam group (root index in
    ``w.forks`` with ``w.shared_prefix`` shared tokens) is added with the
    shared prefix, forked into its beams, and every beam then appends its own
    tokens one step at a time, so the beams share the prefix blocks through
    reference counts.  Returns the sequence ids in batch order.
    """
    from . import pa_alloc_slots, pa_seq_add, pa_seq_fork

    groups = {root: (extra, shared) for (root, extra), shared in
              zip(w.forks, w.shared_prefix or [None] * len(w.forks))}
    ids, next_id = [], len(w.prompt_lens)
    growing = []          # (ids of a group, own tokens still to append)
    for i, n in enumerate(w.prompt_lens):
        if i not in groups:
            pa_seq_add(pool, i, n, want_slots=False)
            ids.append(i)
            continue
        extra, shared = groups[i]
        shared = n if shared is None else shared
        pa_seq_add(pool, i, shared, want_slots=False)
        members = [i]
        for _ in range(extra):
            pa_seq_fork(pool, i, next_id)
            members.append(next_id)
            next_id += 1
        ids.extend(members)
        if n > shared:
            growing.append((members, n - shared))
    for t in range(max((g[1] for g in growing), default=0)):
        batch = [s for members, own in growing if own > t for s in members]
        if batch:
            pa_alloc_slots(pool, batch)
    return ids


class BeamGroups:
    """Applies a BeamChurn's survivor draws to a pool through the block
    manager: forks for repeated survivors, frees for pruned beams, one
    pa_beam_prune call per step.  Keeps the batch (beam sequence ids,
    group-major) for the next decode step."""

    def __init__(self, pool, churn):
        from . import pa_seq_add, pa_seq_fork
        self.pool, self.churn = pool, churn
        G, W = len(churn.prompt_lens), churn.width
        self.beams = np.empty((G, W), np.int32)
        self.next_id = 0
        for g, n in enumerate(churn.prompt_lens):
            root = self.next_id
            pa_seq_add(pool, root, n, want_slots=False)
            for j in range(1, W):
                pa_seq_fork(pool, root, root + j)
            self.beams[g] = np.arange(root, root + W, dtype=np.int32)
            self.next_id += W

    def ids(self):
        return self.beams.ravel().tolist()

    def id_array(self):
        """The batch as an int32 array (a view; valid until the next prune)."""
        return self.beams.reshape(-1)

    def prune(self, survivors):
        """survivors[g]: beam indices kept by group g (with repeats), or an
        int [groups, width] array of how often each beam is kept.  Returns
        (forks, frees) performed."""
        from . import pa_beam_prune
        W = self.beams.shape[1]
        if isinstance(survivors, np.ndarray):
            counts = survivors
        else:
            counts = np.zeros(self.beams.shape, np.int32)
            for g, keep in enumerate(survivors):
                counts[g] = np.bincount(keep, minlength=W)
        frees = int((counts == 0).sum())
        nid = pa_beam_prune(self.pool, self.beams, counts, self.next_id)
        forks = nid - self.next_id
        self.next_id = nid
        return forks, frees
