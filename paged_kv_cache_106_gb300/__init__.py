"""GB300 paged KV cache decode step: thin Python binding of libpagedkv.so.

Every function here has the name of the C entry point it calls
(``include/pagedkv.h``) and only marshals arguments: host arrays go in as
numpy arrays, device buffers as CUDA torch tensors (or raw device addresses),
streams as torch streams (default: torch's current stream).  All the work --
block management on the host, slot write, block copy and decode attention on
the GPU -- runs in the library.  There is no fallback: if the library is
missing, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# always the library that the package's own build step writes next to it
_LIB_PATH = os.path.join(_PKG, "libpagedkv.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_OUT_OF_BLOCKS = 2
PA_ERR_NO_SEQ = 3
PA_ERR_CUDA = 4
PA_ERR_TIMEOUT = 5
PA_ERR_BAD_BLOCK = 6
PA_DTYPE_F16 = 0
PA_POOL_PREFIX_CACHING = 1
PA_DEFAULT_PARTITION_TOKENS = 512
PA_NOALLOC_SCRATCH_BYTES = 32 << 20

_ERR_NAMES = {1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_OUT_OF_BLOCKS", 3: "PA_ERR_NO_SEQ",
              4: "PA_ERR_CUDA", 5: "PA_ERR_TIMEOUT", 6: "PA_ERR_BAD_BLOCK"}


class PagedKVError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


class OutOfBlocks(PagedKVError):
    pass


class pa_pool_desc(ctypes.Structure):
    _fields_ = [
        ("num_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_layers", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("partition_tokens", ctypes.c_int32),
        ("flags", ctypes.c_int32),
        ("free_order", ctypes.POINTER(ctypes.c_int32)),
    ]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "(or python paged_kv_cache_106_gb300/_build.py)")
    lib = ctypes.CDLL(_LIB_PATH)
    i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "pa_last_error_string": (ctypes.c_char_p, []),
        "pa_pool_create": (i32, [P(pa_pool_desc), P(vp)]),
        "pa_pool_destroy": (i32, [vp]),
        "pa_seq_add": (i32, [vp, i32, i32, vp]),
        "pa_seq_add_tokens": (i32, [vp, i32, i32, vp, i64, vp, P(i32)]),
        "pa_pool_cached_blocks": (i32, [vp, P(i32)]),
        "pa_swap_out": (i32, [vp, vp, i32, vp, vp, i32, P(i32)]),
        "pa_swap_in": (i32, [vp, vp, i32, vp, vp, i32, P(i32)]),
        "pa_swap_blocks": (i32, [vp, vp, i32, vp, vp, i32, i32, vp, i32, P(pa_pool_desc), vp, vp]),
        "pa_seq_fork": (i32, [vp, i32, i32]),
        "pa_seq_fork_batch": (i32, [vp, i32, vp, vp]),
        "pa_seq_free_batch": (i32, [vp, i32, vp]),
        "pa_seq_free": (i32, [vp, i32]),
        "pa_beam_prune": (i32, [vp, i32, i32, vp, vp, P(i32)]),
        "pa_alloc_slots": (i32, [vp, i32, vp, vp, vp, i32, P(i32)]),
        "pa_alloc_slots_n": (i32, [vp, i32, vp, vp, vp, vp, i32, P(i32)]),
        "pa_get_block_tables": (i32, [vp, i32, vp, i32, vp, vp]),
        "pa_decode_step_prepare": (i32, [vp, i32, vp, i32, vp, vp, vp, vp, i32, P(i32)]),
        "pa_decode_step_prepare_rows": (i32, [vp, i32, vp, i32, vp, vp, vp, vp, vp, i32, P(i32)]),
        "pa_seq_info": (i32, [vp, i32, P(i32), P(i32)]),
        "pa_pool_num_free": (i32, [vp, P(i32)]),
        "pa_pool_free_queue": (i32, [vp, vp, i32, P(i32)]),
        "pa_pool_refcounts": (i32, [vp, vp]),
        "pa_write_kv": (i32, [vp, vp, vp, i32, vp, vp, P(pa_pool_desc), vp, vp]),
        "pa_copy_blocks": (i32, [vp, vp, i32, vp, i32, P(pa_pool_desc), vp, vp]),
        "pa_decode_workspace_bytes": (sz, [i32, i32, P(pa_pool_desc)]),
        "pa_decode_attention": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, ctypes.c_float, vp, sz,
                                      vp, P(pa_pool_desc), vp]),
        "pa_decode_step_attention": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                           ctypes.c_float, vp, sz, vp, P(pa_pool_desc), vp]),
        "pa_decode_attention_noalloc": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, ctypes.c_float,
                                              vp, P(pa_pool_desc), vp]),
        "pa_prefill_attention": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                       ctypes.c_float, vp, P(pa_pool_desc), vp]),
        "pa_prefill_step_attention": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                            i32, ctypes.c_float, vp, P(pa_pool_desc), vp]),
        "pa_selftest_bounded_wait": (i32, [vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
LIB_PATH = _LIB_PATH


def pa_last_error_string() -> str:
    return _lib.pa_last_error_string().decode()


def _check(rc: int):
    if rc != PA_OK:
        msg = pa_last_error_string()
        if rc == PA_ERR_OUT_OF_BLOCKS:
            raise OutOfBlocks(rc, msg)
        raise PagedKVError(rc, msg)


def _need_elems(n_elems: int, **tensors):
    """Refuses a tensor holding fewer elements than the call reads from it
    (None is left to the library, which refuses a NULL it needs)."""
    for name, t in tensors.items():
        if t is not None and t.numel() < n_elems:
            raise ValueError(f"{name} holds {t.numel()} elements, the call reads {n_elems}")


def _host_i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _dev(x):
    """Device address of a CUDA tensor (or an int address / None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x.data_ptr()


def _addr(x):
    """Device-reachable address of a CUDA tensor or of a pinned host tensor."""
    if x is None or isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if not (x.is_cuda or x.is_pinned()):
        raise ValueError("expected a CUDA tensor or a pinned host tensor")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class PoolDesc:
    """Holds a pa_pool_desc (and keeps its free_order array alive)."""

    def __init__(self, num_blocks, block_size, num_layers=1, num_heads=1, head_dim=8,
                 partition_tokens=0, free_order=None, flags=0):
        self._free = None if free_order is None else _host_i32(free_order)
        self.c = pa_pool_desc(int(num_blocks), int(block_size), int(num_layers), int(num_heads),
                              int(head_dim), PA_DTYPE_F16, int(partition_tokens), int(flags),
                              None if self._free is None else
                              self._free.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))

    def __getattr__(self, name):
        return getattr(self.__dict__["c"], name)

    @property
    def ref(self):
        return ctypes.byref(self.c)


# ---------------------------------------------------------------- host calls
def pa_pool_create(desc: PoolDesc):
    h = ctypes.c_void_p()
    _check(_lib.pa_pool_create(desc.ref, ctypes.byref(h)))
    return h


def pa_pool_destroy(pool) -> None:
    _check(_lib.pa_pool_destroy(pool))


def pa_seq_add(pool, seq_id: int, n_tokens: int, want_slots: bool = True):
    slots = np.empty(max(int(n_tokens), 0), np.int64) if want_slots else None
    _check(_lib.pa_seq_add(pool, int(seq_id), int(n_tokens),
                           None if slots is None else slots.ctypes.data))
    return slots


def pa_seq_add_tokens(pool, seq_id: int, token_ids, extra_key: int = 0, want_slots: bool = True):
    """Returns (slots int64[n] or None, n_cached_tokens)."""
    toks = _host_i32(token_ids)
    n = int(toks.shape[0])
    slots = np.empty(n, np.int64) if want_slots else None
    nc = ctypes.c_int32(0)
    _check(_lib.pa_seq_add_tokens(pool, int(seq_id), n, toks.ctypes.data if n else None,
                                  int(extra_key), None if slots is None else slots.ctypes.data,
                                  ctypes.byref(nc)))
    return slots, nc.value


def pa_pool_cached_blocks(pool) -> int:
    n = ctypes.c_int32()
    _check(_lib.pa_pool_cached_blocks(pool, ctypes.byref(n)))
    return n.value


def _group_move(fn, src_pool, dst_pool, seq_ids):
    ids = _host_i32(seq_ids)
    cap = 0
    # room for every distinct block: at most the sum of the tables' lengths
    for s in ids.tolist():
        cap += pa_seq_info(src_pool, s)[1]
    pairs = np.empty((max(cap, 1), 2), np.int32)
    n = ctypes.c_int32(0)
    _check(fn(src_pool, dst_pool, ids.shape[0], ids.ctypes.data, pairs.ctypes.data, cap,
              ctypes.byref(n)))
    return pairs[: n.value]


def pa_swap_out(gpu_pool, cpu_pool, seq_ids):
    """Move a sequence group to the CPU pool; returns the (gpu, cpu) block pairs."""
    return _group_move(_lib.pa_swap_out, gpu_pool, cpu_pool, seq_ids)


def pa_swap_in(cpu_pool, gpu_pool, seq_ids):
    """Move a sequence group back to the GPU pool; returns the (cpu, gpu) block pairs."""
    return _group_move(_lib.pa_swap_in, cpu_pool, gpu_pool, seq_ids)


def pa_swap_blocks(src_k, src_v, src_num_blocks, dst_k, dst_v, dst_num_blocks, pairs,
                   desc: PoolDesc, status=None, stream=None, n_pairs: int | None = None) -> None:
    L = len(src_k)
    arr = lambda xs: (ctypes.c_void_p * L)(*[_addr(x) for x in xs])
    n = int(pairs.shape[0]) if n_pairs is None else int(n_pairs)
    _check(_lib.pa_swap_blocks(arr(src_k), arr(src_v), int(src_num_blocks), arr(dst_k),
                               arr(dst_v), int(dst_num_blocks), L, _addr(pairs), n, desc.ref,
                               _dev(status), _stream(stream)))


def pa_seq_fork(pool, parent: int, child: int) -> None:
    _check(_lib.pa_seq_fork(pool, int(parent), int(child)))


def pa_seq_fork_batch(pool, parents, children) -> None:
    p, c = _host_i32(parents), _host_i32(children)
    if p.shape != c.shape:
        raise ValueError("parents and children differ in length")
    _check(_lib.pa_seq_fork_batch(pool, p.shape[0], p.ctypes.data, c.ctypes.data))


def pa_seq_free_batch(pool, seq_ids) -> None:
    ids = _host_i32(seq_ids)
    _check(_lib.pa_seq_free_batch(pool, ids.shape[0], ids.ctypes.data))


def pa_beam_prune(pool, beams, counts, next_id: int) -> int:
    """beams: int32 [groups, width] (contiguous, updated in place); counts:
    int32 [groups, width], each row summing to width.  Returns the new next_id."""
    if beams.dtype != np.int32 or not beams.flags.c_contiguous or beams.ndim != 2:
        raise ValueError("beams must be a contiguous int32 [groups, width] array")
    cnt = _host_i32(counts)
    if cnt.shape != beams.shape:
        raise ValueError("counts and beams differ in shape")
    nid = ctypes.c_int32(int(next_id))
    _check(_lib.pa_beam_prune(pool, beams.shape[0], beams.shape[1], beams.ctypes.data,
                              cnt.ctypes.data, ctypes.byref(nid)))
    return nid.value


def pa_seq_free(pool, seq_id: int) -> None:
    _check(_lib.pa_seq_free(pool, int(seq_id)))


def pa_alloc_slots(pool, seq_ids, copies_cap: int | None = None, slot_out=None, copies_out=None):
    """Returns (slot_mapping int64[n], copies int32[n_copies, 2])."""
    ids = _host_i32(seq_ids)
    n = ids.shape[0]
    cap = n if copies_cap is None else int(copies_cap)
    slots = np.empty(n, np.int64) if slot_out is None else slot_out
    copies = np.empty((max(cap, 1), 2), np.int32) if copies_out is None else copies_out
    nc = ctypes.c_int32(0)
    _check(_lib.pa_alloc_slots(pool, n, ids.ctypes.data, slots.ctypes.data, copies.ctypes.data,
                               cap, ctypes.byref(nc)))
    return slots, copies[: nc.value]


def pa_alloc_slots_n(pool, seq_ids, counts, copies_cap: int | None = None):
    """counts[i] new tokens for seq_ids[i]; returns (slot_mapping int64[sum], copies)."""
    ids, cnt = _host_i32(seq_ids), _host_i32(counts)
    if ids.shape != cnt.shape:
        raise ValueError("seq_ids and counts differ in length")
    n = ids.shape[0]
    cap = n if copies_cap is None else int(copies_cap)
    slots = np.empty(max(int(cnt.sum()), 1), np.int64)
    copies = np.empty((max(cap, 1), 2), np.int32)
    nc = ctypes.c_int32(0)
    _check(_lib.pa_alloc_slots_n(pool, n, ids.ctypes.data, cnt.ctypes.data, slots.ctypes.data,
                                 copies.ctypes.data, cap, ctypes.byref(nc)))
    return slots[: int(cnt.sum())], copies[: nc.value]


def pa_get_block_tables(pool, seq_ids, max_blocks: int, tables_out=None, ctx_out=None):
    """Returns (tables int32[n, max_blocks] padded with -1, ctx_lens int32[n])."""
    ids = _host_i32(seq_ids)
    n = ids.shape[0]
    tables = np.empty((n, max_blocks), np.int32) if tables_out is None else tables_out
    ctx = np.empty(n, np.int32) if ctx_out is None else ctx_out
    _check(_lib.pa_get_block_tables(pool, n, ids.ctypes.data, int(max_blocks),
                                    tables.ctypes.data, ctx.ctypes.data))
    return tables, ctx


def pa_decode_step_prepare(pool, seq_ids, max_blocks: int, slot_out=None, ctx_out=None,
                           tables_out=None, copies_out=None, copies_cap: int | None = None):
    """One token appended to every sequence, then the batch's tables.
    Returns (slot_mapping int64[n], ctx_lens int32[n], tables int32[n, max_blocks],
    copies int32[n_copies, 2]); the *_out arrays (e.g. views of a pinned
    staging buffer) are written in place when given."""
    ids = _host_i32(seq_ids)
    n = ids.shape[0]
    cap = n if copies_cap is None else int(copies_cap)
    slots = np.empty(n, np.int64) if slot_out is None else slot_out
    ctx = np.empty(n, np.int32) if ctx_out is None else ctx_out
    tables = np.empty((n, max_blocks), np.int32) if tables_out is None else tables_out
    copies = np.empty((max(cap, 1), 2), np.int32) if copies_out is None else copies_out
    nc = ctypes.c_int32(0)
    _check(_lib.pa_decode_step_prepare(pool, n, ids.ctypes.data, int(max_blocks),
                                       slots.ctypes.data, ctx.ctypes.data, tables.ctypes.data,
                                       copies.ctypes.data, cap, ctypes.byref(nc)))
    return slots, ctx, tables, copies[: nc.value]


def pa_decode_step_prepare_rows(pool, seq_ids, max_blocks: int, tables, row_versions,
                                slot_out=None, ctx_out=None, copies_out=None,
                                copies_cap: int | None = None):
    """pa_decode_step_prepare into a ``tables`` array (int32[n, max_blocks])
    that the caller keeps from step to step, with its ``row_versions``
    (uint64[n], zeros at first): only rows whose sequence's table changed are
    rewritten.  Returns (slot_mapping, ctx_lens, tables, copies)."""
    ids = _host_i32(seq_ids)
    n = ids.shape[0]
    if tables.dtype != np.int32 or tables.shape != (n, max_blocks) or not tables.flags.c_contiguous:
        raise ValueError("tables must be a contiguous int32 array of shape (n, max_blocks)")
    if row_versions.dtype != np.uint64 or row_versions.shape != (n,) or \
            not row_versions.flags.c_contiguous:
        raise ValueError("row_versions must be a contiguous uint64 array of length n")
    cap = n if copies_cap is None else int(copies_cap)
    slots = np.empty(n, np.int64) if slot_out is None else slot_out
    ctx = np.empty(n, np.int32) if ctx_out is None else ctx_out
    copies = np.empty((max(cap, 1), 2), np.int32) if copies_out is None else copies_out
    nc = ctypes.c_int32(0)
    _check(_lib.pa_decode_step_prepare_rows(pool, n, ids.ctypes.data, int(max_blocks),
                                            slots.ctypes.data, ctx.ctypes.data, tables.ctypes.data,
                                            row_versions.ctypes.data, copies.ctypes.data, cap,
                                            ctypes.byref(nc)))
    return slots, ctx, tables, copies[: nc.value]


def pa_decode_step_prepare_into(pool, n_seqs: int, ids_addr: int, max_blocks: int,
                                slots_addr: int, ctx_addr: int, tables_addr: int,
                                copies_addr: int, copies_cap: int, n_copies) -> int:
    """pa_decode_step_prepare on raw host addresses (a serving loop's
    preallocated staging buffers); ``n_copies`` is a ctypes.c_int32 that
    receives the copy count.  Returns it."""
    _check(_lib.pa_decode_step_prepare(pool, n_seqs, ids_addr, max_blocks, slots_addr, ctx_addr,
                                       tables_addr, copies_addr, copies_cap, ctypes.byref(n_copies)))
    return n_copies.value


def pa_decode_step_prepare_rows_into(pool, n_seqs: int, ids_addr: int, max_blocks: int,
                                     slots_addr: int, ctx_addr: int, tables_addr: int,
                                     versions_addr: int, copies_addr: int, copies_cap: int,
                                     n_copies) -> int:
    """pa_decode_step_prepare_rows on raw host addresses: table rows whose
    sequence's table is unchanged since this call last wrote them (per the
    caller's ``versions_addr`` array, one uint64 per row) are left as they
    are.  ``n_copies`` is a ctypes.c_int32 that receives the copy count."""
    _check(_lib.pa_decode_step_prepare_rows(pool, n_seqs, ids_addr, max_blocks, slots_addr,
                                            ctx_addr, tables_addr, versions_addr, copies_addr,
                                            copies_cap, ctypes.byref(n_copies)))
    return n_copies.value


def pa_seq_info(pool, seq_id: int):
    nt, nb = ctypes.c_int32(), ctypes.c_int32()
    _check(_lib.pa_seq_info(pool, int(seq_id), ctypes.byref(nt), ctypes.byref(nb)))
    return nt.value, nb.value


def pa_pool_num_free(pool) -> int:
    n = ctypes.c_int32()
    _check(_lib.pa_pool_num_free(pool, ctypes.byref(n)))
    return n.value


def pa_pool_free_queue(pool, num_blocks: int):
    out = np.empty(max(int(num_blocks), 1), np.int32)
    n = ctypes.c_int32()
    _check(_lib.pa_pool_free_queue(pool, out.ctypes.data, int(num_blocks), ctypes.byref(n)))
    return out[: n.value]


def pa_pool_refcounts(pool, num_blocks: int):
    out = np.empty(max(int(num_blocks), 1), np.int32)
    _check(_lib.pa_pool_refcounts(pool, out.ctypes.data))
    return out[: int(num_blocks)]


# -------------------------------------------------------------- device calls
def pa_write_kv(k, v, slot_mapping, k_cache, v_cache, desc: PoolDesc, status=None,
                stream=None, n_tokens: int | None = None) -> None:
    n = int(slot_mapping.shape[0]) if n_tokens is None else int(n_tokens)
    _check(_lib.pa_write_kv(_dev(k), _dev(v), _dev(slot_mapping), n, _dev(k_cache),
                            _dev(v_cache), desc.ref, _dev(status), _stream(stream)))


def pa_copy_blocks(k_caches, v_caches, pairs, desc: PoolDesc, status=None, stream=None,
                   n_pairs: int | None = None) -> None:
    L = len(k_caches)
    kp = (ctypes.c_void_p * L)(*[_dev(x) for x in k_caches])
    vp = (ctypes.c_void_p * L)(*[_dev(x) for x in v_caches])
    n = int(pairs.shape[0]) if n_pairs is None else int(n_pairs)
    _check(_lib.pa_copy_blocks(kp, vp, L, _dev(pairs), n, desc.ref, _dev(status),
                               _stream(stream)))


def pa_decode_workspace_bytes(n_seqs: int, max_blocks: int, desc: PoolDesc) -> int:
    return int(_lib.pa_decode_workspace_bytes(int(n_seqs), int(max_blocks), desc.ref))


def pa_decode_attention(out, q, k_cache, v_cache, block_tables, ctx_lens, scale: float,
                        desc: PoolDesc, workspace=None, status=None, stream=None,
                        n_seqs: int | None = None, max_blocks: int | None = None) -> None:
    n = int(q.shape[0]) if n_seqs is None else int(n_seqs)
    mb = int(block_tables.shape[1]) if max_blocks is None else int(max_blocks)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.pa_decode_attention(_dev(out), _dev(q), _dev(k_cache), _dev(v_cache),
                                    _dev(block_tables), _dev(ctx_lens), n, mb,
                                    ctypes.c_float(scale), _dev(workspace), ws_bytes,
                                    _dev(status), desc.ref, _stream(stream)))


def pa_decode_step_attention(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                             ctx_lens, scale: float, desc: PoolDesc, workspace=None, status=None,
                             stream=None, n_seqs: int | None = None,
                             max_blocks: int | None = None) -> None:
    """The step's slot write (one new token per sequence, at slot_mapping[s])
    and decode attention in one call."""
    n = int(q.shape[0]) if n_seqs is None else int(n_seqs)
    mb = int(block_tables.shape[1]) if max_blocks is None else int(max_blocks)
    _need_elems(n * desc.num_heads * desc.head_dim, k_new=k_new, v_new=v_new)
    _need_elems(n, slot_mapping=slot_mapping)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.pa_decode_step_attention(_dev(out), _dev(q), _dev(k_new), _dev(v_new),
                                         _dev(slot_mapping), _dev(k_cache), _dev(v_cache),
                                         _dev(block_tables), _dev(ctx_lens), n, mb,
                                         ctypes.c_float(scale), _dev(workspace), ws_bytes,
                                         _dev(status), desc.ref, _stream(stream)))


def pa_prefill_attention(out, q, k_cache, v_cache, block_tables, ctx_lens, q_starts,
                         scale: float, desc: PoolDesc, max_q_len: int, status=None, stream=None,
                         n_seqs: int | None = None, max_blocks: int | None = None,
                         q_rows: int | None = None) -> None:
    """Causal paged prefill: rows q_starts[s]..q_starts[s+1]-1 of q are the last
    positions of sequence s's context of ctx_lens[s] tokens.  ``max_q_len``
    (host int) bounds every q_len; ``q_rows`` defaults to the rows of q and out."""
    n = int(ctx_lens.shape[0]) if n_seqs is None else int(n_seqs)
    mb = int(block_tables.shape[1]) if max_blocks is None else int(max_blocks)
    rows = min(int(q.shape[0]), int(out.shape[0])) if q_rows is None else int(q_rows)
    _check(_lib.pa_prefill_attention(_dev(out), _dev(q), _dev(k_cache), _dev(v_cache),
                                     _dev(block_tables), _dev(ctx_lens), _dev(q_starts), n, mb,
                                     int(max_q_len), rows, ctypes.c_float(scale), _dev(status),
                                     desc.ref, _stream(stream)))


def pa_prefill_step_attention(out, q, k_new, v_new, k_cache, v_cache, block_tables, ctx_lens,
                              q_starts, scale: float, desc: PoolDesc, max_q_len: int, status=None,
                              stream=None, n_seqs: int | None = None, max_blocks: int | None = None,
                              q_rows: int | None = None) -> None:
    """Whole prompts: their keys and values (k_new, v_new, rows as q) stored
    into their blocks and causal prefill attention over them, one call."""
    n = int(ctx_lens.shape[0]) if n_seqs is None else int(n_seqs)
    mb = int(block_tables.shape[1]) if max_blocks is None else int(max_blocks)
    rows = min(int(q.shape[0]), int(out.shape[0])) if q_rows is None else int(q_rows)
    # the new rows are read as [rows][num_heads][head_dim] tensors, like q
    _need_elems(rows * desc.num_heads * desc.head_dim, k_new=k_new, v_new=v_new)
    _check(_lib.pa_prefill_step_attention(_dev(out), _dev(q), _dev(k_new), _dev(v_new),
                                          _dev(k_cache), _dev(v_cache), _dev(block_tables),
                                          _dev(ctx_lens), _dev(q_starts), n, mb, int(max_q_len),
                                          rows, ctypes.c_float(scale), _dev(status), desc.ref,
                                          _stream(stream)))


def pa_selftest_bounded_wait(status, stream=None) -> None:
    """One thread waits, with the kernels' bounded wait, for an mbarrier phase
    that nothing completes; after the limit it writes PA_ERR_TIMEOUT into
    status (device int32)."""
    _check(_lib.pa_selftest_bounded_wait(_dev(status), _stream(stream)))


def pa_decode_attention_noalloc(out, q, k_cache, v_cache, block_tables, ctx_lens, scale: float,
                                desc: PoolDesc, status=None, stream=None,
                                n_seqs: int | None = None, max_blocks: int | None = None) -> None:
    """pa_decode_attention without a workspace argument, for callers that cannot
    allocate device memory when they run attention: the library's fixed
    scratch (PA_NOALLOC_SCRATCH_BYTES, shared by all calls) stands in for it.
    Calls that overlap on the GPU race on that scratch."""
    n = int(q.shape[0]) if n_seqs is None else int(n_seqs)
    mb = int(block_tables.shape[1]) if max_blocks is None else int(max_blocks)
    _check(_lib.pa_decode_attention_noalloc(_dev(out), _dev(q), _dev(k_cache), _dev(v_cache),
                                            _dev(block_tables), _dev(ctx_lens), n, mb,
                                            ctypes.c_float(scale), _dev(status), desc.ref,
                                            _stream(stream)))
