"""ORACLE -- test infrastructure only.

Python entry to the plain C fp64 paged-attention oracle (``paged_attention.c``).
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this module.

The oracle computes softmax attention of one query per (sequence, head) over
the sequence's valid context, gathering every key and value through the
block table (PagedAttention notes, unpurerationalist.github.io, §3.1,
blockwise attention equation; paged KV cache tutorial,
llm-systems-engineering.pages.dev/posts/paged-kv-cache, Fig. 2 and Fig. 4).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attention.c")
_LIB = os.path.join(_HERE, "liboracle_attention.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP) into ``liboracle_attention.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_paged_attention.restype = ctypes.c_int32
            lib.oracle_paged_attention.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_double, ctypes.c_int32,
            ]
            lib.oracle_paged_prefill.restype = ctypes.c_int32
            lib.oracle_paged_prefill.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_double, ctypes.c_int32,
            ]
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def half_bits_to_double(bits: int) -> float:
    """The oracle's own binary16 decoder (exposed so tests can pin it)."""
    return _load().oracle_half_to_double(int(bits) & 0xFFFF)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def paged_attention(q, k_cache, v_cache, block_tables, ctx_lens, scale: float,
                    num_threads: int = 0) -> np.ndarray:
    """fp64 paged decode attention.

    q: float16 [S, H, D]; k_cache, v_cache: float16 [num_blocks, H, B, D];
    block_tables: int32 [S, max_blocks]; ctx_lens: int32 [S].
    Returns float64 [S, H, D].  ``scale`` multiplies q.k (1/sqrt(D) in the
    pages); it is used as given, in double precision.
    """
    q = np.ascontiguousarray(q, dtype=np.float16)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.float16)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.float16)
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx_lens = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    S, H, D = q.shape
    NB, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape does not match q")
    if block_tables.ndim != 2 or block_tables.shape[0] != S or ctx_lens.shape != (S,):
        raise ValueError("block_tables / ctx_lens shape mismatch")
    max_blocks = block_tables.shape[1]
    out = np.empty((S, H, D), dtype=np.float64)
    rc = _load().oracle_paged_attention(
        out.ctypes.data, q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
        block_tables.ctypes.data, ctx_lens.ctypes.data,
        S, H, D, B, NB, max_blocks, float(scale), int(num_threads),
    )
    if rc == -2:
        raise IndexError("block table entry outside the pool")
    if rc != 0:
        raise ValueError(f"oracle_paged_attention rejected its arguments ({rc})")
    return out


def paged_prefill(q, k_cache, v_cache, block_tables, ctx_lens, q_starts, scale: float,
                  num_threads: int = 0) -> np.ndarray:
    """fp64 causal paged prefill: q float16 [T, H, D] (rows of sequence s are
    q_starts[s]..q_starts[s+1]-1, the last positions of its context);
    returns float64 [T, H, D]."""
    q = np.ascontiguousarray(q, dtype=np.float16)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.float16)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.float16)
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx_lens = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    q_starts = np.ascontiguousarray(q_starts, dtype=np.int32)
    T, H, D = q.shape
    NB, H2, B, D2 = k_cache.shape
    S = ctx_lens.shape[0]
    if (H2, D2) != (H, D) or q_starts.shape != (S + 1,) or int(q_starts[-1]) != T:
        raise ValueError("shape mismatch")
    out = np.empty((T, H, D), dtype=np.float64)
    rc = _load().oracle_paged_prefill(
        out.ctypes.data, q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
        block_tables.ctypes.data, ctx_lens.ctypes.data, q_starts.ctypes.data,
        S, H, D, B, NB, block_tables.shape[1], float(scale), int(num_threads))
    if rc == -2:
        raise IndexError("block table entry outside the pool")
    if rc != 0:
        raise ValueError(f"oracle_paged_prefill rejected its arguments ({rc})")
    return out

