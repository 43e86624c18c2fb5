"""ORACLE -- test infrastructure, not part of the product.

A plain, slow, independently written CPU definition of the paged KV cache's
decode-step hot path, used only to check the CUDA path:

* ``alloc``       -- block manager model (free queue, refcounts, block tables,
                     #filled, copy-on-write, fork / append / free);
* ``cache_ops``   -- byte-image models of the slot write and the block copy;
* ``attention``   -- fp64 paged decode attention (C source ``paged_attention.c``).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import, call, link or execute
anything here.  The oracle imports nothing from the product package and the
product imports nothing from here.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against the pages' worked examples (``tests/golden/``), closed forms,
invariants, library routines on special cases and brute force.  No function
here is "parity unpinned".
"""
