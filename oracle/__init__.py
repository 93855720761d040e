"""CPU oracle for the Hybrid HiSparse decode step: TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the decode hot path
computes, in fp64 / exact integer arithmetic with numpy. It shares no code with
the CUDA path (``sparse_mla_kv_indexer_gb300/csrc``) and neither imports the
other; both consume the same seeded inputs from
``sparse_mla_kv_indexer_gb300.workload`` and the same host residency schedule
from ``sparse_mla_kv_indexer_gb300.schedule``.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it. The product path never routes through it.

Modules
  formats       FP8 e4m3 / bf16 / 656-byte row decoding
  indexer       exact integer indexer scores and full-sort top-K
  resolver      top-K residency resolution with the hot buffer and LRU
  attention     sparse MLA decode (masked softmax attention) in fp64
  engine        whole decode steps over a workload and its schedule
  closed_forms  the byte and FLOP closed forms printed by the pages

Parity status: every function is pinned by tests in tests/test_oracle_*.py
against hand-worked cases, brute force, closed forms, library routines or
invariants. The pressure-eviction order and the hot-lease growth rule are
readings of the pages, not printed by them; they live in the shared schedule and
are pinned only by invariants (tail never evicted, capacity bound, byte
identity of every resolved row).
"""
