"""GB300 decode-step hot path of Hybrid HiSparse (sparse-MLA KV offloading).

The compute path is the C-ABI library ``libhisparse.so`` (hand-written CUDA for
sm_103a) declared in ``include/hisparse.h``; ``hisparse`` is its thin ctypes
binding. ``workload`` and ``schedule`` build seeded synthetic inputs and the
host-side residency schedule. Importing this package loads nothing native;
importing ``hisparse`` does, and fails loudly when the library is missing.
"""
